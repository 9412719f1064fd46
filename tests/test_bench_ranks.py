"""The multi-process side of bench.py on the CPU (gloo, world size 2): rank
setup from the torchrun environment, the job time as the maximum over ranks,
the bytes as the sum over ranks, the whole-job value computed from those,
and the reference arm printing on rank 0 only."""
import importlib.util
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    # CPU ranks even on a GPU machine: no device visible -> bench picks gloo
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    b = _bench()
    ws, r, local = b.dist_setup()
    ms = 10.0 + 5.0 * rank                 # this rank's timed region
    byts = 1e9 * (rank + 1)                # this rank's bytes
    t = b.max_over_ranks(ms, ws)
    total = b.sum_over_ranks(byts, ws)
    b.barrier(ws)
    # reference arm: only rank 0 runs and prints
    class A:
        M, steps, warmup, gpus = 1, 1, 1, world
    out = io.StringIO()
    if rank != 0:
        with redirect_stdout(out):
            b.reference_arm(A, ws, r)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((rank, ws, r, t, total, total / (t * 1e-3) / 1e9, out.getvalue()))


@pytest.mark.timeout(300)
def test_two_ranks_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ws, r, t, total, value, out in res:
        assert (ws, r) == (world, rank)
        assert t == 15.0                   # the slowest rank's time
        assert total == 3e9                # every rank's bytes
        assert abs(value - 3e9 / 15e-3 / 1e9) < 1e-9
        if rank != 0:
            assert out == ""               # the reference arm prints on rank 0 only
