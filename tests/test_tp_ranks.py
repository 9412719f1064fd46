"""The tensor-parallel layer step (bandwidth_bound_fp8_gb300/tp.py) on two
CPU ranks over gloo: each rank's partial is the oracle's layer on its shard
(fp64, stored as fp32), the all-gather keeps rank order (slot r of the
gathered tensor is rank r's own partial), and the rank-order sum rounded to
bf16 is the same bits on both ranks and within SPEC plus half a bf16 ulp of
the unsharded oracle layer."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    import torch.distributed as dist
    import oracle as orc
    import synth
    from bandwidth_bound_fp8_gb300 import tp
    from test_oracle_layer import _tiny_layer
    from test_oracle_tp import oracle_shard
    dist.init_process_group("gloo", rank=rank, world_size=world)
    E, H, I, k, M = 8, 256, 512, 2, 3
    experts = _tiny_layer(orc, E, H, I, seed=11)
    xb = synth.activations_bf16(M, H, 41, 3, 30.0)
    lg = synth.logits_f32(M, E, 42)
    x_np = xb.view(torch.uint16).numpy()

    class Shard:   # the orchestration reads R and the slice width only
        R, I_shard = world, I // world

    def partial_fn(partial):
        sh = orc.moe_layer(x_np, lg.numpy(), k, oracle_shard(experts, I, world, rank), H, I // world)
        partial.copy_(torch.from_numpy(sh.out64.astype(np.float32)))

    def reduce_fn(parts, out):
        acc = parts[0].clone()
        for r in range(1, parts.shape[0]):
            acc += parts[r]      # fp32, rank order
        bits = np.array([orc.f64_to_bf16_bits(float(v)) for v in acc.numpy().ravel()], np.uint16)
        out.copy_(torch.from_numpy(bits.view(np.int16).reshape(out.shape)).view(torch.bfloat16))

    out = torch.empty((M, H), dtype=torch.bfloat16)
    parts = tp.tp_moe_layer(xb, lg, E, k, Shard, out, None, partial_fn=partial_fn, reduce_fn=reduce_fn)
    own = torch.empty((M, H), dtype=torch.float32)
    partial_fn(own)
    outs = [torch.empty_like(out) for _ in range(world)]
    dist.all_gather(outs, out)
    dist.destroy_process_group()
    q.put((rank, parts.numpy(), own.numpy(), [o.view(torch.int16).numpy() for o in outs]))


@pytest.mark.timeout(300)
def test_tp_layer_two_ranks_gloo(orc):
    import synth
    from moeq_testlib import SPEC_ABS, SPEC_REL, half_ulp_bf16
    from test_oracle_layer import _tiny_layer
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict((r[0], r[1:]) for r in [q.get(timeout=240) for _ in range(world)])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        parts, own, outs = res[r]
        for s in range(world):
            assert np.array_equal(parts[s], res[s][1]), f"rank {r}: gathered slot {s} is not rank {s}'s partial"
        assert np.array_equal(outs[0], outs[1]), "the ranks' outputs differ"
    # against the unsharded oracle layer
    E, H, I, k, M = 8, 256, 512, 2, 3
    experts = _tiny_layer(orc, E, H, I, seed=11)
    x = synth.activations_bf16(M, H, 41, 3, 30.0).view(torch.uint16).numpy()
    full = orc.moe_layer(x, synth.logits_f32(M, E, 42).numpy(), k, experts, H, I)
    o = orc.bf16_bits_to_f32_array(res[0][2][0].view(np.uint16)).astype(np.float64)
    r16 = orc.bf16_bits_to_f32_array(full.out_bf16).astype(np.float64)
    bound = SPEC_REL * full.Tout + SPEC_ABS + half_ulp_bf16(o, r16)
    assert (np.abs(o - full.out64) <= bound).all()
