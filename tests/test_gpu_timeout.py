"""Failure detection without a GPU fault: every device wait in the engine is
bounded (2 s) and ends in MOEQ_ERR_TIMEOUT in the workspace status word, with
the kernel draining its copies and returning, so the context stays usable.

The test makes one wait run out on purpose: the input-quantisation counter
in the workspace header (byte offset 16) is set far below anything the
launch can reach, so the chunk-preparing warps of every CTA give up after
the limit (a down call whose N is not a multiple of 256, which the
persistent engine serves).  It then checks the status, re-initialises the workspace and
checks that a normal call on the same context still matches the oracle.
A second case does the same to the count that the persistent engine's
one-token layer waits for before its final combine (the engine serves one
token when MOEQ_MTOK_KERNEL=0 and MOEQ_TOKEN_KERNEL=0), in a child process
with that setting."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import synth
from moeq_testlib import STRICT, Experts, assert_close, device_plan, to_np
from test_gpu_gemm import check_h, oracle_down, oracle_gateup

pytestmark = pytest.mark.gpu

A_CNT_INT_OFFSET = 16 // 4   # int32 index of the input-quantisation counter


@pytest.mark.parametrize("M", [1, 8])
def test_bounded_wait_reports_timeout_and_the_context_survives(orc, M):
    from bandwidth_bound_fp8_gb300 import moeq
    K, N = 256, 128
    ex = Experts(1, N, K, base_seed=71, which=1)
    a = synth.activations_bf16(M, K, 73, 2, 20.0, device="cuda")
    du, do, _, dn = device_plan([0], [0, M], [0])
    ws = moeq.Workspace(moeq.moeq_gemm_workspace_size(N, K, M, 1, 0))
    ws.t.view(torch.int32)[A_CNT_INT_OFFSET] = -(1 << 30)   # a count the launch can never reach
    y = torch.zeros((M, N), device="cuda")
    moeq.moeq_expert_gemm_down(a, K, N, ex.q, ex.s, 1, du, do, dn, 1, M, y, ws)
    torch.cuda.synchronize()   # returns: the kernel gave up instead of hanging
    assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == moeq.MOEQ_ERR_TIMEOUT

    # the same context, a fresh workspace state: a normal call is correct
    moeq.moeq_workspace_init(ws.t, ws.nbytes)
    y = torch.full((M, N), float("nan"), device="cuda")
    moeq.moeq_expert_gemm_down(a, K, N, ex.q, ex.s, 1, du, do, dn, 1, M, y, ws)
    torch.cuda.synchronize()
    assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == 0
    y_ref, T, _, _ = oracle_down(orc, to_np(a.contiguous().view(torch.uint16)), ex, [0], [0, M])
    assert_close(to_np(y), y_ref, T, STRICT, what="after a timeout")


DC_CNT_INT_OFFSET = 20 // 4  # int32 index of the down-by-K-group count


def test_layer_combine_wait_reports_timeout_and_the_context_survives(orc):
    """One token without y on the persistent engine: the combine after down by
    K group waits for every CTA's count.  With the count set out of reach that
    wait gives up, the status says so, and after a re-initialisation the layer
    is correct."""
    if os.environ.get("MOEQ_TOKEN_KERNEL") != "0" or os.environ.get("MOEQ_MTOK_KERNEL") != "0":
        env = dict(os.environ, MOEQ_TOKEN_KERNEL="0", MOEQ_MTOK_KERNEL="0")
        here = os.path.dirname(os.path.abspath(__file__))
        cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
               os.path.abspath(__file__), "-k", "combine_wait"]
        r = subprocess.run(cmd, env=env, cwd=os.path.dirname(here), capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, f"{r.stdout[-3000:]}\n{r.stderr[-2000:]}"
        return
    from test_gpu_layer import Layer, check_layer
    from bandwidth_bound_fp8_gb300 import moeq
    E, H, I, k = 8, 512, 256, 2
    lay = Layer(E, H, I, seed=91)
    x = synth.activations_bf16(1, H, 92, 2, 20.0, device="cuda")
    logits = synth.logits_f32(1, E, 93, device="cuda")
    out = torch.empty((1, H), dtype=torch.bfloat16, device="cuda")
    ws = moeq.Workspace(moeq.moeq_workspace_size(1, H, I, E + 1, k))
    ws.t.view(torch.int32)[DC_CNT_INT_OFFSET] = -(1 << 30)
    moeq.moeq_moe_layer(x, logits, H, I, E, k, lay.gu.q, lay.gu.s, lay.dn.q, lay.dn.s, out, ws)
    torch.cuda.synchronize()   # returns: the combine gave up instead of hanging
    assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == moeq.MOEQ_ERR_TIMEOUT
    moeq.moeq_workspace_init(ws.t, ws.nbytes)
    moeq.moeq_moe_layer(x, logits, H, I, E, k, lay.gu.q, lay.gu.s, lay.dn.q, lay.dn.s, out, ws)
    torch.cuda.synchronize()
    assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == 0
    check_layer(orc, lay, x, logits, k, with_y=False)


@pytest.mark.parametrize("M,which", [(1, 0), (4, 0), (2, 1)])
def test_layer_kernel_wait_reports_timeout_and_the_context_survives(orc, M, which):
    """The multi-token kernel (every layer of 1..16 tokens by default): one
    of the counts it waits on -- x's K group 0 (released to the producer
    once every token's group is in) or output unit 0 (summed once every
    column's partials are in) -- is set far out of reach in the workspace.
    The wait gives up after its limit, every role stops and drains, the
    status says MOEQ_ERR_TIMEOUT, and after a re-initialisation the layer
    on the same context matches the oracle."""
    from test_gpu_layer import Layer, check_layer
    from bandwidth_bound_fp8_gb300 import moeq
    E, H, I, k = 8, 512, 256, 2
    off = moeq.moeq_layer_ws_count_offset(M, H, I, E + 1, k, which)
    if off == 0:
        pytest.skip("the multi-token kernel does not serve this shape here")
    lay = Layer(E, H, I, seed=95 + M)
    x = synth.activations_bf16(M, H, 96 + M, 2, 20.0, device="cuda")
    logits = synth.logits_f32(M, E, 97 + M, device="cuda")
    out = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    ws = moeq.Workspace(moeq.moeq_workspace_size(M, H, I, E + 1, k))
    assert off % 4 == 0 and off < ws.nbytes
    ws.t.view(torch.int32)[off // 4] = -(1 << 30)
    moeq.moeq_moe_layer(x, logits, H, I, E, k, lay.gu.q, lay.gu.s, lay.dn.q, lay.dn.s, out, ws)
    torch.cuda.synchronize()   # returns: the kernel gave up instead of hanging
    assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == moeq.MOEQ_ERR_TIMEOUT
    moeq.moeq_workspace_init(ws.t, ws.nbytes)
    ref = check_layer(orc, lay, x, logits, k, with_y=False)   # against the oracle, a fresh workspace
    moeq.moeq_moe_layer(x, logits, H, I, E, k, lay.gu.q, lay.gu.s, lay.dn.q, lay.dn.s, out, ws)
    torch.cuda.synchronize()
    assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))   # the re-initialised one, same bits



@pytest.mark.parametrize("gate_up,which", [(0, 1), (1, 0)])
def test_gemm_kernel_wait_reports_timeout_and_the_context_survives(orc, gate_up, which):
    """The standalone GEMM calls on the multi-token kernel: the count of
    x's K group 0 (gate_up), or of output unit 0 (down, whose pieces
    quantise their own rows of a), set out of reach in the call's
    workspace.  The wait gives up, the status says
    MOEQ_ERR_TIMEOUT, and after a re-initialisation the call on the same
    context matches the oracle."""
    from bandwidth_bound_fp8_gb300 import moeq
    K, rows_out, M = 256, 256 if not gate_up else 128, 3
    off = moeq.moeq_gemm_ws_count_offset(rows_out, K, M, 1, gate_up, which)
    if off == 0:
        pytest.skip("the multi-token kernel does not serve this call here")
    ws = moeq.Workspace(moeq.moeq_gemm_workspace_size(rows_out, K, M, 1, gate_up))
    assert off % 4 == 0 and off < ws.nbytes
    a = synth.activations_bf16(M, K, 75 + which, 2, 20.0, device="cuda")
    if gate_up:
        ex = Experts(1, 2 * rows_out, K, base_seed=77, which=0)
        du, do, dp, dn = device_plan([0], [0, M], list(range(M)))
        out = torch.zeros((M, rows_out), device="cuda")
        call = lambda: moeq.moeq_expert_gemm_gateup_swiglu(a, K, rows_out, ex.q, ex.s, 1, du, do, dp, dn, 1, M, out, ws)
    else:
        ex = Experts(1, rows_out, K, base_seed=79, which=1)
        du, do, _, dn = device_plan([0], [0, M], [0])
        out = torch.zeros((M, rows_out), device="cuda")
        call = lambda: moeq.moeq_expert_gemm_down(a, K, rows_out, ex.q, ex.s, 1, du, do, dn, 1, M, out, ws)
    ws.t.view(torch.int32)[off // 4] = -(1 << 30)
    call()
    torch.cuda.synchronize()   # returns: the kernel gave up instead of hanging
    assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == moeq.MOEQ_ERR_TIMEOUT
    moeq.moeq_workspace_init(ws.t, ws.nbytes)
    out.fill_(float("nan"))
    call()
    torch.cuda.synchronize()
    assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == 0
    a_np = to_np(a.contiguous().view(torch.uint16))
    if gate_up:
        g, u, Tg, Tu, h_ref, _, _ = oracle_gateup(orc, a_np, ex, [0], [0, M], list(range(M)), rows_out)
        check_h(to_np(out), g, u, Tg, Tu, h_ref)
    else:
        y_ref, T, _, _ = oracle_down(orc, a_np, ex, [0], [0, M])
        assert_close(to_np(out), y_ref, T, STRICT, what="after a timeout")
