"""GPU parity of the two expert GEMM calls against the oracle.

Each case hands both sides the same inputs (a plan chosen by the test, the
same fp32 weights quantised by each side, the same activations): codes and
scales of the fused quantisation prologue must match bit for bit, outputs
within STRICT (see moeq_testlib) -- and therefore within SPEC.  Shapes span
several 128-blocks in N and K with ragged group counts, experts with 1, 2,
3 and 5+ tokens (every accumulation mode), split-K with many contributors
per row block (few units per CTA) and CTAs spanning several row blocks.
"""
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import synth
from moeq_testlib import SPEC_ABS, SPEC_REL, STRICT, Experts, assert_close, bf16_bits, device_plan, to_np

pytestmark = pytest.mark.gpu


def _act_np(a):
    return bf16_bits(a) if a.dtype == torch.bfloat16 else to_np(a)


def run_down(a, ex, uniq, offs, want_dump=True):
    from bandwidth_bound_fp8_gb300 import moeq
    P, K = a.shape
    N = ex.N
    du, do, _, dn = device_plan(uniq, offs, [0])
    y = torch.full((P, N), float("nan"), device="cuda")
    qd = torch.zeros((P, K), dtype=torch.uint8, device="cuda") if want_dump else None
    sd = torch.zeros((P, K // 128), dtype=torch.float32, device="cuda") if want_dump else None
    ws = moeq.Workspace(moeq.moeq_gemm_workspace_size(N, K, P, len(uniq), 0))
    moeq.moeq_expert_gemm_down(a, K, N, ex.q, ex.s, ex.E, du, do, dn, len(uniq), P, y, ws, qd, sd)
    torch.cuda.synchronize()
    assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == 0
    return to_np(y), (to_np(qd) if want_dump else None), (to_np(sd) if want_dump else None)


def oracle_down(orc, a_np, ex, uniq, offs):
    P = a_np.shape[0]
    qa, sa = orc.quant_act(a_np)
    y = np.zeros((P, ex.N))
    T = np.zeros((P, ex.N))
    cache = {}
    for u, e in enumerate(uniq):
        if e not in cache:
            cache[e] = ex.oracle(orc, e)
        qw, sw = cache[e]
        for p in range(offs[u], offs[u + 1]):
            y[p], T[p] = [v[0] for v in orc.gemm(qa[p:p + 1], sa[p:p + 1], qw, sw)]
    return y, T, qa, sa


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("K,N,uniq,offs", [
    (640, 384, [3, 0, 4], [0, 1, 3, 8]),          # 1, 2, 5 tokens
    (256, 128, [1], [0, 3]),                       # 3 tokens, tiny: T < grid
    (1280, 512, [2, 5, 0, 1, 3, 4], [0, 1, 2, 3, 4, 5, 21]),   # 16 tokens on one expert
    (768, 512, [2, 0, 1], [0, 5, 21, 28]),         # 16 rows on one expert from pair row 5
    # 64 experts x 8 K groups = 512 one-stage columns on the multi-token
    # kernel: 3-4 pieces per CTA, so each of its two shared-memory B operands
    # is quantised into more than once
    (1024, 256, list(range(63, -1, -1)), [0] + [1 + i + i // 3 for i in range(64)]),
])
def test_down_small(orc, dtype, K, N, uniq, offs):
    # N a multiple of 256 runs the multi-token kernel's down mode (each
    # expert's rows one MMA's B operand, their codes swizzled for their place
    # in it); other N the persistent engine
    E = max(uniq) + 1
    ex = Experts(E, N, K, base_seed=11 + K + N, which=1)
    P = offs[-1]
    if dtype == "bf16":
        a = synth.activations_bf16(P, K, 17 + P, 3, 30.0, device="cuda")
    else:
        a = synth.activations_f32(P, K, 19 + P, device="cuda", std=0.3)
    y, qd, sd = run_down(a, ex, uniq, offs)
    y_ref, T, qa, sa = oracle_down(orc, _act_np(a), ex, uniq, offs)
    assert np.array_equal(qd, qa) and np.array_equal(sd.view(np.uint32), sa.view(np.uint32))
    assert_close(y, y_ref, T, STRICT, what="y")
    assert_close(y, y_ref, T, SPEC_REL, SPEC_ABS, what="y spec")


def test_down_dense_projection_full_size(orc):
    """Dense single projection at its full size: M = 1, K = 2048, N = 4096,
    bf16 x ~ N(0,1) with 4 outlier channels x50, fp32 output."""
    cfg = synth.DENSE_PROJ
    ex = Experts(1, cfg["N"], cfg["K"], base_seed=cfg["seed"], which=1)
    x = synth.activations_bf16(1, cfg["K"], cfg["seed"], cfg["n_outlier"], cfg["outlier_scale"], device="cuda")
    y, qd, sd = run_down(x, ex, [0], [0, 1])
    y_ref, T, qa, sa = oracle_down(orc, bf16_bits(x), ex, [0], [0, 1])
    assert np.array_equal(qd, qa) and np.array_equal(sd.view(np.uint32), sa.view(np.uint32))
    assert_close(y, y_ref, T, STRICT, what="dense y")


def run_gateup(x, ex, uniq, offs, pair_tok, I):
    from bandwidth_bound_fp8_gb300 import moeq
    M, H = x.shape
    P = offs[-1]
    du, do, dp, dn = device_plan(uniq, offs, pair_tok)
    h = torch.full((P, I), float("nan"), device="cuda")
    qx = torch.zeros((M, H), dtype=torch.uint8, device="cuda")
    sx = torch.zeros((M, H // 128), dtype=torch.float32, device="cuda")
    ws = moeq.Workspace(moeq.moeq_gemm_workspace_size(I, H, M, len(uniq), 1))
    moeq.moeq_expert_gemm_gateup_swiglu(x, H, I, ex.q, ex.s, ex.E, du, do, dp, dn, len(uniq), P, h, ws, qx, sx)
    torch.cuda.synchronize()
    assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == 0
    return to_np(h), to_np(qx), to_np(sx)


def oracle_gateup(orc, x_np, ex, uniq, offs, pair_tok, I):
    qx, sx = orc.quant_act(x_np)
    P = offs[-1]
    g = np.zeros((P, I)); u = np.zeros((P, I)); Tg = np.zeros((P, I)); Tu = np.zeros((P, I))
    for ui, e in enumerate(uniq):
        qw, sw = ex.oracle(orc, e)
        for p in range(offs[ui], offs[ui + 1]):
            t = pair_tok[p]
            y, T = orc.gemm(qx[t:t + 1], sx[t:t + 1], qw, sw)
            g[p], u[p], Tg[p], Tu[p] = y[0, :I], y[0, I:], T[0, :I], T[0, I:]
    return g, u, Tg, Tu, orc.swiglu_vec(g, u), qx, sx


def h_bound(g, u, Tg, Tu, rel):
    """|silu(g) u - silu(g') u'| for |g-g'| <= rel*Tg, |u-u'| <= rel*Tu (|silu'| < 1.1),
    plus the fp32 evaluation of silu and the product."""
    eg, eu = rel * Tg, rel * Tu
    sg = np.abs(g * expit(g))
    return 1.1 * eg * (np.abs(u) + eu) + (sg + 1.1 * eg) * eu + 1e-6 * sg * np.abs(u) + 1e-37


def check_h(h, g, u, Tg, Tu, h_ref):
    err = np.abs(h.astype(np.float64) - h_ref.astype(np.float64))
    b = h_bound(g, u, Tg, Tu, STRICT)
    assert (err <= b).all(), f"h: {(err > b).sum()} outside; worst {np.max(err - b)}"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("H,I,uniq,offs,pair_tok,M", [
    (640, 384, [3, 0, 4, 5], [0, 1, 3, 6, 11], [2, 0, 1, 0, 1, 2, 0, 1, 2, 3, 4], 5),
    (256, 128, [0], [0, 1], [0], 1),
    (1152, 256, [1, 0], [0, 2, 18], [3, 9] + list(range(16)), 16),
    (512, 10240, [1, 0], [0, 3, 7], [0, 1, 2, 0, 1, 2, 3], 4),   # 160 columns: split between CTAs
    # 100 columns of 12 stages dealt over 152 CTAs (7.9 stages each): ranges
    # inside one column (middle pieces) take and hand on the sums
    (1536, 6400, [1, 0], [0, 2, 4], [0, 1, 0, 1], 2),
])
def test_gateup_small(orc, dtype, H, I, uniq, offs, pair_tok, M):
    E = max(uniq) + 1
    ex = Experts(E, 2 * I, H, base_seed=23 + H + I, which=0)
    if dtype == "bf16":
        x = synth.activations_bf16(M, H, 29 + M, 4, 50.0, device="cuda")
    else:
        x = synth.activations_f32(M, H, 31 + M, device="cuda")
    h, qx, sx = run_gateup(x, ex, uniq, offs, pair_tok, I)
    g, u, Tg, Tu, h_ref, qx_ref, sx_ref = oracle_gateup(orc, _act_np(x), ex, uniq, offs, pair_tok, I)
    # the dump covers the tokens of the last unique expert
    toks = sorted(set(pair_tok[offs[-2]:offs[-1]]))
    assert np.array_equal(qx[toks], qx_ref[toks])
    assert np.array_equal(sx[toks].view(np.uint32), sx_ref[toks].view(np.uint32))
    check_h(h, g, u, Tg, Tu, h_ref)


def test_dense_ffn_full_size(orc):
    """Dense fused gate_up + SwiGLU + down at full size (hidden 6144,
    intermediate 12288, M = 1, 61 outlier channels x30): gate_up stage
    STRICT on h; down stage STRICT given the same h on both sides (the
    oracle's); end to end SPEC."""
    from bandwidth_bound_fp8_gb300 import moeq
    cfg = synth.DENSE_FFN
    H, I = cfg["H"], cfg["I"]
    gu = Experts(1, 2 * I, H, base_seed=cfg["seed"], which=0)
    dn = Experts(1, H, I, base_seed=cfg["seed"], which=1)
    x = synth.activations_bf16(1, H, cfg["seed"], cfg["n_outlier"], cfg["outlier_scale"], device="cuda")
    h, qx, sx = run_gateup(x, gu, [0], [0, 1], [0], I)
    g, u, Tg, Tu, h_ref, qx_ref, sx_ref = oracle_gateup(orc, bf16_bits(x), gu, [0], [0, 1], [0], I)
    assert np.array_equal(qx, qx_ref) and np.array_equal(sx.view(np.uint32), sx_ref.view(np.uint32))
    check_h(h, g, u, Tg, Tu, h_ref)
    # down on the oracle's h (same input both sides)
    y, qd, sd = run_down(torch.from_numpy(h_ref).cuda(), dn, [0], [0, 1])
    y_ref, T, qa, sa = oracle_down(orc, h_ref, dn, [0], [0, 1])
    assert np.array_equal(qd, qa) and np.array_equal(sd.view(np.uint32), sa.view(np.uint32))
    assert_close(y, y_ref, T, STRICT, what="down(h_ref)")
    # end to end: down on the GPU's own h, then the bf16 cast via moeq_combine (top_k = 0)
    y2, _, _ = run_down(torch.from_numpy(h).cuda(), dn, [0], [0, 1], want_dump=False)
    assert_close(y2, y_ref, T, SPEC_REL, SPEC_ABS, what="end-to-end y")
    plan = moeq.RoutePlan(1, 1, 1)
    plan.pair_of.view(-1)[0] = 0
    out = torch.empty((1, H), dtype=torch.bfloat16, device="cuda")
    moeq.moeq_combine(torch.from_numpy(y2).cuda().float(), H, plan, 1, 0, out)
    torch.cuda.synchronize()
    ref_bits = np.array([orc.f64_to_bf16_bits(v) for v in y2[0].astype(np.float32).astype(np.float64)])
    assert np.array_equal(bf16_bits(out)[0], ref_bits)


def test_gemm_deterministic(orc):
    """Two runs of the same call give bit-identical outputs."""
    ex = Experts(5, 256, 1152, base_seed=41, which=0)
    x = synth.activations_bf16(4, 1152, 43, 2, 30.0, device="cuda")
    args = ([4, 1, 3], [0, 2, 3, 7], [0, 2, 1, 0, 1, 2, 3], 128)
    h1, _, _ = run_gateup(x, ex, *args)
    h2, _, _ = run_gateup(x, ex, *args)
    assert np.array_equal(h1.view(np.uint32), h2.view(np.uint32))


def _status_after(call):
    from bandwidth_bound_fp8_gb300 import moeq
    ws = call()
    torch.cuda.synchronize()
    return moeq.moeq_read_device_status(ws.t, ws.nbytes)


@pytest.mark.skipif(os.environ.get("MOEQ_MTOK_KERNEL") == "0", reason="the multi-token kernel's own plan check")
@pytest.mark.parametrize("defect", ["expert", "rows", "order", "n_uniq"])
def test_down_plan_check(defect):
    """A plan that breaks the down call's contract leaves MOEQ_ERR_INVALID_ARG
    in the workspace status: an expert out of range, more than 16 rows on
    one expert, pair ranges out of order, n_uniq above max_uniq."""
    from bandwidth_bound_fp8_gb300 import moeq
    K, N = 256, 256
    ex = Experts(2, N, K, base_seed=5, which=1)
    uniq, offs, n = {"expert": ([0, 2], [0, 1, 2], 2), "rows": ([1], [0, 17], 1),
                     "order": ([0, 1], [0, 3, 2], 2), "n_uniq": ([0, 1], [0, 1, 2], 3)}[defect]
    P = max(offs)
    a = synth.activations_bf16(P, K, 3, 0, 1.0, device="cuda")
    du, do, _, _ = device_plan(uniq, offs, [0])
    dn = torch.tensor([n], dtype=torch.int32, device="cuda")
    y = torch.zeros((P, N), device="cuda")

    def call():
        ws = moeq.Workspace(moeq.moeq_gemm_workspace_size(N, K, P, len(uniq), 0))
        moeq.moeq_expert_gemm_down(a, K, N, ex.q, ex.s, ex.E, du, do, dn, len(uniq), P, y, ws)
        return ws
    assert _status_after(call) == moeq.MOEQ_ERR_INVALID_ARG


@pytest.mark.skipif(os.environ.get("MOEQ_MTOK_KERNEL") == "0", reason="the multi-token kernel's own plan check")
@pytest.mark.parametrize("defect", ["expert", "token", "twice", "n_uniq"])
def test_gateup_plan_check(defect):
    """As test_down_plan_check for the gate_up call: an expert out of range,
    a token out of range, a token twice on one expert, n_uniq above
    max_uniq."""
    from bandwidth_bound_fp8_gb300 import moeq
    H, I, M = 256, 256, 3
    ex = Experts(2, 2 * I, H, base_seed=7, which=0)
    uniq, offs, pair_tok, n = {"expert": ([5, 0], [0, 1, 4], [0, 0, 1, 2], 2),
                               "token": ([1, 0], [0, 1, 4], [3, 0, 1, 2], 2),
                               "twice": ([1, 0], [0, 2, 5], [1, 1, 0, 1, 2], 2),
                               "n_uniq": ([1, 0], [0, 1, 4], [0, 0, 1, 2], 3)}[defect]
    x = synth.activations_bf16(M, H, 9, 0, 1.0, device="cuda")
    du, do, dp, _ = device_plan(uniq, offs, pair_tok)
    dn = torch.tensor([n], dtype=torch.int32, device="cuda")
    h = torch.zeros((offs[-1], I), device="cuda")

    def call():
        ws = moeq.Workspace(moeq.moeq_gemm_workspace_size(I, H, M, len(uniq), 1))
        moeq.moeq_expert_gemm_gateup_swiglu(x, H, I, ex.q, ex.s, ex.E, du, do, dp, dn, len(uniq), offs[-1], h, ws)
        return ws
    assert _status_after(call) == moeq.MOEQ_ERR_INVALID_ARG
