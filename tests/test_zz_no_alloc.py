"""moeq_expert_gemm_down_noalloc (static scratch, no workspace) against
moeq_expert_gemm_down (caller workspace): the same inputs through both, two
no-alloc calls in a row, outputs within the tests' STRICT tolerance of the
workspace call's, quantisation dumps identical, device status 0; a problem
beyond the static scratch is refused.  Named to be collected last, so it runs
both after every other GPU test and alone in a fresh process."""
import numpy as np
import pytest
import torch

import synth
from moeq_testlib import STRICT, Experts, assert_close, device_plan, to_np

pytestmark = pytest.mark.gpu


def _oracle_T(orc, a_np, ex, uniq, offs):
    qa, sa = orc.quant_act(a_np)
    T = np.zeros((offs[-1], ex.N))
    for u, e in enumerate(uniq):
        qw, sw = ex.oracle(orc, e)
        for p in range(offs[u], offs[u + 1]):
            T[p] = orc.gemm(qa[p:p + 1], sa[p:p + 1], qw, sw)[1][0]
    return T


def _act_np(a):
    return to_np(a.contiguous().view(torch.uint16)) if a.dtype == torch.bfloat16 else to_np(a)


@pytest.mark.parametrize("case", ["dense_projection", "experts_bf16", "experts_f32"])
def test_noalloc_matches_workspace_call(orc, case):
    from bandwidth_bound_fp8_gb300 import moeq
    if case == "dense_projection":
        cfg = synth.DENSE_PROJ
        K, N, uniq, offs = cfg["K"], cfg["N"], [0], [0, 1]
        ex = Experts(1, N, K, base_seed=cfg["seed"], which=1)
        a = synth.activations_bf16(1, K, cfg["seed"], cfg["n_outlier"], cfg["outlier_scale"], device="cuda")
    else:
        K, N, uniq, offs = 640, 384, [3, 0, 4], [0, 1, 3, 8]
        ex = Experts(5, N, K, base_seed=97, which=1)
        P = offs[-1]
        a = (synth.activations_bf16(P, K, 61, 3, 30.0, device="cuda") if case == "experts_bf16"
             else synth.activations_f32(P, K, 67, device="cuda", std=0.3))
    P = offs[-1]
    du, do, _, dn = device_plan(uniq, offs, [0])

    # the existing entry, with a caller workspace
    y_ws = torch.full((P, N), float("nan"), device="cuda")
    q_ws = torch.zeros((P, K), dtype=torch.uint8, device="cuda")
    s_ws = torch.zeros((P, K // 128), dtype=torch.float32, device="cuda")
    ws = moeq.Workspace(moeq.moeq_gemm_workspace_size(N, K, P, len(uniq), 0))
    moeq.moeq_expert_gemm_down(a, K, N, ex.q, ex.s, ex.E, du, do, dn, len(uniq), P, y_ws, ws, q_ws, s_ws)
    torch.cuda.synchronize()
    assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == 0

    T = _oracle_T(orc, _act_np(a), ex, uniq, offs)
    ref = to_np(y_ws).astype(np.float64)
    for call in range(2):   # two calls in a row on the same static scratch
        y = torch.full((P, N), float("nan"), device="cuda")
        q = torch.zeros((P, K), dtype=torch.uint8, device="cuda")
        s = torch.zeros((P, K // 128), dtype=torch.float32, device="cuda")
        st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        moeq.moeq_expert_gemm_down_noalloc(a, K, N, ex.q, ex.s, ex.E, du, do, dn, len(uniq), P, y, q, s,
                                           device_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, f"call {call}: device status {int(st.item())}"
        assert np.array_equal(to_np(q), to_np(q_ws)), f"call {call}: codes differ"
        assert np.array_equal(to_np(s).view(np.uint32), to_np(s_ws).view(np.uint32)), f"call {call}: scales"
        assert_close(to_np(y), ref, T, STRICT, what=f"no-alloc call {call} vs workspace call")


def test_noalloc_refuses_beyond_static_scratch():
    """K = 32768 with 64 pair rows needs ~13 MiB of scratch (> 8 MiB):
    refused with MOEQ_ERR_WORKSPACE before anything is launched."""
    from bandwidth_bound_fp8_gb300 import moeq
    K, N, P = 32768, 128, 64
    w = torch.zeros((1, N, K), dtype=torch.uint8, device="cuda")
    sw = torch.zeros((1, N // 128, K // 128), dtype=torch.float32, device="cuda")
    a = torch.zeros((P, K), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((P, N), dtype=torch.float32, device="cuda")
    du, do, _, dn = device_plan([0], [0, 16], [0])
    with pytest.raises(moeq.MoeqError) as err:
        moeq.moeq_expert_gemm_down_noalloc(a, K, N, w, sw, 1, du, do, dn, 1, P, y)
    assert err.value.status == moeq.MOEQ_ERR_WORKSPACE
