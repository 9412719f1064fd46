"""moeq_expert_gemm_down_noalloc (static scratch, no workspace) against the
oracle and against moeq_expert_gemm_down (caller workspace).

The same inputs go through both calls, and the no-alloc call runs twice in a
row on the same static scratch.  Its outputs are within the tests' STRICT
tolerance of the oracle's GEMM and bit-identical to the workspace call's
(the two run the same kernel path in the same order); its quantisation dumps
equal the workspace call's, and its device status is 0.  The cases cover the
dense projection, experts with 1 to 5 rows, and one expert with 16 rows,
which takes the tcgen05 path by default; child processes re-run every case
with the tcgen05 crossover forced to 1 row (everything on the tensor cores)
and to 17 (everything on the CUDA cores).  A problem beyond the static
scratch is refused.  Named to be collected last, so it runs both after every
other GPU test and alone in a fresh process."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import synth
from moeq_testlib import STRICT, Experts, assert_close, device_plan, to_np

pytestmark = pytest.mark.gpu


def _oracle(orc, a_np, ex, uniq, offs):
    qa, sa = orc.quant_act(a_np)
    y = np.zeros((offs[-1], ex.N))
    T = np.zeros((offs[-1], ex.N))
    for u, e in enumerate(uniq):
        qw, sw = ex.oracle(orc, e)
        for p in range(offs[u], offs[u + 1]):
            yy, tt = orc.gemm(qa[p:p + 1], sa[p:p + 1], qw, sw)
            y[p], T[p] = yy[0], tt[0]
    return y, T


def _act_np(a):
    return to_np(a.contiguous().view(torch.uint16)) if a.dtype == torch.bfloat16 else to_np(a)


@pytest.mark.parametrize("case", ["dense_projection", "experts_bf16", "experts_f32", "sixteen_rows"])
def test_noalloc_matches_oracle_and_workspace_call(orc, case):
    from bandwidth_bound_fp8_gb300 import moeq
    if case == "dense_projection":
        cfg = synth.DENSE_PROJ
        K, N, uniq, offs = cfg["K"], cfg["N"], [0], [0, 1]
        ex = Experts(1, N, K, base_seed=cfg["seed"], which=1)
        a = synth.activations_bf16(1, K, cfg["seed"], cfg["n_outlier"], cfg["outlier_scale"], device="cuda")
    elif case == "sixteen_rows":
        K, N, uniq, offs = 768, 256, [1], [0, 16]
        ex = Experts(2, N, K, base_seed=83, which=1)
        a = synth.activations_bf16(16, K, 89, 4, 30.0, device="cuda")
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

    y_ref, T = _oracle(orc, _act_np(a), ex, uniq, offs)
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
        assert_close(to_np(y), y_ref, T, STRICT, what=f"no-alloc call {call} vs the oracle")
        assert np.array_equal(to_np(y).view(np.uint32), to_np(y_ws).view(np.uint32)), \
            f"no-alloc call {call} is not bit-identical to the workspace call"


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


@pytest.mark.skipif(os.environ.get("MOEQ_MMA_MIN_TOKENS") is not None, reason="already a forced-path child")
@pytest.mark.parametrize("crossover", ["1", "17"])
def test_noalloc_with_forced_path(crossover):
    env = dict(os.environ, MOEQ_MMA_MIN_TOKENS=crossover)
    here = os.path.dirname(os.path.abspath(__file__))
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.abspath(__file__), "-k", "matches_oracle"]
    r = subprocess.run(cmd, env=env, cwd=os.path.dirname(here), capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, f"crossover {crossover}:\n{r.stdout[-3000:]}\n{r.stderr[-2000:]}"
