"""GPU parity of an FP8 LM-head projection (GLM-5.2 x10, §8b: the LM head
in FP8 is one of the runtime changes behind the decode speed-up).  A
vocabulary-sized weight, N = 151,552 rows of K = 6144 (931 MB of E4M3
codes), goes through the down GEMM call with one expert and the trivial
plan: the same live-quantised weight stream as the experts'.  One token,
and four (a draft-verification batch).  The prologue's codes and scales
are checked bit for bit, and sampled 128-row blocks of the output within
STRICT: the first and last blocks and two inside.  The oracle quantises
those blocks from the same fp32 rows; a block scale covers 128 rows, so a
128-row slab quantises on its own."""
import numpy as np
import pytest
import torch

import synth
from moeq_testlib import STRICT, Experts, assert_close, bf16_bits, to_np
from test_gpu_gemm import run_down

pytestmark = pytest.mark.gpu

VOCAB, HIDDEN = 151552, 6144


@pytest.fixture(scope="module")
def lm_head():
    return Experts(1, VOCAB, HIDDEN, base_seed=3100, which=1)


@pytest.mark.parametrize("M", [1, 4])
def test_lm_head_fp8(orc, lm_head, M):
    ex = lm_head
    x = synth.activations_bf16(M, HIDDEN, 3101 + M, 61, 30.0, device="cuda")
    y, qd, sd = run_down(x, ex, [0], [0, M])
    qa, sa = orc.quant_act(bf16_bits(x))
    assert np.array_equal(qd, qa) and np.array_equal(sd.view(np.uint32), sa.view(np.uint32))
    w = torch.empty((VOCAB, HIDDEN), dtype=torch.float32, device="cuda")
    ex._draw(0, w)
    for nb in (0, 517, 1000, VOCAB // 128 - 1):
        qw, sw = orc.quant_weight(to_np(w[nb * 128:(nb + 1) * 128]))
        y_ref, T = orc.gemm(qa, sa, qw, sw)
        assert_close(y[:, nb * 128:(nb + 1) * 128], y_ref, T, STRICT, what=f"logits {nb * 128}..{nb * 128 + 127}")
