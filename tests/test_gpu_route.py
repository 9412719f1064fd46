"""GPU parity: moeq_route against the oracle -- expert ids, unique list,
offsets and pair bookkeeping bit for bit; routing weights within fp32
rounding of the softmax (|d| <= 1e-6, weights are in [0, 1])."""
import numpy as np
import pytest
import torch

import synth
from moeq_testlib import to_np

pytestmark = pytest.mark.gpu


def _gpu_route(logits, k):
    from bandwidth_bound_fp8_gb300 import moeq
    M, E = logits.shape
    plan = moeq.RoutePlan(M, E, k)
    moeq.moeq_route(logits, plan, k)
    torch.cuda.synchronize()
    return plan


def _compare(plan, ref, M, k):
    U = int(to_np(plan.n_uniq)[0])
    P = M * k + M
    assert U == ref.n_uniq
    assert np.array_equal(to_np(plan.topk_id), ref.topk_id)
    assert np.allclose(to_np(plan.topk_w), ref.topk_w, rtol=0, atol=1e-6)
    assert np.array_equal(to_np(plan.uniq)[:U], ref.uniq)
    assert np.array_equal(to_np(plan.offs)[:U + 1], ref.offs)
    assert np.array_equal(to_np(plan.pair_tok)[:P], ref.pair_tok)
    assert np.array_equal(to_np(plan.pair_of), ref.pair_of)


@pytest.mark.parametrize("M,E,k", [(1, 256, 8), (2, 256, 8), (4, 256, 8), (16, 256, 8),
                                   (3, 8, 2), (16, 64, 1), (5, 1024, 16), (16, 16, 16)])
def test_route_matches_oracle(orc, M, E, k):
    logits = synth.logits_f32(M, E, 300 + M * E + k, device="cuda")
    plan = _gpu_route(logits, k)
    _compare(plan, orc.route(to_np(logits), k), M, k)


def test_route_ties_and_shared_tokens(orc):
    # integer logits: many ties, resolved to the lower id; tokens share experts
    g = torch.Generator().manual_seed(9)
    logits = torch.randint(0, 4, (16, 256), generator=g).float().cuda()
    plan = _gpu_route(logits, 8)
    _compare(plan, orc.route(to_np(logits), 8), 16, 8)
    # every token identical: 8 unique experts shared by all 16 tokens
    one = synth.logits_f32(1, 256, 77, device="cuda").repeat(16, 1)
    plan = _gpu_route(one, 8)
    ref = orc.route(to_np(one), 8)
    _compare(plan, ref, 16, 8)
    assert ref.n_uniq == 9
