"""Pin of the tensor-parallel split on the oracle: I cut into R slices of
whole 128-wide groups (GLM-5.2 x10, bandwidth model: TP8).  Rank r's shard
of every expert is gate_up's gate rows and up rows of its slice and down's
columns of its slice.  The R shard layers' fp64 outputs add up to the
unsharded layer's fp64 output (the per-pair sums only regroup), and each
shard's live quantisation of h -- codes and scales -- is exactly the
unsharded layer's on its slice (an h group never straddles slices)."""
import numpy as np
import pytest
import torch

import synth
from test_oracle_layer import _tiny_layer


def oracle_shard(experts: dict, I: int, R: int, r: int) -> dict:
    """Rank r's slice of row-major oracle weights (codes and block scales)."""
    Is = I // R
    out = {}
    for e, (qgu, sgu, qd, sd) in experts.items():
        rows = np.r_[r * Is:(r + 1) * Is, I + r * Is:I + (r + 1) * Is]
        brow = np.r_[r * Is // 128:(r + 1) * Is // 128, (I + r * Is) // 128:(I + (r + 1) * Is) // 128]
        out[e] = (qgu[rows], sgu[brow], qd[:, r * Is:(r + 1) * Is], sd[:, r * Is // 128:(r + 1) * Is // 128])
    return out


@pytest.mark.parametrize("R,M", [(2, 1), (4, 3), (2, 5)])
def test_shards_add_up_to_the_layer(orc, R, M):
    E, H, I, k = 8, 256, 512, 2
    experts = _tiny_layer(orc, E, H, I, seed=11)
    x = synth.activations_bf16(M, H, 31 + M, 3, 30.0).view(torch.uint16).numpy()
    logits = synth.logits_f32(M, E, 32 + M).numpy()
    full = orc.moe_layer(x, logits, k, experts, H, I)
    total = np.zeros_like(full.out64)
    Is = I // R
    for r in range(R):
        sh = orc.moe_layer(x, logits, k, oracle_shard(experts, I, R, r), H, Is)
        total += sh.out64
        # the same plan and the same live quantisation of x on every rank
        assert np.array_equal(sh.route.uniq, full.route.uniq) and np.array_equal(sh.qx, full.qx)
        # h's codes and scales of the slice are the unsharded layer's
        assert np.array_equal(sh.qh, full.qh[:, r * Is:(r + 1) * Is])
        assert np.array_equal(sh.sh.view(np.uint32), full.sh[:, r * Is // 128:(r + 1) * Is // 128].view(np.uint32))
    assert np.all(np.abs(total - full.out64) <= 1e-12 * full.Tout + 1e-300)
    # and not trivially: a shard alone is far from the layer
    assert np.max(np.abs(sh.out64 - full.out64)) > 1e-3 * np.max(np.abs(full.out64))
