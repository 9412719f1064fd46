"""GPU parity of the tensor-parallel layer (GLM-5.2 x10, bandwidth model:
TP8), with R ranks emulated one after another on one GPU -- no kernel waits
for another rank's, so nothing needs the ranks to run at the same time.

Checked: the shards moeq_tp_shard_weights cuts are, byte for byte, the
slices of the full weights (codes through the tile layout, and scales);
each rank's fp32 partial is within SPEC of the oracle's layer on that shard;
the live quantisation of h on each rank is, bit for bit, the oracle's
quantisation of that rank's own h; moeq_tp_reduce adds the partials in rank
order (a case where any other order gives another value); and the reduced
bf16 output is within SPEC plus half a bf16 ulp of the oracle's unsharded
layer, for R = 2 and 4 at one and at several tokens, and at the full MoE
shape."""
import numpy as np
import pytest
import torch

import synth
from moeq_testlib import SPEC_ABS, SPEC_REL, bf16_bits, half_ulp_bf16, tiles_to_rows, to_np
from test_gpu_layer import Layer
from test_oracle_tp import oracle_shard

pytestmark = pytest.mark.gpu


def _check_shard_bytes(lay, sh, R, r):
    E1, H, I, Is = lay.E + 1, lay.H, lay.I, lay.I // R
    full_gu = tiles_to_rows(to_np(lay.gu.q).ravel(), E1, 2 * I, H)
    shard_gu = tiles_to_rows(to_np(sh.w_gu).ravel(), E1, 2 * Is, H)
    rows = np.r_[r * Is:(r + 1) * Is, I + r * Is:I + (r + 1) * Is]
    assert np.array_equal(shard_gu, full_gu[:, rows]), "gate_up shard codes"
    brow = np.r_[r * Is // 128:(r + 1) * Is // 128, (I + r * Is) // 128:(I + (r + 1) * Is) // 128]
    assert np.array_equal(to_np(sh.s_gu), to_np(lay.gu.s)[:, brow]), "gate_up shard scales"
    full_d = tiles_to_rows(to_np(lay.dn.q).ravel(), E1, H, I)
    shard_d = tiles_to_rows(to_np(sh.w_d).ravel(), E1, H, Is)
    assert np.array_equal(shard_d, full_d[:, :, r * Is:(r + 1) * Is]), "down shard codes"
    assert np.array_equal(to_np(sh.s_d), to_np(lay.dn.s)[:, :, r * Is // 128:(r + 1) * Is // 128]), "down shard scales"


def _run_tp(orc, lay, x, logits, k, R, check_bytes=True):
    from bandwidth_bound_fp8_gb300 import moeq, tp
    M, H, I, E = x.shape[0], lay.H, lay.I, lay.E
    Is = I // R
    parts = torch.full((R, M, H), float("nan"), device="cuda")
    x_bits, lg = bf16_bits(x), to_np(logits)
    r_plan = orc.route(lg, k)
    experts = lay.oracle_weights(orc, r_plan.uniq)
    for r in range(R):
        sh = tp.TPShard(E + 1, H, I, R, r, lay.gu.q, lay.gu.s, lay.dn.q, lay.dn.s)
        if check_bytes:
            _check_shard_bytes(lay, sh, R, r)
        ws = moeq.Workspace(moeq.moeq_workspace_size(M, H, Is, E + 1, k))
        P = moeq.moeq_max_pairs(M, k)
        h = torch.full((P, Is), float("nan"), device="cuda")
        qh = torch.zeros((P, Is), dtype=torch.uint8, device="cuda")
        shs = torch.zeros((P, Is // 128), dtype=torch.float32, device="cuda")
        moeq.moeq_moe_layer_shard(x, logits, H, Is, E, k, sh.w_gu, sh.s_gu, sh.w_d, sh.s_d, parts[r], ws,
                                  h=h, q_h=qh, s_h=shs)
        torch.cuda.synchronize()
        assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == 0
        ref = orc.moe_layer(x_bits, lg, k, oracle_shard(experts, I, R, r), H, Is)
        err = np.abs(to_np(parts[r]).astype(np.float64) - ref.out64)
        assert (err <= SPEC_REL * ref.Tout + SPEC_ABS).all(), f"rank {r} partial: worst {np.max(err)}"
        npairs = r_plan.n_pairs
        qh_ref, sh_ref = orc.quant_act(to_np(h)[:npairs])
        assert np.array_equal(to_np(qh)[:npairs], qh_ref), f"rank {r}: h codes"
        assert np.array_equal(to_np(shs)[:npairs].view(np.uint32), sh_ref.view(np.uint32)), f"rank {r}: h scales"
    out = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    moeq.moeq_tp_reduce(parts, out)
    torch.cuda.synchronize()
    full = orc.moe_layer(x_bits, lg, k, experts, H, I)
    o = orc.bf16_bits_to_f32_array(bf16_bits(out)).astype(np.float64)
    r16 = orc.bf16_bits_to_f32_array(full.out_bf16).astype(np.float64)
    bound = SPEC_REL * full.Tout + SPEC_ABS + half_ulp_bf16(o, r16)
    err = np.abs(o - full.out64)
    assert (err <= bound).all(), f"reduced out: {(err > bound).sum()} outside, worst {np.max(err - bound)}"
    # the reduce is the rank-order fp32 sum of the partials, rounded once
    acc = to_np(parts[0]).copy()
    for r in range(1, R):
        acc += to_np(parts[r])
    ref16 = np.array([orc.f64_to_bf16_bits(float(v)) for v in acc.ravel()], np.uint16).reshape(M, H)
    assert np.array_equal(bf16_bits(out), ref16)


@pytest.mark.parametrize("M,R", [(1, 2), (1, 4), (4, 2), (4, 4), (16, 2)])
def test_tp_reduced(orc, M, R):
    E, H, I, k = 16, 1024, 512, 4
    lay = Layer(E, H, I, seed=900 + M)
    x = synth.activations_bf16(M, H, 910 + M, 10, 30.0, device="cuda")
    logits = synth.logits_f32(M, E, 920 + M, device="cuda")
    _run_tp(orc, lay, x, logits, k, R)


def test_tp_full_shape_m1(orc):
    c = synth.MOE_LAYER
    lay = Layer(c["E"], c["H"], c["I"], seed=c["seed"] + 50)
    x = synth.activations_bf16(1, c["H"], c["seed"] + 51, c["n_outlier"], c["outlier_scale"], device="cuda")
    logits = synth.logits_f32(1, c["E"], c["seed"] + 52, device="cuda")
    _run_tp(orc, lay, x, logits, c["top_k"], 4, check_bytes=False)


def test_tp_reduce_adds_in_rank_order():
    """Partials 1e8, 1, -1e8, 1: in rank order fp32 gives ((1e8 + 1) - 1e8)
    + 1 = 1 (1e8 + 1 rounds to 1e8); other orders give 0 or 2."""
    from bandwidth_bound_fp8_gb300 import moeq
    vals = [1e8, 1.0, -1e8, 1.0]
    parts = torch.stack([torch.full((2, 256), v, device="cuda") for v in vals])
    out = torch.empty((2, 256), dtype=torch.bfloat16, device="cuda")
    moeq.moeq_tp_reduce(parts, out)
    torch.cuda.synchronize()
    assert torch.all(out.float() == 1.0)


def test_tp_shard_rejects_uneven_split():
    from bandwidth_bound_fp8_gb300 import moeq
    w = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(moeq.MoeqError) as e:
        moeq.moeq_tp_shard_weights(2, 256, 384, 2, 0, w, w, w, w, w, w, w, w)
    assert e.value.status == moeq.MOEQ_ERR_UNSUPPORTED_SHAPE
