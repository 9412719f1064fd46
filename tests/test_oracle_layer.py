"""Pins of the oracle's MoE layer composition.

Pinned to brute force on tiny shapes -- the layer rebuilt from library
routines (numpy argsort / softmax via scipy, numpy float64 matmul over the
dequantised operands, scipy's expit) and the separately pinned quantiser --
and to invariants: tokens are independent (row m of an M-token layer equals
the one-token layer of token m, exactly), an all-zero gate weight gives
an all-zero output, and doubling the down weights' scales doubles the output.
"""
import numpy as np
import torch
from scipy.special import expit, softmax

import synth


def _tiny_layer(orc, E=8, H=256, I=128, seed=0):
    experts = {}
    for e in range(E + 1):
        wgu = synth.weight_f32(2 * I, H, synth.expert_seed(seed, 0, e, 0)).numpy()
        wd = synth.weight_f32(H, I, synth.expert_seed(seed, 0, e, 1)).numpy()
        qgu, sgu = orc.quant_weight(wgu)
        qd, sd = orc.quant_weight(wd)
        experts[e] = (qgu, sgu, qd, sd)
    return experts


def _deq(orc, q, s):
    dec = orc.e4m3_decode_table()
    return dec[q] * np.kron(s.astype(np.float64), np.ones((128, 128)))


def test_layer_brute_force(orc):
    E, H, I, k, M = 8, 256, 128, 2, 3
    experts = _tiny_layer(orc, E, H, I)
    x = synth.activations_bf16(M, H, 21, 3, 30.0).view(torch.uint16).numpy()
    logits = synth.logits_f32(M, E, 22).numpy()
    r = orc.moe_layer(x, logits, k, experts, H, I)
    dec = orc.e4m3_decode_table()

    order = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :k]
    w = softmax(np.take_along_axis(logits.astype(np.float64), order, axis=1), axis=1)
    qx, sx = orc.quant_act(x)
    xq = dec[qx] * np.repeat(sx.astype(np.float64), 128, axis=1)
    out = np.zeros((M, H))
    for m in range(M):
        for j, e in enumerate(list(order[m]) + [E]):
            qgu, sgu, qd, sd = experts[e]
            gu = _deq(orc, qgu, sgu) @ xq[m]
            g, u = gu[:I], gu[I:]
            h = (g * expit(g) * u).astype(np.float32)
            qh, sh = orc.quant_act(h[None, :])
            hq = dec[qh[0]] * np.repeat(sh[0].astype(np.float64), 128)
            y = _deq(orc, qd, sd) @ hq
            out[m] += (1.0 if e == E else w[m, j]) * y
    scale = r.Tout.max()
    assert np.allclose(r.out64, out, rtol=0, atol=1e-12 * scale)
    # the per-pair h of the oracle equals the brute-force h to fp32 rounding
    assert np.array_equal(r.route.topk_id, order)


def test_layer_token_independence(orc):
    E, H, I, k, M = 8, 256, 128, 2, 4
    experts = _tiny_layer(orc, E, H, I, seed=1)
    x = synth.activations_bf16(M, H, 31, 3, 30.0).view(torch.uint16).numpy()
    logits = synth.logits_f32(M, E, 32).numpy()
    r = orc.moe_layer(x, logits, k, experts, H, I)
    for m in range(M):
        r1 = orc.moe_layer(x[m:m + 1].copy(), logits[m:m + 1].copy(), k, experts, H, I)
        assert np.array_equal(r1.out64[0], r.out64[m])
        assert np.array_equal(r1.out_bf16[0], r.out_bf16[m])


def test_layer_zero_gate_and_scale_linearity(orc):
    E, H, I, k, M = 4, 256, 128, 2, 2
    experts = _tiny_layer(orc, E, H, I, seed=2)
    x = synth.activations_bf16(M, H, 41, 0, 1.0).view(torch.uint16).numpy()
    logits = synth.logits_f32(M, E, 42).numpy()
    base = orc.moe_layer(x, logits, k, experts, H, I)
    doubled = {e: (a, b, c, (d * np.float32(2)).astype(np.float32)) for e, (a, b, c, d) in experts.items()}
    r2 = orc.moe_layer(x, logits, k, doubled, H, I)
    assert np.array_equal(r2.out64, 2 * base.out64)
    zero_gate = {}
    for e, (qgu, sgu, qd, sd) in experts.items():
        sgu0 = sgu.copy()
        sgu0[: I // 128] = 0                                 # gate rows [0, I)
        zero_gate[e] = (qgu, sgu0, qd, sd)
    r0 = orc.moe_layer(x, logits, k, zero_gate, H, I)
    assert not np.any(r0.out64) and not np.any(r0.h)
