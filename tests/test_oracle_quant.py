"""Pins of the oracle's live activation quantisation and weight quantisation.

Pinned to hand-derived worked cases (tests/golden/quant_hand.json), to the
power-of-two invariance the scale convention implies, to the bound
|s*decode(q) - x| <= half an E4M3 step of x/s (closed form of RNE), and to
the special case where a group's amax/448 is an exact power of two.
"""
import json
import os

import numpy as np
import pytest


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_quant_hand_cases(orc, golden_dir):
    doc = _load(golden_dir, "quant_hand.json")
    assert doc["citation"]
    for case in doc["cases"]:
        K = case["K"]
        x = np.zeros((1, K), np.float32)
        for i, v in case["x_nonzero"].items():
            x[0, int(i)] = v
        codes = np.zeros(K, np.uint8)
        for i, c in case["codes_nonzero"].items():
            codes[int(i)] = int(c, 16)
        q, s = orc.quant_act(x)
        assert np.array_equal(s[0], np.array(case["s"], np.float32)), case["name"]
        assert np.array_equal(q[0], codes), case["name"]


def _step(v):
    """Spacing of the E4M3 grid at magnitude v (closed form of the format)."""
    v = abs(v)
    if v < 2.0 ** -6:
        return 2.0 ** -9
    e = int(np.floor(np.log2(v)))
    return 2.0 ** (e - 3)


def test_quant_rounding_bound_and_scale(orc):
    rng = np.random.default_rng(5)
    x = rng.normal(0, 1, (4, 512)).astype(np.float32)
    x[:, 7] *= 50
    q, s = orc.quant_act(x)
    dec = orc.e4m3_decode_table()
    for m in range(4):
        for g in range(4):
            grp = x[m, g * 128:(g + 1) * 128]
            amax = np.float32(np.max(np.abs(grp)))
            assert s[m, g] == np.float32(amax / np.float32(448.0))
            v = (grp / s[m, g]).astype(np.float32)
            d = dec[q[m, g * 128:(g + 1) * 128]]
            for vi, di in zip(v, d):
                assert abs(di - vi) <= 0.5 * _step(vi) + 1e-12
            # the amax element maps to the top of the grid
            assert np.max(np.abs(d)) == 448.0


def test_quant_power_of_two_invariance(orc):
    rng = np.random.default_rng(9)
    x = rng.normal(0, 1, (3, 384)).astype(np.float32)
    q0, s0 = orc.quant_act(x)
    for j in (-20, -3, 1, 7, 30):
        q1, s1 = orc.quant_act((x * np.float32(2.0 ** j)).astype(np.float32))
        assert np.array_equal(q0, q1)
        assert np.array_equal(s1, (s0 * np.float32(2.0 ** j)).astype(np.float32))


def test_quant_bf16_equals_widened_f32(orc):
    import torch
    xb = torch.randn(2, 256, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    bits = xb.view(torch.uint16).numpy()
    q0, s0 = orc.quant_act(bits)
    q1, s1 = orc.quant_act(orc.bf16_bits_to_f32_array(bits))
    assert np.array_equal(q0, q1) and np.array_equal(s0, s1)


def test_quant_scale_underflow_gives_zero_scale(orc):
    """amax/448 below half the smallest fp32 subnormal rounds to 0: the group
    gets s = 0 and signed-zero codes; a subnormal-but-nonzero s still works."""
    x = np.zeros((1, 256), np.float32)
    x[0, 0] = np.float32(1e-44)       # amax/448 -> 0
    x[0, 1] = np.float32(-1e-45)
    x[0, 128] = np.float32(1e-38)     # amax/448 is a subnormal fp32
    x[0, 129] = np.float32(-5e-39)
    q, s = orc.quant_act(x)
    assert s[0, 0] == 0.0 and q[0, 0] == 0x00 and q[0, 1] == 0x80
    assert s[0, 1] > 0 and s[0, 1] < np.finfo(np.float32).tiny
    assert q[0, 128] == 0x7E
    assert q[0, 129] & 0x80


def test_weight_quant_block_structure(orc):
    """A 256x256 weight with four blocks of different magnitude: each block
    gets amax/448 of its own entries; the codes equal the activation codec
    applied to w/s; a zero block gets s = 0 and zero codes."""
    rng = np.random.default_rng(2)
    w = rng.normal(0, 0.02, (256, 256)).astype(np.float32)
    w[:128, 128:] *= 100
    w[128:, :128] = 0
    q, s = orc.quant_weight(w)
    assert s.shape == (2, 2)
    for nb in range(2):
        for kb in range(2):
            blk = w[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            assert s[nb, kb] == np.float32(np.float32(np.max(np.abs(blk))) / np.float32(448))
    assert s[1, 0] == 0.0 and not q[128:, :128].any()
    # the block codec agrees with the activation codec row by row where the
    # row's own amax equals the block amax (scaled to the same s)
    blk = w[:128, :128]
    r = int(np.argmax(np.max(np.abs(blk), axis=1)))
    qa, sa = orc.quant_act(blk[r:r + 1].copy())
    assert sa[0, 0] == s[0, 0]
    assert np.array_equal(qa[0], q[r, :128])
