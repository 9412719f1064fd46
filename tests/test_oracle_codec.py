"""Pins of the oracle's E4M3FN codec and bf16 rounding (no GPU).

The codec is pinned to (a) the field formula's closed-form values, (b) torch's
float8_e4m3fn decode for all 256 codes (a library routine on the special case
of decoding), (c) torch's float8_e4m3fn encode inside the finite range, (d) the
RNE tie rule at every midpoint, and (e) agreement of the bisection encoder with
the linear-scan definition.
"""
import math

import numpy as np
import pytest
import torch


def test_decode_closed_forms(orc):
    d = orc.e4m3_decode
    assert d(0x00) == 0.0 and math.copysign(1, d(0x80)) == -1.0
    assert d(0x01) == 2.0 ** -9            # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9        # largest subnormal
    assert d(0x08) == 2.0 ** -6            # smallest normal
    assert d(0x38) == 1.0
    assert d(0x40) == 2.0
    assert d(0x7E) == 448.0                # largest finite
    assert d(0xFE) == -448.0
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))


def test_decode_matches_torch_all_codes(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = orc.e4m3_decode_table()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(ours[~nan]))


def test_encode_decode_roundtrip_all_finite_codes(orc):
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        v = orc.e4m3_decode(c)
        assert orc.e4m3_encode(v) == c, hex(c)
        assert orc.e4m3_encode_scan(v) == c, hex(c)


def test_midpoints_round_to_even(orc):
    """Every midpoint between neighbours goes to the even code; one fp32 ulp
    either side goes to the nearer neighbour."""
    for c in range(0x7E):
        lo, hi = orc.e4m3_decode(c), orc.e4m3_decode(c + 1)
        mid = 0.5 * (lo + hi)
        even = c if c % 2 == 0 else c + 1
        assert orc.e4m3_encode(mid) == even and orc.e4m3_encode_scan(mid) == even
        assert orc.e4m3_encode(-mid) == 0x80 | even
        below = float(np.nextafter(np.float32(mid), np.float32(0)))
        above = float(np.nextafter(np.float32(mid), np.float32(1000)))
        assert orc.e4m3_encode(below) == c
        assert orc.e4m3_encode(above) == c + 1


def test_saturation_and_signed_zero(orc):
    assert orc.e4m3_encode(448.0) == 0x7E
    assert orc.e4m3_encode(463.99) == 0x7E
    assert orc.e4m3_encode(1e30) == 0x7E
    assert orc.e4m3_encode(-1e30) == 0xFE
    assert orc.e4m3_encode(0.0) == 0x00
    assert orc.e4m3_encode(-0.0) == 0x80
    assert orc.e4m3_encode(-1e-30) == 0x80
    assert orc.e4m3_encode(2.0 ** -10) == 0x00          # tie between 0 and 2^-9 -> even (0)
    assert orc.e4m3_encode(2.0 ** -10 * 1.0000001) == 0x01


def test_bisection_equals_scan_random(orc):
    rng = np.random.default_rng(7)
    mags = np.exp(rng.uniform(np.log(1e-6), np.log(600.0), 4000)).astype(np.float32)
    vals = mags * rng.choice([-1, 1], 4000).astype(np.float32)
    for v in vals:
        assert orc.e4m3_encode(float(v)) == orc.e4m3_encode_scan(float(v))


def test_encode_matches_torch_in_range(orc):
    """torch's float8_e4m3fn cast rounds to nearest even; inside [-448, 448]
    it must agree with the oracle code for code (outside, torch gives NaN where
    the satfinite convention clamps)."""
    rng = np.random.default_rng(11)
    v = np.concatenate([
        rng.uniform(-448, 448, 20000),
        rng.normal(0, 1, 20000),
        rng.normal(0, 1e-2, 5000),
        np.exp(rng.uniform(np.log(1e-5), np.log(448), 5000)),
    ]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([orc.e4m3_encode(float(x)) for x in v], np.uint8)
    assert np.array_equal(ref, ours)


def test_bf16_rounding(orc):
    assert orc.f64_to_bf16_bits(1.0) == 0x3F80
    assert orc.f64_to_bf16_bits(-2.0) == 0xC000
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7: ties to even -> 1.0
    assert orc.f64_to_bf16_bits(1.0 + 2.0 ** -8) == 0x3F80
    assert orc.f64_to_bf16_bits(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert orc.f64_to_bf16_bits(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    # agreement with torch's bf16 cast on fp32-representable values
    rng = np.random.default_rng(3)
    v = rng.normal(0, 10, 5000).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.uint16).numpy()
    ours = np.array([orc.f64_to_bf16_bits(float(x)) for x in v], np.uint16)
    assert np.array_equal(ref, ours)
