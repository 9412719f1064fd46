"""Pins of the oracle's block-scaled FP8 GEMM.

Pinned to a hand-derived cancelling case (tests/golden/gemm_hand.json), the
all-ones closed form, single-block isolation, zero-scale blocks, additivity
over K groups (catches transposed block scales and a transposed weight
operand), and brute force: numpy's float64 matmul over the dequantised
operands (a library routine) on tiny shapes that span several blocks.
"""
import json
import os

import numpy as np


def test_gemm_hand_case(orc, golden_dir):
    with open(os.path.join(golden_dir, "gemm_hand.json")) as f:
        c = json.load(f)
    M, N, K = c["M"], c["N"], c["K"]
    qa = np.zeros((M, K), np.uint8)
    qw = np.zeros((N, K), np.uint8)
    for g in range(K // 128):
        qa[:, g * 128:(g + 1) * 128] = int(c["qa_group_codes"][g], 16)
        qw[:, g * 128:(g + 1) * 128] = int(c["qw_group_codes"][g], 16)
    sa = np.array([c["sa"]], np.float32)
    sw = np.array(c["sw"], np.float32)
    y, T = orc.gemm(qa, sa, qw, sw)
    assert np.all(y == c["y"]) and np.all(T == c["T"])


def test_gemm_all_ones(orc):
    K, N = 384, 256
    qa = np.full((2, K), 0x38, np.uint8)                  # 1.0
    qw = np.full((N, K), 0x38, np.uint8)
    y, T = orc.gemm(qa, np.ones((2, 3), np.float32), qw, np.ones((2, 3), np.float32))
    assert np.all(y == K) and np.all(T == K)


def test_gemm_single_block_isolation(orc):
    rng = np.random.default_rng(0)
    K, N = 512, 384
    qa = rng.integers(0, 256, (1, K)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x38
    qw = rng.integers(0, 256, (N, K)).astype(np.uint8)
    qw[(qw & 0x7F) == 0x7F] = 0x38
    sa = np.zeros((1, 4), np.float32)
    sw = np.zeros((3, 4), np.float32)
    sa[0, 2] = 0.5
    sw[1, 2] = 3.0
    y, _ = orc.gemm(qa, sa, qw, sw)
    dec = orc.e4m3_decode_table()
    expect = np.zeros(N)
    for n in range(128, 256):
        expect[n] = 1.5 * float(np.sum(dec[qa[0, 256:384]] * dec[qw[n, 256:384]]))
    assert np.array_equal(y[0], expect)


def test_gemm_zero_scale_block_contributes_nothing(orc):
    rng = np.random.default_rng(1)
    K, N = 256, 128
    qa = np.full((1, K), 0x7E, np.uint8)
    qw = np.full((N, K), 0x7E, np.uint8)
    sw = np.array([[0.0, 1.0]], np.float32)
    y, T = orc.gemm(qa, np.ones((1, 2), np.float32), qw, sw)
    assert np.all(y == 128 * 448.0 * 448.0) and np.all(T == y)


def test_gemm_brute_force_numpy(orc):
    dec = orc.e4m3_decode_table()
    rng = np.random.default_rng(4)
    for (M, N, K) in [(1, 128, 128), (3, 256, 256), (2, 384, 512)]:
        qa = rng.integers(0, 256, (M, K)).astype(np.uint8)
        qw = rng.integers(0, 256, (N, K)).astype(np.uint8)
        qa[(qa & 0x7F) == 0x7F] = 0
        qw[(qw & 0x7F) == 0x7F] = 0
        sa = rng.uniform(0.01, 2, (M, K // 128)).astype(np.float32)
        sw = rng.uniform(0.01, 2, (N // 128, K // 128)).astype(np.float32)
        A = dec[qa] * np.repeat(sa.astype(np.float64), 128, axis=1)
        W = dec[qw] * np.kron(sw.astype(np.float64), np.ones((128, 128)))
        ref = A @ W.T
        Tref = np.abs(A) @ np.abs(W).T
        y, T = orc.gemm(qa, sa, qw, sw)
        assert np.allclose(y, ref, rtol=0, atol=1e-12 * Tref.max())
        assert np.allclose(T, Tref, rtol=1e-13)


def test_gemm_is_the_sum_of_its_k_groups(orc):
    """y over all of K equals the sum, in group order, of the GEMMs limited to
    one 128-wide K group each (with that group's activation and block
    scales), the way a split over K decomposes it.  A scale taken from the
    wrong group or row block breaks the equality."""
    rng = np.random.default_rng(7)
    M, N, K = 2, 384, 640
    qa = rng.integers(0, 256, (M, K)).astype(np.uint8)
    qw = rng.integers(0, 256, (N, K)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0
    qw[(qw & 0x7F) == 0x7F] = 0
    sa = rng.uniform(0.01, 2, (M, K // 128)).astype(np.float32)
    sw = rng.uniform(0.01, 2, (N // 128, K // 128)).astype(np.float32)
    y, T = orc.gemm(qa, sa, qw, sw)
    acc, acc_T = np.zeros_like(y), np.zeros_like(T)
    for g in range(K // 128):
        k = slice(g * 128, (g + 1) * 128)
        y_g, T_g = orc.gemm(qa[:, k], sa[:, g:g + 1], qw[:, k], sw[:, g:g + 1])
        acc += y_g
        acc_T += T_g
    assert np.allclose(acc, y, rtol=0, atol=1e-14 * T.max())
    assert np.allclose(acc_T, T, rtol=1e-14)
