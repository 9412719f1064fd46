"""GPU parity: moeq_quant_act and moeq_quant_weight against the oracle, bit
for bit on codes and scales (including signed zeros, zero groups, subnormal
and underflowing scales, outlier channels)."""
import numpy as np
import pytest
import torch

import synth
from moeq_testlib import Experts, bf16_bits, rows_to_tiles, tiles_to_rows, to_np

pytestmark = pytest.mark.gpu


def _gpu_quant(x):
    from bandwidth_bound_fp8_gb300 import moeq
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    s = torch.empty((M, K // 128), dtype=torch.float32, device="cuda")
    moeq.moeq_quant_act(x, q, s)
    torch.cuda.synchronize()
    return to_np(q), to_np(s)


@pytest.mark.parametrize("M,K,n_out,scale", [(1, 128, 0, 1.0), (1, 2048, 4, 50.0), (3, 640, 6, 30.0),
                                             (16, 6144, 61, 30.0), (5, 12288, 0, 1.0)])
def test_quant_act_bf16_bit_exact(orc, M, K, n_out, scale):
    x = synth.activations_bf16(M, K, 100 + M + K, n_out, scale, device="cuda")
    q, s = _gpu_quant(x)
    q_ref, s_ref = orc.quant_act(bf16_bits(x))
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q, q_ref)


@pytest.mark.parametrize("M,K,std", [(1, 128, 1.0), (7, 384, 1e-3), (16, 2048, 40.0), (144, 2048, 0.05)])
def test_quant_act_f32_bit_exact(orc, M, K, std):
    x = synth.activations_f32(M, K, 7 * M + K, device="cuda", std=std)
    q, s = _gpu_quant(x)
    q_ref, s_ref = orc.quant_act(to_np(x))
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q, q_ref)


def test_quant_act_edge_cases(orc):
    """Zero group with negative zeros, a group of ties, subnormal scale, a
    scale that underflows to zero, and huge values."""
    K = 128 * 6
    x = np.zeros((2, K), np.float32)
    x[0, 3] = -0.0
    x[0, 128:256] = np.arange(128, dtype=np.float32) * np.float32(2.0 ** -7) * np.float32(0.5)  # many ties
    x[0, 128] = np.float32(3.5)
    x[0, 256:384] = np.float32(1e-39) * np.linspace(-1, 1, 128, dtype=np.float32)            # subnormal s
    x[0, 384] = np.float32(1e-44)                                                                 # s -> 0
    x[0, 385] = np.float32(-1e-45)
    x[0, 512:640] = np.float32(3e38) * np.linspace(-1, 1, 128, dtype=np.float32)
    x[1] = np.float32(-0.0)
    x[1, 700] = np.float32(1.0)
    xg = torch.from_numpy(x).cuda()
    q, s = _gpu_quant(xg)
    q_ref, s_ref = orc.quant_act(x)
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q, q_ref)
    assert q[0, 3] == 0x80 and s[0, 0] == 0 and s[0, 3] == 0 and q[0, 385] == 0x80
    # bf16 input of the same values (rounded to bf16 first)
    xb = xg.to(torch.bfloat16)
    q, s = _gpu_quant(xb)
    q_ref, s_ref = orc.quant_act(bf16_bits(xb))
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q, q_ref)


def test_quant_weight_bit_exact(orc):
    ex = Experts(3, 256, 384, base_seed=5, which=0,
                 scale_blocks={(0, 1, 2): 0.0, (1, 0, 0): 1e4, (2, 1, 1): 1e-30})
    q, s = tiles_to_rows(to_np(ex.q), 3, 256, 384), to_np(ex.s)
    for e in range(3):
        q_ref, s_ref = ex.oracle(orc, e)
        assert np.array_equal(s[e].view(np.uint32), s_ref.view(np.uint32)), e
        assert np.array_equal(q[e], q_ref), e
    assert s[0, 1, 2] == 0.0 and set(np.unique(q[0, 128:, 256:]).tolist()) <= {0x00, 0x80}


def test_pack_weight_is_the_tile_permutation():
    """moeq_pack_weight moves row-major codes to the tile-major layout; the
    test's own permutation (tests/moeq_testlib.rows_to_tiles) must agree."""
    from bandwidth_bound_fp8_gb300 import moeq
    g = torch.Generator().manual_seed(3)
    rows = torch.randint(0, 256, (2, 384, 256), generator=g, dtype=torch.uint8)
    tiles = torch.empty_like(rows).cuda()
    moeq.moeq_pack_weight(rows.cuda(), tiles)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(tiles), rows_to_tiles(rows.numpy()))
    assert np.array_equal(tiles_to_rows(to_np(tiles), 2, 384, 256), rows.numpy())
