"""Helpers shared by the GPU parity tests: seeded expert weights on both
sides (CUDA path quantises them with moeq_quant_weight, the oracle with its
own codec, from the same fp32 draw) and the tolerances.

Tolerances (floating point outputs; codes, scales and indices are compared
bit for bit):
  * SPEC:   |gpu - ref| <= 1e-3 * T + 1e-5, T = sum of |scaled terms| of the
            output element (the oracle returns T with every GEMM);
  * STRICT: |gpu - ref| <= 2e-5 * T.  The CUDA path sums every term in fp32
            through at most ~115 dependent roundings (16 products per lane in
            two interleaved chains, one scale multiply and one running-sum
            update per K group for up to 96 groups, a 3-level shuffle tree and
            a split-K sum over a few partials), so its error is below
            115 * 2^-24 * T = 6.9e-6 * T; STRICT leaves a 3x margin.  STRICT
            applies wherever both sides quantise the same input; the layer
            output after the second live quantisation (of h, which the two
            sides compute with different rounding) is held to SPEC.
"""
from __future__ import annotations

import numpy as np
import torch

import synth

STRICT = 2e-5
SPEC_REL, SPEC_ABS = 1e-3, 1e-5


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def tiles_to_rows(q_tiles: np.ndarray, E: int, N: int, K: int) -> np.ndarray:
    """Undo the tile-major weight layout (a byte permutation, no arithmetic):
    tile (e, nb, kb) holds rows of 128 bytes whose 16-byte chunk c sits at
    chunk position c ^ (r % 8)."""
    t = np.asarray(q_tiles, np.uint8).reshape(E, N // 128, K // 128, 128, 8, 16)
    r = np.arange(128)[:, None]
    c = np.arange(8)[None, :]
    t = t[:, :, :, r, c ^ (r & 7), :]                      # logical chunk order
    return t.transpose(0, 1, 3, 2, 4, 5).reshape(E, N, K)


def rows_to_tiles(q_rows: np.ndarray) -> np.ndarray:
    """Inverse of tiles_to_rows."""
    E, N, K = q_rows.shape
    t = np.asarray(q_rows, np.uint8).reshape(E, N // 128, 128, K // 128, 8, 16).transpose(0, 1, 3, 2, 4, 5)
    r = np.arange(128)[:, None]
    c = np.arange(8)[None, :]
    out = np.empty_like(t)
    out[:, :, :, r, c ^ (r & 7), :] = t
    return out.reshape(E, N, K)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return to_np(t.contiguous().view(torch.uint16))


class Experts:
    """E expert matrices [N, K] drawn per expert from its own seed, quantised
    on the GPU by libmoeq (codes tile-major in self.q, E*N*K bytes); the
    oracle view re-draws the same fp32 weights and quantises them on the CPU."""

    def __init__(self, E: int, N: int, K: int, base_seed: int, which: int, layer: int = 0,
                 scale_blocks: dict | None = None):
        from bandwidth_bound_fp8_gb300 import moeq
        self.E, self.N, self.K, self.base, self.which, self.layer = E, N, K, base_seed, which, layer
        self.scale_blocks = scale_blocks or {}
        self.q = torch.empty((E, N, K), dtype=torch.uint8, device="cuda")
        self.s = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device="cuda")
        buf = torch.empty((N, K), dtype=torch.float32, device="cuda")
        for e in range(E):
            self._draw(e, buf)
            moeq.moeq_quant_weight(buf[None], self.q[e:e + 1], self.s[e:e + 1])
        torch.cuda.synchronize()

    def _draw(self, e, buf):
        synth.weight_f32(self.N, self.K, synth.expert_seed(self.base, self.layer, e, self.which),
                         device="cuda", out=buf)
        for (ee, nb, kb), f in self.scale_blocks.items():
            if ee == e:
                buf[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128] *= f

    def f32(self, e: int) -> np.ndarray:
        buf = torch.empty((self.N, self.K), dtype=torch.float32, device="cuda")
        self._draw(e, buf)
        return to_np(buf)

    def oracle(self, orc, e: int):
        return orc.quant_weight(self.f32(e))


def half_ulp_bf16(*vals) -> np.ndarray:
    """Half a bf16 ulp at the larger magnitude of the given values (arrays of
    the same shape), from the exponent: a value in [2^e, 2^(e+1)) has ulp
    2^(e-7) in bf16 (8 significant bits), so half of it is 2^(e-8); zero and
    subnormal magnitudes take the subnormal spacing's half, 2^-134.  This
    bounds the final rounding of a result to bf16: |RN(g) - g| is at most
    half an ulp at |RN(g)|."""
    m = np.max(np.abs(np.stack([np.asarray(v, np.float64) for v in vals])), axis=0)
    e = np.floor(np.log2(np.maximum(m, 2.0 ** -126)))
    return np.where(m >= 2.0 ** -126, 2.0 ** (e - 8), 2.0 ** -134)


def assert_close(gpu, ref, T, rel, absl=0.0, what=""):
    gpu = np.asarray(gpu, np.float64)
    err = np.abs(gpu - ref)
    bound = rel * T + absl
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside |d| <= {rel}*T + {absl}; "
                             f"worst at {i}: gpu={gpu[i]!r} ref={ref[i]!r} T={T[i]!r}")
    return float(np.max(err / np.maximum(T, 1e-300))) if err.size else 0.0


def device_plan(uniq, offs, pair_tok, device="cuda"):
    """A plan given by the test (host lists) as device int32 tensors."""
    t = lambda a: torch.tensor(np.asarray(a, np.int32), device=device)
    return t(uniq), t(offs), t(pair_tok), t([len(uniq)])
