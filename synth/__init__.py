"""Seeded synthetic inputs shared by the tests, smoke() and bench.py.

This module holds none of the method's arithmetic: it only draws the raw
inputs (fp32 weights, bf16 activations with outlier channels, fp32 router
logits) with torch's seeded generators.  Quantisation, routing and every later
step are done separately by the oracle (CPU) and by the CUDA path.

torch's CPU and CUDA generators give different streams for the same seed, so a
parity test draws each input on ONE device and copies it to the other.

Workload recipe (shapes and distributions of the FP8 MoE decode workloads):
  * weights  ~ N(0, 0.02) in fp32, one independent seed per (layer, expert,
    matrix), later block-quantised to E4M3 with 128x128 scales;
  * x        ~ N(0, 1) in fp32 with a seeded set of outlier channels scaled by
    a constant factor (the same channels for every token), rounded to bf16;
  * logits   ~ N(0, 1) in fp32.
"""
from __future__ import annotations

import torch

WEIGHT_STD = 0.02


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def expert_seed(base: int, layer: int, expert: int, which: int) -> int:
    """Distinct seed for (layer, expert, matrix); which = 0 gate_up, 1 down."""
    return (int(base) * 1_000_003 + layer * 65_537 + expert * 4 + which) & 0x7FFFFFFF


def weight_f32(N: int, K: int, seed: int, device="cpu", std: float = WEIGHT_STD,
               out: torch.Tensor | None = None) -> torch.Tensor:
    """fp32 [N, K] ~ N(0, std^2)."""
    g = _gen(seed, device)
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=device)
    out.normal_(0.0, std, generator=g)
    return out


def outlier_channels(K: int, n_outlier: int, seed: int) -> torch.Tensor:
    """n_outlier distinct channel indices in [0, K), drawn on the CPU generator."""
    g = _gen(seed ^ 0x5A5A5A5A, "cpu")
    return torch.randperm(K, generator=g)[:n_outlier]


def activations_bf16(M: int, K: int, seed: int, n_outlier: int, outlier_scale: float,
                     device="cpu") -> torch.Tensor:
    """bf16 [M, K]: N(0,1) with n_outlier seeded channels multiplied by outlier_scale."""
    g = _gen(seed, device)
    x = torch.randn((M, K), generator=g, dtype=torch.float32, device=device)
    if n_outlier:
        ch = outlier_channels(K, n_outlier, seed).to(device)
        x[:, ch] *= outlier_scale
    return x.to(torch.bfloat16)


def activations_f32(M: int, K: int, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    """fp32 [M, K] ~ N(0, std^2) (stand-in for the fp32 h between the GEMMs)."""
    g = _gen(seed, device)
    return torch.randn((M, K), generator=g, dtype=torch.float32, device=device) * std


def logits_f32(M: int, E: int, seed: int, device="cpu") -> torch.Tensor:
    """fp32 [M, E] router logits ~ N(0,1)."""
    g = _gen(seed, device)
    return torch.randn((M, E), generator=g, dtype=torch.float32, device=device)


# Workload presets: the shapes of the dense and MoE FP8 decode projections.
DENSE_PROJ = dict(name="dense_proj_m1_k2048_n4096", M=1, K=2048, N=4096, n_outlier=4,
                  outlier_scale=50.0, seed=1000)
DENSE_FFN = dict(name="dense_ffn_m1_h6144_i12288", M=1, H=6144, I=12288, n_outlier=61,
                 outlier_scale=30.0, seed=1001)
MOE_LAYER = dict(name="moe_layer_h6144_i2048_e256_top8_shared1", H=6144, I=2048, E=256,
                 top_k=8, n_outlier=61, outlier_scale=30.0, seed=1002)
