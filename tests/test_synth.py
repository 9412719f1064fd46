"""The seeded input recipe (the one module the oracle and the CUDA path
share; it draws inputs and holds none of the method's arithmetic): seeds
give identical draws and distinct seeds differ, the outlier channels are
the stated count of distinct channels shared by every token and scaled by
the stated factor before the bf16 rounding, every (layer, expert, matrix)
of the 8-layer stack gets its own seed, and the distributions have the
stated moments."""
import numpy as np
import torch

import synth


def test_draws_are_seeded():
    a = synth.activations_bf16(3, 1024, 5, 10, 30.0)
    assert torch.equal(a, synth.activations_bf16(3, 1024, 5, 10, 30.0))
    assert not torch.equal(a, synth.activations_bf16(3, 1024, 6, 10, 30.0))
    assert torch.equal(synth.logits_f32(2, 256, 9), synth.logits_f32(2, 256, 9))
    assert torch.equal(synth.weight_f32(128, 256, 3), synth.weight_f32(128, 256, 3))
    assert not torch.equal(synth.weight_f32(128, 256, 3), synth.weight_f32(128, 256, 4))


def test_outlier_channels_are_scaled_before_rounding():
    M, K, seed, n, f = 4, 2048, 11, 20, 50.0
    ch = synth.outlier_channels(K, n, seed)
    assert len(set(ch.tolist())) == n and 0 <= int(ch.min()) and int(ch.max()) < K
    g = torch.Generator().manual_seed(seed)
    base = torch.randn((M, K), generator=g, dtype=torch.float32)
    want = base.clone()
    want[:, ch] *= f                        # the same channels for every token
    assert torch.equal(synth.activations_bf16(M, K, seed, n, f), want.to(torch.bfloat16))
    assert torch.equal(synth.activations_bf16(M, K, seed, 0, f), base.to(torch.bfloat16))


def test_presets_follow_the_recipe():
    c = synth.MOE_LAYER
    assert c["n_outlier"] == round(0.01 * c["H"]) == 61          # "1 % outlier channels"
    assert (c["H"], c["I"], c["E"], c["top_k"]) == (6144, 2048, 256, 8)
    assert synth.DENSE_FFN["n_outlier"] == round(0.01 * synth.DENSE_FFN["H"])


def test_every_matrix_of_the_stack_has_its_own_seed():
    seeds = {synth.expert_seed(2000, l, e, w) for l in range(8) for e in range(257) for w in range(2)}
    assert len(seeds) == 8 * 257 * 2


def test_moments():
    w = synth.weight_f32(1024, 1024, 21).double()
    assert abs(w.mean().item()) < 1e-4 and abs(w.std().item() - synth.WEIGHT_STD) < 1e-4
    lg = synth.logits_f32(64, 1024, 22).double()
    assert abs(lg.mean().item()) < 0.01 and abs(lg.std().item() - 1.0) < 0.01
    x = synth.activations_bf16(64, 1024, 23, 0, 1.0).double()
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1.0) < 0.01
    assert np.isfinite(x.numpy()).all()
