"""moeq_moe_stack: L MoE layers in sequence as one CUDA graph (GLM-5.2 x10
§8b, graph replay of a decode step), against the oracle layer by layer.

Each layer's output is the next layer's x; each layer has its own weights
and logits.  Checked for every layer: the route plan the stack leaves in its
workspace (bit for bit against the oracle's routing of that layer's
logits), and the bf16 output against the oracle's layer fed the GPU's own
previous output (SPEC plus half a bf16 ulp).  The graph call (capture, then
replay), the eager call (MOEQ_STACK_EAGER) and a chain of moeq_moe_layer
calls give the same bits: layers after the first route before they wait for
the layer ahead, which changes when routing happens, not what it computes.
A stack call made inside the caller's own capture lands in the caller's
graph.  One and four tokens run the multi-token kernel, and
the full MoE shape runs two layers at one token."""
import numpy as np
import pytest
import torch

import synth
from moeq_testlib import SPEC_ABS, SPEC_REL, bf16_bits, half_ulp_bf16, to_np
from test_gpu_layer import Layer

pytestmark = pytest.mark.gpu


def _weights(layers):
    return ([l.gu.q for l in layers], [l.gu.s for l in layers], [l.dn.q for l in layers], [l.dn.s for l in layers])


def _check_vs_oracle(orc, moeq, layers, ws, x0, logits, out, E, H, I, k):
    L, M = len(layers), x0.shape[0]
    xin = bf16_bits(x0)
    for l, lay in enumerate(layers):
        lg = to_np(logits[l])
        r = orc.route(lg, k)
        plan = moeq.moeq_stack_plan(ws, L, M, H, I, E, k, l)
        U = int(to_np(plan.n_uniq)[0])
        assert U == r.n_uniq, f"layer {l}: unique experts"
        assert np.array_equal(to_np(plan.topk_id), r.topk_id), f"layer {l}: top-k ids"
        assert np.allclose(to_np(plan.topk_w), r.topk_w, rtol=0, atol=1e-6), f"layer {l}: routing weights"
        assert np.array_equal(to_np(plan.uniq)[:U], r.uniq), f"layer {l}: unique list"
        assert np.array_equal(to_np(plan.offs)[:U + 1], r.offs), f"layer {l}: offsets"
        assert np.array_equal(to_np(plan.pair_of), r.pair_of), f"layer {l}: pair map"
        ref = orc.moe_layer(xin, lg, k, lay.oracle_weights(orc, r.uniq), H, I)
        o = orc.bf16_bits_to_f32_array(bf16_bits(out[l])).astype(np.float64)
        r16 = orc.bf16_bits_to_f32_array(ref.out_bf16).astype(np.float64)
        bound = SPEC_REL * ref.Tout + SPEC_ABS + half_ulp_bf16(o, r16)
        err = np.abs(o - ref.out64)
        assert (err <= bound).all(), f"layer {l}: {(err > bound).sum()} outside, worst {np.max(err - bound)}"
        xin = bf16_bits(out[l])


def _run_all_ways(moeq, layers, x0, logits, E, H, I, k):
    """The stack as a graph (first call captures, second replays), eagerly,
    and as a chain of layer calls; returns the graph call's outputs and
    workspace after asserting that all agree bit for bit."""
    L, M = len(layers), x0.shape[0]
    ws = moeq.Workspace(moeq.moeq_stack_workspace_size(L, M, H, I, E + 1, k))
    w = _weights(layers)
    results = []
    for flags in (0, 0, moeq.MOEQ_STACK_EAGER):
        out = torch.full((L, M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        moeq.moeq_moe_stack(x0, logits, H, I, E, k, *w, out, ws, flags=flags)
        torch.cuda.synchronize()
        assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == 0
        results.append(out)
    lw = moeq.Workspace(moeq.moeq_workspace_size(M, H, I, E + 1, k))
    chain = torch.empty((L, M, H), dtype=torch.bfloat16, device="cuda")
    x = x0
    for l, lay in enumerate(layers):
        moeq.moeq_moe_layer(x, logits[l], H, I, E, k, lay.gu.q, lay.gu.s, lay.dn.q, lay.dn.s, chain[l], lw)
        x = chain[l]
    torch.cuda.synchronize()
    results.append(chain)
    names = ["graph capture", "graph replay", "eager", "layer calls"]
    for n, r in zip(names[1:], results[1:]):
        assert torch.equal(results[0].view(torch.int16), r.view(torch.int16)), f"{n} differs from the first call"
    return results[0], ws


@pytest.mark.parametrize("M", [1, 4])
def test_stack_matches_oracle_per_layer(orc, M):
    from bandwidth_bound_fp8_gb300 import moeq
    E, H, I, k, L = 16, 1024, 256, 4, 4
    layers = [Layer(E, H, I, seed=700 + l, layer=l) for l in range(L)]
    x0 = synth.activations_bf16(M, H, 710 + M, 10, 30.0, device="cuda")
    logits = torch.stack([synth.logits_f32(M, E, 720 + 10 * M + l, device="cuda") for l in range(L)])
    out, ws = _run_all_ways(moeq, layers, x0, logits, E, H, I, k)
    _check_vs_oracle(orc, moeq, layers, ws, x0, logits, out, E, H, I, k)


def test_stack_full_shape_two_layers(orc):
    from bandwidth_bound_fp8_gb300 import moeq
    c = synth.MOE_LAYER
    E, H, I, k, L = c["E"], c["H"], c["I"], c["top_k"], 2
    layers = [Layer(E, H, I, seed=c["seed"] + 7, layer=l) for l in range(L)]
    x0 = synth.activations_bf16(1, H, c["seed"] + 3, c["n_outlier"], c["outlier_scale"], device="cuda")
    logits = torch.stack([synth.logits_f32(1, E, c["seed"] + 30 + l, device="cuda") for l in range(L)])
    out, ws = _run_all_ways(moeq, layers, x0, logits, E, H, I, k)
    _check_vs_oracle(orc, moeq, layers, ws, x0, logits, out, E, H, I, k)


def test_stack_inside_caller_capture_and_release():
    """Inside the caller's torch.cuda.graph the stack's launches join the
    caller's graph; after moeq_stack_release_graphs a call captures anew."""
    from bandwidth_bound_fp8_gb300 import moeq
    E, H, I, k, L, M = 16, 512, 256, 4, 3, 1
    layers = [Layer(E, H, I, seed=760 + l, layer=l) for l in range(L)]
    x0 = synth.activations_bf16(M, H, 770, 5, 30.0, device="cuda")
    logits = torch.stack([synth.logits_f32(M, E, 780 + l, device="cuda") for l in range(L)])
    ws = moeq.Workspace(moeq.moeq_stack_workspace_size(L, M, H, I, E + 1, k))
    w = _weights(layers)
    ref = torch.empty((L, M, H), dtype=torch.bfloat16, device="cuda")
    moeq.moeq_moe_stack(x0, logits, H, I, E, k, *w, ref, ws)
    torch.cuda.synchronize()
    out = torch.zeros_like(ref)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        moeq.moeq_moe_stack(x0, logits, H, I, E, k, *w, out, ws)   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moeq.moeq_moe_stack(x0, logits, H, I, E, k, *w, out, ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    moeq.moeq_stack_release_graphs()
    out.zero_()
    moeq.moeq_moe_stack(x0, logits, H, I, E, k, *w, out, ws)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_stack_rejects_bad_arguments():
    from bandwidth_bound_fp8_gb300 import moeq
    E, H, I, k, L, M = 16, 512, 256, 4, 2, 1
    layers = [Layer(E, H, I, seed=790 + l, layer=l) for l in range(L)]
    x0 = synth.activations_bf16(M, H, 795, 5, 30.0, device="cuda")
    logits = torch.stack([synth.logits_f32(M, E, 796 + l, device="cuda") for l in range(L)])
    ws = moeq.Workspace(moeq.moeq_stack_workspace_size(L, M, H, I, E + 1, k))
    out = torch.empty((L, M, H), dtype=torch.bfloat16, device="cuda")
    gq, gs, dq, ds = _weights(layers)
    small = moeq.Workspace(moeq.moeq_stack_workspace_size(1, M, H, I, E + 1, k))
    with pytest.raises(moeq.MoeqError) as e:
        moeq.moeq_moe_stack(x0, logits, H, I, E, k, gq, gs, dq, ds, out, small)
    assert e.value.status == moeq.MOEQ_ERR_WORKSPACE
    with pytest.raises(moeq.MoeqError) as e:   # layer 1's down weights misaligned
        moeq.moeq_moe_stack(x0, logits, H, I, E, k, gq, gs, dq[:1] + [dq[1].data_ptr() + 1], ds, out, ws)
    assert e.value.status == moeq.MOEQ_ERR_INVALID_ARG
    with pytest.raises(moeq.MoeqError) as e:
        moeq.moeq_moe_stack(x0, logits, H, I, E, k, gq, gs, dq, ds, out, ws, flags=2)
    assert e.value.status == moeq.MOEQ_ERR_INVALID_ARG
