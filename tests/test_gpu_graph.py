"""A chain of MoE layers captured in one CUDA graph (GLM-5.2 x10, §8b: CUDA
graphs are one of the runtime changes that took host-side cost out of each
decode step).  Each layer's output is the next layer's x, and each layer
routes its own logits.  The layer kernels keep their per-launch state in the
workspace and leave it ready for the next launch, so a replay needs no host
work.  Every layer of a replay matches the oracle's layer fed the GPU's own
previous bf16 output (SPEC plus half a bf16 ulp), and replaying the graph
twice gives, bit for bit, the outputs of the same calls made eagerly, at one
token (the multi-token kernel, launched with programmatic dependent launch)
and at four (the persistent engine)."""
import numpy as np
import pytest
import torch

import synth
from moeq_testlib import SPEC_ABS, SPEC_REL, bf16_bits, half_ulp_bf16, to_np
from test_gpu_layer import Layer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M", [1, 4])
def test_layer_chain_in_a_cuda_graph(orc, M):
    from bandwidth_bound_fp8_gb300 import moeq
    E, H, I, k, L = 16, 1024, 256, 4, 4
    layers = [Layer(E, H, I, seed=400 + l, layer=l) for l in range(L)]
    x0 = synth.activations_bf16(M, H, 410 + M, 10, 30.0, device="cuda")
    logits = [synth.logits_f32(M, E, 420 + 10 * M + l, device="cuda") for l in range(L)]
    ws = moeq.Workspace(moeq.moeq_workspace_size(M, H, I, E + 1, k))
    outs = [torch.empty((M, H), dtype=torch.bfloat16, device="cuda") for _ in range(L)]

    def chain():
        x = x0
        for l, lay in enumerate(layers):
            moeq.moeq_moe_layer(x, logits[l], H, I, E, k, lay.gu.q, lay.gu.s, lay.dn.q, lay.dn.s, outs[l], ws)
            x = outs[l]

    chain()
    torch.cuda.synchronize()
    assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == 0
    eager = [o.clone() for o in outs]

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        chain()   # the first calls on the capture's stream happen outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    for rep in range(2):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == 0
        for l in range(L):
            assert torch.equal(outs[l].view(torch.int16), eager[l].view(torch.int16)), (rep, l)
    # every layer of the replay against the oracle, fed the GPU's own input
    xin = bf16_bits(x0)
    for l, lay in enumerate(layers):
        lg = to_np(logits[l])
        r = orc.route(lg, k)
        ref = orc.moe_layer(xin, lg, k, lay.oracle_weights(orc, r.uniq), H, I)
        o = orc.bf16_bits_to_f32_array(bf16_bits(outs[l])).astype(np.float64)
        r16 = orc.bf16_bits_to_f32_array(ref.out_bf16).astype(np.float64)
        bound = SPEC_REL * ref.Tout + SPEC_ABS + half_ulp_bf16(o, r16)
        err = np.abs(o - ref.out64)
        assert (err <= bound).all(), f"layer {l}: {(err > bound).sum()} outside, worst {np.max(err - bound)}"
        xin = bf16_bits(outs[l])
