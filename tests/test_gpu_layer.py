"""GPU parity of moeq_moe_layer (route -> quant+gate_up+SwiGLU -> quant+down
-> combine) against the oracle's layer.

Checked on every case, for every token and every (token, expert) pair:
  * routing bookkeeping bit for bit (ids, unique list, offsets, pair lists),
    routing weights within 1e-6;
  * the live quantisation of x (a2): the layer's own codes and scales,
    dumped by the kernel, bit for bit against the oracle's quantisation of x;
  * h per pair within the STRICT bound propagated through SwiGLU, against
    the oracle's gate_up GEMM of the same token on the oracle's own weights;
  * the live quantisation of h (a5): the codes and scales the down GEMM
    multiplies, dumped by the kernel, bit for bit against the oracle's
    quantisation of the GPU's own fp32 h (the two sides' h may differ by an
    fp32 ulp, which can move a code, so each side's codes are checked
    against its own h);
  * the bf16 output within SPEC of the fp64 reference plus half a bf16 ulp
    at the output's magnitude (the final rounding), end to end from the same
    x, logits and fp32 weights.
Reduced shapes span several blocks and ragged group counts; the full MoE
shape (hidden 6144, 256 routed experts of 4096x6144 + 6144x2048, top-8 + 1
shared) runs at M = 1 (every output), and at M = 4 and 16 with the whole plan
and every pair's h and codes checked and the outputs of sampled tokens (tokens
are independent, a property pinned in the oracle).

Without the per-pair y output a layer of 1..16 tokens runs the multi-token
kernel; asking for y keeps the persistent engine's row-block down path, so
both are checked (and test_gpu_paths re-runs the cases without y on the
engine, and the one-token ones on the one-token kernel).
"""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import synth
from moeq_testlib import SPEC_ABS, SPEC_REL, STRICT, Experts, bf16_bits, half_ulp_bf16, to_np
from test_gpu_gemm import h_bound

pytestmark = pytest.mark.gpu


class Layer:
    def __init__(self, E, H, I, seed, layer=0):
        self.E, self.H, self.I = E, H, I
        self.gu = Experts(E + 1, 2 * I, H, base_seed=seed, which=0, layer=layer)
        self.dn = Experts(E + 1, H, I, base_seed=seed, which=1, layer=layer)
        self._oracle_w = {}

    def run(self, x, logits, k, with_y=True, dumps=True):
        from bandwidth_bound_fp8_gb300 import moeq
        M = x.shape[0]
        plan = moeq.RoutePlan(M, self.E, k)
        P = plan.max_pairs
        h = torch.full((P, self.I), float("nan"), device="cuda")
        y = torch.full((P, self.H), float("nan"), device="cuda") if with_y else None
        out = torch.empty((M, self.H), dtype=torch.bfloat16, device="cuda")
        d = {}
        if dumps:
            d["q_x"] = torch.zeros((M, self.H), dtype=torch.uint8, device="cuda")
            d["s_x"] = torch.zeros((M, self.H // 128), dtype=torch.float32, device="cuda")
            d["q_h"] = torch.zeros((P, self.I), dtype=torch.uint8, device="cuda")
            d["s_h"] = torch.zeros((P, self.I // 128), dtype=torch.float32, device="cuda")
        ws = moeq.Workspace(moeq.moeq_workspace_size(M, self.H, self.I, self.E + 1, k))
        moeq.moeq_moe_layer(x, logits, self.H, self.I, self.E, k, self.gu.q, self.gu.s, self.dn.q, self.dn.s,
                            out, ws, plan=plan, h=h, y=y, **d)
        torch.cuda.synchronize()
        assert moeq.moeq_read_device_status(ws.t, ws.nbytes) == 0
        return out, plan, h, y, d

    def oracle_weights(self, orc, ids):
        """The oracle's own quantisation of the fp32 draws of the given
        experts (gate_up and down), in parallel host threads, cached."""
        todo = [int(e) for e in ids if int(e) not in self._oracle_w]
        with cf.ThreadPoolExecutor(max_workers=16) as ex:
            for b0 in range(0, len(todo), 8):   # 8 experts' fp32 draws in host memory at a time
                f32 = {e: (self.gu.f32(e), self.dn.f32(e)) for e in todo[b0:b0 + 8]}
                fut = {e: (ex.submit(orc.quant_weight, a), ex.submit(orc.quant_weight, b)) for e, (a, b) in f32.items()}
                for e, (fa, fb) in fut.items():
                    self._oracle_w[e] = (*fa.result(), *fb.result())
        return {int(e): self._oracle_w[int(e)] for e in ids}


def check_layer(orc, lay, x, logits, k, rows=None, with_y=True):
    M = x.shape[0]
    out, plan, h, y, d = lay.run(x, logits, k, with_y=with_y)
    rows = list(range(M)) if rows is None else rows
    x_bits, lg = bf16_bits(x), to_np(logits)

    # routing bookkeeping, every token
    r = orc.route(lg, k)
    U = int(to_np(plan.n_uniq)[0])
    assert U == r.n_uniq
    assert np.array_equal(to_np(plan.topk_id), r.topk_id)
    assert np.allclose(to_np(plan.topk_w), r.topk_w, rtol=0, atol=1e-6)
    assert np.array_equal(to_np(plan.uniq)[:U], r.uniq)
    assert np.array_equal(to_np(plan.offs)[:U + 1], r.offs)
    assert np.array_equal(to_np(plan.pair_tok)[:r.n_pairs], r.pair_tok)
    assert np.array_equal(to_np(plan.pair_of), r.pair_of)

    # live quantisation of x (a2): the kernel's own codes and scales
    qx, sx = orc.quant_act(x_bits)
    assert np.array_equal(to_np(d["q_x"]), qx), "x codes"
    assert np.array_equal(to_np(d["s_x"]).view(np.uint32), sx.view(np.uint32)), "x scales"

    # h of every pair, and the codes of its live quantisation (a5)
    experts = lay.oracle_weights(orc, r.uniq)
    I, P = lay.I, r.n_pairs
    hg = to_np(h)[:P]
    for ui, e in enumerate(r.uniq):
        qgu, sgu = experts[int(e)][:2]
        for p in range(r.offs[ui], r.offs[ui + 1]):
            t = r.pair_tok[p]
            gy, gT = orc.gemm(qx[t:t + 1], sx[t:t + 1], qgu, sgu)
            b = h_bound(gy[0, :I], gy[0, I:], gT[0, :I], gT[0, I:], STRICT)
            h_ref = orc.swiglu_vec(gy[0, :I], gy[0, I:]).astype(np.float64)
            err = np.abs(hg[p].astype(np.float64) - h_ref)
            assert (err <= b).all(), f"h pair {p}: worst {np.max(err - b)}"
    qh, sh = orc.quant_act(hg.astype(np.float32))
    assert np.array_equal(to_np(d["q_h"])[:P], qh), "h codes"
    assert np.array_equal(to_np(d["s_h"])[:P].view(np.uint32), sh.view(np.uint32)), "h scales"

    # the bf16 output of the checked tokens
    for group in ([rows] if rows == list(range(M)) else [[m] for m in rows]):
        sub_x, sub_l = x_bits[group], lg[group]
        ref_r = orc.route(sub_l, k)
        ref = orc.moe_layer(sub_x, sub_l, k, lay.oracle_weights(orc, ref_r.uniq), lay.H, lay.I)
        o = orc.bf16_bits_to_f32_array(bf16_bits(out)[group]).astype(np.float64)
        r16 = orc.bf16_bits_to_f32_array(ref.out_bf16).astype(np.float64)
        bound = SPEC_REL * ref.Tout + SPEC_ABS + half_ulp_bf16(o, r16)
        err = np.abs(o - ref.out64)
        assert (err <= bound).all(), f"out: {(err > bound).sum()} outside, worst {np.max(err - bound)}"
        # how close in practice (reported): most elements equal the reference bf16
        same = np.mean(bf16_bits(out)[group] == ref.out_bf16)
        assert same > 0.9, same
    return out


@pytest.mark.parametrize("M,E,H,I,k,with_y", [(1, 16, 1024, 256, 4, True), (1, 16, 1024, 256, 4, False),
                                              (1, 12, 1280, 384, 3, False), (1, 8, 640, 256, 2, False),
                                              (1, 16, 512, 2432, 7, False), (1, 16, 512, 2432, 7, True),
                                              (3, 16, 640, 384, 2, True), (16, 32, 512, 256, 8, True),
                                              (5, 8, 768, 128, 8, True),
                                              (2, 16, 1024, 256, 4, False), (3, 16, 512, 384, 2, False),
                                              (5, 8, 768, 128, 8, False), (16, 32, 512, 256, 8, False),
                                              (8, 32, 512, 2560, 8, False), (13, 64, 256, 1280, 6, False),
                                              (2, 8, 256, 128, 2, False), (3, 4, 512, 256, 2, False)])
def test_layer_reduced(orc, M, E, H, I, k, with_y):
    # (1, 8, 640, ...): an odd number of output row blocks keeps one token
    # on the persistent engine; (1, 16, 512, 2432, 7): 8 unique experts x 19
    # K groups of down = 152 columns, one per CTA on 152 SMs.  Two or more
    # tokens without y run the multi-token kernel: (8, 32, 512, 2560, 8) and
    # (13, 64, 256, 1280, 6) have several hundred columns of 6 (3) stages, so
    # the even split of the stages over the CTAs cuts columns inside gate_up
    # and inside down; (2, 8, 256, 128, 2) and (3, 4, 512, 256, 2) have
    # fewer columns than SMs: one column per CTA, many CTAs idle
    lay = Layer(E, H, I, seed=50 + M + E)
    x = synth.activations_bf16(M, H, 51 + M, max(1, H // 100), 30.0, device="cuda")
    logits = synth.logits_f32(M, E, 52 + M, device="cuda")
    check_layer(orc, lay, x, logits, k, with_y=with_y)


@pytest.fixture(scope="module")
def full_layer():
    c = synth.MOE_LAYER
    return Layer(c["E"], c["H"], c["I"], seed=c["seed"])


@pytest.mark.parametrize("with_y", [True, False])
def test_layer_full_m1(orc, full_layer, with_y):
    c = synth.MOE_LAYER
    x = synth.activations_bf16(1, c["H"], c["seed"], c["n_outlier"], c["outlier_scale"], device="cuda")
    logits = synth.logits_f32(1, c["E"], c["seed"] + 1, device="cuda")
    out = check_layer(orc, full_layer, x, logits, c["top_k"], with_y=with_y)
    if not with_y:
        # determinism of the sums over K groups: a second run is bit-identical
        out2 = full_layer.run(x, logits, c["top_k"], with_y=False, dumps=False)[0]
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("M,rows,with_y", [(4, [0, 3], True), (16, [5], True), (2, [0, 1], False),
                                           (4, [1, 2], False), (16, [0, 15], False)])
def test_layer_full_multi_token(orc, full_layer, M, rows, with_y):
    # with y: the persistent engine's row-block down; without: the
    # multi-token kernel (the path of every bench layer with 2..16 tokens)
    c = synth.MOE_LAYER
    x = synth.activations_bf16(M, c["H"], c["seed"] + M, c["n_outlier"], c["outlier_scale"], device="cuda")
    logits = synth.logits_f32(M, c["E"], c["seed"] + 100 + M, device="cuda")
    out = check_layer(orc, full_layer, x, logits, c["top_k"], rows=rows, with_y=with_y)
    # determinism: a second run is bit-identical
    out2 = full_layer.run(x, logits, c["top_k"], with_y=with_y, dumps=False)[0]
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
