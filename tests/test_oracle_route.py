"""Pins of the oracle's top-k routing and expert deduplication.

Pinned to hand-derived cases with ties (tests/golden/route_hand.json), to
numpy's stable argsort (a library routine) for the selection, scipy's softmax
for the weights, and to invariants: weights sum to one, permuting expert ids
permutes the plan, M = 1 gives k + 1 unique experts with one pair each, and
the unique set is the union of the per-token picks.
"""
import json
import math
import os

import numpy as np
from scipy.special import softmax


def _check_plan_consistency(r, M, E, k):
    P = M * k + M
    assert r.n_pairs == P
    assert r.uniq[-1] == E
    assert list(r.uniq[:-1]) == sorted(set(int(e) for e in r.topk_id.ravel()))
    assert r.offs[0] == 0 and r.offs[-1] == P
    for u, e in enumerate(r.uniq):
        toks = r.pair_tok[r.offs[u]:r.offs[u + 1]]
        assert list(toks) == sorted(toks)
        if e == E:
            assert list(toks) == list(range(M))
        else:
            assert list(toks) == [m for m in range(M) if e in r.topk_id[m]]
    for m in range(M):
        for j in range(k + 1):
            p = r.pair_of[m, j]
            assert r.pair_tok[p] == m
            e = E if j == k else r.topk_id[m, j]
            u = int(np.searchsorted(r.offs, p, side="right")) - 1
            assert r.uniq[u] == e


def test_route_hand_cases(orc, golden_dir):
    with open(os.path.join(golden_dir, "route_hand.json")) as f:
        doc = json.load(f)
    assert doc["citation"]
    c = doc["cases"][0]
    r = orc.route(np.array(c["logits"], np.float32), c["k"])
    den = 2 + math.exp(-2)
    assert r.topk_id.tolist() == c["topk_id"]
    assert np.allclose(r.topk_w[0], [1 / den, 1 / den, math.exp(-2) / den], rtol=1e-15)
    assert r.uniq.tolist() == c["uniq"] and r.offs.tolist() == c["offs"]
    assert r.pair_tok.tolist() == c["pair_tok"] and r.pair_of.tolist() == c["pair_of"]
    c = doc["cases"][1]
    r = orc.route(np.array(c["logits"], np.float32), c["k"])
    a = 1 / (1 + math.exp(-1))
    assert r.topk_id.tolist() == c["topk_id"]
    assert np.allclose(r.topk_w, [[a, 1 - a], [a, 1 - a]], rtol=1e-15)
    assert r.uniq.tolist() == c["uniq"] and r.offs.tolist() == c["offs"]
    assert r.pair_tok.tolist() == c["pair_tok"] and r.pair_of.tolist() == c["pair_of"]


def test_route_matches_argsort_and_softmax(orc):
    rng = np.random.default_rng(12)
    for M in (1, 2, 4, 16):
        logits = rng.normal(0, 1, (M, 256)).astype(np.float32)
        logits[0, 10] = logits[0, 200] = logits[0].max() + 1   # a tie at the top
        r = orc.route(logits, 8)
        order = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :8]
        assert np.array_equal(r.topk_id, order)
        w = softmax(np.take_along_axis(logits.astype(np.float64), order, axis=1), axis=1)
        assert np.allclose(r.topk_w, w, rtol=1e-14, atol=0)
        assert np.allclose(r.topk_w.sum(axis=1), 1.0, rtol=0, atol=1e-15)
        _check_plan_consistency(r, M, 256, 8)


def test_route_m1_and_union(orc):
    rng = np.random.default_rng(13)
    r = orc.route(rng.normal(0, 1, (1, 256)).astype(np.float32), 8)
    assert r.n_uniq == 9 and r.n_pairs == 9
    assert np.all(np.diff(r.offs) == 1)
    r = orc.route(rng.normal(0, 1, (16, 256)).astype(np.float32), 8)
    assert r.n_uniq - 1 == len(set(r.topk_id.ravel().tolist()))


def test_route_permutation_equivariance(orc):
    rng = np.random.default_rng(14)
    logits = rng.normal(0, 1, (4, 64)).astype(np.float32)
    perm = rng.permutation(64)
    r0 = orc.route(logits, 4)
    r1 = orc.route(logits[:, perm], 4)          # expert i of r1 is expert perm[i] of r0
    assert np.array_equal(perm[r1.topk_id], r0.topk_id)
    assert np.allclose(r1.topk_w, r0.topk_w, rtol=0, atol=0)


def test_swiglu_closed_forms(orc):
    from scipy.special import expit
    assert orc.swiglu(0.0, 5.0) == 0.0
    assert orc.swiglu(3.0, 0.0) == 0.0
    for g, u in [(1.0, 2.0), (-2.5, 0.3), (10.0, -1.0), (-40.0, 2.0)]:
        ref = np.float32(g * expit(g) * u)
        assert orc.swiglu(g, u) == ref
