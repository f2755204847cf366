"""Pins of the oracle's routing (logits, top-k, weights, permutation) against hand cases,
brute force and library softmax."""
import itertools
import json
import os

import numpy as np
import pytest
import scipy.special

import oracle
from sparse_moe_fine_gb300 import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))


@pytest.mark.parametrize("case", GOLD["route"])
def test_route_hand_cases(case):
    l = np.array(case["logits"], np.float32)
    idx, w = oracle.route_topk(l, case["k"], renorm=1)
    assert idx.tolist() == case["idx"]
    if "w_renorm" in case:
        np.testing.assert_allclose(w, np.array(case["w_renorm"]), rtol=0, atol=1e-15)


def _brute_topk(row, k):
    # exhaustive: the k-subset whose sorted logits dominate, ties to lower indices
    E = len(row)
    best = None
    for sub in itertools.combinations(range(E), k):
        key = sorted(((-float(row[e]), e) for e in sub))
        if best is None or key < best:
            best = key
    return [e for _, e in best]


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(5)
    for _ in range(200):
        E = int(rng.integers(2, 8))
        k = int(rng.integers(1, E + 1))
        row = rng.integers(-3, 3, size=E).astype(np.float32)  # many ties
        idx, _ = oracle.route_topk(row[None, :], k)
        assert idx[0].tolist() == _brute_topk(row, k)


def test_renorm_weights_equal_library_softmax():
    cfg = synth.small_config("r", T=64, H=32, E=16, k=4, I=8, bf16=False)
    inp = synth.moe_inputs(cfg, seed=3)
    l = oracle.router_logits(inp["x"], inp["w_router"])
    idx, w = oracle.route_topk(l, 4, renorm=1)
    idx0, w0 = oracle.route_topk(l, 4, renorm=0)
    assert (idx == idx0).all()
    full = scipy.special.softmax(l.astype(np.float64), axis=1)
    sel = np.take_along_axis(full, idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-13)
    np.testing.assert_allclose(w0, sel, rtol=1e-13)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert (w > 0).all()
    # selected logits descending, distinct experts
    ls = np.take_along_axis(l, idx.astype(np.int64), axis=1)
    assert (np.diff(ls, axis=1) <= 0).all()
    assert all(len(set(r)) == 4 for r in idx.tolist())


def test_k_equals_E_is_full_softmax():
    l = np.random.default_rng(1).standard_normal((10, 6)).astype(np.float32)
    idx, w = oracle.route_topk(l, 6, renorm=1)
    full = scipy.special.softmax(l.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(full, idx.astype(np.int64), axis=1),
                               rtol=1e-13)


def test_router_logits_fp64_then_fp32():
    x = np.array([[1.0, 2.0**-30]], np.float32)
    wr = np.array([[1.0, 1.0]], np.float32)
    # fp64 accumulation keeps the tiny term until the single final rounding
    assert oracle.router_logits(x, wr)[0, 0] == np.float32(1.0 + 2.0**-30)
    x = np.random.default_rng(2).standard_normal((7, 5)).astype(np.float32)
    wr = np.random.default_rng(3).standard_normal((3, 5)).astype(np.float32)
    ref = np.einsum("th,eh->te", x.astype(np.float64), wr.astype(np.float64))
    np.testing.assert_array_equal(oracle.router_logits(x, wr), ref.astype(np.float32))


def test_permutation_invariants():
    rng = np.random.default_rng(0)
    T, E, k = 50, 7, 3
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, lists = oracle.permutation(topk, E)
    assert counts.tolist() == np.bincount(topk.reshape(-1), minlength=E).tolist()
    allslots = np.concatenate(lists)
    assert sorted(allslots.tolist()) == list(range(T * k))
    for e, sl in enumerate(lists):
        toks = sl // k
        assert (np.diff(toks) > 0).all()
        assert (topk.reshape(-1)[sl] == e).all()
