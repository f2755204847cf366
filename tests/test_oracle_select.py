"""Pins of the oracle's importance selection and RigL swap: hand cases, brute force on small N,
the threshold form on larger N with injected ties, and the set invariants; plus the parameter
counts the USAF README prints."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from sparse_moe_fine_gb300 import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))
PAGE = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_param_counts.json")))


@pytest.mark.parametrize("case", GOLD["select"])
def test_select_hand_cases(case):
    g = np.array(case["g"], np.float32)
    assert oracle.importance_select(g, case["K"]).tolist() == case["idx"]
    assert oracle.importance_select_threshold(g, case["K"]).tolist() == case["idx"]


def _brute_select(g, K):
    items = sorted(range(len(g)), key=lambda i: (-abs(float(g[i])), i))
    return sorted(items[:K])


def test_select_brute_force_small():
    rng = np.random.default_rng(0)
    for _ in range(100):
        n = int(rng.integers(1, 60))
        K = int(rng.integers(1, n + 1))
        g = (rng.integers(-4, 5, n) * 0.25).astype(np.float32)  # heavy ties, signed zeros
        assert oracle.importance_select(g, K).tolist() == _brute_select(g, K)


def test_select_threshold_form_and_invariants():
    n = 2_000_000
    g = synth.student_t3(n, seed=1)
    g[::1000] = 3.0  # a block of exact ties near the threshold
    K = math.ceil(0.005 * n)
    a = oracle.importance_select(g, K)
    b = oracle.importance_select_threshold(g, K)
    assert a.size == K and (a == b).all()
    key = np.abs(g)
    sel = np.zeros(n, bool)
    sel[a] = True
    assert key[sel].min() >= key[~sel].max()
    tau = key[sel].min()
    # at the threshold every selected index precedes every unselected tied index
    tied_sel = np.nonzero(sel & (key == tau))[0]
    tied_un = np.nonzero(~sel & (key == tau))[0]
    if tied_un.size and tied_sel.size:
        assert tied_sel.max() < tied_un.min()


def test_page_param_counts():
    L = PAGE["layer"]
    N = L["E"] * 3 * L["I"] * L["H"]
    K = math.ceil(PAGE["frac"] * N)
    router = L["E"] * L["H"]
    layers = round(PAGE["expert_params_total"] / N)
    assert layers == 8  # TRAIN_FROM=40 of a 48-layer model
    r = PAGE["rounding"]
    assert abs(layers * N - PAGE["expert_params_total"]) <= r["expert_params_total"] / 2
    assert abs(layers * (K + router) - PAGE["trained_params_total"]) <= r["trained_params_total"] / 2
    assert abs(layers * router - PAGE["router_params_total"]) <= r["router_params_total"] / 2
    assert N == synth.CONFIGS["qwen3_30b_a3b"].N and K == synth.CONFIGS["qwen3_30b_a3b"].K


@pytest.mark.parametrize("case", GOLD["rigl"])
def test_rigl_hand_case(case):
    g = np.array(case["g"], np.float32)
    w = np.arange(case["N"], dtype=np.float32) * 0.5
    act = np.array(case["act_idx"], np.int64)
    p = np.array(case["p"], np.float32)
    m = np.arange(len(act), dtype=np.float32) + 1
    v = m * 2
    new, p2, m2, v2, ns = oracle.rigl_swap(act, p, m, v, g, case["D"], lambda i: w[i])
    assert new.tolist() == case["new_idx"] and ns == case["D"]
    for i, f in enumerate(new.tolist()):
        if f in case["grown"]:
            assert p2[i] == w[f] and m2[i] == 0 and v2[i] == 0
        else:
            j = case["act_idx"].index(f)
            assert p2[i] == p[j] and m2[i] == m[j] and v2[i] == v[j]


def _brute_rigl(act, p, g, D):
    act = list(act)
    drop = sorted(range(len(act)), key=lambda i: (abs(float(p[i])), act[i]))[:D]
    dropped = {act[i] for i in drop}
    inactive = [f for f in range(len(g)) if f not in set(act)]
    grow = sorted(inactive, key=lambda f: (-abs(float(g[f])), f))[:D]
    return sorted((set(act) - dropped) | set(grow)), dropped, set(grow)


def test_rigl_brute_force_and_invariants():
    rng = np.random.default_rng(1)
    for _ in range(60):
        N = int(rng.integers(4, 80))
        K = int(rng.integers(1, N))
        D = int(rng.integers(0, min(K, N - K) + 1))
        act = np.sort(rng.choice(N, K, replace=False)).astype(np.int64)
        p = (rng.integers(-3, 4, K) * 0.5).astype(np.float32)
        m = rng.standard_normal(K).astype(np.float32)
        v = np.abs(rng.standard_normal(K)).astype(np.float32)
        g = (rng.integers(-3, 4, N) * 0.5).astype(np.float32)
        wd = rng.standard_normal(N).astype(np.float32)
        new, p2, m2, v2, ns = oracle.rigl_swap(act, p, m, v, g, D, lambda i: wd[i])
        ref, dropped, grown = _brute_rigl(act, p, g, D)
        assert new.tolist() == ref
        assert new.size == K and ns == D
        assert dropped <= set(act.tolist()) and not (grown & set(act.tolist()))
        old = {f: i for i, f in enumerate(act.tolist())}
        for i, f in enumerate(new.tolist()):
            if f in old:
                j = old[f]
                assert (p2[i], m2[i], v2[i]) == (p[j], m[j], v[j])
            else:
                assert (p2[i], m2[i], v2[i]) == (wd[f], 0, 0)


def test_rigl_threshold_form_equals_sort_form():
    """The threshold form of the grow set (used for full-size layers) gives the sort form's result,
    also when the threshold key is shared by entries inside and outside the active set and when
    many outside entries tie at it; brute force on the small cases too."""
    rng = np.random.default_rng(7)
    for N, K, D in ((60, 20, 7), (500, 120, 0), (500, 120, 120), (2_000_000, 10_000, 3_000)):
        act = np.sort(rng.choice(N, K, replace=False)).astype(np.int64)
        g = (rng.integers(-40, 41, N) * 0.25).astype(np.float32)
        if N > 1000:
            g[::13] = 20.0          # a tied group larger than D: the threshold key
            g[act[::2]] = 20.0      # the same key inside the set, never grown
        p = (rng.integers(-3, 4, K) * 0.5).astype(np.float32)
        m = rng.standard_normal(K).astype(np.float32)
        v = np.abs(rng.standard_normal(K)).astype(np.float32)
        wd = rng.standard_normal(N).astype(np.float32)
        a = oracle.rigl_swap(act, p, m, v, g, D, lambda i: wd[i])
        b = oracle.rigl_swap(act, p, m, v, g, D, lambda i: wd[i], grow_by="threshold")
        for x, y in zip(a[:4], b[:4]):
            assert np.array_equal(x, y)
        assert a[4] == b[4] == D
        if N < 1000:
            assert a[0].tolist() == _brute_rigl(act, p, g, D)[0]


def test_reselect_full_hand_case():
    # |g| ranks: idx 7 (9.0), 2 (-8.0), 5 and 9 tie at 5.0 (lower index first), then 0 (4.0)
    g = np.array([4.0, 0.5, -8.0, 1.0, 0.0, 5.0, -0.25, 9.0, 3.0, -5.0], np.float32)
    act = np.array([0, 2, 3, 8], np.int64)
    p = np.array([10.0, 20.0, 30.0, 80.0], np.float32)
    m = np.array([1.0, 2.0, 3.0, 8.0], np.float32)
    v = np.array([0.1, 0.2, 0.3, 0.8], np.float32)
    w = np.arange(10, dtype=np.float32) * 100.0
    new, p2, m2, v2, kept = oracle.reselect_full(act, p, m, v, g, 4, lambda i: w[i])
    assert new.tolist() == [2, 5, 7, 9]
    assert p2.tolist() == [20.0, 500.0, 700.0, 900.0]
    assert m2.tolist() == [2.0, 0.0, 0.0, 0.0] and v2.tolist() == [np.float32(0.2), 0.0, 0.0, 0.0]
    assert kept == 1


def test_reselect_full_brute_force():
    rng = np.random.default_rng(11)
    for trial in range(30):
        N = int(rng.integers(5, 60))
        K_old = int(rng.integers(0, N + 1))
        K_new = int(rng.integers(0, N + 1))
        g = rng.integers(-4, 5, N).astype(np.float32)  # many ties, signed zeros below
        g[rng.random(N) < 0.2] = -0.0
        act = np.sort(rng.choice(N, K_old, replace=False)).astype(np.int64)
        p = rng.standard_normal(K_old).astype(np.float32)
        m = rng.standard_normal(K_old).astype(np.float32)
        v = rng.random(K_old).astype(np.float32)
        w = rng.standard_normal(N).astype(np.float32)
        new, p2, m2, v2, kept = oracle.reselect_full(act, p, m, v, g, K_new, lambda i: w[i])
        # brute force: rank by (|g| descending, index ascending) with plain Python
        ranked = sorted(range(N), key=lambda i: (-abs(float(g[i])), i))
        want = sorted(ranked[:K_new])
        assert new.tolist() == want
        old = {int(f): t for t, f in enumerate(act)}
        n_k = 0
        for t, f in enumerate(want):
            if f in old:
                n_k += 1
                assert (p2[t], m2[t], v2[t]) == (p[old[f]], m[old[f]], v[old[f]])
            else:
                assert (p2[t], m2[t], v2[t]) == (w[f], 0.0, 0.0)
        assert kept == n_k


def test_reselect_full_keeps_a_set_that_still_ranks_first():
    rng = np.random.default_rng(12)
    N, K = 1000, 50
    act = np.sort(rng.choice(N, K, replace=False)).astype(np.int64)
    g = rng.standard_normal(N).astype(np.float32) * 0.1
    g[act] = 10.0 + rng.random(K).astype(np.float32)
    p, m, v = (rng.standard_normal(K).astype(np.float32) for _ in range(3))
    new, p2, m2, v2, kept = oracle.reselect_full(act, p, m, v, g, K, lambda i: np.zeros(len(i)))
    assert kept == K and (new == act).all()
    assert (p2 == p).all() and (m2 == m).all() and (v2 == v).all()
