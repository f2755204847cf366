"""GPU importance selection and RigL swap against the oracle: selected sets, dropped/grown sets
and the merged active set are bit-exact; state carried or reset exactly."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_moe_fine_gb300 import binding as B
from sparse_moe_fine_gb300 import synth

from _gpu import device, to_dev

pytestmark = pytest.mark.gpu

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))


def gpu_select(g_np, K, dev):
    g = to_dev(g_np, dev)
    out = torch.full((K,), -1, dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    B.importance_select(g, K, out, dev_status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("case", GOLD["select"])
def test_select_hand_cases(case):
    dev = device()
    got, _ = gpu_select(np.array(case["g"], np.float32), case["K"], dev)
    assert got.tolist() == case["idx"]


def test_select_small_random_with_ties():
    dev = device()
    rng = np.random.default_rng(0)
    for n in (1, 7, 100, 4097, 100_000):
        for K in {1, max(1, n // 3), n}:
            g = (rng.integers(-6, 7, n) * 0.125).astype(np.float32)
            got, _ = gpu_select(g, K, dev)
            assert (got == oracle.importance_select(g, K)).all(), (n, K)


def test_select_sampled_path_with_threshold_ties():
    dev = device()
    n = 1 << 23
    g = synth.student_t3(n, seed=2)
    K = math.ceil(0.005 * n)
    ref = oracle.importance_select_threshold(g, K)
    tau = np.abs(g[ref]).min()
    g[::997] = tau  # many exact ties at the threshold
    ref = oracle.importance_select_threshold(g, K)
    got, st = gpu_select(g, K, dev)
    assert (got == ref).all()
    assert st & B.DEV_SELECT_EXACT_PATH == 0


def test_select_with_nonfinite_gradients():
    """NaN and infinite magnitudes rank above every finite one (the key is the bit pattern with the
    sign cleared: a NaN above inf), and the call flags the non-finite gradient: a few of each on
    the sampled path, then so many NaNs that the threshold falls among them."""
    dev = device()
    n = 1 << 23
    g = synth.student_t3(n, seed=4)
    K = math.ceil(0.005 * n)
    rng = np.random.default_rng(4)
    pos = rng.choice(n, 200, replace=False)
    g[pos[:100]] = np.inf
    g[pos[100:150]] = -np.inf
    g[pos[150:]] = np.nan
    got, st = gpu_select(g, K, dev)
    assert (got == oracle.importance_select_threshold(g, K)).all()
    assert st & B.DEV_NONFINITE
    g2 = g.copy()
    g2[rng.choice(n, 2 * K, replace=False)] = np.nan
    got, st = gpu_select(g2, K, dev)
    assert (got == oracle.importance_select_threshold(g2, K)).all()
    assert st & B.DEV_NONFINITE
    # no non-finite value: no flag
    _, st = gpu_select(synth.student_t3(n, seed=5), K, dev)
    assert not st & B.DEV_NONFINITE


@pytest.mark.parametrize("kind", ["sorted", "constant"])
def test_select_adversarial_inputs_take_exact_path(kind):
    dev = device()
    n = 1 << 23
    if kind == "sorted":
        g = np.linspace(0, 1, n, dtype=np.float32)
    else:
        g = np.full(n, 0.5, np.float32)
    K = math.ceil(0.005 * n)
    got, st = gpu_select(g, K, dev)
    assert (got == oracle.importance_select_threshold(g, K)).all()
    assert st & B.DEV_SELECT_EXACT_PATH


def test_select_full_qwen3_layer():
    """N = 603,979,776 Student-t(3) gradient, K = ceil(0.005 N)."""
    dev = device()
    cfg = synth.CONFIGS["qwen3_30b_a3b"]
    g = synth.student_t3(cfg.N, seed=0)
    got, st = gpu_select(g, cfg.K, dev)
    ref = oracle.importance_select_threshold(g, cfg.K)
    assert got.size == cfg.K and (got == ref).all()
    assert st == 0


def gpu_rigl(g_np, act, p, m, v, w_np, n0, D, dev):
    g = to_dev(g_np, dev)
    a = to_dev(act, dev)
    w = to_dev(w_np, dev, True)
    K = act.size
    outs = [torch.empty(K, dtype=torch.int64, device=dev)] + [torch.empty(K, device=dev)
                                                              for _ in range(3)]
    ns = torch.zeros(1, dtype=torch.int64, device=dev)
    B.rigl_swap(g, a, D, to_dev(p, dev), to_dev(m, dev), to_dev(v, dev), w[:n0], n0, w[n0:],
                *outs, ns)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in outs] + [int(ns.item())]


def test_rigl_hand_case():
    dev = device()
    c = GOLD["rigl"][0]
    act = np.array(c["act_idx"], np.int64)
    w = synth.to_bf16_values(np.arange(c["N"], dtype=np.float32) * 0.5)
    p = np.array(c["p"], np.float32)
    m = np.arange(4, dtype=np.float32) + 1
    v = 2 * m
    new, p2, m2, v2, ns = gpu_rigl(np.array(c["g"], np.float32), act, p, m, v, w, 4, c["D"], dev)
    assert new.tolist() == c["new_idx"] and ns == c["D"]


@pytest.mark.parametrize("N,K,D", [(50, 20, 6), (5000, 700, 200), (5000, 700, 0),
                                   (1 << 23, 41944, 12583)])
def test_rigl_against_oracle(N, K, D):
    dev = device()
    rng = np.random.default_rng(N)
    act = synth.uniform_mask(N, K, seed=N % 97)
    if N < 10000:
        g = (rng.integers(-5, 6, N) * 0.25).astype(np.float32)
        p = (rng.integers(-3, 4, K) * 0.01).astype(np.float32)
    else:
        g = synth.student_t3(N, seed=3)
        p = synth.to_bf16_values(rng.standard_normal(K).astype(np.float32) * 0.02)
    m = rng.standard_normal(K).astype(np.float32)
    v = np.abs(rng.standard_normal(K)).astype(np.float32)
    w = synth.to_bf16_values(rng.standard_normal(N).astype(np.float32))
    n0 = N // 3 * 2
    got = gpu_rigl(g, act, p, m, v, w, n0, D, dev)
    ref = oracle.rigl_swap(act, p, m, v, g, D, lambda i: w[i])
    for a, b in zip(got[:4], ref[:4]):
        assert np.array_equal(a, b)
    assert got[4] == ref[4] == D


def test_rigl_full_qwen3_layer():
    """N = 603,979,776, K = 3,019,899, D = floor(0.3 K) = 905,969: the oracle's RigL swap (grow
    set by its threshold form, pinned to the sort form on the CPU) and the device's agree on the
    new set and on every carried or reset state entry."""
    dev = device()
    cfg = synth.CONFIGS["qwen3_30b_a3b"]
    N, K = cfg.N, cfg.K
    D = int(0.3 * K)
    g = synth.student_t3(N, seed=0)
    act = oracle.importance_select_threshold(synth.student_t3(N, seed=1), K)
    wgu = synth.normal((cfg.N_gu,), 0.02, 0, "w_gate_up", True)
    wd = synth.normal((N - cfg.N_gu,), 0.02, 0, "w_down", True)
    w = np.concatenate([wgu, wd])
    p = w[act].copy()
    m, v = synth.adam_state(K, seed=0)
    got = gpu_rigl(g, act, p, m, v, w, cfg.N_gu, D, dev)
    ref = oracle.rigl_swap(act, p, m, v, g, D, lambda i: w[i], grow_by="threshold")
    for a, b in zip(got[:4], ref[:4]):
        assert np.array_equal(a, b)
    assert got[4] == ref[4] == D


def gpu_reselect(g_np, K, act, p, m, v, w_np, n0, dev):
    g = to_dev(g_np, dev)
    w = to_dev(w_np, dev, True)
    outs = [torch.empty(K, dtype=torch.int64, device=dev)] + [torch.empty(K, device=dev)
                                                              for _ in range(3)]
    nk = torch.zeros(1, dtype=torch.int64, device=dev)
    B.reselect_full(g, K, to_dev(act, dev), to_dev(p, dev), to_dev(m, dev), to_dev(v, dev),
                    w[:n0], n0, w[n0:], *outs, nk)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in outs] + [int(nk.item())]


@pytest.mark.parametrize("N,K_old,K", [(40, 12, 9), (6000, 800, 900), (1 << 23, 41944, 41944)])
def test_reselect_full_against_oracle(N, K_old, K):
    """Full re-ranking reselection: new set bit-exact; state carried for kept entries, weights
    and zero moments for new ones; kept count. The large case takes the sampled path."""
    dev = device()
    rng = np.random.default_rng(N + 1)
    act = synth.uniform_mask(N, K_old, seed=N % 89)
    if N < 10000:
        g = (rng.integers(-4, 5, N) * 0.5).astype(np.float32)
    else:
        g = synth.student_t3(N, seed=5)
        # the previous set overlaps the new one: half of it from the top of this gradient
        top = oracle.importance_select_threshold(g, K_old // 2)
        act = np.union1d(top, act)[:K_old]
        act = np.sort(act)
    p = rng.standard_normal(act.size).astype(np.float32)
    m = rng.standard_normal(act.size).astype(np.float32)
    v = np.abs(rng.standard_normal(act.size)).astype(np.float32)
    w = synth.to_bf16_values(rng.standard_normal(N).astype(np.float32))
    n0 = N // 3 * 2
    got = gpu_reselect(g, K, act, p, m, v, w, n0, dev)
    ref = oracle.reselect_full(act, p, m, v, g, K, lambda i: w[i])
    for a, b in zip(got[:4], ref[:4]):
        assert np.array_equal(a, b)
    assert got[4] == ref[4]
    if N >= 10000:
        assert 0 < got[4] < K
