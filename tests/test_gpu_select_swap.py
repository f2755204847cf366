"""The importance selection and the RigL swap from one pass over g (usaf_select_and_swap) against
the oracle: the selected set, the new active set and every carried or reset state entry are
bit-exact, on the shared-candidate path (random and top-K active sets, K_sel unlike K, threshold
ties), on the exact path it falls back to for adversarial gradients, and on the inputs that run the
two selections one after the other (small N, D = 0)."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_moe_fine_gb300 import binding as B
from sparse_moe_fine_gb300 import synth

from _gpu import device, to_dev

pytestmark = pytest.mark.gpu


def gpu_select_and_swap(g_np, K_sel, act, p, m, v, w_np, n0, D, dev):
    g = to_dev(g_np, dev)
    w = to_dev(w_np, dev, True)
    K = act.size
    sel = torch.full((K_sel,), -1, dtype=torch.int64, device=dev)
    outs = [torch.empty(K, dtype=torch.int64, device=dev)] + [torch.empty(K, device=dev)
                                                              for _ in range(3)]
    ns = torch.zeros(1, dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    B.select_and_swap(g, sel, to_dev(act, dev), D, to_dev(p, dev), to_dev(m, dev),
                      to_dev(v, dev), w[:n0], n0, w[n0:], *outs, ns, dev_status=st)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), [o.cpu().numpy() for o in outs] + [int(ns.item())], int(st.item())


def _state(N, K, seed):
    rng = np.random.default_rng(seed)
    p = synth.to_bf16_values(rng.standard_normal(K).astype(np.float32) * 0.02)
    m = rng.standard_normal(K).astype(np.float32)
    v = np.abs(rng.standard_normal(K)).astype(np.float32)
    w = synth.to_bf16_values(rng.standard_normal(N).astype(np.float32))
    return p, m, v, w


def _check(g, K_sel, act, p, m, v, w, n0, D, dev):
    sel, swap, st = gpu_select_and_swap(g, K_sel, act, p, m, v, w, n0, D, dev)
    assert np.array_equal(sel, oracle.importance_select_threshold(g, K_sel))
    ref = oracle.rigl_swap(act, p, m, v, g, D, lambda i: w[i], grow_by="threshold")
    for a, b in zip(swap[:4], ref[:4]):
        assert np.array_equal(a, b)
    assert swap[4] == ref[4] == D
    return st


@pytest.mark.parametrize("N,K_sel,K,D,act_kind", [
    (1 << 23, 41944, 41944, 12583, "uniform"),
    # the active set is this gradient's own top-K: every excluded key lies above the grow set
    (1 << 23, 41944, 41944, 12583, "top"),
    # a ragged N (the last region short), K_sel unlike K
    ((1 << 22) + 12345, 30000, 20000, 6000, "uniform"),
    # N too small for the sampled path, and D = 0: the two selections run one after the other
    (5000, 700, 700, 200, "uniform"),
    (1 << 23, 41944, 41944, 0, "uniform"),
])
def test_select_and_swap_against_oracle(N, K_sel, K, D, act_kind):
    dev = device()
    g = synth.student_t3(N, seed=5)
    if act_kind == "top":
        act = oracle.importance_select_threshold(g, K)
    else:
        act = synth.uniform_mask(N, K, seed=N % 89)
    p, m, v, w = _state(N, K, N % 101)
    st = _check(g, K_sel, act, p, m, v, w, N // 3 * 2, D, dev)
    assert st & B.DEV_SELECT_EXACT_PATH == 0


def test_select_and_swap_threshold_ties():
    """Thousands of exact ties at both thresholds, of which each selection takes a few dozen: the
    lowest indices win in each."""
    dev = device()
    N = 1 << 23
    g = synth.student_t3(N, seed=6)
    K = math.ceil(0.005 * N)
    D = int(0.3 * K)
    act = synth.uniform_mask(N, K, seed=3)
    one, zero = np.ones(K, np.float32), np.zeros(K, np.float32)

    def grown(g):
        new = oracle.rigl_swap(act, one, zero, zero, g, D, lambda i: np.zeros(i.size, np.float32),
                               grow_by="threshold")[0]
        return np.setdiff1d(new, act)

    # ties at the grow threshold, then (on active entries only, which the grow set never sees)
    # ties at the selection's
    g[np.arange(1, N, 1009)] = np.abs(g[grown(g)]).min()
    g[act[::5]] = np.abs(g[oracle.importance_select_threshold(g, K)]).min()
    a = np.abs(g)
    t_sel = a[oracle.importance_select_threshold(g, K)].min()
    t_grow = a[grown(g)].min()
    outside = np.ones(N, bool)
    outside[act] = False
    assert (a == t_sel).sum() > 1000 and ((a == t_grow) & outside).sum() > 1000
    p, m, v, w = _state(N, K, 7)
    st = _check(g, K, act, p, m, v, w, N // 2, D, dev)
    assert st & B.DEV_SELECT_EXACT_PATH == 0


@pytest.mark.parametrize("kind", ["sorted", "constant"])
def test_select_and_swap_adversarial_inputs_take_exact_path(kind):
    dev = device()
    N = 1 << 23
    g = np.linspace(0, 1, N, dtype=np.float32) if kind == "sorted" else np.full(N, 0.5, np.float32)
    K = math.ceil(0.005 * N)
    D = int(0.3 * K)
    act = synth.uniform_mask(N, K, seed=11)
    p, m, v, w = _state(N, K, 13)
    st = _check(g, K, act, p, m, v, w, N // 2, D, dev)
    assert st & B.DEV_SELECT_EXACT_PATH


def test_select_and_swap_full_qwen3_layer():
    """N = 603,979,776, K_sel = K = 3,019,899, D = 905,969 (the layer's importance pass): the
    active set is the top-K of another seed's gradient, as after an earlier selection."""
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
    st = _check(g, K, act, p, m, v, w, cfg.N_gu, D, dev)
    assert st & B.DEV_SELECT_EXACT_PATH == 0
