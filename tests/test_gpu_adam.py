"""GPU SparseAdam against the oracle (same g fed to both sides): fp32 state max-rel <= 1e-5 (for
m, whose update b1*m + (1-b1)*g can cancel, relative to the magnitude of the terms), the
dense weight at each index equals the nearest bf16 of the oracle's p (or is 1 bf16 ulp away where
p sits on a rounding boundary), entries outside the index set bit-unchanged, NaN steps skipped."""
import numpy as np
import pytest
import torch

import oracle
from sparse_moe_fine_gb300 import binding as B
from sparse_moe_fine_gb300 import synth

from _gpu import device, max_rel, to_dev

pytestmark = pytest.mark.gpu


def _bf16_ulp_diff(a, b):
    ua = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    ub = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    return np.abs(ua - ub) >> 16


@pytest.mark.parametrize("n_gu,n_d,K", [(4000, 2000, 300), (402653184 // 64, 201326592 // 64, 47186)])
def test_sparse_adam_multi_step_two_segments(n_gu, n_d, K):
    dev = device()
    N = n_gu + n_d
    idx = synth.uniform_mask(N, K, seed=2)
    w_gu = synth.normal((n_gu,), 0.02, 2, "w_gate_up", True)
    w_d = synth.normal((n_d,), 0.02, 2, "w_down", True)
    W = np.concatenate([w_gu, w_d])
    p = W[idx].copy()
    m, v = synth.adam_state(K, seed=2)
    gwgu, gwd = to_dev(w_gu, dev, True), to_dev(w_d, dev, True)
    gi = to_dev(idx, dev)
    gp, gm, gv = to_dev(p, dev), to_dev(m, dev), to_dev(v, dev)
    rng = np.random.default_rng(9)
    m_scale = np.zeros(K)
    for step in range(1, 4):
        g = (rng.standard_normal(K) * 1e-3).astype(np.float32)
        g[::5] = 0.0
        B.sparse_adam_step(gi, to_dev(g, dev), gp, gm, gv, gwgu, n_gu, gwd, 1e-4, 0.9, 0.999,
                           1e-8, step)
        m_scale = np.maximum(m_scale, 0.9 * np.abs(m) + 0.1 * np.abs(g))
        p, m, v = oracle.sparse_adam(g, p, m, v, 1e-4, 0.9, 0.999, 1e-8, step)
    torch.cuda.synchronize()
    assert max_rel(gp.cpu().numpy(), p) <= 1e-5
    gm_ = gm.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(gm_ - m) / np.maximum(np.abs(m), m_scale)) <= 1e-5
    assert max_rel(gv.cpu().numpy(), v) <= 1e-5
    Wg = np.concatenate([gwgu.float().cpu().numpy(), gwd.float().cpu().numpy()])
    assert (_bf16_ulp_diff(Wg[idx], oracle.bf16_round(p)) <= 1).all()
    assert (Wg[idx] == oracle.bf16_round(p)).mean() > 0.999
    out = np.ones(N, bool)
    out[idx] = False
    assert (Wg[out] == W[out]).all()


def test_dense_router_update_fp32():
    dev = device()
    E, H = 128, 2048
    w = synth.normal((E * H,), 0.02, 3, "w_router", False)
    g = (np.random.default_rng(1).standard_normal(E * H) * 1e-2).astype(np.float32)
    gw = to_dev(w, dev)
    gp = gw.clone()
    gm = torch.zeros_like(gw)
    gv = torch.zeros_like(gw)
    B.sparse_adam_step(None, to_dev(g, dev), gp, gm, gv, gw, E * H, None, 1e-4, 0.9, 0.999, 1e-8, 1)
    torch.cuda.synchronize()
    p, m, v = oracle.sparse_adam(g, w, np.zeros_like(w), np.zeros_like(w), 1e-4, 0.9, 0.999, 1e-8, 1)
    assert max_rel(gp.cpu().numpy(), p) <= 1e-5
    assert max_rel(gw.cpu().numpy(), p) <= 1e-5
    assert max_rel(gm.cpu().numpy(), m) <= 1e-5 and max_rel(gv.cpu().numpy(), v) <= 1e-5


def test_nonfinite_step_is_skipped():
    dev = device()
    K, N = 1000, 10000
    idx = to_dev(synth.uniform_mask(N, K, seed=4), dev)
    w = to_dev(synth.normal((N,), 0.02, 4, "w_gate_up", True), dev, True)
    w0 = w.clone()
    g = torch.randn(K, device=dev)
    g[17] = float("nan")
    p = torch.ones(K, device=dev)
    m = torch.zeros(K, device=dev)
    v = torch.zeros(K, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    B.sparse_adam_step(idx, g, p, m, v, w, N, None, 1e-3, 0.9, 0.999, 1e-8, 1,
                       skip_if_nonfinite=1, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & B.DEV_NONFINITE
    assert torch.equal(w, w0) and (p == 1).all() and (m == 0).all() and (v == 0).all()
    # a flag already raised by the backward also skips a finite step
    g[17] = 0.0
    B.sparse_adam_step(idx, g, p, m, v, w, N, None, 1e-3, 0.9, 0.999, 1e-8, 1,
                       skip_if_nonfinite=1, dev_status=st)
    torch.cuda.synchronize()
    assert torch.equal(w, w0)
    st.zero_()
    B.sparse_adam_step(idx, g, p, m, v, w, N, None, 1e-3, 0.9, 0.999, 1e-8, 1,
                       skip_if_nonfinite=1, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and not torch.equal(w, w0)
