"""Pins of the oracle's SparseAdam (closed form at step 1, torch.optim.SparseAdam as a library
routine over several steps, masking invariants) and of its bf16 rounding (torch's cast)."""
import numpy as np
import torch

import oracle
from sparse_moe_fine_gb300 import synth


def test_step_one_closed_form():
    rng = np.random.default_rng(0)
    g = (rng.standard_normal(1000) * 10.0 ** rng.integers(-9, 1, 1000)).astype(np.float32)
    p = rng.standard_normal(1000).astype(np.float32)
    lr, b1, b2, eps = 1e-3, 0.9, 0.999, 1e-8
    p1, m1, v1 = oracle.sparse_adam(g, p, np.zeros(1000), np.zeros(1000), lr, b1, b2, eps, 1)
    g64 = g.astype(np.float64)
    # with zero state: p1 = p0 - lr * g / (|g| + eps / sqrt(1 - b2))
    ref = p.astype(np.float64) - lr * g64 / (np.abs(g64) + eps / np.sqrt(1 - b2))
    np.testing.assert_allclose(p1, ref.astype(np.float32), rtol=1e-7, atol=0)
    np.testing.assert_allclose(m1, (0.1 * g64).astype(np.float32), rtol=1e-7)
    np.testing.assert_allclose(v1, (0.001 * g64 * g64).astype(np.float32), rtol=1e-7)


def test_matches_torch_sparse_adam_multi_step():
    N, K = 500, 60
    idx = synth.uniform_mask(N, K, seed=1)
    rng = np.random.default_rng(2)
    w0 = rng.standard_normal(N).astype(np.float32)
    param = torch.nn.Parameter(torch.tensor(w0))
    opt = torch.optim.SparseAdam([param], lr=1e-2, betas=(0.8, 0.99), eps=1e-6)
    p = w0[idx].copy()
    m = np.zeros(K, np.float32)
    v = np.zeros(K, np.float32)
    for step in range(1, 5):
        g = rng.standard_normal(K).astype(np.float32)
        g[::7] = 0.0  # present but zero: m, v still decay and p still moves
        param.grad = torch.sparse_coo_tensor(torch.tensor(idx)[None, :], torch.tensor(g), (N,))
        opt.step()
        p, m, v = oracle.sparse_adam(g, p, m, v, 1e-2, 0.8, 0.99, 1e-6, step)
        st = opt.state[param]
        np.testing.assert_allclose(p, param.detach().numpy()[idx], rtol=2e-6, atol=1e-7)
        np.testing.assert_allclose(m, st["exp_avg"].numpy()[idx], rtol=2e-6, atol=1e-9)
        np.testing.assert_allclose(v, st["exp_avg_sq"].numpy()[idx], rtol=2e-6, atol=1e-12)
        out = np.setdiff1d(np.arange(N), idx)
        assert (param.detach().numpy()[out] == w0[out]).all()


def test_sparse_equals_dense_restricted():
    rng = np.random.default_rng(3)
    N = 300
    g = rng.standard_normal(N).astype(np.float32)
    p = rng.standard_normal(N).astype(np.float32)
    m, v = synth.adam_state(N, seed=3)
    idx = synth.uniform_mask(N, 40, seed=5)
    dense = oracle.sparse_adam(g, p, m, v, 1e-3, 0.9, 0.999, 1e-8, 7)
    sub = oracle.sparse_adam(g[idx], p[idx], m[idx], v[idx], 1e-3, 0.9, 0.999, 1e-8, 7)
    for a, b in zip(dense, sub):
        np.testing.assert_array_equal(a[idx], b)


def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(4)
    a = (rng.standard_normal(100000) * 10.0 ** rng.integers(-30, 30, 100000)).astype(np.float32)
    # exact ties: bf16 value plus half an ulp, both parities
    base = synth.to_bf16_values(rng.standard_normal(1000).astype(np.float32))
    ties = (base.view(np.uint32) | np.uint32(0x8000)).view(np.float32)
    for arr in (a, ties):
        ref = torch.tensor(arr).to(torch.bfloat16).to(torch.float32).numpy()
        np.testing.assert_array_equal(oracle.bf16_round(arr), ref)
