"""The seeded input recipe: determinism, the drawn distributions, bf16 rounding, the uniform
active-set mask and the skewed-routing bias, checked on the host."""
import numpy as np
import pytest
import torch
from scipy import stats

from sparse_moe_fine_gb300 import synth


def test_draws_depend_only_on_seed_stream_and_shape(monkeypatch):
    n = synth.CHUNK + 12_345  # two chunks
    monkeypatch.setattr(synth, "_threads", lambda: 1)
    a = synth.normal((n,), 1.0, 3, "x", False)
    monkeypatch.setattr(synth, "_threads", lambda: 4)
    b = synth.normal((n,), 1.0, 3, "x", False)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, synth.normal((n,), 1.0, 3, "dy", False))  # streams differ
    assert not np.array_equal(a, synth.normal((n,), 1.0, 4, "x", False))   # seeds differ


def test_normal_scale_and_bf16_values():
    a = synth.normal((1 << 20,), 0.02, 0, "w_gate_up", False)
    assert a.dtype == np.float32
    assert abs(a.mean()) < 1e-4 and a.std() == pytest.approx(0.02, rel=5e-3)
    b = synth.normal((1 << 20,), 0.02, 0, "w_gate_up", True)
    ref = torch.from_numpy(a).to(torch.bfloat16).float().numpy()
    assert np.array_equal(b, ref)  # nearest bf16, ties to even, as torch's cast


def test_bf16_rounding_ties_go_to_even():
    # 1 + 2^-8 lies halfway between bf16 neighbours 1 and 1 + 2^-7: ties to the even mantissa (1)
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: ties to 1 + 2^-6
    v = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8)], np.float32)
    assert synth.to_bf16_values(v).tolist() == [1.0, 1 + 2.0 ** -6, -1.0]


def test_student_t3_distribution():
    g = synth.student_t3(1 << 20, seed=0)
    assert g.dtype == np.float32 and np.isfinite(g).all()
    ks = stats.kstest(g.astype(np.float64), stats.t(df=3).cdf)
    assert ks.statistic < 2e-3
    # heavy tail: the fraction beyond 5 matches t(3)'s two-sided tail
    assert np.mean(np.abs(g) > 5) == pytest.approx(2 * stats.t(df=3).sf(5), rel=0.05)


@pytest.mark.parametrize("N,K", [(1000, 400), (1 << 20, 5243)])  # dense and sparse branches
def test_uniform_mask(N, K):
    m = synth.uniform_mask(N, K, seed=2)
    assert m.dtype == np.int64 and m.size == K
    assert np.all(np.diff(m) > 0) and m[0] >= 0 and m[-1] < N
    assert np.array_equal(m, synth.uniform_mask(N, K, seed=2))
    counts = np.bincount(m * 16 // N, minlength=16)  # 16 equal buckets
    assert stats.chisquare(counts).pvalue > 1e-3


def test_skew_bias_and_its_realisation():
    E, dead, s = 32, 4, 1.2
    b = synth.skew_bias(E, s, dead, seed=0)
    assert np.sum(b == -1e3) == dead
    live = np.sort(b[b > -1e3])[::-1]
    np.testing.assert_allclose(live, -s * np.log(np.arange(1, E - dead + 1)), rtol=1e-6)
    cfg = synth.small_config("skew", T=16, H=64, E=E, k=2, I=64)
    inp = synth.moe_inputs(cfg, seed=0)
    synth.apply_skew(inp, b)
    assert np.all(inp["x"][:, 0] == 1.0) and np.array_equal(inp["w_router"][:, 0], b)


def test_workload_sizes_follow_the_recipe():
    tiny = synth.CONFIGS["tiny_fp32"]
    assert (tiny.N, tiny.K) == (49_152, 2_458)
    q = synth.CONFIGS["qwen3_30b_a3b"]
    assert (q.N_gu, q.N, q.K) == (402_653_184, 603_979_776, 3_019_899)
    mx = synth.CONFIGS["mixtral_8x7b"]
    assert (mx.N_gu, mx.N, mx.K) == (939_524_096, 1_409_286_144, 7_046_431)


def test_concentrated_mask():
    """hot_frac of K on the given experts' weights (both tensors), the rest on the others; sorted,
    distinct, inside [0, N), and the same draw for the same seed."""
    cfg = synth.small_config("conc", T=64, H=64, E=16, k=2, I=32, frac=0.05)
    hot = [3, 7, 11]
    a = synth.concentrated_mask(cfg, hot, 0.8, seed=4)
    assert a.size == cfg.K and (np.diff(a) > 0).all() and a[0] >= 0 and a[-1] < cfg.N
    gu = a < cfg.N_gu
    e = np.where(gu, a // (2 * cfg.I * cfg.H), (a - cfg.N_gu) // (cfg.H * cfg.I))
    assert np.isin(e, hot).sum() == int(0.8 * cfg.K)
    assert gu[np.isin(e, hot)].any() and (~gu[np.isin(e, hot)]).any()
    assert np.array_equal(a, synth.concentrated_mask(cfg, hot, 0.8, seed=4))
