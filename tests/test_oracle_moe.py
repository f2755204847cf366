"""Pins of the oracle's expert forward/backward: a dense SwiGLU MLP through torch.nn.functional,
torch.autograd on an independently written per-token layer, central finite differences, and the
invariants of the sparse backward."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from sparse_moe_fine_gb300 import synth


def _layer(T=24, H=16, E=5, k=2, I=6, seed=0):
    cfg = synth.small_config("t", T=T, H=H, E=E, k=k, I=I, bf16=False, dy_std=1.0)
    inp = synth.moe_inputs(cfg, seed=seed)
    # larger weights than the workload's 0.02 so every term is well above rounding
    for key in ("w_gate_up", "w_down"):
        inp[key] = (inp[key] * 20).astype(np.float32)
    inp["w_router"] = (inp["w_router"] * 20).astype(np.float32)
    return cfg, inp


def test_single_expert_is_dense_swiglu_mlp():
    cfg, inp = _layer(E=1, k=1)
    T = cfg.T
    idx = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1))
    out = oracle.moe_forward(inp["x"], inp["w_gate_up"], inp["w_down"], idx, w)
    x = torch.tensor(inp["x"], dtype=torch.float64)
    wgu = torch.tensor(inp["w_gate_up"][0], dtype=torch.float64)
    wd = torch.tensor(inp["w_down"][0], dtype=torch.float64)
    gate = F.linear(x, wgu[: cfg.I])
    up = F.linear(x, wgu[cfg.I:])
    ref = F.linear(F.silu(gate) * up, wd)
    np.testing.assert_allclose(out["Y"], ref.numpy(), rtol=1e-12, atol=1e-12)


def _torch_layer(inp, idx, renorm):
    """Per-token loop in torch, differentiated by autograd; the selection idx is held fixed."""
    x = torch.tensor(inp["x"], dtype=torch.float64, requires_grad=True)
    wr = torch.tensor(inp["w_router"], dtype=torch.float64, requires_grad=True)
    wgu = torch.tensor(inp["w_gate_up"], dtype=torch.float64, requires_grad=True)
    wd = torch.tensor(inp["w_down"], dtype=torch.float64, requires_grad=True)
    I = wgu.shape[1] // 2
    logits = x @ wr.T
    rows = []
    for t in range(x.shape[0]):
        sel = torch.tensor(idx[t].astype(np.int64))
        if renorm:
            wt = torch.softmax(logits[t, sel], dim=0)
        else:
            wt = torch.softmax(logits[t], dim=0)[sel]
        acc = torch.zeros(x.shape[1], dtype=torch.float64)
        for j in range(sel.numel()):
            e = int(sel[j])
            hh = wgu[e] @ x[t]
            a = F.silu(hh[:I]) * hh[I:]
            acc = acc + wt[j] * (wd[e] @ a)
        rows.append(acc)
    Y = torch.stack(rows)
    dY = torch.tensor(inp["dy"], dtype=torch.float64)
    (Y * dY).sum().backward()
    return Y.detach().numpy(), x.grad.numpy(), wr.grad.numpy(), wgu.grad.numpy(), wd.grad.numpy()


@pytest.mark.parametrize("renorm", [1, 0])
def test_backward_matches_torch_autograd(renorm):
    cfg, inp = _layer()
    logits = oracle.router_logits(inp["x"], inp["w_router"])
    idx, w = oracle.route_topk(logits, cfg.k, renorm=renorm)
    Y, gx, gwr, gwgu, gwd = _torch_layer(inp, idx, renorm)
    b = oracle.moe_backward(inp["x"], inp["w_router"], inp["w_gate_up"], inp["w_down"], idx, w,
                            logits, inp["dy"], renorm=renorm, dense_wgrad=True)
    # torch recomputes logits in fp64; the oracle ranks on fp32 logits but its weights use the
    # fp32-rounded logits, so compare with a tolerance at fp32 logit resolution
    np.testing.assert_allclose(b["Y"], Y, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(b["dx"], gx, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(b["g_router"], gwr, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(b["dW_gate_up"], gwgu, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(b["dW_down"], gwd, rtol=1e-5, atol=1e-6)


def _loss(inp, idx, renorm, **over):
    d = dict(inp)
    d.update(over)
    l = np.asarray(d["x"], np.float64) @ np.asarray(d["w_router"], np.float64).T
    # weights from fp64 logits for a smooth loss (selection held fixed)
    z = l - l.max(axis=1, keepdims=True)
    if renorm:
        sel = np.take_along_axis(z, idx.astype(np.int64), axis=1)
        w = np.exp(sel) / np.exp(sel).sum(axis=1, keepdims=True)
    else:
        p = np.exp(z) / np.exp(z).sum(axis=1, keepdims=True)
        w = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    Y = oracle.moe_forward(d["x"], d["w_gate_up"], d["w_down"], idx, w)["Y"]
    return float(np.sum(np.asarray(d["dy"], np.float64) * Y))


def _fd_inputs(inp):
    return {k: np.asarray(v, np.float64) for k, v in inp.items()}


@pytest.mark.parametrize("renorm", [1, 0])
def test_backward_central_finite_differences(renorm):
    cfg, inp = _layer(T=12, H=8, E=4, k=2, I=4, seed=1)
    inp64 = _fd_inputs(inp)
    logits = (inp64["x"] @ inp64["w_router"].T)
    idx, _ = oracle.route_topk(logits.astype(np.float32), cfg.k, renorm)
    z = logits - logits.max(axis=1, keepdims=True)
    if renorm:
        sel = np.take_along_axis(z, idx.astype(np.int64), axis=1)
        w = np.exp(sel) / np.exp(sel).sum(axis=1, keepdims=True)
    else:
        p = np.exp(z) / np.exp(z).sum(axis=1, keepdims=True)
        w = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    b = oracle.moe_backward(inp64["x"], inp64["w_router"], inp64["w_gate_up"], inp64["w_down"],
                            idx, w, logits, inp64["dy"], renorm=renorm, dense_wgrad=True)
    rng = np.random.default_rng(7)
    eps = 1e-6
    checks = [("w_gate_up", b["dW_gate_up"]), ("w_down", b["dW_down"]),
              ("w_router", b["g_router"]), ("x", b["dx"])]
    for name, grad in checks:
        for _ in range(6):
            pos = tuple(int(rng.integers(0, s)) for s in inp64[name].shape)
            plus = inp64[name].copy()
            plus[pos] += eps
            minus = inp64[name].copy()
            minus[pos] -= eps
            # the selection must not flip at +-eps
            for arr in (plus, minus):
                d = dict(inp64)
                d[name] = arr
                l2 = (d["x"] @ d["w_router"].T).astype(np.float32)
                assert (oracle.route_topk(l2, cfg.k, renorm)[0] == idx).all()
            num = (_loss(inp64, idx, renorm, **{name: plus})
                   - _loss(inp64, idx, renorm, **{name: minus})) / (2 * eps)
            assert abs(num - grad[pos]) <= 1e-6 * max(1.0, abs(num)), (name, pos, num, grad[pos])


def test_masked_grad_equals_dense_gathered_and_dead_experts_zero():
    cfg, inp = _layer(T=20, H=8, E=6, k=2, I=4, seed=2)
    logits = oracle.router_logits(inp["x"], inp["w_router"])
    idx, w = oracle.route_topk(logits, cfg.k)
    # force expert 5 to receive no token
    idx = np.where(idx == 5, -1, idx)
    for t in range(cfg.T):
        for j in range(cfg.k):
            if idx[t, j] < 0:
                idx[t, j] = [e for e in range(5) if e not in idx[t]][0]
    b = oracle.moe_backward(inp["x"], inp["w_router"], inp["w_gate_up"], inp["w_down"], idx, w,
                            logits, inp["dy"], dense_wgrad=True)
    N = cfg.N
    act = synth.uniform_mask(N, N // 3, seed=4)
    g = oracle.masked_expert_grad(act, inp["x"], inp["w_gate_up"], inp["w_down"], idx, w,
                                  inp["dy"])
    dense = np.concatenate([b["dW_gate_up"].reshape(-1), b["dW_down"].reshape(-1)])
    np.testing.assert_allclose(g, dense[act], rtol=1e-12, atol=1e-14)
    t_, e_, r_, c_ = oracle.split_flat_index(act, cfg.E, cfg.I, cfg.H)
    assert (g[e_ == 5] == 0).all() and (e_ == 5).any()
    # flat index split round trip
    Ngu = cfg.N_gu
    back = np.where(t_ == 0, e_ * 2 * cfg.I * cfg.H + r_ * cfg.H + c_,
                    Ngu + e_ * cfg.H * cfg.I + r_ * cfg.I + c_)
    assert (back == act).all()


def test_router_grad_invariants():
    cfg, inp = _layer(seed=3)
    logits = oracle.router_logits(inp["x"], inp["w_router"])
    idx, w = oracle.route_topk(logits, cfg.k)
    b = oracle.moe_backward(inp["x"], inp["w_router"], inp["w_gate_up"], inp["w_down"], idx, w,
                            logits, inp["dy"])
    np.testing.assert_allclose(b["dlogit"].sum(axis=1), 0.0, atol=1e-12)
    mask = np.zeros_like(b["dlogit"], dtype=bool)
    np.put_along_axis(mask, idx.astype(np.int64), True, axis=1)
    assert (b["dlogit"][~mask] == 0).all()


def _bf16_inputs(seed=3):
    cfg = synth.small_config("bf", T=96, H=32, E=6, k=2, I=16, bf16=True, dy_std=1.0)
    inp = synth.moe_inputs(cfg, seed=seed)
    for key in ("w_gate_up", "w_down"):
        inp[key] = synth.to_bf16_values(inp[key] * 20)
    logits = oracle.router_logits(inp["x"], inp["w_router"])
    idx, w = oracle.route_topk(logits, cfg.k)
    act = synth.uniform_mask(cfg.N, cfg.K, seed=seed)
    return cfg, inp, logits, idx, w, act


def _all_outputs(cfg, inp, logits, idx, w, act, rnd):
    b = oracle.moe_backward(inp["x"], inp["w_router"], inp["w_gate_up"], inp["w_down"], idx, w,
                            logits, inp["dy"], dense_wgrad=True, rnd=rnd)
    g = oracle.masked_expert_grad(act, inp["x"], inp["w_gate_up"], inp["w_down"], idx, w,
                                  inp["dy"], rnd=rnd)
    return b, g


def test_bf16_emulating_mode_with_identity_rounding_is_the_fp64_oracle():
    """With a rounding function that changes nothing, the bf16-emulating code path gives the fp64
    oracle's results (up to the order of the routing-weight product), so the mode adds nothing but
    its rounding points."""
    cfg, inp, logits, idx, w, act = _bf16_inputs()
    ref_b, ref_g = _all_outputs(cfg, inp, logits, idx, w, act, None)
    got_b, got_g = _all_outputs(cfg, inp, logits, idx, w, act, lambda a: np.array(a, np.float64))
    for key in ("Y", "dx", "dw", "dh", "dlogit", "g_router", "dW_gate_up", "dW_down"):
        np.testing.assert_allclose(got_b[key], ref_b[key], rtol=1e-11, atol=1e-13, err_msg=key)
    np.testing.assert_allclose(got_g, ref_g, rtol=1e-11, atol=1e-13)


def test_bf16_emulating_mode_rounds_at_the_storage_points():
    """With bf16 rounding (pinned against torch's cast): the stored h is the nearest bf16 of the
    fp64 h, w*A is the nearest bf16 of the fp64 w*A, every stored dh is a bf16 value, and each
    result stays within a few bf16 half-ulps (2^-9 relative) of the fp64 oracle."""
    cfg, inp, logits, idx, w, act = _bf16_inputs()
    ref_b, ref_g = _all_outputs(cfg, inp, logits, idx, w, act, None)
    rb, rg = _all_outputs(cfg, inp, logits, idx, w, act, oracle.bf16_round)
    f64 = oracle.moe_forward(inp["x"], inp["w_gate_up"], inp["w_down"], idx, w)
    f16 = oracle.moe_forward(inp["x"], inp["w_gate_up"], inp["w_down"], idx, w,
                             rnd=oracle.bf16_round)
    assert np.array_equal(f16["h"], oracle.bf16_round(f64["h"]))
    assert np.array_equal(f16["wA"], oracle.bf16_round(f64["wA"]))
    assert np.array_equal(rb["dh"], oracle.bf16_round(rb["dh"]))
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    for key in ("Y", "dx", "dw", "g_router", "dW_gate_up", "dW_down"):
        e = rel(rb[key], ref_b[key])
        assert 1e-5 < e < 2e-2, (key, e)  # rounded somewhere, and only by bf16 steps
    assert 1e-5 < rel(rg, ref_g) < 2e-2
    # the masked gradient is the dense one gathered at the mask in this mode too
    dense = np.concatenate([rb["dW_gate_up"].reshape(-1), rb["dW_down"].reshape(-1)])
    np.testing.assert_allclose(rg, dense[act], rtol=1e-10, atol=1e-12)
