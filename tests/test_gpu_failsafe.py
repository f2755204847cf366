"""Failure paths on the GPU, each made to happen without any fault: a bounded wait that runs out,
active sets that break their contract, and the status word of a step run on a stream that is not
the current one. Every case here is reported through the device status word and leaves the
context usable for the next call."""
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_moe_fine_gb300 import binding as B
from sparse_moe_fine_gb300 import synth

from _gpu import device, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def _status(dev):
    return torch.zeros(1, dtype=torch.int32, device=dev)


def test_bounded_wait_times_out_and_context_survives():
    """usaf_diag_bounded_wait: one CTA waits on an mbarrier nothing arrives on, with a limit of
    about five milliseconds. The timeout bit is set, and the next ordinary calls run and agree
    with the oracle."""
    dev = device()
    st = _status(dev)
    B.diag_bounded_wait(10_000_000, st)
    torch.cuda.synchronize()
    assert int(st.item()) == B.DEV_TIMEOUT
    # a second run after the first: the barrier, tensor memory and status path are per launch
    st2 = _status(dev)
    B.diag_bounded_wait(1_000_000, st2)
    cfg = synth.small_config("after_timeout", T=128, H=128, E=8, k=2, I=64, bf16=True)
    inp = synth.moe_inputs(cfg, seed=21)
    s = B.shape(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I)
    rt = B.Routing.empty(s, dev)
    logits = torch.empty(cfg.T, cfg.E, device=dev)
    st3 = _status(dev)
    B.route_topk(s, to_dev(inp["x"], dev, True), to_dev(inp["w_router"], dev), rt,
                 logits_out=logits, dev_status=st3)
    torch.cuda.synchronize()
    assert int(st2.item()) == B.DEV_TIMEOUT and int(st3.item()) == 0
    idx, _ = oracle.route_topk(logits.cpu().numpy(), cfg.k)
    assert (rt.topk_idx.cpu().numpy().reshape(cfg.T, cfg.k) == idx).all()


@pytest.mark.parametrize("case", ["good", "unsorted", "repeat", "too_large", "negative",
                                  "empty"])
def test_validate_active(case):
    dev = device()
    N = 10_000
    a = synth.uniform_mask(N, 500, seed=3)
    want_bad = True
    if case == "good":
        want_bad = False
    elif case == "unsorted":
        a[[100, 101]] = a[[101, 100]]
    elif case == "repeat":
        a[300] = a[299]
    elif case == "too_large":
        a[-1] = N
    elif case == "negative":
        a[0] = -1
    else:
        a = a[:0]
        want_bad = False
    st = _status(dev)
    B.validate_active(to_dev(a, dev) if a.size else None, N, st)
    torch.cuda.synchronize()
    assert bool(int(st.item()) & B.DEV_BAD_INDEX) == want_bad
    assert int(st.item()) & ~B.DEV_BAD_INDEX == 0


def test_adam_updates_nothing_after_a_bad_index():
    """With USAF_DEV_BAD_INDEX already in the status word, SparseAdam returns before touching
    anything, with or without skip_if_nonfinite; with the word clear the same call updates."""
    dev = device()
    K, N = 1000, 10000
    idx = to_dev(synth.uniform_mask(N, K, seed=5), dev)
    w = to_dev(synth.normal((N,), 0.02, 5, "w_gate_up", True), dev, True)
    w0 = w.clone()
    g = torch.randn(K, device=dev)
    p, m, v = torch.ones(K, device=dev), torch.zeros(K, device=dev), torch.zeros(K, device=dev)
    st = _status(dev)
    for skip in (0, 1):
        st.fill_(B.DEV_BAD_INDEX)
        B.sparse_adam_step(idx, g, p, m, v, w, N, None, 1e-3, 0.9, 0.999, 1e-8, 1,
                           skip_if_nonfinite=skip, dev_status=st)
        torch.cuda.synchronize()
        assert torch.equal(w, w0) and (p == 1).all() and (m == 0).all() and (v == 0).all()
    st.zero_()
    B.sparse_adam_step(idx, g, p, m, v, w, N, None, 1e-3, 0.9, 0.999, 1e-8, 1,
                       skip_if_nonfinite=1, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and not torch.equal(w, w0) and (m != 0).any()


def _masked_grad(cfg, inp, act_np, dev, debug=False):
    """Route (from the oracle's logits), forward, sparse backward; returns g_act and status."""
    s = B.shape(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I)
    x, wr = to_dev(inp["x"], dev, True), to_dev(inp["w_router"], dev)
    wgu, wd = to_dev(inp["w_gate_up"], dev, True), to_dev(inp["w_down"], dev, True)
    dy = to_dev(inp["dy"], dev, True)
    li = to_dev(oracle.router_logits(inp["x"], inp["w_router"]), dev)
    rt = B.Routing.empty(s, dev)
    B.route_topk(s, x, wr, rt, logits_in=li)
    cap = B.routed_rows_capacity(s)
    bf = torch.bfloat16
    xp = torch.empty(cfg.H, cap, dtype=bf, device=dev)
    h = torch.empty(2 * cfg.I, cap, dtype=bf, device=dev)
    wa = torch.empty(cfg.I, cap, dtype=bf, device=dev)
    y = torch.empty(cfg.T, cfg.H, dtype=bf, device=dev)
    B.moe_fwd(s, x, wgu, wd, rt, xp, h, wa, y)
    act = to_dev(act_np, dev)
    g_act = torch.full((act.numel(),), float("nan"), device=dev)
    g_r = torch.empty(cfg.E, cfg.H, device=dev)
    st = _status(dev)
    old = os.environ.get("USAF_DEBUG")
    if debug:
        os.environ["USAF_DEBUG"] = "1"
    try:
        B.moe_bwd_sparse(s, x, wr, wgu, wd, rt, xp, h, wa, dy, act, g_act, g_r, dev_status=st)
    finally:
        if debug:
            if old is None:
                del os.environ["USAF_DEBUG"]
            else:
                os.environ["USAF_DEBUG"] = old
    torch.cuda.synchronize()
    return g_act.cpu().numpy(), int(st.item())


def test_masked_gradient_skips_an_out_of_range_entry():
    """An active index past the last expert weight is range-checked in the masked-gradient kernel
    before it is decoded into addresses: the entry gets 0, USAF_DEV_BAD_INDEX is set, and every
    other entry is still the expert gradient."""
    dev = device()
    cfg = synth.small_config("bad_entry", T=256, H=128, E=8, k=2, I=64, bf16=True, frac=0.05)
    inp = synth.moe_inputs(cfg, seed=22)
    act = synth.uniform_mask(cfg.N, cfg.K, seed=22)
    ref, st_ref = _masked_grad(cfg, inp, act, dev)
    bad = np.concatenate([act, [cfg.N + 100]]).astype(np.int64)
    got, st = _masked_grad(cfg, inp, bad, dev)
    assert st_ref == 0 and st == B.DEV_BAD_INDEX
    assert got[-1] == 0.0
    assert rel_l2(got[:-1], ref) <= 1e-5


def test_debug_mode_validates_the_active_set():
    """USAF_DEBUG=1: the backward validates its active set first. A repeated (in-range) entry is
    harmless to the kernels but breaks the contract, so only the debug run reports it."""
    dev = device()
    cfg = synth.small_config("debug_set", T=128, H=128, E=4, k=2, I=64, bf16=True, frac=0.05)
    inp = synth.moe_inputs(cfg, seed=23)
    act = synth.uniform_mask(cfg.N, cfg.K, seed=23)
    act[10] = act[9]
    _, st_plain = _masked_grad(cfg, inp, act, dev)
    _, st_debug = _masked_grad(cfg, inp, act, dev, debug=True)
    assert st_plain == 0 and st_debug == B.DEV_BAD_INDEX


def test_layer_refuses_a_bad_active_set():
    from sparse_moe_fine_gb300.layer import MoELayer
    dev = device()
    cfg = synth.small_config("bad_set", T=64, H=128, E=4, k=2, I=64, bf16=True, frac=0.05)
    inp = synth.moe_inputs(cfg, seed=24)
    act = synth.uniform_mask(cfg.N, cfg.K, seed=24)
    bf = lambda a: torch.from_numpy(a).to(dev).to(torch.bfloat16)
    L = MoELayer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, bf(inp["w_gate_up"]), bf(inp["w_down"]),
                 torch.from_numpy(inp["w_router"]).to(dev), torch.from_numpy(act).to(dev),
                 lr=1e-3, device=dev)
    bad = act[::-1].copy()
    with pytest.raises(ValueError):
        L.set_active(torch.from_numpy(bad).to(dev))
    assert torch.equal(L.act.cpu(), torch.from_numpy(act))


def test_train_step_on_a_stream_that_is_not_current():
    """A train step given a stream other than the current one clears its status word on that
    stream: a non-finite upstream gradient there skips the step, and the next finite step on the
    same stream is applied and matches a step on the current stream."""
    from sparse_moe_fine_gb300.layer import MoELayer
    dev = device()
    cfg = synth.small_config("stream", T=256, H=128, E=8, k=2, I=64, bf16=True, frac=0.05)
    inp = synth.moe_inputs(cfg, seed=25)
    act = torch.from_numpy(synth.uniform_mask(cfg.N, cfg.K, seed=25)).to(dev)
    bf = lambda a: torch.from_numpy(a).to(dev).to(torch.bfloat16)

    def make():
        return MoELayer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, bf(inp["w_gate_up"]),
                        bf(inp["w_down"]), torch.from_numpy(inp["w_router"]).to(dev), act,
                        lr=1e-3, device=dev)
    x, dy = bf(inp["x"]), bf(inp["dy"])
    dy_nan = dy.clone()
    dy_nan[3, 5] = float("nan")
    a, b = make(), make()
    other = torch.cuda.Stream(device=dev)
    other.wait_stream(torch.cuda.current_stream(dev))
    w0 = b.w_gate_up.clone()
    b.train_step(x, dy_nan, stream=other)
    b.wait_optimizer(other)
    other.synchronize()
    assert int(b.status.item()) & B.DEV_NONFINITE
    assert torch.equal(b.w_gate_up, w0)
    b.train_step(x, dy, stream=other)
    b.wait_optimizer(other)
    other.synchronize()
    assert int(b.status.item()) == 0 and not torch.equal(b.w_gate_up, w0)
    a.train_step(x, dy_nan)  # the same two steps on the current stream
    ya, _ = a.train_step(x, dy)
    a.wait_optimizer()
    torch.cuda.synchronize()
    assert rel_l2(b.y.float().cpu().numpy(), ya.float().cpu().numpy()) <= 1e-3
    assert rel_l2(b.p.cpu().numpy(), a.p.cpu().numpy()) <= 1e-5
