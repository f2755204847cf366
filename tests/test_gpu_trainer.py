"""The training loop on the GPU: micro-batch accumulation, a two-layer stack and the
reselection cadence, against the oracle composed the same way."""
import numpy as np
import pytest
import torch

import oracle
from sparse_moe_fine_gb300 import synth
from sparse_moe_fine_gb300.layer import MoELayer
from sparse_moe_fine_gb300.trainer import StackTrainer, cosine_lr

from _gpu import device, rel_l2

pytestmark = pytest.mark.gpu

CFG = synth.small_config("stack", T=256, H=128, E=8, k=2, I=128, bf16=True, frac=0.05)
# the upper layer of the two-layer stack routes every token to all its experts, so its routing
# has no discrete choice that the bf16 rounding of the lower layer's output could flip
CFG_TOP = synth.small_config("stack_top", T=256, H=128, E=4, k=4, I=128, bf16=True, frac=0.05)


def make_layer(dev, seed, cfg=CFG):
    inp = synth.moe_inputs(cfg, seed=seed)
    bf = lambda a: torch.from_numpy(a).to(dev).to(torch.bfloat16)
    act = synth.uniform_mask(cfg.N, cfg.K, seed=seed)
    L = MoELayer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, bf(inp["w_gate_up"]), bf(inp["w_down"]),
                 torch.from_numpy(inp["w_router"]).to(dev), torch.from_numpy(act).to(dev),
                 device=dev)
    return L, inp, act


def micro(seed):
    m = synth.moe_inputs(CFG, seed=seed)
    return m["x"], m["dy"]


def oracle_grads(inp, act, x, dy, k=CFG.k):
    logits = oracle.router_logits(x, inp["w_router"])
    idx, w = oracle.route_topk(logits, k)
    b = oracle.moe_backward(x, inp["w_router"], inp["w_gate_up"], inp["w_down"], idx, w, logits,
                            dy)
    g = oracle.masked_expert_grad(act, x, inp["w_gate_up"], inp["w_down"], idx, w, dy)
    return g, b


def test_microbatches_accumulate_and_schedule():
    dev = device()
    L, inp, act = make_layer(dev, 30)
    p0 = L.p.cpu().numpy().copy()
    tr = StackTrainer([L], total_steps=10, lr_peak=2e-4, reselect_every=0)
    mbs = [micro(31), micro(32)]
    bf = lambda a: torch.from_numpy(a).to(dev).to(torch.bfloat16)
    tr.step([bf(x) for x, _ in mbs], [bf(dy) for _, dy in mbs])
    L.wait_optimizer()
    torch.cuda.synchronize()
    g_sum = 0
    gr_sum = 0
    for x, dy in mbs:
        g, b = oracle_grads(inp, act, x, dy)
        g_sum = g_sum + g
        gr_sum = gr_sum + b["g_router"]
    assert rel_l2(L.g_act.cpu().numpy(), g_sum) <= 1e-2
    assert rel_l2(L.g_router.cpu().numpy(), gr_sum) <= 1e-2
    lr = cosine_lr(1, 10, 2e-4)
    assert L.lr == lr
    # SparseAdam step 1 of the accumulated gradient from the initial master values
    z = np.zeros(act.size, np.float32)
    p_ref, _, _ = oracle.sparse_adam(L.g_act.cpu().numpy(), p0, z, z, lr, 0.9, 0.999, 1e-8, 1)
    np.testing.assert_allclose(L.p.cpu().numpy(), p_ref, rtol=1e-5, atol=1e-9)
    assert tr.metrics()[0]["skipped"] == [False]


def test_two_layer_stack_chains_inputs_and_gradients():
    dev = device()
    L0, inp0, act0 = make_layer(dev, 40)
    L1, inp1, act1 = make_layer(dev, 41, CFG_TOP)
    x, dy = micro(42)
    # oracle chain with the stack's bf16 interfaces: y0 -> x1, dx1 -> dy0
    l0 = oracle.router_logits(x, inp0["w_router"])
    i0, w0 = oracle.route_topk(l0, CFG.k)
    y0 = oracle.bf16_round(oracle.moe_forward(x, inp0["w_gate_up"], inp0["w_down"], i0, w0)["Y"])
    g1, b1 = oracle_grads(inp1, act1, y0, dy, k=CFG_TOP.k)
    dy0 = oracle.bf16_round(b1["dx"])
    g0, b0 = oracle_grads(inp0, act0, x, dy0)
    tr = StackTrainer([L0, L1], total_steps=10, reselect_every=0)
    bf = lambda a: torch.from_numpy(a).to(dev).to(torch.bfloat16)
    tr.step([bf(x)], [bf(dy)])
    torch.cuda.synchronize()
    assert rel_l2(L1.g_act.cpu().numpy(), g1) <= 1e-2
    assert rel_l2(L1.g_router.cpu().numpy(), b1["g_router"]) <= 1e-2
    assert rel_l2(L0.g_act.cpu().numpy(), g0) <= 1e-2
    assert rel_l2(L0.g_router.cpu().numpy(), b0["g_router"]) <= 1e-2


@pytest.mark.parametrize("mode", ["rigl", "full"])
def test_reselection_every_two_steps(mode):
    dev = device()
    L, inp, act = make_layer(dev, 50)
    tr = StackTrainer([L], total_steps=10, reselect_every=2, reselect=mode)
    bf = lambda a: torch.from_numpy(a).to(dev).to(torch.bfloat16)
    for s in range(2):
        x, dy = micro(51 + s)
        tr.step([bf(x)], [bf(dy)])
    met = tr.metrics()
    assert met[0]["turnover"] is None and met[1]["turnover"] is not None
    new = L.act.cpu().numpy()
    assert new.size == CFG.K and (np.diff(new) > 0).all()
    if mode == "rigl":
        assert met[1]["turnover"][0] == pytest.approx(int(0.3 * CFG.K) / CFG.K)
    else:
        assert 0.0 < met[1]["turnover"][0] <= 1.0
        assert np.setdiff1d(new, act).size > 0
    assert met[1]["load_balance"][0] >= 1.0


def test_checkpoint_resume_continues_bit_exactly():
    """Save after one step, rebuild the layer from the saved state (through torch.save and
    torch.load), run two more steps: every piece of training state equals, bit for bit, that of a
    layer that ran the three steps without interruption. (The state evolves without
    order-dependent sums: dw is summed from per-tile partials in a fixed order; only y and dx,
    which are outputs, are summed by atomics.)"""
    import io
    dev = device()
    xs, dys = zip(*[micro(40 + i) for i in range(3)])
    bf = lambda a: torch.from_numpy(a).to(dev).to(torch.bfloat16)
    a, _, _ = make_layer(dev, 41)
    b, _, _ = make_layer(dev, 41)
    for i in range(3):
        ya, _ = a.train_step(bf(xs[i]), bf(dys[i]))
    b.train_step(bf(xs[0]), bf(dys[0]))
    buf = io.BytesIO()
    torch.save(b.checkpoint(), buf)
    del b
    buf.seek(0)
    c = MoELayer.from_checkpoint(torch.load(buf), device=dev)
    assert c.step_count == 1
    for i in (1, 2):
        yc, _ = c.train_step(bf(xs[i]), bf(dys[i]))
    ka, kc = a.checkpoint(), c.checkpoint()
    for key in ("w_gate_up", "w_down", "w_router", "act", "p", "m", "v", "r_p", "r_m", "r_v"):
        assert torch.equal(ka[key], kc[key]), key
    assert ka["step_count"] == kc["step_count"] == 3
    assert rel_l2(yc.float().cpu().numpy(), ya.float().cpu().numpy()) <= 1e-3
