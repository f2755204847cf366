"""GPU routing (router logits, top-k, weights, permutation) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from sparse_moe_fine_gb300 import binding as B
from sparse_moe_fine_gb300 import synth

from _gpu import device, max_rel, to_dev

pytestmark = pytest.mark.gpu


def _route(cfg, inp, dev, logits_in=None, renorm=1):
    s = B.shape(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I)
    rt = B.Routing.empty(s, dev)
    logits = torch.empty(cfg.T, cfg.E, device=dev)
    x = to_dev(inp["x"], dev, cfg.bf16)
    wr = to_dev(inp["w_router"], dev)
    li = None if logits_in is None else to_dev(logits_in, dev)
    B.route_topk(s, x, wr, rt, logits_in=li, logits_out=logits, renorm=renorm)
    torch.cuda.synchronize()
    return s, rt, logits.cpu().numpy()


def _check_perm(cfg, rt, idx):
    cnt, lists = oracle.permutation(idx, cfg.E)
    gc = rt.expert_count.cpu().numpy()
    off = rt.expert_offset.cpu().numpy()
    ptok = rt.perm_tok.cpu().numpy()
    pslot = rt.perm_slot.cpu().numpy()
    srow = rt.slot_row.cpu().numpy()
    assert (gc == cnt).all()
    assert off[0] == 0 and (off % B.ROW_ALIGN == 0).all()
    for e in range(cfg.E):
        seg = pslot[off[e]:off[e + 1]]
        assert (seg[:cnt[e]] == lists[e]).all()
        assert (seg[cnt[e]:] == -1).all()
        assert (ptok[off[e]:off[e] + cnt[e]] == lists[e] // cfg.k).all()
        assert off[e + 1] - off[e] == -(-cnt[e] // B.ROW_ALIGN) * B.ROW_ALIGN
        assert (srow[lists[e]] == np.arange(off[e], off[e] + cnt[e])).all()
    assert (pslot[off[cfg.E]:] == -1).all() and (ptok[off[cfg.E]:] == 0).all()


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen3_30b_a3b", "mixtral_8x7b"])
@pytest.mark.parametrize("renorm", [1, 0])
def test_topk_bit_exact_given_logits(name, renorm):
    dev = device()
    cfg = synth.CONFIGS[name]
    # logits with the layer's statistics, plus injected ties (and a signed zero pair)
    rng = np.random.default_rng(3)
    l = (rng.standard_normal((cfg.T, cfg.E)) * 0.9).astype(np.float32)
    l[::7, : min(cfg.E, 5)] = 0.25
    l[1, 0], l[1, 1] = -0.0, 0.0
    inp = {"x": np.zeros((cfg.T, cfg.H), np.float32), "w_router": np.zeros((cfg.E, cfg.H),
                                                                            np.float32)}
    s, rt, _ = _route(cfg, inp, dev, logits_in=l, renorm=renorm)
    oi, ow = oracle.route_topk(l, cfg.k, renorm)
    gi = rt.topk_idx.cpu().numpy().reshape(cfg.T, cfg.k)
    assert (gi == oi).all()
    gw = rt.topk_w.cpu().numpy().reshape(cfg.T, cfg.k)
    assert max_rel(gw, ow) < 1e-5
    _check_perm(cfg, rt, oi)


SMALL = {"bf16_ragged": dict(T=300, H=256, E=8, k=2, I=64),
         "bf16_two_m_tiles": dict(T=1000, H=128, E=160, k=4, I=64),
         # 3 k-blocks for 4 K splits (one split empty), E not a multiple of 4, one short tile
         "bf16_short_k_odd_e": dict(T=70, H=64, E=6, k=2, I=64)}


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen3_30b_a3b", "bf16_ragged",
                                  "bf16_two_m_tiles", "bf16_short_k_odd_e"])
def test_router_logits_and_routing_from_x(name):
    """fp32 tokens: CUDA-core FFMA logits; bf16 tokens: three bf16 tensor-core products of the
    split fp32 router weight. Both within the fp32 dot-product error bound of the oracle."""
    dev = device()
    cfg = synth.CONFIGS[name] if name in synth.CONFIGS else synth.small_config(
        name, bf16=True, **SMALL[name])
    inp = synth.moe_inputs(cfg, seed=0)
    s, rt, gl = _route(cfg, inp, dev)
    ol = oracle.router_logits(inp["x"], inp["w_router"])
    # fp32 FFMA over H terms against the fp64 sum rounded once
    scale = np.abs(inp["x"]).astype(np.float64) @ np.abs(inp["w_router"]).T.astype(np.float64)
    assert np.max(np.abs(gl - ol) / np.maximum(scale, 1e-30)) < 4 * cfg.H * 2.0**-24
    # ranking on the device's own logits is bit-exact against the oracle fed the same logits
    oi, ow = oracle.route_topk(gl, cfg.k)
    gi = rt.topk_idx.cpu().numpy().reshape(cfg.T, cfg.k)
    assert (gi == oi).all()
    _check_perm(cfg, rt, oi)
    # against the oracle's own logits, a slot may differ only where two logits nearly tie
    oi2, _ = oracle.route_topk(ol, cfg.k)
    diff = np.nonzero((gi != oi2).any(axis=1))[0]
    for t in diff:
        srt = np.sort(ol[t])[::-1]
        assert np.min(np.abs(np.diff(srt[: cfg.k + 1]))) < 1e-4


def test_routing_is_deterministic():
    dev = device()
    cfg = synth.CONFIGS["qwen3_30b_a3b"]
    inp = synth.moe_inputs(cfg, seed=1)
    a = _route(cfg, inp, dev)[1]
    b = _route(cfg, inp, dev)[1]
    for f in ("topk_idx", "expert_offset", "perm_tok", "perm_slot", "slot_row"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f
