"""The allocation-free routing entry point (usaf_route_topk_noalloc) against the workspace one.

usaf_route_topk_noalloc serves callers that cannot allocate device memory where they route (a
fixed, pre-planned memory pool; code running inside another runtime's allocator); it keeps its
scratch in a fixed array inside the library instead of a caller workspace. Two calls in a row on
different inputs must each give exactly the routing that usaf_route_topk gives (the routing
tables are integers and are compared bit for bit; logits and weights are compared exactly too,
since both entry points run the same kernels). A layer too large for the fixed array is refused
before anything runs.
"""
import ctypes

import pytest
import torch

from sparse_moe_fine_gb300 import binding as B
from sparse_moe_fine_gb300 import synth

from _gpu import device, to_dev

pytestmark = pytest.mark.gpu

FIELDS = ("topk_idx", "topk_w", "expert_count", "expert_offset", "perm_tok", "perm_slot",
          "slot_row")


def _inputs(cfg, seed, dev):
    inp = synth.moe_inputs(cfg, seed=seed)
    return to_dev(inp["x"], dev, cfg.bf16), to_dev(inp["w_router"], dev)


def test_noalloc_routing_matches_workspace_routing_on_two_calls():
    dev = device()
    cfg = synth.CONFIGS["qwen3_30b_a3b"]
    s = B.shape(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I)
    runs = []
    for seed in (0, 1):
        x, wr = _inputs(cfg, seed, dev)
        rt = B.Routing.empty(s, dev)
        logits = torch.empty(cfg.T, cfg.E, device=dev)
        B.route_topk_noalloc(s, x, wr, rt, logits_out=logits)
        runs.append((x, wr, rt, logits))
    torch.cuda.synchronize()
    for x, wr, rt, logits in runs:
        ref = B.Routing.empty(s, dev)
        ref_logits = torch.empty(cfg.T, cfg.E, device=dev)
        B.route_topk(s, x, wr, ref, logits_out=ref_logits)
        torch.cuda.synchronize()
        assert torch.equal(logits, ref_logits)
        for f in FIELDS:
            a, b = getattr(rt, f), getattr(ref, f)
            if f in ("perm_tok", "perm_slot"):
                n = int(ref.expert_offset[-1].item())
                a, b = a[:n], b[:n]
            assert torch.equal(a, b), f
    # the two calls routed different inputs, so the second did not reuse the first's results
    assert not torch.equal(runs[0][2].topk_idx, runs[1][2].topk_idx)


def test_noalloc_fp32_layer_and_size_limit():
    dev = device()
    cfg = synth.CONFIGS["tiny_fp32"]
    s = B.shape(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I)
    x, wr = _inputs(cfg, 2, dev)
    rt, ref = B.Routing.empty(s, dev), B.Routing.empty(s, dev)
    la, lb = torch.empty(cfg.T, cfg.E, device=dev), torch.empty(cfg.T, cfg.E, device=dev)
    B.route_topk_noalloc(s, x, wr, rt, logits_out=la, renorm=0)
    B.route_topk(s, x, wr, ref, logits_out=lb, renorm=0)
    torch.cuda.synchronize()
    assert torch.equal(la, lb)
    for f in ("topk_idx", "topk_w", "expert_count", "expert_offset", "slot_row"):
        assert torch.equal(getattr(rt, f), getattr(ref, f)), f
    # a router of E*H = 1024*4096 needs 24 MiB of split weights: more than the fixed array
    big = B.shape(16, 4096, 1024, 2, 64)
    r = B._Routing(*[1] * 7)
    code = B.lib().usaf_route_topk_noalloc(ctypes.byref(big), 1, B.BF16, 1, None, 1, 1,
                                           ctypes.byref(r), None, None)
    assert code == 3
    # the same layer routed from given logits, or with fp32 tokens, needs no split weights and
    # fits: both calls run and agree with the workspace entry point
    E, H, T = 1024, 4096, 16
    bs = B.shape(T, H, E, 2, 64)
    gen = torch.Generator().manual_seed(3)
    xb = torch.randn(T, H, generator=gen).to(dev)
    wrb = (0.02 * torch.randn(E, H, generator=gen)).to(dev)
    got, want = B.Routing.empty(bs, dev), B.Routing.empty(bs, dev)
    lg, lw = torch.empty(T, E, device=dev), torch.empty(T, E, device=dev)
    B.route_topk_noalloc(bs, xb, wrb, got, logits_out=lg)
    B.route_topk(bs, xb, wrb, want, logits_out=lw)
    torch.cuda.synchronize()
    assert torch.equal(lg, lw)
    assert torch.equal(got.topk_idx, want.topk_idx)
    got2 = B.Routing.empty(bs, dev)
    B.route_topk_noalloc(bs, None, None, got2, logits_in=lw)
    torch.cuda.synchronize()
    assert torch.equal(got2.topk_idx, want.topk_idx)
    assert torch.equal(got2.perm_slot, want.perm_slot)
