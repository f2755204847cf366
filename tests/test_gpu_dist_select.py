"""The selection spread over ranks on the GPU: the library's per-part calls (usaf_shard_*), driven
by dist_select over several parts held in one process, give the single-GPU selection and the
oracle's set bit for bit; RigL's drop and merge with the grow set found over the parts
(usaf_rigl_apply) and the state carry for a set found over the parts (usaf_reselect_carry) equal
usaf_rigl_swap and usaf_reselect_full on every output. The trainer's reduce-scatter exchange runs
through a one-rank NCCL group."""
import math
import os
import socket

import numpy as np
import pytest
import torch

import oracle
from sparse_moe_fine_gb300 import binding as B
from sparse_moe_fine_gb300 import dist_select as DS
from sparse_moe_fine_gb300 import synth

from _gpu import device, to_dev

pytestmark = pytest.mark.gpu


def over_parts(g, cuts, K, act=None, st=None):
    """topk_over_parts on the parts [cuts[j], cuts[j+1]) of the device tensor g, one process."""
    parts = []
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        ex = None if act is None else DS.part_bitmap(act, lo, hi - lo)
        parts.append((g[lo:hi], lo, ex))
    out = DS.topk_over_parts(parts, K, DS.LibShardOps(dev_status=st), DS.LocalComm())
    torch.cuda.synchronize()
    return out


def whole(g, K):
    out = torch.full((K,), -1, dtype=torch.int64, device=g.device)
    st = torch.zeros(1, dtype=torch.int32, device=g.device)
    B.importance_select(g, K, out, dev_status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def gradient(kind, N):
    if kind == "ties":
        rng = np.random.default_rng(N)
        return (rng.integers(-6, 7, N) * 0.125).astype(np.float32)
    g = synth.student_t3(N, seed=11)
    K = math.ceil(0.005 * N)
    if kind == "t3_ties":
        tau = np.abs(g[oracle.importance_select_threshold(g, K)]).min()
        g[::997] = tau  # exact ties at the threshold in every part
    elif kind == "clustered":
        # the largest entries crowd one compaction region: that part's emission takes the
        # whole-part path
        g[1000:1000 + 2 * K] *= 1000.0
    return g


@pytest.mark.parametrize("kind,N,cuts", [
    # a one-entry part and bases that are not 16-byte aligned
    ("ties", 100_000, [0, 33_333, 33_334, 70_001, 100_000]),
    ("t3_ties", 9_000_003, [0, 4_500_001, 9_000_003]),
    ("clustered", 9_000_003, [0, 4_500_001, 9_000_003]),
    ("t3_ties", 9_000_003, [0, 1_000_000, 1_000_000, 9_000_003]),  # an empty part
])
def test_parts_match_the_single_gpu_selection(kind, N, cuts):
    dev = device()
    g_np = gradient(kind, N)
    K = N // 3 if kind == "ties" else math.ceil(0.005 * N)
    g = to_dev(g_np, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    got = over_parts(g, cuts, K, st=st).cpu().numpy()
    ref = oracle.importance_select_threshold(g_np, K)
    assert got.size == K and np.array_equal(got, ref)
    assert np.array_equal(whole(g, K), ref)
    # the large parts emit from their candidate regions, except where the winners crowd one
    assert int(st.item()) == (B.DEV_SELECT_EXACT_PATH if kind == "clustered" else 0)


def state(K, seed):
    rng = np.random.default_rng(seed)
    p = synth.to_bf16_values(rng.standard_normal(K).astype(np.float32) * 0.02)
    m = rng.standard_normal(K).astype(np.float32)
    v = np.abs(rng.standard_normal(K)).astype(np.float32)
    return p, m, v


@pytest.mark.parametrize("N,K,D,cuts", [
    (5000, 700, 200, [0, 1234, 2500, 5000]),
    (5000, 700, 0, [0, 2500, 5000]),
    (1 << 23, 41944, 12583, [0, 5_000_000, 1 << 23]),
])
def test_rigl_apply_with_the_grow_set_over_parts(N, K, D, cuts):
    dev = device()
    rng = np.random.default_rng(N + D)
    act = synth.uniform_mask(N, K, seed=N % 89)
    g = (gradient("ties", N) if N < 10000 else synth.student_t3(N, seed=4))
    p, m, v = state(K, N)
    w = synth.to_bf16_values(rng.standard_normal(N).astype(np.float32))
    n0 = N // 3 * 2
    a, gd, wd = to_dev(act, dev), to_dev(g, dev), to_dev(w, dev, True)
    pd, md, vd = to_dev(p, dev), to_dev(m, dev), to_dev(v, dev)
    grown = over_parts(gd, cuts, D, act=a)

    def outs():
        return ([torch.empty(K, dtype=torch.int64, device=dev)]
                + [torch.empty(K, device=dev) for _ in range(3)]
                + [torch.zeros(1, dtype=torch.int64, device=dev)])
    o1, o2 = outs(), outs()
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    B.rigl_apply(a, D, grown, pd, md, vd, wd[:n0], n0, wd[n0:], *o1, dev_status=st)
    B.rigl_swap(gd, a, D, pd, md, vd, wd[:n0], n0, wd[n0:], *o2)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for x, y in zip(o1, o2):
        assert torch.equal(x, y)
    ref = oracle.rigl_swap(act, p, m, v, g, D, lambda i: w[i], grow_by="threshold")
    for x, y in zip(o1[:4], ref[:4]):
        assert np.array_equal(x.cpu().numpy(), y)
    assert int(o1[4].item()) == ref[4] == D


@pytest.mark.parametrize("N,K_old,K,cuts", [
    (6000, 800, 900, [0, 3001, 6000]),
    (1 << 23, 41944, 41944, [0, 4_194_304, 6_000_000, 1 << 23]),
])
def test_reselect_carry_for_a_set_over_parts(N, K_old, K, cuts):
    dev = device()
    rng = np.random.default_rng(N + 7)
    g = gradient("ties", N) if N < 10000 else synth.student_t3(N, seed=6)
    act = synth.uniform_mask(N, K_old, seed=N % 83)
    if N >= 10000:
        act = np.sort(np.union1d(oracle.importance_select_threshold(g, K_old // 2), act)[:K_old])
    p, m, v = state(act.size, N + 1)
    w = synth.to_bf16_values(rng.standard_normal(N).astype(np.float32))
    n0 = N // 3 * 2
    a, gd, wd = to_dev(act, dev), to_dev(g, dev), to_dev(w, dev, True)
    pd, md, vd = to_dev(p, dev), to_dev(m, dev), to_dev(v, dev)
    new = over_parts(gd, cuts, K)
    o1 = [torch.empty(K, device=dev) for _ in range(3)] + [torch.zeros(1, dtype=torch.int64,
                                                                        device=dev)]
    o2 = ([torch.empty(K, dtype=torch.int64, device=dev)]
          + [torch.empty(K, device=dev) for _ in range(3)]
          + [torch.zeros(1, dtype=torch.int64, device=dev)])
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    B.reselect_carry(new, a, pd, md, vd, wd[:n0], n0, wd[n0:], *o1, dev_status=st)
    B.reselect_full(gd, K, a, pd, md, vd, wd[:n0], n0, wd[n0:], *o2)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(new, o2[0])
    for x, y in zip(o1, o2[1:]):
        assert torch.equal(x, y)
    ref = oracle.reselect_full(act, p, m, v, g, K, lambda i: w[i])
    assert np.array_equal(new.cpu().numpy(), ref[0])
    for x, y in zip(o1[:3], ref[1:4]):
        assert np.array_equal(x.cpu().numpy(), y)
    assert int(o1[3].item()) == ref[4]


def test_given_sets_out_of_range_are_flagged_not_read():
    """A grow set or a new set holding an entry past the last weight: that entry's p is 0 and
    USAF_DEV_BAD_INDEX is set; the weights are never read there, and the other entries are as for
    the set without it."""
    dev = device()
    N, K = 4000, 300
    act = synth.uniform_mask(N, K, seed=5)
    p, m, v = state(K, 5)
    w = synth.to_bf16_values(np.random.default_rng(5).standard_normal(N).astype(np.float32))
    a, wd = to_dev(act, dev), to_dev(w, dev, True)
    pd, md, vd = to_dev(p, dev), to_dev(m, dev), to_dev(v, dev)
    free = np.setdiff1d(np.arange(N), act)
    grown = np.concatenate([free[:9], [N + 3]]).astype(np.int64)
    outs = ([torch.empty(K, dtype=torch.int64, device=dev)]
            + [torch.empty(K, device=dev) for _ in range(3)]
            + [torch.zeros(1, dtype=torch.int64, device=dev)])
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    B.rigl_apply(a, 10, to_dev(grown, dev), pd, md, vd, wd[:N // 2], N // 2, wd[N // 2:], *outs,
                 dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == B.DEV_BAD_INDEX
    new = outs[0].cpu().numpy()
    assert new[-1] == N + 3 and outs[1][-1].item() == 0.0
    j = np.searchsorted(new, free[:9])
    assert np.array_equal(outs[1].cpu().numpy()[j], w[free[:9]])
    # the state carry
    newset = np.concatenate([act[:K - 1], [N + 5]]).astype(np.int64)
    o = [torch.empty(K, device=dev) for _ in range(3)] + [torch.zeros(1, dtype=torch.int64,
                                                                       device=dev)]
    st.zero_()
    B.reselect_carry(to_dev(newset, dev), a, pd, md, vd, wd[:N // 2], N // 2, wd[N // 2:], *o,
                     dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == B.DEV_BAD_INDEX
    assert o[0][-1].item() == 0.0 and int(o[3].item()) == K - 1
    assert np.array_equal(o[0].cpu().numpy()[:-1], p[:-1])


@pytest.mark.parametrize("mode", ["rigl", "full"])
def test_trainer_reduce_scatter_exchange_one_rank(mode):
    """A one-rank NCCL group: the trainer's reduce-scatter exchange and selection over parts
    install the same active set and state as the all-reduce exchange."""
    import torch.distributed as dist
    from sparse_moe_fine_gb300.layer import MoELayer
    from sparse_moe_fine_gb300.trainer import StackTrainer
    dev = device()
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    torch.cuda.set_device(dev)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        cfg = synth.small_config("rs", T=256, H=128, E=8, k=2, I=128, bf16=True, frac=0.05)
        inp = synth.moe_inputs(cfg, seed=60)
        act = synth.uniform_mask(cfg.N, cfg.K, seed=60)
        bf = lambda x: torch.from_numpy(x).to(dev).to(torch.bfloat16)

        def run(exchange):
            L = MoELayer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, bf(inp["w_gate_up"]),
                         bf(inp["w_down"]), torch.from_numpy(inp["w_router"]).to(dev),
                         torch.from_numpy(act).to(dev), device=dev, group=dist.group.WORLD)
            tr = StackTrainer([L], total_steps=10, reselect_every=2, reselect=mode,
                              dense_exchange=exchange)
            for s in range(2):
                m = synth.moe_inputs(cfg, seed=61 + s)
                tr.step([bf(m["x"])], [bf(m["dy"])])
            torch.cuda.synchronize()
            return L, tr.metrics()
        La, ma = run("allreduce")
        Lb, mb = run("reduce_scatter")
        assert torch.equal(La.act, Lb.act)
        for x, y in ((La.p, Lb.p), (La.m, Lb.m), (La.v, Lb.v)):
            assert torch.equal(x, y)
        assert ma[1]["turnover"] == mb[1]["turnover"] and mb[1]["turnover"][0] > 0
        assert not np.array_equal(La.act.cpu().numpy(), act)
    finally:
        dist.destroy_process_group()
