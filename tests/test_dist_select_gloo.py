"""The selection spread over ranks (sparse_moe_fine_gb300.dist_select) on three CPU ranks (gloo):
each rank holds one part of the gradient, the digit histograms are summed over the ranks, the
ties at the threshold go to the lowest global indices across the part boundaries, and the set
every rank ends with is the oracle's. The per-part work runs here in numpy (the same contract as
the library's usaf_shard_* calls, whose GPU parity is in test_gpu_dist_select.py)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from sparse_moe_fine_gb300 import dist_select as DS

WORLD = 3


def _keys(g):
    return g.numpy().view(np.uint32) & np.uint32(0x7FFFFFFF)


def _kept(excl, n):
    if excl is None:
        return np.ones(n, bool)
    bits = np.unpackbits(excl.numpy().view(np.uint8), bitorder="little")[:n]
    return bits == 0


class NumpyShardOps:
    """The usaf_shard_* contract on host tensors."""

    def histogram(self, g, excl, prefix, shift, bits):
        k = _keys(g)[_kept(excl, g.numel())].astype(np.int64)
        hs = shift + bits
        if hs < 32:
            k = k[(k >> hs) == (prefix >> hs)]
        d = (k >> shift) & ((1 << bits) - 1)
        return torch.from_numpy(np.bincount(d, minlength=1 << bits).astype(np.int64))

    def emit(self, g, excl, tau, take_eq, gt, count, base):
        k = _keys(g)
        ok = _kept(excl, g.numel())
        above = np.nonzero(ok & (k > tau))[0]
        eq = np.nonzero(ok & (k == tau))[0][:take_eq]
        assert above.size == gt and count == gt + int((ok & (k == tau)).sum())
        return torch.from_numpy(np.sort(np.concatenate([above, eq])).astype(np.int64) + base)


def _bitmap(act, lo, n):
    bits = np.zeros(((n + 31) // 32) * 32, np.uint8)
    a = act[(act >= lo) & (act < lo + n)] - lo
    bits[a] = 1
    return torch.from_numpy(np.packbits(bits, bitorder="little").view(np.int32).copy())


def tied_gradient(N, seed):
    """Magnitudes from a few dozen values, so the threshold falls inside a large tie group that
    spans the parts; random signs (the selection ranks |g|)."""
    rng = np.random.default_rng(seed)
    mags = np.float32(2.0) ** rng.integers(-6, 6, 40).astype(np.float32)
    g = mags[rng.integers(0, 40, N)] * rng.choice(np.float32([-1, 1]), N)
    return g.astype(np.float32)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run(rank, port, fn, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        out[rank] = fn(rank)
    finally:
        dist.destroy_process_group()


def _spawn(fn):
    out = mp.Manager().dict()
    mp.spawn(_run, args=(_free_port(), fn, out), nprocs=WORLD, join=True)
    return [out[r] for r in range(WORLD)]


N, K, D = 5003, 700, 150  # N not a multiple of the world: the last part is shorter


def _select(rank):
    g = tied_gradient(N, 7)
    act = np.sort(np.random.default_rng(8).choice(N, 400, replace=False)).astype(np.int64)
    comm = DS.TorchComm()
    # the dense gradient: each rank adds its share, the reduce-scatter leaves it one summed part
    share = torch.from_numpy(g / WORLD if rank else g - (WORLD - 1) * (g / WORLD))
    part, lo = DS.reduce_scatter_part(share)
    top = DS.topk_over_parts([(part, lo, None)], K, NumpyShardOps(), comm)
    grow = DS.topk_over_parts([(part, lo, _bitmap(act, lo, part.numel()))], D, NumpyShardOps(),
                              comm)
    # this rank's own part alone, as two sub-parts: the split inside a rank is free too
    half = part.numel() // 2
    two = [(part[:half], lo, None), (part[half:], lo + half, None)]
    top2 = DS.topk_over_parts(two, K, NumpyShardOps(), comm)
    return (lo, part.numel(), part.numpy().copy(), top.numpy().copy(), grow.numpy().copy(),
            top2.numpy().copy())


def test_topk_over_ranks_matches_the_oracle():
    res = _spawn(_select)
    # the parts tile [0, N) in rank order, the last one shorter
    assert [r[0] for r in res] == [DS.shard_range(N, i, WORLD)[0] for i in range(WORLD)]
    assert sum(r[1] for r in res) == N and res[-1][1] < res[0][1]
    g = np.concatenate([r[2] for r in res])
    want = oracle.importance_select(g, K)
    key = oracle.abs_key(g)
    tau = np.sort(key)[::-1][K - 1]
    # the threshold's tie group is larger than what is taken from it and spans parts
    eq = np.nonzero(key == tau)[0]
    assert eq.size > K - (key > tau).sum() and eq[0] < res[0][1] <= eq[-1]
    act = np.sort(np.random.default_rng(8).choice(N, 400, replace=False)).astype(np.int64)
    p = np.ones(act.size, np.float32)
    z = np.zeros(act.size, np.float32)
    new = oracle.rigl_swap(act, p, z, z, g, D, lambda i: np.zeros(i.size, np.float32))[0]
    want_grow = np.setdiff1d(new, act)
    for _, _, _, top, grow, top2 in res:
        np.testing.assert_array_equal(top, want)
        np.testing.assert_array_equal(top2, want)
        np.testing.assert_array_equal(grow, want_grow)


def _edge(rank):
    """K = every entry; K = 0; a rank whose part is empty (fewer entries than ranks' parts)."""
    comm = DS.TorchComm()
    g = torch.from_numpy(tied_gradient(5, 9))
    lo, hi = DS.shard_range(5, rank, WORLD)  # parts of 2, 2, 1
    part = g[lo:hi]
    alln = DS.topk_over_parts([(part, lo, None)], 5, NumpyShardOps(), comm)
    none = DS.topk_over_parts([(part, lo, None)], 0, NumpyShardOps(), comm)
    lo2, hi2 = DS.shard_range(2, rank, WORLD)  # parts of 1, 1, 0
    one = DS.topk_over_parts([(g[lo2:hi2], lo2, None)], 1, NumpyShardOps(), comm)
    return alln.numpy().copy(), none.numpy().copy(), one.numpy().copy()


def test_degenerate_sizes():
    res = _spawn(_edge)
    g = tied_gradient(5, 9)
    for alln, none, one in res:
        np.testing.assert_array_equal(alln, np.arange(5))
        assert none.size == 0
        np.testing.assert_array_equal(one, oracle.importance_select(g[:2], 1))


def test_pick_digit_and_tie_quota():
    # bins 3, 2, 1 hold 2, 1, 3 keys; the 4th largest key is in bin 1, 1st of it
    assert DS.pick_digit([5, 3, 1, 2], 4) == (1, 1)
    assert DS.pick_digit([5, 3, 1, 2], 2) == (3, 2)
    assert DS.pick_digit([5, 0, 0, 0], 3) == (0, 3)  # all in bin 0
    # ties 2, 3, 1 at the threshold over three parts, 4 wanted: the lowest indices first
    assert DS.tie_quota([(1, 2), (0, 3), (5, 1)], 4) == [2, 2, 0]
    assert DS.tie_quota([(0, 0), (0, 3)], 0) == [0, 0]


@pytest.mark.parametrize("n,world", [(10, 3), (9, 3), (2, 4), (0, 2)])
def test_shard_range_tiles(n, world):
    spans = [DS.shard_range(n, r, world) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == n
    assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
    assert all(lo <= hi for lo, hi in spans)
