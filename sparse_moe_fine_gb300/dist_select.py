"""Top-K selection spread over data-parallel ranks: the host side of the importance pass and of
RigL's grow step when the dense gradient is reduce-scattered instead of all-reduced.

USAF README: the trainable weights are the 0.5% with the largest gradient magnitude ("Not all
weights matter"), chosen again every 50 steps ("Sparsity adapts"), and the multi-GPU mode is
DataParallel (feature table). Every rank holds the same weights and active set; each rank's dense
gradient covers its own tokens. A reduce-scatter leaves rank r with the sum over ranks of one
contiguous part of the gradient (half the bytes of an all-reduce). The top-K of |g| over all
parts (ties to the lower global index) is then found as the single-GPU radix selection finds it,
with every digit histogram summed over the ranks:

  for each digit of the 31-bit key (11, 11 and 9 bits, most significant first):
      every rank counts its keys that match the digits found so far, by their next digit;
      the counts are summed over the ranks (one all-reduce of at most 2048 integers);
      every rank takes the same digit: the largest one whose keys, with those above it, reach K;
  tau = the K-th largest key. A rank's own histograms also count its keys above tau (those whose
  digit exceeded the chosen one in some round) and at tau (the last round's bin); one all-gather
  of these counts lets every rank give the ties at tau to the lowest global indices first, i.e.
  to the parts in rank order; every rank emits its winners in index order, and an all-gather
  concatenates them (sorted).

The device work per part is the library's usaf_shard_* calls (`LibShardOps`); the exchanges go
through `comm` (torch.distributed, or a single process holding several parts for tests). RigL's
grow step is the same selection over the entries outside the active set (`excl` bitmaps).
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B

ROUNDS = ((20, 11), (9, 11), (0, 9))


def pick_digit(hist, krem):
    """The largest digit d whose bins from d up hold at least krem keys, and krem minus the keys
    above d. Falls to digit 0 when the counts cannot reach krem."""
    h = np.asarray(hist, np.int64)
    top = np.cumsum(h[:0:-1])  # top[j]: keys in the bins from the highest down to nb - 1 - j
    j = int(np.searchsorted(top, krem))  # the first j with top[j] >= krem (top is nondecreasing)
    if j == top.size:
        return 0, krem - (int(top[-1]) if top.size else 0)
    return h.size - 1 - j, krem - (int(top[j - 1]) if j else 0)


def tie_quota(counts, need):
    """counts: (gt, eq) of every part in global index order; the ties each part gives, lowest
    indices first."""
    out, before = [], 0
    for _, eq in counts:
        out.append(max(0, min(eq, need - before)))
        before += eq
    return out


class LibShardOps:
    """The per-part kernels through the library (device tensors, the given or current stream)."""

    def __init__(self, stream=None, dev_status=None):
        self.stream = stream
        self.dev_status = dev_status

    def histogram(self, g, excl, prefix, shift, bits):
        h = torch.zeros(1 << bits, dtype=torch.int64, device=g.device)
        B.shard_key_histogram(g, excl, prefix, shift, bits, h, stream=self.stream)
        return h

    def emit(self, g, excl, tau, take_eq, gt, count, base):
        out = torch.empty(gt + take_eq, dtype=torch.int64, device=g.device)
        if out.numel():
            B.shard_emit(g, excl, tau, take_eq, count, base, out, dev_status=self.dev_status,
                         stream=self.stream)
        return out


class TorchComm:
    """The exchanges over a torch.distributed group (NCCL with device tensors, gloo with host
    tensors)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def allreduce(self, t):
        self.dist.all_reduce(t, op=self.dist.ReduceOp.SUM, group=self.group)
        return t

    def allgather_cat(self, t):
        """Every rank's 1-D tensor (sizes may differ) concatenated in rank order, and the sizes."""
        n = torch.tensor([t.numel()], dtype=torch.int64, device=t.device)
        sizes = [torch.zeros_like(n) for _ in range(self.world)]
        self.dist.all_gather(sizes, n, group=self.group)
        sizes = [int(v) for v in torch.cat(sizes).tolist()]
        pad = torch.zeros(max(sizes), dtype=t.dtype, device=t.device)
        pad[:t.numel()] = t
        bufs = [torch.empty_like(pad) for _ in sizes]
        self.dist.all_gather(bufs, pad, group=self.group)
        return torch.cat([b[:m] for b, m in zip(bufs, sizes)]), sizes


class LocalComm:
    """One process holding every part (world size 1): the exchanges are identities."""

    rank, world = 0, 1

    def allreduce(self, t):
        return t

    def allgather_cat(self, t):
        return t, [t.numel()]


def topk_over_parts(parts, K, ops, comm):
    """The K entries with the largest |g| over every rank's parts (ties to the lower global
    index), sorted by global index; the same tensor on every rank.

    parts: this rank's parts as (g_part, base, excl_part) in index order, g_part a 1-D fp32
    tensor holding the global entries base .. base + len - 1, excl_part a bitmap of its entries to
    leave out (usaf_active_bitmap) or None. Every rank calls this with the same K, and the parts
    of all ranks, taken in rank order, cover the entries in index order. K must not exceed the
    number of entries left in."""
    if not parts:
        raise ValueError("every rank needs at least one part")
    dev = parts[0][0].device
    if K <= 0:
        return torch.empty(0, dtype=torch.int64, device=dev)
    prefix, krem = 0, int(K)
    gt, eq = [0] * len(parts), [0] * len(parts)
    for shift, bits in ROUNDS:
        hs = [ops.histogram(g, ex, prefix, shift, bits) for g, _, ex in parts]
        total = hs[0].clone()
        for h in hs[1:]:
            total += h
        rows = torch.stack(hs + [comm.allreduce(total)]).cpu().numpy()  # one copy to the host
        d, krem = pick_digit(rows[-1], krem)
        for j, row in enumerate(rows[:-1]):
            gt[j] += int(row[d + 1:].sum())  # above tau: a larger digit where the prefix matched
            eq[j] = int(row[d])
        prefix |= d << shift
    tau = prefix
    local = torch.tensor([v for j in range(len(parts)) for v in (gt[j], eq[j])],
                         dtype=torch.int64, device=dev)
    every, sizes = comm.allgather_cat(local)
    quota = tie_quota(every.view(-1, 2).tolist(), krem)
    first = sum(sizes[:comm.rank]) // 2  # this rank's first part among all ranks' parts
    outs = [ops.emit(g, ex, tau, quota[first + j], gt[j], gt[j] + eq[j], base)
            for j, (g, base, ex) in enumerate(parts)]
    return comm.allgather_cat(torch.cat(outs))[0]


def shard_range(N, rank, world):
    """The part [lo, hi) of N entries that rank holds after a reduce-scatter (equal parts, the
    last one shorter)."""
    per = (N + world - 1) // world
    lo = min(N, rank * per)
    return lo, min(N, lo + per)


def part_bitmap(act_idx, lo, n):
    """The bitmap of the active entries that fall in the part [lo, lo + n) (None for an empty
    part: nothing to leave out)."""
    if n == 0:
        return None
    bm = torch.empty((n + 31) // 32, dtype=torch.int32, device=act_idx.device)
    B.active_bitmap(act_idx, lo, n, bm)
    return bm


def reduce_scatter_part(g, group=None):
    """Rank r's part of the sum over ranks of g (1-D), by reduce-scatter where the backend has
    it and by all-reduce otherwise (gloo)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    N = g.numel()
    per = (N + world - 1) // world
    lo, hi = shard_range(N, rank, world)
    if dist.get_backend(group) == "nccl":
        src = g
        if per * world != N:  # the collective wants equal parts
            src = torch.zeros(per * world, dtype=g.dtype, device=g.device)
            src[:N] = g
        out = torch.empty(per, dtype=g.dtype, device=g.device)
        dist.reduce_scatter_tensor(out, src, op=dist.ReduceOp.SUM, group=group)
        return out[:hi - lo], lo
    t = g.clone()  # gloo has no reduce-scatter: the sum everywhere, this rank's part kept
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return t[lo:hi].contiguous(), lo
