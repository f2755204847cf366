"""Seeded synthetic inputs for the USAF MoE-layer workloads.

This module only draws random numbers and shapes them: it holds none of the method's arithmetic
(no routing, no selection, no optimizer), so both the CUDA path and the CPU oracle can be fed from
it. Every tensor is drawn from numpy's PCG64 in fixed chunks of 2^22 elements, chunk c of stream s
seeded with ``default_rng([s, c])``; chunks are filled by a thread pool, so the values depend only
on (seed, stream, shape) and not on the thread count. Values that a workload stores in bf16 are
drawn in fp32 and rounded to the nearest bf16 (ties to even), and returned as float32 arrays
holding exactly those bf16 values.

Per-tensor streams (base seed s): x = s+1, router weight = s+2, gate_up_proj = s+3,
down_proj = s+4, upstream gradient dY = s+5, dense gradient g = s+6, mask = s+7.

The workloads are the Qwen3-30B-A3B-shaped layer the USAF README trains (its "used in all
benchmarks" model), a Mixtral-8x7B-shaped layer (listed among the README's model families), and a
tiny fp32 layer for exhaustive checks. No dataset or trained weight is involved: the README's own
workload is private code data, which these draws stand in for.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

CHUNK = 1 << 22
STREAM = {"x": 1, "w_router": 2, "w_gate_up": 3, "w_down": 4, "dy": 5, "g": 6, "mask": 7,
          "state": 8}


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _fill(n: int, seed: int, stream: int, draw) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK

    def work(c: int) -> None:
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        rng = np.random.default_rng([seed + stream, c])
        out[lo:hi] = draw(rng, hi - lo)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def to_bf16_values(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32 holding them."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = a.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (b.astype(np.uint32) << 16).view(np.float32).reshape(a.shape)


def normal(shape, std: float, seed: int, stream: str, bf16: bool) -> np.ndarray:
    n = int(np.prod(shape))
    a = _fill(n, seed, STREAM[stream],
              lambda rng, m: rng.standard_normal(m, dtype=np.float32) * np.float32(std))
    a = a.reshape(shape)
    return to_bf16_values(a) if bf16 else a


def student_t3(n: int, seed: int, stream: str = "g") -> np.ndarray:
    """Student-t with 3 degrees of freedom: Z / sqrt(chi2_3 / 3), drawn per chunk."""
    def draw(rng, m):
        z = rng.standard_normal(m, dtype=np.float64)
        c = rng.chisquare(3.0, m)
        return (z / np.sqrt(c / 3.0)).astype(np.float32)
    return _fill(n, seed, STREAM[stream], draw)


def uniform_mask(N: int, K: int, seed: int) -> np.ndarray:
    """K distinct flat indices in [0, N), uniformly without replacement, sorted ascending."""
    rng = np.random.default_rng([seed + STREAM["mask"], 0])
    if K * 4 >= N:
        return np.sort(rng.permutation(N)[:K]).astype(np.int64)
    got = np.empty(0, dtype=np.int64)
    while got.size < K:
        extra = rng.integers(0, N, size=int((K - got.size) * 1.2) + 64, dtype=np.int64)
        got = np.unique(np.concatenate([got, extra]))
    # drop a seeded random surplus so the kept set stays uniform
    keep = np.sort(rng.permutation(got.size)[:K])
    return got[keep]


@dataclass
class MoEConfig:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    bf16: bool
    x_std: float = 1.0
    w_router_std: float = 0.02
    w_std: float = 0.02
    dy_std: float = 1.0
    frac: float = 0.005
    lr: float = 1e-4
    betas: tuple = (0.9, 0.999)
    eps: float = 1e-8
    renorm: int = 1
    extra: dict = field(default_factory=dict)

    @property
    def N_gu(self) -> int:
        return self.E * 2 * self.I * self.H

    @property
    def N(self) -> int:
        return self.E * 3 * self.I * self.H

    @property
    def K(self) -> int:
        return int(math.ceil(self.frac * self.N))


CONFIGS = {
    # tiny fp32 layer: H=64, E=8, top-2, I=32, T=128; 5% random mask; lr 1e-3
    "tiny_fp32": MoEConfig("tiny_fp32", T=128, H=64, E=8, k=2, I=32, bf16=False, dy_std=1.0,
                           frac=0.05, lr=1e-3),
    # Qwen3-30B-A3B-shaped layer: H=2048, E=128, top-8, I=768, T=4096
    "qwen3_30b_a3b": MoEConfig("qwen3_30b_a3b", T=4096, H=2048, E=128, k=8, I=768, bf16=True,
                               dy_std=1e-2),
    # the same layer under skewed routing, T=16384
    "qwen3_skewed": MoEConfig("qwen3_skewed", T=16384, H=2048, E=128, k=8, I=768, bf16=True,
                              dy_std=1e-2, extra={"zipf_s": 1.2, "dead_experts": 10}),
    # Mixtral-8x7B-shaped layer: H=4096, E=8, top-2, I=14336, T=8192
    "mixtral_8x7b": MoEConfig("mixtral_8x7b", T=8192, H=4096, E=8, k=2, I=14336, bf16=True,
                              w_std=0.015, dy_std=1e-2),
}


def small_config(name: str, T: int, H: int, E: int, k: int, I: int, bf16: bool = True,
                 frac: float = 0.05, dy_std: float = 1e-2) -> MoEConfig:
    """A reduced layer of the same recipe, for tests that must finish on the CPU oracle."""
    return MoEConfig(name, T=T, H=H, E=E, k=k, I=I, bf16=bf16, dy_std=dy_std, frac=frac,
                     lr=1e-3)


def moe_inputs(cfg: MoEConfig, seed: int = 0) -> dict:
    """x [T,H], w_router [E,H] fp32, w_gate_up [E,2I,H], w_down [E,H,I], dy [T,H]."""
    b = cfg.bf16
    return {
        "x": normal((cfg.T, cfg.H), cfg.x_std, seed, "x", b),
        "w_router": normal((cfg.E, cfg.H), cfg.w_router_std, seed, "w_router", False),
        "w_gate_up": normal((cfg.E, 2 * cfg.I, cfg.H), cfg.w_std, seed, "w_gate_up", b),
        "w_down": normal((cfg.E, cfg.H, cfg.I), cfg.w_std, seed, "w_down", b),
        "dy": normal((cfg.T, cfg.H), cfg.dy_std, seed, "dy", b),
    }


def skew_bias(E: int, zipf_s: float, dead: int, seed: int) -> np.ndarray:
    """Per-expert logit offsets for skewed routing: the `dead` experts get -1e3 (never routed),
    the others log(rank^-s) in a seeded random rank order. Realised loads are measured, not
    assumed."""
    rng = np.random.default_rng([seed + STREAM["w_router"], 1])
    order = rng.permutation(E)
    b = np.empty(E, dtype=np.float32)
    live = order[: E - dead]
    ranks = np.arange(1, live.size + 1, dtype=np.float64)
    b[live] = (-zipf_s * np.log(ranks)).astype(np.float32)
    b[order[E - dead:]] = -1e3
    return b


def _union_sample(ranges, n: int, rng) -> np.ndarray:
    """n distinct indices drawn uniformly from a union of disjoint [lo, hi) ranges, sorted."""
    sizes = np.array([hi - lo for lo, hi in ranges], dtype=np.int64)
    starts = np.concatenate([[0], np.cumsum(sizes)[:-1]])
    got = np.empty(0, dtype=np.int64)
    while got.size < n:
        got = np.unique(np.concatenate([got, rng.integers(0, sizes.sum(), n - got.size + 64)]))
    got = got[np.sort(rng.permutation(got.size)[:n])]
    r = np.searchsorted(starts, got, side="right") - 1
    return np.array([lo for lo, _ in ranges], dtype=np.int64)[r] + (got - starts[r])


def concentrated_mask(cfg: "MoEConfig", hot_experts, hot_frac: float, seed: int) -> np.ndarray:
    """The skewed workload's active set: hot_frac of K uniformly over the weights (both tensors)
    of the given experts, the rest uniformly over the other experts' weights; sorted."""
    rng = np.random.default_rng([seed + STREAM["mask"], 2])
    hot = sorted(set(int(e) for e in hot_experts))
    cold = [e for e in range(cfg.E) if e not in set(hot)]
    pgu, pd = 2 * cfg.I * cfg.H, cfg.H * cfg.I

    def ranges(es):
        return ([(e * pgu, (e + 1) * pgu) for e in es] +
                [(cfg.N_gu + e * pd, cfg.N_gu + (e + 1) * pd) for e in es])
    n_hot = int(hot_frac * cfg.K)
    a = _union_sample(ranges(hot), n_hot, rng)
    b = _union_sample(ranges(cold), cfg.K - n_hot, rng)
    return np.sort(np.concatenate([a, b]))


def apply_skew(inputs: dict, bias: np.ndarray) -> None:
    """Realise a router logit bias without a bias term: x[:,0] := 1 and w_router[:,0] := bias."""
    inputs["x"][:, 0] = 1.0
    inputs["w_router"][:, 0] = bias


def adam_state(K: int, seed: int) -> tuple:
    """Nonzero (m, v) state for multi-step optimizer checks: m ~ N(0,1e-3), v ~ |N(0,1e-6)|."""
    rng = np.random.default_rng([seed + STREAM["state"], 0])
    m = (rng.standard_normal(K) * 1e-3).astype(np.float32)
    v = np.abs(rng.standard_normal(K) * 1e-6).astype(np.float32)
    return m, v
