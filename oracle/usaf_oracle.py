"""CPU oracle of the USAF sparse MoE fine-tuning hot path.

TEST INFRASTRUCTURE ONLY. This is a plain, slow, deliberately obvious restatement of what one
MoE layer's USAF train step computes, written from the pages and checked against closed forms,
brute force, finite differences and library routines by the tests. Only the test suite, the smoke
check and the benchmark's CPU-baseline leg may import it; the product library never calls it and
shares no code with it.

Arithmetic: numpy, float64 for every floating-point step. Inputs stored in bf16 are upcast
exactly. Where a floating-point value decides an integer (the expert ranking, the |g| and |p|
orders), the decision is taken on the fp32 values, as the device does. A library matmul or sort
serves as a step; nothing is blocked, fused or reordered beyond the definitions below.

Sources (page title and section):
  * USAF README (tsuyu122/usaf): "Not all weights matter" (importance phase, 0.5% by gradient
    magnitude), "The router is leverage" (router trained in full), "Sparsity adapts" (RigL
    reselection every 50 steps), the A100 operations table (SparseAdam over the trained 26M),
    the results table (steps with NaN are skipped).
  * "USAF Open Source: 12G VRAM Fine-Tuning Qwen3-30B MoE", section on the key differences
    (only part of the weights of each routed expert is trained, and only that part has optimizer
    state; experts that receive no token get no gradient).
  * experts4bit-qlora page, "The abstraction that fails, and what replaces it" (fused layouts
    gate_up_proj [E,2I,H], down_proj [E,H,I]) and its epilogue-contract bullet (act(gate)*up).

Readings taken where the pages are silent (each also listed in the design notes): softmax then
top-k then renormalise routing, ranked on fp32 logits with ties to the lower expert; gate = the
first I rows of gate_up_proj; act = SiLU; SparseAdam with torch.optim.SparseAdam's formula (eps
added to the uncorrected sqrt(v)); K = ceil(0.005 N); RigL drops the smallest |p| and grows the
largest |g| outside the old set, ties to the lower flat index.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


# ----------------------------------------------------------------------------------------------
# Routing
# ----------------------------------------------------------------------------------------------

def router_logits(x: np.ndarray, w_router: np.ndarray) -> np.ndarray:
    """logits[t,e] = sum_h x[t,h] * Wr[e,h]; accumulated in fp64, rounded once to fp32.

    The router is the gating network the USAF README trains in full ("The router is leverage").
    """
    return (np.asarray(x, F64) @ np.asarray(w_router, F64).T).astype(np.float32)


def route_topk(logits: np.ndarray, k: int, renorm: int = 1):
    """Top-k experts per token and their routing weights.

    Ranking: fp32 logits descending, ties to the lower expert index (stable sort of -logit).
    renorm=1: w_j = exp(l_j - max) / sum over the k selected (softmax, top-k, renormalise);
    renorm=0: w_j = softmax over all E evaluated at the selected experts.
    Returns (idx [T,k] int32, w [T,k] float64).
    """
    l32 = np.asarray(logits, np.float32)
    T, E = l32.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=F64)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(l32[t, e]), e))
        sel = np.array(order[:k], dtype=np.int64)
        idx[t] = sel
        l = l32[t].astype(F64)
        if renorm:
            z = np.exp(l[sel] - l[sel].max())
            w[t] = z / z.sum()
        else:
            z = np.exp(l - l.max())
            w[t] = z[sel] / z.sum()
    return idx, w


def permutation(topk_idx: np.ndarray, E: int):
    """For e = 0..E-1, the slots s = t*k + j routed to e, in ascending token order.

    Returns (counts [E] int64, lists: list of E int64 arrays of slots)."""
    flat = np.asarray(topk_idx).reshape(-1)
    lists = []
    for e in range(E):
        # flat slot order t*k+j is token-major and an expert occurs once per token, so
        # ascending slot order is ascending token order
        lists.append(np.nonzero(flat == e)[0].astype(np.int64))
    counts = np.array([len(s) for s in lists], dtype=np.int64)
    return counts, lists


# ----------------------------------------------------------------------------------------------
# Expert forward / backward (SwiGLU experts over the fused layouts)
# ----------------------------------------------------------------------------------------------

def silu(z):
    return z / (1.0 + np.exp(-z))


def silu_grad(z):
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def _expert_rows(topk_idx, e):
    rows, slots = np.nonzero(topk_idx == e)
    return rows, slots


def _keep(a):
    return a


def moe_forward(x, w_gate_up, w_down, topk_idx, topk_w, rnd=None):
    """Y[t] = sum_j w[t,j] * down[e_j] . (silu(gate) * up), [gate; up] = gate_up[e_j] . x[t].

    rnd (bf16-emulating mode, for narrowing a failing comparison): None keeps every value in
    fp64; bf16_round rounds where the bf16 device path stores an intermediate: h (gate|up, from
    which the backward works) and w * A (what the down projection reads; A itself is formed from
    the unrounded h). Then Y[t] = sum_j down[e_j] . rnd(w[t,j] * A_j), the same sum with the
    routing weight moved inside the linear map.

    Returns dict(Y [T,H], h [T,k,2I], A [T,k,I], wA [T,k,I]) in float64 (h and wA as rounded)."""
    rnd = _keep if rnd is None else rnd
    x = np.asarray(x, F64)
    Wgu = np.asarray(w_gate_up, F64)
    Wd = np.asarray(w_down, F64)
    w = np.asarray(topk_w, F64)
    T, H = x.shape
    E, I2, _ = Wgu.shape
    I = I2 // 2
    k = topk_idx.shape[1]
    Y = np.zeros((T, H))
    h = np.zeros((T, k, I2))
    A = np.zeros((T, k, I))
    wA = np.zeros((T, k, I))
    for e in range(E):
        rows, slots = _expert_rows(topk_idx, e)
        if rows.size == 0:
            continue
        he = x[rows] @ Wgu[e].T
        gate, up = he[:, :I], he[:, I:]
        Ae = silu(gate) * up
        we = w[rows, slots][:, None]
        if rnd is _keep:
            Y[rows] += we * (Ae @ Wd[e].T)
            wAe = we * Ae
        else:
            wAe = np.asarray(rnd(we * Ae), F64)
            Y[rows] += wAe @ Wd[e].T
        h[rows, slots] = rnd(he)
        A[rows, slots] = Ae
        wA[rows, slots] = wAe
    return {"Y": Y, "h": h, "A": A, "wA": wA}


def moe_backward(x, w_router, w_gate_up, w_down, topk_idx, topk_w, logits, dY, renorm=1,
                 dense_wgrad=False, rnd=None):
    """Gradients of L = sum(dY * Y) with the expert selection held fixed.

    gvec = down[e]^T dY[t]; dw_j = <gvec, A_j>; dA = w_j gvec;
    dgate = dA * up * silu'(gate); dup = dA * silu(gate);
    dlogit: renorm=1 -> w_j (dw_j - sum_i w_i dw_i) at the selected experts, 0 elsewhere;
            renorm=0 -> p_e (dw_e [e selected] - sum_i p_{e_i} dw_i) for every e;
    g_router = dlogit^T x; dx = sum_j gate_up[e_j]^T dh_j + dlogit . Wr.
    Only routed experts receive gradient (the news article's key differences).
    rnd (bf16-emulating mode, see moe_forward): the backward reads the rounded h (for A in dw and
    for the SwiGLU derivative), rounds dh where the device stores it (dx and the gate_up weight
    gradient read the rounded dh), and the down weight gradient reads the rounded w * A.
    Returns dict(dw, dh, dlogit, g_router, dx [, dW_gate_up, dW_down])."""
    x = np.asarray(x, F64)
    Wr = np.asarray(w_router, F64)
    Wgu = np.asarray(w_gate_up, F64)
    Wd = np.asarray(w_down, F64)
    w = np.asarray(topk_w, F64)
    dY = np.asarray(dY, F64)
    T, H = x.shape
    E, I2, _ = Wgu.shape
    I = I2 // 2
    k = topk_idx.shape[1]
    fwd = moe_forward(x, Wgu, Wd, topk_idx, w, rnd=rnd)
    rnd = _keep if rnd is None else rnd
    dw = np.zeros((T, k))
    dh = np.zeros((T, k, I2))
    dx = np.zeros((T, H))
    dWgu = np.zeros_like(Wgu) if dense_wgrad else None
    dWd = np.zeros_like(Wd) if dense_wgrad else None
    for e in range(E):
        rows, slots = _expert_rows(topk_idx, e)
        if rows.size == 0:
            continue
        he = fwd["h"][rows, slots]
        gate, up = he[:, :I], he[:, I:]
        # A from the h the backward reads (the rounded one in bf16-emulating mode)
        Ae = fwd["A"][rows, slots] if rnd is _keep else silu(gate) * up
        gvec = dY[rows] @ Wd[e]
        dw[rows, slots] = np.sum(gvec * Ae, axis=1)
        dA = w[rows, slots][:, None] * gvec
        dge = np.asarray(rnd(np.concatenate([dA * up * silu_grad(gate), dA * silu(gate)],
                                            axis=1)), F64)
        dh[rows, slots] = dge
        dx[rows] += dge @ Wgu[e]
        if dense_wgrad:
            dWgu[e] = dge.T @ x[rows]
            if rnd is _keep:
                dWd[e] = (w[rows, slots][:, None] * dY[rows]).T @ Ae
            else:
                dWd[e] = dY[rows].T @ fwd["wA"][rows, slots]
    dlogit = np.zeros((T, E))
    if renorm:
        s = np.sum(w * dw, axis=1, keepdims=True)
        for j in range(k):
            dlogit[np.arange(T), topk_idx[:, j]] = w[:, j] * (dw[:, j] - s[:, 0])
    else:
        l = np.asarray(logits, F64)
        p = np.exp(l - l.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        s = np.sum(w * dw, axis=1, keepdims=True)
        dsel = np.zeros((T, E))
        for j in range(k):
            dsel[np.arange(T), topk_idx[:, j]] = dw[:, j]
        dlogit = p * (dsel - s)
    g_router = dlogit.T @ x
    dx += dlogit @ Wr
    out = {"dw": dw, "dh": dh, "dlogit": dlogit, "g_router": g_router, "dx": dx,
           "Y": fwd["Y"], "h": fwd["h"], "A": fwd["A"]}
    if dense_wgrad:
        out["dW_gate_up"] = dWgu
        out["dW_down"] = dWd
    return out


def split_flat_index(f, E, I, H):
    """Flat index -> (tensor, e, r, c): tensor 0 = gate_up [E,2I,H], 1 = down [E,H,I]."""
    f = np.asarray(f, np.int64)
    Ngu = E * 2 * I * H
    gu = f < Ngu
    out_t = np.where(gu, 0, 1)
    fg = np.where(gu, f, 0)
    fd = np.where(gu, 0, f - Ngu)
    e = np.where(gu, fg // (2 * I * H), fd // (H * I))
    r = np.where(gu, (fg // H) % (2 * I), (fd // I) % H)
    c = np.where(gu, fg % H, fd % I)
    return out_t, e, r, c


def masked_expert_grad(act_idx, x, w_gate_up, w_down, topk_idx, topk_w, dY, experts=None,
                       rnd=None):
    """Expert weight gradients at the active flat indices only (the USAF sparse backward):

    gate_up entry (e, r, c): sum over tokens routed to e of dh[t, r] * x[t, c]
    down entry (e, r, c):    sum over tokens routed to e of w[t] * dY[t, r] * A[t, c]
    Experts with no routed token give 0. If `experts` is given, only actives of those experts are
    computed and the others are returned as NaN (for sampled checks of large layers).
    rnd (bf16-emulating mode, see moe_forward and moe_backward): dh from the rounded h, then
    rounded; the down entries read the rounded w * A."""
    rnd = _keep if rnd is None else rnd
    x = np.asarray(x, F64)
    Wgu = np.asarray(w_gate_up, F64)
    Wd = np.asarray(w_down, F64)
    w = np.asarray(topk_w, F64)
    dY = np.asarray(dY, F64)
    E, I2, H = Wgu.shape
    I = I2 // 2
    act_idx = np.asarray(act_idx, np.int64)
    tens, ee, rr, cc = split_flat_index(act_idx, E, I, H)
    g = np.full(act_idx.shape[0], np.nan)
    todo = range(E) if experts is None else experts
    for e in todo:
        sel = np.nonzero(ee == e)[0]
        if sel.size == 0:
            continue
        rows, slots = _expert_rows(topk_idx, e)
        if rows.size == 0:
            g[sel] = 0.0
            continue
        he_exact = x[rows] @ Wgu[e].T
        we = w[rows, slots][:, None]
        he = np.asarray(rnd(he_exact), F64)
        gate, up = he[:, :I], he[:, I:]
        Ae = silu(gate) * up
        gvec = dY[rows] @ Wd[e]
        dA = we * gvec
        dge = np.asarray(rnd(np.concatenate([dA * up * silu_grad(gate), dA * silu(gate)],
                                            axis=1)), F64)
        gu = sel[tens[sel] == 0]
        dn = sel[tens[sel] == 1]
        if gu.size:
            g[gu] = np.einsum("ta,ta->a", dge[:, rr[gu]], x[rows][:, cc[gu]])
        if dn.size:
            if rnd is _keep:
                wdy = we * dY[rows]
                g[dn] = np.einsum("ta,ta->a", wdy[:, rr[dn]], Ae[:, cc[dn]])
            else:
                # w * A from the unrounded h, rounded where the forward stores it
                ge, ue = he_exact[:, :I], he_exact[:, I:]
                wAe = np.asarray(rnd(we * silu(ge) * ue), F64)
                g[dn] = np.einsum("ta,ta->a", dY[rows][:, rr[dn]], wAe[:, cc[dn]])
    return g


# ----------------------------------------------------------------------------------------------
# SparseAdam (USAF README A100 operations table; torch.optim.SparseAdam's update rule)
# ----------------------------------------------------------------------------------------------

def sparse_adam(g, p, m, v, lr, beta1, beta2, eps, step):
    """One SparseAdam step over the given entries (every given entry counts as present):

    m <- b1 m + (1-b1) g; v <- b2 v + (1-b2) g^2;
    p <- p - lr * sqrt(1-b2^t)/(1-b1^t) * m / (sqrt(v) + eps).
    Evaluated in fp64 from fp32 inputs; returns fp32 (p, m, v)."""
    g = np.asarray(g, np.float32).astype(F64)
    p = np.asarray(p, np.float32).astype(F64)
    m = np.asarray(m, np.float32).astype(F64)
    v = np.asarray(v, np.float32).astype(F64)
    m2 = beta1 * m + (1.0 - beta1) * g
    v2 = beta2 * v + (1.0 - beta2) * g * g
    step_size = lr * np.sqrt(1.0 - beta2 ** step) / (1.0 - beta1 ** step)
    p2 = p - step_size * m2 / (np.sqrt(v2) + eps)
    return p2.astype(np.float32), m2.astype(np.float32), v2.astype(np.float32)


def bf16_round(a):
    """Nearest bf16 value of each fp32 value (ties to even), returned as float32."""
    a = np.ascontiguousarray(np.asarray(a, np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) >> 16
    return (u.astype(np.uint32) << 16).view(np.float32).reshape(a.shape)


# ----------------------------------------------------------------------------------------------
# Importance selection and RigL (USAF README: "Not all weights matter", "Sparsity adapts")
# ----------------------------------------------------------------------------------------------

def abs_key(a):
    """|a| as the fp32 bit pattern with the sign cleared (orders like |a| for finite values)."""
    return np.ascontiguousarray(np.asarray(a, np.float32)).view(np.uint32) & np.uint32(0x7FFFFFFF)


def importance_select(g, K):
    """Sort all N entries by (|g| descending, index ascending); the first K, sorted by index."""
    key = abs_key(g).astype(np.int64)
    idx = np.arange(key.size, dtype=np.int64)
    order = np.lexsort((idx, -key))
    return np.sort(order[:K])


def importance_select_threshold(g, K):
    """The same set as importance_select, by its threshold form (for large N): with tau the K-th
    largest key, all entries with key > tau plus the lowest-index entries with key == tau."""
    key = abs_key(g)
    n = key.size
    tau = np.partition(key, n - K)[n - K]
    above = np.nonzero(key > tau)[0]
    eq = np.nonzero(key == tau)[0]
    need = K - above.size
    return np.sort(np.concatenate([above, eq[:need]])).astype(np.int64)


def rigl_swap(act_idx, p, m, v, g, D, dense_weight_at, grow_by="sort"):
    """RigL drop/grow with a fixed count D:

    drop = the D entries of the active set S with the smallest |p| (ties: lower flat index first);
    grow = the D entries outside S with the largest |g| (ties: lower flat index first);
    S' = (S minus drop) union grow, sorted. Kept entries keep (p, m, v); grown entries get
    p = dense weight value (dense_weight_at(idx) -> float32 array), m = v = 0.
    grow_by="threshold" finds the same grow set by its threshold form (for large N): with tau the
    D-th largest key outside S, every outside entry with key > tau plus the lowest-index outside
    entries with key == tau.
    Returns (new_idx, p', m', v', n_swapped)."""
    act_idx = np.asarray(act_idx, np.int64)
    K = act_idx.size
    pk = abs_key(p).astype(np.int64)
    pos = np.arange(K)
    drop_order = np.lexsort((act_idx, pk))
    drop_pos = np.sort(drop_order[:D])
    keep_mask = np.ones(K, dtype=bool)
    keep_mask[drop_pos] = False
    gk = abs_key(g).astype(np.int64)
    N = gk.size
    inactive = np.ones(N, dtype=bool)
    inactive[act_idx] = False
    if grow_by == "sort":
        cand = np.nonzero(inactive)[0]
        grow_order = np.lexsort((cand, -gk[cand]))
        grow = np.sort(cand[grow_order[:D]])
    else:
        outk = np.where(inactive, gk, -1)  # entries of S can never be grown
        tau = np.partition(outk, N - D)[N - D] if D > 0 else np.iinfo(np.int64).max
        above = np.nonzero(outk > tau)[0]
        eq = np.nonzero(outk == tau)[0]
        grow = np.sort(np.concatenate([above, eq[:D - above.size]])).astype(np.int64)
    kept = act_idx[keep_mask]
    new_idx = np.concatenate([kept, grow])
    p_new = np.concatenate([np.asarray(p, np.float32)[keep_mask],
                            np.asarray(dense_weight_at(grow), np.float32)])
    m_new = np.concatenate([np.asarray(m, np.float32)[keep_mask], np.zeros(D, np.float32)])
    v_new = np.concatenate([np.asarray(v, np.float32)[keep_mask], np.zeros(D, np.float32)])
    order = np.argsort(new_idx, kind="stable")
    n_swapped = int(K - np.intersect1d(act_idx, new_idx).size)
    del pos
    return new_idx[order], p_new[order], m_new[order], v_new[order], n_swapped


def reselect_full(act_idx, p, m, v, g, K_new, dense_weight_at):
    """Full reselection by re-ranking (USAF README, "Sparsity adapts": the active set is chosen
    again from fresh gradient magnitudes; the README reports about 92% turnover at the first
    reselections, which a full re-rank allows and a fixed-fraction swap does not):

    S' = the K_new entries with the largest |g| (ties: lower flat index first), sorted. Entries in
    both S and S' keep (p, m, v); entries new to S' get p = dense weight value, m = v = 0.
    Returns (new_idx, p', m', v', n_kept)."""
    act_idx = np.asarray(act_idx, np.int64)
    new_idx = importance_select(g, K_new)
    p = np.asarray(p, np.float32)
    m = np.asarray(m, np.float32)
    v = np.asarray(v, np.float32)
    old_pos = {int(f): i for i, f in enumerate(act_idx)}
    p_new = np.empty(K_new, np.float32)
    m_new = np.zeros(K_new, np.float32)
    v_new = np.zeros(K_new, np.float32)
    fresh = [t for t, f in enumerate(new_idx) if int(f) not in old_pos]
    kept = [t for t, f in enumerate(new_idx) if int(f) in old_pos]
    for t in kept:
        i = old_pos[int(new_idx[t])]
        p_new[t], m_new[t], v_new[t] = p[i], m[i], v[i]
    if fresh:
        fresh = np.asarray(fresh, np.int64)
        p_new[fresh] = np.asarray(dense_weight_at(new_idx[fresh]), np.float32)
    return new_idx, p_new, m_new, v_new, len(kept)

