"""Training loop around the layer calls: a stack of USAF MoE layers, several micro-batches per
step, a cosine learning-rate schedule, and reselection of the active sets every few steps.

The schedule and cadence follow the USAF README: learning rate peaking at LR_PEAK with cosine
decay, MICROBATCH micro-batches accumulated per optimizer step, the active set reselected every
RESELECT_EVERY steps from an accumulated dense gradient (RigL drop/grow, or a full re-rank), and
steps with a non-finite gradient skipped and counted. Every tensor operation on the path is one of
the library's calls; this module sequences them and keeps the counters.
"""
from __future__ import annotations

import math

import torch

from . import binding as B
from . import dist_select as DS
from .layer import allreduce_dense_grad


def cosine_lr(step: int, total_steps: int, peak: float, warmup_steps: int = 0,
              floor: float = 0.0) -> float:
    """Learning rate of optimizer step `step` (counted from 1): linear warm-up to `peak` over
    `warmup_steps`, then cosine decay from `peak` to `floor` at `total_steps`."""
    if warmup_steps > 0 and step <= warmup_steps:
        return peak * step / warmup_steps
    span = max(1, total_steps - warmup_steps)
    prog = min(max((step - warmup_steps) / span, 0.0), 1.0)
    return floor + 0.5 * (peak - floor) * (1.0 + math.cos(math.pi * prog))


def reselect_due(step: int, every: int) -> bool:
    """Whether optimizer step `step` (from 1) ends with a reselection of the active sets."""
    return every > 0 and step % every == 0


class StackTrainer:
    """Steps a stack of MoELayer objects: the output y of layer i is the input x of layer i+1, and
    the input gradient dx of layer i+1 is the upstream gradient dy of layer i."""

    def __init__(self, layers, total_steps, lr_peak=2e-4, warmup_steps=0, reselect_every=50,
                 reselect="rigl", drop_frac=0.3, skip_nonfinite=True, dense_exchange="allreduce"):
        """dense_exchange (data parallel only): how the replicas agree on the importance phase's
        gradient. "allreduce": every rank sums the whole dense gradient and selects alone;
        "reduce_scatter": every rank sums one part and the selection runs over the parts
        (dist_select), moving half the bytes and ranking 1/world of the entries per rank."""
        if reselect not in ("rigl", "full"):
            raise ValueError("reselect must be 'rigl' or 'full'")
        if dense_exchange not in ("allreduce", "reduce_scatter"):
            raise ValueError("dense_exchange must be 'allreduce' or 'reduce_scatter'")
        self.dense_exchange = dense_exchange
        self.layers = list(layers)
        self.total_steps = total_steps
        self.lr_peak, self.warmup_steps = lr_peak, warmup_steps
        self.reselect_every, self.reselect = reselect_every, reselect
        self.drop_frac = drop_frac
        self.skip_nonfinite = skip_nonfinite
        self.step_no = 0
        self.history = []  # per step: lr, status words, turnover (device tensors until read)
        self._g_dense = [None] * len(self.layers)

    # ------------------------------------------------------------------ one micro-batch
    def _forward(self, x):
        inputs = []
        for L in self.layers:
            inputs.append(x)
            L.route(x)
            x = L.forward(x)
        return inputs

    def _backward(self, inputs, dy, first, dense):
        for i in reversed(range(len(self.layers))):
            L = self.layers[i]
            x = inputs[i]
            dx = L.dx if i > 0 else None  # the bottom layer's input needs no gradient
            L.backward_into(x, dy, accumulate=0 if first else 1, dx=dx)
            if dense:
                # the importance phase's dense gradient of this micro-batch, accumulated, from
                # the dh and permuted dy the sparse call just left in the layer's workspace
                if self._g_dense[i] is None:
                    self._g_dense[i] = torch.zeros(L.N, device=L.dev)
                B.moe_wgrad_dense(L.s, L.rt, L.x_perm, L.wa, self._g_dense[i], L.ws_bwd,
                                  accumulate=1, dev_status=L.status)
            dy = L.dx

    # ------------------------------------------------------------------ one optimizer step
    def step(self, x_micro, dy_micro):
        """One optimizer step over the micro-batches: x_micro[j] [T,H] is micro-batch j's input
        to the bottom layer, dy_micro[j] [T,H] the gradient at the top layer's output."""
        if len(x_micro) != len(dy_micro) or not x_micro:
            raise ValueError("need the same number (>= 1) of inputs and upstream gradients")
        self.step_no += 1
        n = self.step_no
        lr = cosine_lr(n, self.total_steps, self.lr_peak, self.warmup_steps)
        dense = reselect_due(n, self.reselect_every)
        for i, L in enumerate(self.layers):
            L.status = L.status2[L.step_count % 2:L.step_count % 2 + 1]
            L.status.zero_()
        for j, (x, dy) in enumerate(zip(x_micro, dy_micro)):
            inputs = self._forward(x)
            self._backward(inputs, dy, first=(j == 0), dense=dense)
        status = []
        for L in self.layers:
            L.lr = lr
            L.optimizer_step(skip_if_nonfinite=1 if self.skip_nonfinite else 0)
            L.wait_optimizer()  # the expert update's status bits are in before they are kept
            status.append(L.status.clone())
        rec = {"step": n, "lr": lr, "status": status, "turnover": None,
               "expert_count": [L.rt.expert_count.clone() for L in self.layers]}
        if dense:
            rec["turnover"] = self._reselect()
        self.history.append(rec)
        return rec

    def _reselect(self):
        """New active sets from the accumulated dense gradients; state carried by the library."""
        turn = []
        for i, L in enumerate(self.layers):
            L.wait_optimizer()
            g = self._g_dense[i]
            K = L.K
            new = torch.empty(K, dtype=torch.int64, device=L.dev)
            p, m, v = (torch.empty(K, device=L.dev) for _ in range(3))
            cnt = torch.zeros(1, dtype=torch.int64, device=L.dev)
            if L.group is not None and self.dense_exchange == "reduce_scatter":
                turn.append(self._reselect_parts(L, g, new, p, m, v, cnt))
                L.set_active(new, p, m, v)
                g.zero_()
                continue
            if L.group is not None:
                # data parallel: rank the whole batch's gradient, so the replicas' sets agree
                allreduce_dense_grad(g, L.group)
            if self.reselect == "rigl":
                D = int(self.drop_frac * K)
                B.rigl_swap(g, L.act, D, L.p, L.m, L.v, L.w_gate_up, L.N_gu, L.w_down, new, p, m,
                            v, cnt)
                turn.append(cnt)  # entries swapped
            else:
                B.reselect_full(g, K, L.act, L.p, L.m, L.v, L.w_gate_up, L.N_gu, L.w_down, new,
                                p, m, v, cnt)
                turn.append(K - cnt)  # entries not kept
            L.set_active(new, p, m, v)
            g.zero_()
        return turn

    def _reselect_parts(self, L, g, new, p, m, v, cnt):
        """Reselection with the dense gradient reduce-scattered: each rank holds the batch's sum
        over one part of the entries; the new set (or RigL's grow set) is selected over the parts
        of all ranks, and every rank carries its state with the library as on one GPU."""
        part, lo = DS.reduce_scatter_part(g, L.group)
        comm, ops = DS.TorchComm(L.group), DS.LibShardOps()
        if self.reselect == "rigl":
            D = int(self.drop_frac * L.K)
            excl = DS.part_bitmap(L.act, lo, part.numel())
            grown = DS.topk_over_parts([(part, lo, excl)], D, ops, comm)
            B.rigl_apply(L.act, D, grown, L.p, L.m, L.v, L.w_gate_up, L.N_gu, L.w_down, new, p,
                         m, v, cnt)
            return cnt
        new.copy_(DS.topk_over_parts([(part, lo, None)], L.K, ops, comm))
        B.reselect_carry(new, L.act, L.p, L.m, L.v, L.w_gate_up, L.N_gu, L.w_down, p, m, v, cnt)
        return L.K - cnt

    # ------------------------------------------------------------------ metrics
    def metrics(self):
        """Host view of the recorded steps (synchronises): learning rate, whether the step was
        skipped for a non-finite gradient, turnover fraction at reselections, and the load
        balance (largest expert count over the mean) per layer."""
        torch.cuda.synchronize()
        out = []
        for r in self.history:
            skipped = [bool(int(s.item()) & 1) for s in r["status"]]
            turnover = None
            if r["turnover"] is not None:
                turnover = [int(t.item()) / L.K for t, L in zip(r["turnover"], self.layers)]
            balance = [float(c.max().item()) / max(1e-9, float(c.float().mean().item()))
                       for c in r["expert_count"]]
            out.append({"step": r["step"], "lr": r["lr"], "skipped": skipped,
                        "turnover": turnover, "load_balance": balance})
        return out
