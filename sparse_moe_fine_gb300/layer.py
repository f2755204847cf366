"""One USAF MoE layer held on the GPU: weights, router, active set and its SparseAdam state, and
the buffers of a train step. Each method is a sequence of C-ABI calls (see include/usaf.h); this
module only allocates with PyTorch and passes pointers.

A train step is: route (router logits, top-k, permutation) -> grouped SwiGLU forward -> sparse
backward (router gradient, input gradient, expert gradients at the active set) -> SparseAdam on
the active expert entries -> SparseAdam on the router (USAF README: the router is trained in
full, expert weights at a 0.5% active set, both under SparseAdam).

Data parallel (the README's DataParallel mode): every rank holds the same weights and active set
and runs the step on its own tokens; before the optimizer, one all-reduce sums the compact
gradients (K active expert entries and the E*H router entries) and one takes the maximum of the
status words, so every replica applies the same update or skips the same step.
"""
from __future__ import annotations

import math

import torch

from . import binding as B


STATUS_BITS = 4  # NONFINITE, SELECT_EXACT_PATH, TIMEOUT, BAD_INDEX (usaf.h USAF_DEV_*)


def allreduce_grads(g_act, g_router, status, group=None):
    """Sum the compact gradients over the ranks of `group` and OR their status words, in place, on
    the current stream. The loss is a sum over tokens, so the sum of the ranks' gradients is the
    gradient of the whole batch; the OR makes a non-finite value seen by any rank skip the step on
    every rank. (The OR is taken bit by bit as a maximum, which every backend reduces.)"""
    import torch.distributed as dist
    dist.all_reduce(g_act, op=dist.ReduceOp.SUM, group=group)
    dist.all_reduce(g_router, op=dist.ReduceOp.SUM, group=group)
    bits = torch.stack([(status >> b) & 1 for b in range(STATUS_BITS)])
    dist.all_reduce(bits, op=dist.ReduceOp.MAX, group=group)
    status.copy_(sum(bits[b] << b for b in range(STATUS_BITS)))


def allreduce_dense_grad(g_dense, group=None):
    """Sum the accumulated dense expert gradient of the importance phase over the ranks of
    `group`, in place, on the current stream. Each rank accumulated the gradient of its own
    tokens; the sum is the whole batch's gradient, so every replica then ranks the same |g| and
    installs the same active set (the compact gradients of later steps index the same weights
    on every rank)."""
    import torch.distributed as dist
    dist.all_reduce(g_dense, op=dist.ReduceOp.SUM, group=group)


class MoELayer:
    def __init__(self, T, H, E, k, I, w_gate_up, w_down, w_router, act_idx, lr=1e-4,
                 betas=(0.9, 0.999), eps=1e-8, renorm=1, device="cuda", group=None,
                 dense_density=0.015):
        self.dev = torch.device(device)
        self.s = B.shape(T, H, E, k, I)
        self.T, self.H, self.E, self.k, self.I = T, H, E, k, I
        self.dtype = w_gate_up.dtype
        self.dt = B.BF16 if self.dtype == torch.bfloat16 else B.F32
        self.w_gate_up = w_gate_up.contiguous()
        self.w_down = w_down.contiguous()
        self.w_router = w_router.contiguous().float()
        self.N_gu = E * 2 * I * H
        self.N = E * 3 * I * H
        self.lr, self.betas, self.eps, self.renorm = lr, betas, eps, renorm
        self.group = group  # data-parallel process group (None: one replica)
        # experts whose active entries are at least this fraction of their weights get their
        # masked gradient from dense tensor-core tiles (usaf_masked_plan_build)
        self.dense_density = dense_density
        self.step_count = 0
        d = self.dev
        cap = B.routed_rows_capacity(self.s)
        self.rt = B.Routing.empty(self.s, d)
        self.logits = torch.empty(T, E, device=d)
        # per-row activations are feature-major: [features, R_cap]
        self.x_perm = torch.empty(H, cap, dtype=self.dtype, device=d)
        self.h = torch.empty(2 * I, cap, dtype=self.dtype, device=d)
        self.wa = torch.empty(I, cap, dtype=self.dtype, device=d)
        self.y = torch.empty(T, H, dtype=self.dtype, device=d)
        self.dx = torch.empty(T, H, dtype=self.dtype, device=d)
        self.g_router = torch.empty(E, H, device=d)
        # one status word per step parity: the expert update of step i may still be reading its
        # word on the side stream while step i+1 clears and fills the other one
        self.status2 = torch.zeros(2, dtype=torch.int32, device=d)
        self.status = self.status2[0:1]
        # the expert SparseAdam update runs on a side stream, overlapping the next step's routing
        self.side = torch.cuda.Stream(device=d)
        # the routing graph is replayed on a stream of the greatest priority, so that its blocks
        # are placed ahead of the expert update's (which runs beside it at the default priority)
        self.hp = torch.cuda.Stream(device=d, priority=torch.cuda.Stream.priority_range()[1])
        self.ev_bwd = torch.cuda.Event()
        # the update is issued in two parts, gate_up's entries first: ev_gu marks that part (the
        # forward's gate_up GEMM waits for it), ev_opt the whole update (its down GEMM waits)
        self.ev_gu = torch.cuda.Event()
        self.ev_opt = torch.cuda.Event()
        for e in (self.ev_gu, self.ev_opt):  # create the events now: captured waits need them
            e.record(self.side)
        self.pending_opt = False
        self.replayed_kernels = 0  # library kernels run by graph replays (graphed_train_step)
        self.ws_route = torch.empty(B.route_topk_workspace_size(self.s), dtype=torch.uint8,
                                    device=d)
        self.ws_fwd = torch.empty(B.moe_fwd_workspace_size(self.s, self.dt), dtype=torch.uint8,
                                  device=d)
        # router SparseAdam state (dense over all E*H entries)
        self.r_p = self.w_router.reshape(-1).clone()
        self.r_m = torch.zeros_like(self.r_p)
        self.r_v = torch.zeros_like(self.r_p)
        self.set_active(act_idx)

    # ------------------------------------------------------------------ active set
    def set_active(self, act_idx, p=None, m=None, v=None):
        """Install a sorted active set; fresh state starts from the weight values. The set is
        checked on the device (usaf_validate_active: ascending, no repeats, inside [0, N)) and
        refused with ValueError before anything reads it; this waits for the device once."""
        act = act_idx.to(self.dev, torch.int64).contiguous()
        chk = torch.zeros(1, dtype=torch.int32, device=self.dev)
        B.validate_active(act, self.N, chk)
        if int(chk.item()) & B.DEV_BAD_INDEX:
            raise ValueError("active set is not strictly ascending inside [0, N)")
        self.act = act
        K = self.act.numel()
        self.K = K
        # the first part of the split update: every gate_up entry, rounded up to four entries so
        # that the second part's state starts on a 16-byte boundary
        self.k_split = min(K, -(-int((act < self.N_gu).sum().item()) // 4) * 4)
        if p is None:
            flat_gu = self.w_gate_up.reshape(-1)
            flat_d = self.w_down.reshape(-1)
            gu = self.act < self.N_gu
            p = torch.empty(K, device=self.dev)
            p[gu] = flat_gu[self.act[gu]].float()
            p[~gu] = flat_d[self.act[~gu] - self.N_gu].float()
            m = torch.zeros(K, device=self.dev)
            v = torch.zeros(K, device=self.dev)
        self.p, self.m, self.v = p, m, v
        # the masked-gradient plan of this set; its expert count is read once, here
        self.plan = torch.empty(max(1, B.masked_plan_size(self.s)), dtype=torch.uint8,
                                device=self.dev)
        if self.dt == B.BF16 and K > 0:
            B.masked_plan_build(self.s, self.act, self.dense_density, self.plan)
            self.n_dense = B.masked_plan_count(self.plan)
        else:
            self.n_dense = 0
        self.g_act = torch.empty(K, device=self.dev)
        self.ws_bwd = torch.empty(B.moe_bwd_workspace_size(self.s, self.dt, K),
                                  dtype=torch.uint8, device=self.dev)
        self._graphs = {}  # captured steps hold the old active set's pointers

    # ------------------------------------------------------------------ checkpoint / resume
    def checkpoint(self) -> dict:
        """The layer's whole training state as CPU tensors and host scalars: expert and router
        weights, the active set with its fp32 master copy and Adam moments, the router's Adam
        state, the step count and the optimizer settings. Waits for the last update. A layer
        rebuilt from it (from_checkpoint) continues exactly as this one would."""
        self.wait_optimizer()
        torch.cuda.current_stream(self.dev).synchronize()
        cpu = lambda t: t.detach().to("cpu", copy=True)
        return {"shape": (self.T, self.H, self.E, self.k, self.I),
                "w_gate_up": cpu(self.w_gate_up), "w_down": cpu(self.w_down),
                "w_router": cpu(self.w_router), "act": cpu(self.act), "p": cpu(self.p),
                "m": cpu(self.m), "v": cpu(self.v), "r_p": cpu(self.r_p), "r_m": cpu(self.r_m),
                "r_v": cpu(self.r_v), "step_count": self.step_count, "lr": self.lr,
                "betas": tuple(self.betas), "eps": self.eps, "renorm": self.renorm,
                "dense_density": self.dense_density}

    @classmethod
    def from_checkpoint(cls, ck: dict, device="cuda", group=None) -> "MoELayer":
        T, H, E, k, I = ck["shape"]
        d = torch.device(device)
        L = cls(T, H, E, k, I, ck["w_gate_up"].to(d), ck["w_down"].to(d), ck["w_router"].to(d),
                ck["act"].to(d), lr=ck["lr"], betas=ck["betas"], eps=ck["eps"],
                renorm=ck["renorm"], device=d, group=group,
                dense_density=ck.get("dense_density", 0.015))
        L.set_active(ck["act"].to(d), ck["p"].to(d), ck["m"].to(d), ck["v"].to(d))
        L.r_p.copy_(ck["r_p"])
        L.r_m.copy_(ck["r_m"])
        L.r_v.copy_(ck["r_v"])
        L.step_count = int(ck["step_count"])
        return L

    # ------------------------------------------------------------------ the step
    def _check_tokens(self, **ts):
        """The library reads and writes [T, H] token tensors through bare pointers, so their
        shape, dtype and layout are checked here, before any launch."""
        for name, t in ts.items():
            if t is None:
                continue
            if tuple(t.shape) != (self.T, self.H) or t.dtype != self.dtype:
                raise ValueError(f"{name}: expected a [{self.T}, {self.H}] {self.dtype} tensor, "
                                 f"got {list(t.shape)} {t.dtype}")
            if not (t.is_cuda and t.is_contiguous()):
                raise ValueError(f"{name}: expected a contiguous CUDA tensor")

    def route(self, x, stream=None):
        self._check_tokens(x=x)
        B.route_topk(self.s, x, self.w_router, self.rt, logits_out=self.logits,
                     renorm=self.renorm, dev_status=self.status, ws=self.ws_route, stream=stream)

    def _main(self, stream):
        return torch.cuda.current_stream(self.dev) if stream is None else stream

    def wait_optimizer(self, stream=None):
        """Make `stream` wait for the last expert update (the weights it writes)."""
        if self.pending_opt:
            self._main(stream).wait_event(self.ev_opt)
            self.pending_opt = False

    def forward(self, x, stream=None, y=None):
        """The token gather overlaps the last expert update; the GEMMs wait for it."""
        y = self.y if y is None else y
        self._check_tokens(x=x, y=y)
        gu, dn = (self.ev_gu, self.ev_opt) if self.pending_opt else (None, None)
        B.moe_fwd(self.s, x, self.w_gate_up, self.w_down, self.rt, self.x_perm, self.h, self.wa,
                  y, ws=self.ws_fwd, stream=stream, weights_ready=gu, down_ready=dn,
                  dev_status=self.status)
        self.pending_opt = False  # the stream is ordered after the update from here on
        return y

    def backward(self, x, dy, want_dx=True, stream=None, dx=None):
        dx = self.dx if dx is None else dx
        self._check_tokens(x=x, dy=dy, dx=dx)
        self.backward_into(x, dy, accumulate=0, dx=dx if want_dx else None, stream=stream)

    def backward_into(self, x, dy, accumulate=0, dx=None, stream=None, dev_status=None):
        """The sparse backward with this set's masked-gradient plan; accumulate = 1 adds into
        g_act and g_router (micro-batches)."""
        B.moe_bwd_sparse_planned(self.s, x, self.w_router, self.w_gate_up, self.w_down, self.rt,
                                 self.x_perm, self.h, self.wa, dy, self.act, self.g_act,
                                 self.g_router, plan=self.plan, n_dense=self.n_dense,
                                 accumulate=accumulate, dx=dx, logits=self.logits,
                                 renorm=self.renorm,
                                 dev_status=self.status if dev_status is None else dev_status,
                                 ws=self.ws_bwd, stream=stream)

    def optimizer_step(self, stream=None, skip_if_nonfinite=1):
        """Router update on the calling stream (the next routing reads it); expert update on the
        side stream, which the next forward waits for."""
        self.step_count += 1
        b1, b2 = self.betas
        main = self._main(stream)
        if self.group is not None:
            with torch.cuda.stream(main):
                allreduce_grads(self.g_act, self.g_router, self.status, self.group)
        self.ev_bwd.record(main)
        self.side.wait_event(self.ev_bwd)
        # one scan of the whole gradient, then the update in two parts that only check the status
        # word (a non-finite entry anywhere skips both): gate_up's entries, then down_proj's, so
        # that the next forward's gate_up GEMM waits only for the first part
        if skip_if_nonfinite:
            B.scan_nonfinite(self.g_act, self.status, stream=self.side)
        skip = 2 if skip_if_nonfinite else 0
        for lo, hi, ev in ((0, self.k_split, self.ev_gu), (self.k_split, self.K, self.ev_opt)):
            if hi > lo:
                B.sparse_adam_step(self.act[lo:hi], self.g_act[lo:hi], self.p[lo:hi],
                                   self.m[lo:hi], self.v[lo:hi], self.w_gate_up, self.N_gu,
                                   self.w_down, self.lr, b1, b2, self.eps, self.step_count, skip,
                                   self.status, stream=self.side)
            ev.record(self.side)
        self.pending_opt = True
        B.sparse_adam_step(None, self.g_router, self.r_p, self.r_m, self.r_v, self.w_router,
                           self.E * self.H, None, self.lr, b1, b2, self.eps, self.step_count,
                           skip_if_nonfinite, self.status, stream=main)

    def train_step(self, x, dy, stream=None, y=None, dx=None):
        """route -> forward -> sparse backward -> SparseAdam (experts, router). y and dx may name
        other output buffers than the layer's own."""
        # per-step non-finite flag (a non-finite gradient skips this step), alternating words;
        # cleared on the step's own stream, ahead of the kernels that set its bits
        self.status = self.status2[self.step_count % 2:self.step_count % 2 + 1]
        with torch.cuda.stream(self._main(stream)):
            self.status.zero_()
        self.route(x, stream)
        y = self.forward(x, stream, y=y)
        self.backward(x, dy, stream=stream, dx=dx)
        self.optimizer_step(stream)
        return y, (self.dx if dx is None else dx)

    def graphed_train_step(self, x, dy, stream=None):
        """train_step with the routing and the forward + sparse backward replayed from CUDA graphs,
        captured on first use for these x and dy buffers (one pair per status-word parity), so
        their dependent launches run without per-launch gaps. The expert update of the previous
        step overlaps the routing and token-gather graph; the gate_up GEMM's graph waits for the
        update's gate_up part only, and the rest of the step's graph for its down_proj part. The two SparseAdam
        updates stay ordinary launches, since their step sizes change every step. Outputs are
        the layer's own y and dx buffers. One graph pair is kept per distinct (x, dy) buffer pair
        and parity, so a caller cycles through a fixed set of input buffers."""
        self._check_tokens(x=x, dy=dy)
        main = self._main(stream)
        par = self.step_count % 2
        key = (x.data_ptr(), dy.data_ptr(), par)
        if key not in self._graphs:
            self._graphs[key] = self._capture(x, dy, par, main)
        g_route, g_up, g_body, n_kernels = self._graphs[key]
        self.status = self.status2[par:par + 1]
        with torch.cuda.stream(main):
            # routing and the token gather, beside the last expert update, at high priority
            self.hp.wait_stream(main)
            with torch.cuda.stream(self.hp):
                g_route.replay()
            main.wait_stream(self.hp)
            if self.pending_opt:
                main.wait_event(self.ev_gu)
            g_up.replay()     # the gate_up GEMM, beside the update's down_proj part
            if self.pending_opt:
                main.wait_event(self.ev_opt)
            g_body.replay()
        self.pending_opt = False
        self.replayed_kernels += n_kernels
        self.optimizer_step(main)
        return self.y, self.dx

    def _capture(self, x, dy, par, main):
        status = self.status2[par:par + 1]
        cs = torch.cuda.Stream(device=self.dev)
        cs.wait_stream(main)
        g_route, g_up, g_body = (torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(),
                                 torch.cuda.CUDAGraph())
        n0 = B.launch_count()
        fwd = lambda stages: B.moe_fwd_stage(self.s, x, self.w_gate_up, self.w_down, self.rt,
                                             self.x_perm, self.h, self.wa, self.y, stages,
                                             self.ws_fwd, stream=cs, dev_status=status)
        # three graphs, so that the replays can wait for the expert update's two parts between
        # them: routing + token gather | gate_up GEMM | down GEMM + combine + sparse backward
        with torch.cuda.graph(g_route, stream=cs):
            status.zero_()
            B.route_topk(self.s, x, self.w_router, self.rt, logits_out=self.logits,
                         renorm=self.renorm, dev_status=status, ws=self.ws_route, stream=cs)
            fwd(B.FWD_GATHER)
        with torch.cuda.graph(g_up, stream=cs):
            fwd(B.FWD_GATE_UP)
        with torch.cuda.graph(g_body, stream=cs):
            fwd(B.FWD_DOWN)
            self.backward_into(x, dy, accumulate=0, dx=self.dx, stream=cs, dev_status=status)
        main.wait_stream(cs)
        return g_route, g_up, g_body, B.launch_count() - n0  # library kernels in the graphs

    def train_step_host(self, x_host, dy_host, y_host, dx_host, x_dev, dy_dev, stream=None):
        """The same step fed from (pinned) host memory: copy x and dy in, run, copy y and dx out,
        every copy on the step's stream."""
        main = self._main(stream)
        with torch.cuda.stream(main):
            x_dev.copy_(x_host, non_blocking=True)
            dy_dev.copy_(dy_host, non_blocking=True)
        self.train_step(x_dev, dy_dev, main)
        with torch.cuda.stream(main):
            y_host.copy_(self.y, non_blocking=True)
            dx_host.copy_(self.dx, non_blocking=True)


class HostStepper:
    """Train steps fed from pinned host memory with the copies overlapped with compute: a step's
    x and dY are copied in on one copy stream while the previous step computes, and its y and dx
    are copied out on another while the next step computes. Two sets of device buffers alternate;
    every step still moves its own inputs in and its own outputs out."""

    def __init__(self, layer):
        self.L = layer
        d = layer.dev
        shape = (layer.T, layer.H)
        mk = lambda: [torch.empty(shape, dtype=layer.dtype, device=d) for _ in range(2)]
        self.xd, self.dyd, self.yd, self.dxd = mk(), mk(), mk(), mk()
        self.h2d = torch.cuda.Stream(device=d)
        self.d2h = torch.cuda.Stream(device=d)
        ev = lambda: [torch.cuda.Event() for _ in range(2)]
        self.in_ready, self.computed, self.out_done = ev(), ev(), ev()
        self.used = [False, False]
        self.i = 0

    def step(self, x_host, dy_host, y_host, dx_host, stream=None):
        L = self.L
        main = L._main(stream)
        b = self.i % 2
        if self.used[b]:
            self.h2d.wait_event(self.computed[b])  # the step two back has read this input pair
        with torch.cuda.stream(self.h2d):
            self.xd[b].copy_(x_host, non_blocking=True)
            self.dyd[b].copy_(dy_host, non_blocking=True)
            self.in_ready[b].record(self.h2d)
        main.wait_event(self.in_ready[b])
        if self.used[b]:
            main.wait_event(self.out_done[b])  # its outputs are out before they are overwritten
        L.train_step(self.xd[b], self.dyd[b], stream=main, y=self.yd[b], dx=self.dxd[b])
        self.computed[b].record(main)
        self.d2h.wait_event(self.computed[b])
        with torch.cuda.stream(self.d2h):
            y_host.copy_(self.yd[b], non_blocking=True)
            dx_host.copy_(self.dxd[b], non_blocking=True)
            self.out_done[b].record(self.d2h)
        self.used[b] = True
        self.i += 1

    def finish(self, stream=None):
        """Make `stream` wait for the last outputs on the host and the last optimizer update."""
        main = self.L._main(stream)
        if self.i:
            main.wait_event(self.out_done[(self.i - 1) % 2])
        self.L.wait_optimizer(main)


def active_count(N: int, frac: float = 0.005) -> int:
    return int(math.ceil(frac * N))
