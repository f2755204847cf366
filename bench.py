"""Benchmark of the USAF MoE-layer train step on GB300.

A step is one pass of the whole hot path over one batch: route (router logits, top-k,
permutation) -> grouped SwiGLU forward -> sparse backward (router gradient, dx, expert gradients
at the 0.5% active set) -> SparseAdam on the active expert entries and on the router.
Default workload: the Qwen3-30B-A3B-shaped layer (T=4096 tokens, H=2048, E=128, top-8, I=768,
bf16, router fp32, K = ceil(0.005 * 603,979,776) = 3,019,899 active entries chosen by the
importance selection of a seeded Student-t(3) dense gradient). --workload qwen3_skewed times the
same layer at T=16384 under Zipf(1.2) expert loads with ten dead experts and 80% of the active
set on the 16 most loaded experts; --workload mixtral_8x7b the Mixtral-8x7B-shaped layer (H=4096,
E=8, top-2, I=14336, T=8192, uniform 0.5% active set). Inputs are seeded synthetic data; the
expert weights (1.2 GB and more) are larger than L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload NAME]

Prints one JSON line. Under torchrun each rank runs its own replica (weak scaling, no
collective on the data path); rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_moe_fine_gb300 import synth  # noqa: E402

METRIC = "MoE-layer train-step tokens/s (fwd+sparse bwd+SparseAdam); % of roofline"
WORKLOADS = ("qwen3_30b_a3b", "qwen3_skewed", "mixtral_8x7b")
HOT_EXPERTS, HOT_FRAC = 16, 0.8  # the skewed workload's active-set concentration


def workload_inputs(name):
    """The workload's configuration and its seeded inputs (skewed routing realised through
    x[:, 0] = 1 and the router's first column)."""
    cfg = synth.CONFIGS[name]
    inp = synth.moe_inputs(cfg, seed=0)
    if "zipf_s" in cfg.extra:
        synth.apply_skew(inp, skew_bias(cfg))
    return cfg, inp


def skew_bias(cfg):
    return synth.skew_bias(cfg.E, cfg.extra["zipf_s"], cfg.extra["dead_experts"], seed=0)


def fixed_active_set(name, cfg):
    """The active set of the workloads whose set is drawn rather than selected: the skewed
    layer's concentrated set (hot experts = the largest logit offsets) or a uniform set."""
    if name == "qwen3_skewed":
        hot = np.argsort(-skew_bias(cfg), kind="stable")[:HOT_EXPERTS]
        return synth.concentrated_mask(cfg, hot, HOT_FRAC, seed=0)
    return synth.uniform_mask(cfg.N, cfg.K, seed=0)


def oracle_active_set(name, cfg):
    """The active set the CPU baseline uses, formed on the host only: for the default workload
    the oracle's importance selection of the same seeded Student-t(3) gradient the device selects
    from (the two are the same set; the GPU tests check it bit for bit)."""
    if name == "qwen3_30b_a3b":
        import oracle
        return oracle.importance_select_threshold(synth.student_t3(cfg.N, seed=0), cfg.K)
    return fixed_active_set(name, cfg)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def algorithmic(cfg, sddmm_pairs=None):
    """Algorithmic FLOPs and HBM bytes of one step (unpadded, SDDMM-counted masked dW: 2 flops per
    (active entry, token routed to its expert) pair, from the live routing when given)."""
    T, H, E, k, I, K = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.K
    R = T * k
    pairs = sddmm_pairs if sddmm_pairs is not None else K * (R / E)
    fl = (2 * R * 2 * I * H + 2 * R * I * H          # forward GEMMs
          + 2 * R * I * H + 2 * R * 2 * I * H        # dgrad through down, dx
          + 2 * T * E * H * 3                        # router logits, g_router, dx router term
          + 2 * pairs)                               # masked dW at the active set
    by = (2 * cfg.N * 2                             # expert weights, read in fwd and in bwd
          + 2 * T * H * 2                            # x
          + 2 * R * 2 * I * 2 + 2 * R * I * 2        # h, A (write + read)
          + 3 * T * H * 2                            # y, dy, dx
          + 2 * R * 2 * I * 2                        # dh (write + read)
          + 2 * T * E * 4                            # logits
          + 2 * (K + E * H) * 4                      # gradients at the active set and router
          + 34 * (K + E * H))                        # SparseAdam: idx, g, p/m/v, weight scatter
    return fl, by


def kernel_units(cfg, sddmm_pairs=None, split=None):
    """Per-launch algorithmic work of the main kernels: (flops, HBM bytes).

    Tensor-core GEMMs count 2*M*N*K over the routed rows (no padding) and each operand read or
    result written once; the gathers count one read of the source rows and one write of the
    transposed rows; the masked expert gradient counts 2 flops per (active entry, routed token)
    pair (`sddmm_pairs`, from the live routing) and one read of its four operands, the active
    indices and the gradient it writes. With `split` (from `masked_split`: the experts whose
    entries the masked-gradient plan reads out of dense tensor-core tiles), the masked-gradient
    kernel counts only the other experts, and the two dense-tile kernels count each listed
    expert's whole gradient (2 * rows * cols * routed rows) and one read of its operands.
    """
    T, H, E, k, I, K = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.K
    R = T * k
    Wgu, Wd = E * 2 * I * H * 2, E * H * I * 2
    pairs = sddmm_pairs if sddmm_pairs is not None else K * R / E
    units = {
        "tc_gate_up_swiglu": (2 * R * 2 * I * H, Wgu + R * H * 2 + R * 2 * I * 2 + R * I * 2),
        "tc_down_combine": (2 * R * I * H, Wd + R * I * 2),
        "tc_gvec_swiglu_bwd": (2 * R * I * H, Wd + R * H * 2 + 2 * R * 2 * I * 2),
        "tc_dx": (2 * R * 2 * I * H, Wgu + R * 2 * I * 2),
        "gather_x": (0, T * H * 2 + R * H * 2),
        "gather_dy": (0, T * H * 2 + R * H * 2),
        "wgrad_sddmm": (2 * pairs, R * (2 * I + H + H + I) * 2 + K * (8 + 4)),
    }
    if split is not None and split["dense"].any():
        n, kgu, kd, dense = split["rows"], split["k_gu"], split["k_down"], split["dense"]
        sp = ~dense
        rows_sp = int(n[sp & ((kgu + kd) > 0)].sum())
        k_sp = int((kgu + kd)[sp].sum())
        units["wgrad_sddmm"] = (2 * int((n * (kgu + kd))[sp].sum()),
                                rows_sp * (2 * I + H + H + I) * 2 + k_sp * (8 + 4))
        nd = int(n[dense].sum())
        units["tc_wgrad_gather_gate_up"] = (2 * nd * 2 * I * H,
                                            nd * (2 * I + H) * 2 + int(kgu[dense].sum()) * 12)
        units["tc_wgrad_gather_down"] = (2 * nd * H * I,
                                         nd * (H + I) * 2 + int(kd[dense].sum()) * 12)
    return units


def masked_split(layer, cfg):
    """Per expert: routed rows, active entries in gate_up and in down, and whether the layer's
    masked-gradient plan lists it (at least dense_density * 3*I*H active entries, bf16 layers
    with a non-empty plan)."""
    import numpy as np
    a = layer.act
    gu = a < cfg.N_gu
    e = torch.where(gu, a // (2 * cfg.I * cfg.H), (a - cfg.N_gu) // (cfg.H * cfg.I))
    kgu = torch.bincount(e[gu], minlength=cfg.E).cpu().numpy()
    kd = torch.bincount(e[~gu], minlength=cfg.E).cpu().numpy()
    dense = np.zeros(cfg.E, bool)
    if getattr(layer, "n_dense", 0):
        dense = (kgu + kd) >= layer.dense_density * 3 * cfg.I * cfg.H
    return {"rows": layer.rt.expert_count.to(torch.int64).cpu().numpy(), "k_gu": kgu, "k_down": kd,
            "dense": dense}


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of one ncu capture of the
# kernel on the workload named (profiles/), with the SHA-256 of the kernel's source file at capture
# time; on another workload, or once that file has changed, the traffic is reported null.
NCU_TRAFFIC = {
    # the masked-gradient kernel's code is unchanged since its capture; the file's later changes
    # are host sequencing (staged forward, router gradient on a side stream)
    "wgrad_sddmm": (456482560 + 13689344, "qwen3_30b_a3b", "sparse_moe_fine_gb300/csrc/moe.cu",
                    "cd08276a7866c3678fb154013b547e0b331e89f6e014d22f04436d3b3a7bde2a"),
    "tc_gate_up_swiglu": (946807808 + 140072704, "qwen3_30b_a3b",
                          "sparse_moe_fine_gb300/csrc/moe_tc.cu",
                          "09b3f6edd25128d85ed5df16d125b3f4c7f081890aea944cce53f1f7891ea79c"),
    "tc_dx": (1122077000 + 156789504, "qwen3_30b_a3b", "sparse_moe_fine_gb300/csrc/moe_tc.cu",
              "09b3f6edd25128d85ed5df16d125b3f4c7f081890aea944cce53f1f7891ea79c"),
}


def ncu_traffic(name, workload="qwen3_30b_a3b"):
    if name not in NCU_TRAFFIC:
        return None
    nbytes, wl, src, sha = NCU_TRAFFIC[name]
    if wl != workload:
        return None
    import hashlib
    try:
        with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), src), "rb") as f:
            cur = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    return nbytes if cur == sha else None


def sddmm_pairs(layer, cfg):
    """Sum over active entries of the routed-token count of the entry's expert."""
    cnt = layer.rt.expert_count.to(torch.int64)
    a = layer.act
    gu = a < cfg.N_gu
    e = torch.where(gu, a // (2 * cfg.I * cfg.H), (a - cfg.N_gu) // (cfg.H * cfg.I))
    return int(cnt[e].sum().item())


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return dist, ws, rank, local
    return None, 1, 0, local


def max_over_ranks(dist, value: float, device) -> float:
    """Largest value over all ranks (the slowest rank sets the time)."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_step_sample(cfg, inp, act, p0, tokens):
    """The CPU oracle's layer step on the first `tokens` tokens of the workload (same weights,
    router, active set and its fp32 master values p0): routing, forward, backward, gradients at
    the active entries of the experts those tokens reach, SparseAdam. Returns seconds."""
    import oracle
    x = inp["x"][:tokens]
    dy = inp["dy"][:tokens]
    t0 = time.perf_counter()
    logits = oracle.router_logits(x, inp["w_router"])
    idx, w = oracle.route_topk(logits, cfg.k)
    b = oracle.moe_backward(x, inp["w_router"], inp["w_gate_up"], inp["w_down"], idx, w, logits,
                            dy)
    hit = sorted(set(idx.reshape(-1).tolist()))
    g = oracle.masked_expert_grad(act, x, inp["w_gate_up"], inp["w_down"], idx, w, dy,
                                  experts=hit)
    g = np.nan_to_num(g, nan=0.0)  # entries of experts no sampled token reaches
    oracle.sparse_adam(g, p0, np.zeros_like(p0), np.zeros_like(p0), cfg.lr, 0.9, 0.999, 1e-8, 1)
    oracle.sparse_adam(b["g_router"].reshape(-1), inp["w_router"].reshape(-1),
                       np.zeros(cfg.E * cfg.H), np.zeros(cfg.E * cfg.H), cfg.lr, 0.9, 0.999,
                       1e-8, 1)
    return time.perf_counter() - t0


def master_values(inp, act, N_gu):
    gu = act < N_gu
    p0 = np.empty(act.size, np.float32)
    p0[gu] = inp["w_gate_up"].reshape(-1)[act[gu]]
    p0[~gu] = inp["w_down"].reshape(-1)[act[~gu] - N_gu]
    return p0


def cpu_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        return max(int(i.get("num_threads", 1)) for i in info) if info else os.cpu_count()
    except Exception:
        return os.cpu_count()


def oracle_steps(name, tokens, steps, warmup):
    """The one CPU baseline both arms report: the oracle's step (oracle_step_sample) on the first
    `tokens` tokens of the workload, with the workload's weights and an active set formed on the
    host; `warmup` untimed steps, then `steps` timed ones. Returns (seconds per step, cfg)."""
    cfg, inp = workload_inputs(name)
    act = oracle_active_set(name, cfg)
    p0 = master_values(inp, act, cfg.N_gu)
    inp = {k: v.astype(np.float64) for k, v in inp.items()}  # exact upcast of the bf16 inputs
    for _ in range(warmup):
        oracle_step_sample(cfg, inp, act, p0, tokens)
    times = [oracle_step_sample(cfg, inp, act, p0, tokens) for _ in range(max(1, steps))]
    return sum(times) / len(times), cfg


def cpu_baseline_entry(sec_per_step, tokens, cfg, steps):
    return {"value": tokens / sec_per_step, "unit": "tokens/s", "cores": cpu_threads(),
            "kind": "oracle",
            "sample": f"oracle step on the first {tokens} of {cfg.T} tokens (whole router, "
                      f"every expert those tokens reach, SparseAdam over all {cfg.K} active "
                      f"entries and the router), mean of {steps} steps",
            "ms_per_step": 1e3 * sec_per_step}


def run_reference(args):
    """The oracle on the host cores: the same metric on bounded samples of the workload. Every
    timed step is one oracle step on the same token sample the GPU arm's cpu_baseline uses."""
    dist, ws, rank, local = dist_setup()
    if rank != 0:
        return
    tokens = args.cpu_tokens
    sec, cfg = oracle_steps(args.workload, tokens, args.steps, args.warmup)
    value = tokens / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": ws, "steps": max(1, args.steps), "warmup": args.warmup,
            "ms_per_step": 1e3 * sec,
            "ms_per_step_note": f"time of the {tokens}-token step that ran",
            "est_ms_per_full_batch": 1e3 * sec * cfg.T / tokens,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": workload_config(args.workload, cfg, ws),
            "cpu_baseline": cpu_baseline_entry(sec, tokens, cfg, max(1, args.steps)),
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run(args):
    from sparse_moe_fine_gb300 import binding as B
    from sparse_moe_fine_gb300.layer import MoELayer

    dist, ws, rank, local = dist_setup()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    B.lib()
    hbm, tf_burst, tf_sus, peak_src = peaks()
    cfg, inp = workload_inputs(args.workload)
    bf = lambda a: torch.from_numpy(a).to(dev).to(torch.bfloat16)
    x, dy = bf(inp["x"]), bf(inp["dy"])
    wgu, wd = bf(inp["w_gate_up"]), bf(inp["w_down"])
    wr = torch.from_numpy(inp["w_router"]).to(dev)
    stream = torch.cuda.current_stream()

    # ---- importance pass: the active set is the top 0.5% |g| of a dense gradient (default
    # workload); the other workloads' sets are drawn
    if args.no_importance or args.workload != "qwen3_30b_a3b":
        act = fixed_active_set(args.workload, cfg)
        return run_steps(args, B, MoELayer, dist, ws, rank, local, dev, cfg, inp, x, dy, wgu, wd,
                         wr, torch.from_numpy(act).to(dev), None, hbm, tf_burst, tf_sus,
                         peak_src, stream)
    g_dense = torch.from_numpy(synth.student_t3(cfg.N, seed=0)).to(dev)
    act = torch.empty(cfg.K, dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_sel = torch.empty(B.importance_select_workspace_size(cfg.N, cfg.K), dtype=torch.uint8,
                         device=dev)
    for _ in range(2):
        B.importance_select(g_dense, cfg.K, act, dev_status=st, ws=ws_sel)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    reps = 5
    ev[0].record()
    for _ in range(reps):
        B.importance_select(g_dense, cfg.K, act, dev_status=st, ws=ws_sel)
    ev[1].record()
    torch.cuda.synchronize()
    sel_ms = ev[0].elapsed_time(ev[1]) / reps
    # RigL reselection on the same layer (drop 30% by |p|, grow by |g|)
    D = int(0.3 * cfg.K)
    layer = MoELayer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, wgu, wd, wr, act, lr=cfg.lr, device=dev)
    outs = [torch.empty(cfg.K, dtype=torch.int64, device=dev)] + \
        [torch.empty(cfg.K, device=dev) for _ in range(3)]
    ns = torch.zeros(1, dtype=torch.int64, device=dev)
    ws_rigl = torch.empty(B.rigl_swap_workspace_size(cfg.N, cfg.K, D), dtype=torch.uint8,
                          device=dev)
    rigl = lambda: B.rigl_swap(g_dense, act, D, layer.p, layer.m, layer.v, wgu, cfg.N_gu, wd,
                               *outs, ns, ws=ws_rigl)
    rigl()
    ev[0].record()
    for _ in range(reps):
        rigl()
    ev[1].record()
    torch.cuda.synchronize()
    rigl_ms = ev[0].elapsed_time(ev[1]) / reps
    # both from one pass over g: the top-K of |g| and the RigL swap of the current set
    sel2 = torch.empty(cfg.K, dtype=torch.int64, device=dev)
    ws_fused = torch.empty(B.select_and_swap_workspace_size(cfg.N, cfg.K, cfg.K, D),
                           dtype=torch.uint8, device=dev)
    fused = lambda: B.select_and_swap(g_dense, sel2, act, D, layer.p, layer.m, layer.v, wgu,
                                      cfg.N_gu, wd, *outs, ns, dev_status=st, ws=ws_fused)
    fused()
    ev[0].record()
    for _ in range(reps):
        fused()
    ev[1].record()
    torch.cuda.synchronize()
    fused_ms = ev[0].elapsed_time(ev[1]) / reps
    # dense gradient pass of the importance phase: one micro-batch's dense expert gradient added
    # into the accumulated g (route, forward, dense backward)
    st_d = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_dense = torch.empty(B.moe_bwd_workspace_size(layer.s, layer.dt, 0), dtype=torch.uint8,
                           device=dev)
    layer.route(x)
    layer.forward(x)
    dense = lambda: B.moe_bwd_dense(layer.s, x, layer.w_router, layer.w_gate_up, layer.w_down,
                                    layer.rt, layer.x_perm, layer.h, layer.wa, dy, g_dense,
                                    layer.g_router, accumulate=1, dx=layer.dx,
                                    logits=layer.logits, renorm=layer.renorm, dev_status=st_d,
                                    ws=ws_dense)
    dense()
    ev[0].record()
    for _ in range(reps):
        dense()
    ev[1].record()
    torch.cuda.synchronize()
    dense_ms = ev[0].elapsed_time(ev[1]) / reps
    del ws_dense
    # full reselection: re-rank by |g|, carry the state of entries that stay
    nk = torch.zeros(1, dtype=torch.int64, device=dev)
    ws_res = torch.empty(B.reselect_full_workspace_size(cfg.N, cfg.K), dtype=torch.uint8,
                         device=dev)
    resel = lambda: B.reselect_full(g_dense, cfg.K, act, layer.p, layer.m, layer.v, wgu, cfg.N_gu,
                                    wd, *outs, nk, ws=ws_res)
    resel()
    ev[0].record()
    for _ in range(reps):
        resel()
    ev[1].record()
    torch.cuda.synchronize()
    resel_ms = ev[0].elapsed_time(ev[1]) / reps
    # per-stage device times of one more selection and one more RigL swap (event trace)
    B.trace_enable(True)
    B.importance_select(g_dense, cfg.K, act, dev_status=st, ws=ws_sel)
    torch.cuda.synchronize()
    sel_stages = {n: 1e3 * t / max(1, c) for n, c, t in B.trace_summary()}
    B.trace_enable(True)
    rigl()
    torch.cuda.synchronize()
    rigl_stages = {n: 1e3 * t for n, c, t in B.trace_summary()}
    B.trace_enable(True)
    fused()
    torch.cuda.synchronize()
    fused_stages = {n: 1e3 * t for n, c, t in B.trace_summary()}
    B.trace_enable(False)
    del ws_rigl, ws_sel, outs, ws_res, ws_fused, sel2
    g_bytes = cfg.N * 4
    importance = {
        "select_ms": sel_ms, "select_gbs": g_bytes / sel_ms / 1e6,
        "select_frac": g_bytes / sel_ms / 1e6 / hbm,
        "rigl_ms": rigl_ms, "rigl_gbs": (g_bytes + cfg.N / 8 + cfg.K * 40) / rigl_ms / 1e6,
        "rigl_frac": (g_bytes + cfg.N / 8 + cfg.K * 40) / rigl_ms / 1e6 / hbm,
        # one read of g for both: its bytes as RigL's plus the K selected indices written
        "select_and_swap_ms": fused_ms, "separate_select_plus_swap_ms": sel_ms + rigl_ms,
        "select_and_swap_frac": (g_bytes + cfg.N / 8 + cfg.K * 48) / fused_ms / 1e6 / hbm,
        "select_and_swap_stages_us": fused_stages,
        "reselect_full_ms": resel_ms, "reselect_full_kept": int(nk.item()),
        "dense_grad_bwd_ms": dense_ms,
        "select_exact_path": bool(int(st.item()) & B.DEV_SELECT_EXACT_PATH),
        "select_stages_us": sel_stages, "rigl_stages_us": rigl_stages,
        "N": cfg.N, "K": cfg.K, "D": D}
    del g_dense, layer
    torch.cuda.empty_cache()
    return run_steps(args, B, MoELayer, dist, ws, rank, local, dev, cfg, inp, x, dy, wgu, wd, wr,
                     act, importance, hbm, tf_burst, tf_sus, peak_src, stream)


def run_steps(args, B, MoELayer, dist, ws, rank, local, dev, cfg, inp, x, dy, wgu, wd, wr, act,
              importance, hbm, tf_burst, tf_sus, peak_src, stream):
    # data parallel over ranks: each rank steps on its own T tokens; the compact gradients are
    # summed over the ranks before SparseAdam (one all-reduce per step)
    group = dist.group.WORLD if dist is not None else None
    layer = MoELayer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, wgu, wd, wr, act, lr=cfg.lr, device=dev,
                     group=group)
    # ---- train steps: routing and forward + backward replayed from CUDA graphs (captured in the
    # first warm-up steps), the two SparseAdam updates launched each step
    for _ in range(args.warmup):
        layer.graphed_train_step(x, dy)
    torch.cuda.synchronize()
    n0 = B.launch_count()
    r0 = layer.replayed_kernels
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            layer.graphed_train_step(x, dy)
        layer.wait_optimizer(stream)
        e1.record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    launches = (B.launch_count() - n0 + layer.replayed_kernels - r0) // max(1, args.steps)
    ms = max_over_ranks(dist, e0.elapsed_time(e1) / args.steps, dev)
    value = ws * cfg.T / (ms / 1e3)

    # ---- per-kernel times over a second timed region of the same steps, launched one by one
    # (event-bracketed; the kernels are the ones the graphs replay)
    B.trace_enable(True)
    for _ in range(args.steps):
        layer.train_step(x, dy)
    torch.cuda.synchronize()
    trace = B.trace_summary()
    B.trace_enable(False)
    # the step's path: a scope traced on the library's side stream spans the kernels it runs
    # beside (dx) and is not part of the sum
    tot = sum(t for n, _, t in trace if n not in OVERLAPPED)
    pairs = sddmm_pairs(layer, cfg)
    units = kernel_units(cfg, pairs, masked_split(layer, cfg))
    # the dominant kernel among those with algorithmic units (the ones a roofline applies to)
    dominant = max((r for r in trace if r[0] in units), key=lambda r: r[2], default=trace[0])
    name, nl, tms = dominant
    avg_ms = tms / nl
    if name in units:
        fl, by = units[name]
        t_fl, t_by = fl / (tf_burst * 1e12), by / (hbm * 1e9)
        if t_fl >= t_by and name.startswith("tc_"):
            roof = {"bound": "tensor", "achieved": fl / (avg_ms / 1e3) / 1e12, "peak": tf_burst,
                    "unit": "TFLOP/s"}
        else:
            roof = {"bound": "hbm", "achieved": by / (avg_ms / 1e3) / 1e9, "peak": hbm,
                    "unit": "GB/s"}
    else:
        roof = {"bound": "hbm", "achieved": None, "peak": hbm, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"] if roof["achieved"] else None
    roof.update({"kernel": name, "kernel_ms": avg_ms,
                 "traffic": ncu_traffic(name, args.workload),
                 "peak_source": peak_src, "share": tms / tot if tot else None})
    fl, by = algorithmic(cfg, pairs)
    step_roof_ms = max(fl / (tf_sus * 1e12), by / (hbm * 1e9)) * 1e3

    # ---- end to end: x, dy from pinned host memory, y and dx back, through the layer API
    if args.no_e2e:
        e2e_ms = None
    else:
        e2e_ms = e2e_time(args, layer, x, dy, e0, e1, stream, dist, dev)
    nbytes = x.numel() * 2
    line = make_line(args, cfg, ws, ms, value, step_roof_ms, fl, by, roof, trace, tot,
                     importance, e2e_ms, nbytes, launches, clk, units, hbm, tf_burst)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        del layer, wgu, wd, inp
        # the reference arm's measurement on the same sample (about 10 s of CPU work)
        sec, _ = oracle_steps(args.workload, args.cpu_tokens, args.cpu_steps, 1)
        line["cpu_baseline"] = cpu_baseline_entry(sec, args.cpu_tokens, cfg, args.cpu_steps)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def e2e_time(args, layer, x, dy, e0, e1, stream, dist, dev):
    """Steps through the layer API fed from pinned host memory: every step copies its x and dY in
    and its y and dx out; the copies of one step overlap the compute of its neighbours."""
    from sparse_moe_fine_gb300.layer import HostStepper
    xh = x.cpu().pin_memory()
    dyh = dy.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    dxh = torch.empty_like(xh).pin_memory()
    hs = HostStepper(layer)
    for _ in range(2):
        hs.step(xh, dyh, yh, dxh)
    hs.finish(stream)
    torch.cuda.synchronize()
    e0.record(stream)
    hs.h2d.wait_event(e0)  # the first input copy starts inside the timed region
    for _ in range(args.steps):
        hs.step(xh, dyh, yh, dxh)
    hs.finish(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    return max_over_ranks(dist, e0.elapsed_time(e1) / args.steps, dev)


# trace scopes on the library's side stream (they overlap the main path's kernels)
OVERLAPPED = {"router_grad"}


def kernel_entry(n, l, t, tot, units, hbm, tf_burst, workload="qwen3_30b_a3b"):
    e = {"name": n, "launches": l, "ms": t, "share": None if n in OVERLAPPED else t / tot}
    if n in OVERLAPPED:
        e["overlapped"] = True  # the span beside the main stream's kernels, not its own time
    tr = ncu_traffic(n, workload)
    if tr is not None:
        e["traffic"] = tr
    if n in units:
        fl, by = units[n]
        avg_s = t / l / 1e3
        e["gbs"] = by / avg_s / 1e9
        e["hbm_frac"] = e["gbs"] / hbm
        if n.startswith("tc_"):
            e["tflops"] = fl / avg_s / 1e12
            e["tensor_frac"] = e["tflops"] / tf_burst
    return e


def workload_config(name, cfg, ws):
    """The `config` object of the JSON line; both arms report the same one."""
    c = {"workload": f"{name} layer step", "T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k,
         "I": cfg.I, "active": cfg.K, "router": "fp32",
         "optimizer": "SparseAdam (experts at the active set, router dense)",
         "parallelism": f"dp{ws}" + (" (all-reduce of the compact gradients)"
                                     if ws > 1 else ""),
         "l2": f"inputs larger than L2 ({cfg.N * 2 / 1e9:.1f} GB of expert weights per step)"}
    if name == "qwen3_30b_a3b":
        c["active_set"] = "importance selection of a seeded Student-t(3) dense gradient"
    elif name == "qwen3_skewed":
        c["routing"] = (f"Zipf({cfg.extra['zipf_s']}) expert loads, "
                        f"{cfg.extra['dead_experts']} experts never routed")
        c["active_set"] = (f"{int(HOT_FRAC * 100)}% on the {HOT_EXPERTS} most loaded experts, "
                           "the rest uniform")
    else:
        c["active_set"] = "uniform"
    return c


def make_line(args, cfg, ws, ms, value, step_roof_ms, fl, by, roof, trace, tot, importance,
              e2e_ms, nbytes, launches, clk, units, hbm, tf_burst):
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(args.workload, cfg, ws),
        "step_roofline": {"ms": step_roof_ms, "frac": step_roof_ms / ms,
                          "algorithmic_gflop": fl / 1e9, "algorithmic_gb": by / 1e9},
        "roofline": roof,
        "kernels": [kernel_entry(n, l, t, tot, units, hbm, tf_burst, args.workload)
                    for n, l, t in trace],
        "importance_pass": importance,
        "e2e": None if e2e_ms is None else {
            "value": ws * cfg.T / (e2e_ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": 2 * nbytes, "d2h_bytes_per_step": 2 * nbytes,
            "ms_per_step": e2e_ms},
        "gpu_launches": int(launches) * args.steps,
        "clocks": clk.summary(),
    }
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3_30b_a3b", choices=WORKLOADS)
    ap.add_argument("--cpu-tokens", type=int, default=512)
    ap.add_argument("--cpu-steps", type=int, default=8,
                    help="oracle steps timed for the GPU arm's cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-importance", action="store_true",
                    help="skip the importance/RigL timing; use a seeded uniform 0.5%% mask")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer timing")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run(args)


if __name__ == "__main__":
    main()
