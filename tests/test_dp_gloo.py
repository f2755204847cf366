"""Data-parallel exchange on two CPU ranks (gloo): the layer's gradient all-reduce, and the
composition it relies on -- per-rank gradients of token shards, summed, equal the gradient of the
whole batch, so every replica's SparseAdam update equals the single-replica update."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from sparse_moe_fine_gb300 import synth
from sparse_moe_fine_gb300.layer import allreduce_dense_grad, allreduce_grads

WORLD = 2


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


def _exchange(rank):
    g_act = torch.tensor([1.0, 2.0, -3.0], dtype=torch.float32) * (rank + 1)
    g_r = torch.full((2, 3), float(rank))
    status = torch.tensor([1 if rank == 0 else 4], dtype=torch.int32)  # distinct bits per rank
    allreduce_grads(g_act, g_r, status)
    return g_act.numpy().copy(), g_r.numpy().copy(), int(status.item())


def test_allreduce_grads_sums_and_ors():
    res = _spawn(_exchange)
    for g_act, g_r, st in res:
        np.testing.assert_array_equal(g_act, np.array([3.0, 6.0, -9.0], np.float32))
        np.testing.assert_array_equal(g_r, np.ones((2, 3), np.float32))
        assert st == 5  # NONFINITE from rank 0 and TIMEOUT from rank 1 both survive


CFG = synth.small_config("dp", T=96, H=64, E=4, k=2, I=32, bf16=False, frac=0.05, dy_std=1.0)


def _shard_step(rank):
    """One rank: oracle gradients of its half of the tokens, summed over ranks with the layer's
    exchange, then the oracle SparseAdam step."""
    inp = synth.moe_inputs(CFG, seed=3)
    act = synth.uniform_mask(CFG.N, CFG.K, seed=3)
    sl = slice(rank * CFG.T // WORLD, (rank + 1) * CFG.T // WORLD)
    x, dy = inp["x"][sl], inp["dy"][sl]
    logits = oracle.router_logits(x, inp["w_router"])
    idx, w = oracle.route_topk(logits, CFG.k)
    b = oracle.moe_backward(x, inp["w_router"], inp["w_gate_up"], inp["w_down"], idx, w, logits,
                            dy)
    g = oracle.masked_expert_grad(act, x, inp["w_gate_up"], inp["w_down"], idx, w, dy)
    g_act = torch.from_numpy(np.ascontiguousarray(g, np.float64))
    g_r = torch.from_numpy(np.ascontiguousarray(b["g_router"], np.float64))
    allreduce_grads(g_act, g_r, torch.zeros(1, dtype=torch.int32))
    p0 = np.asarray(inp["w_gate_up"], np.float64).reshape(-1)
    p0 = np.concatenate([p0, np.asarray(inp["w_down"], np.float64).reshape(-1)])[act]
    z = np.zeros(act.size)
    p1, _, _ = oracle.sparse_adam(g_act.numpy(), p0, z, z, CFG.lr, 0.9, 0.999, 1e-8, 1)
    return g_act.numpy().copy(), g_r.numpy().copy(), np.asarray(p1).copy()


def test_sharded_gradients_sum_to_whole_batch():
    res = _spawn(_shard_step)
    inp = synth.moe_inputs(CFG, seed=3)
    act = synth.uniform_mask(CFG.N, CFG.K, seed=3)
    logits = oracle.router_logits(inp["x"], inp["w_router"])
    idx, w = oracle.route_topk(logits, CFG.k)
    b = oracle.moe_backward(inp["x"], inp["w_router"], inp["w_gate_up"], inp["w_down"], idx, w,
                            logits, inp["dy"])
    g = oracle.masked_expert_grad(act, inp["x"], inp["w_gate_up"], inp["w_down"], idx, w,
                                  inp["dy"])
    p0 = np.concatenate([np.asarray(inp["w_gate_up"], np.float64).reshape(-1),
                         np.asarray(inp["w_down"], np.float64).reshape(-1)])[act]
    z = np.zeros(act.size)
    p1, _, _ = oracle.sparse_adam(g, p0, z, z, CFG.lr, 0.9, 0.999, 1e-8, 1)
    for g_act, g_r, p in res:
        np.testing.assert_allclose(g_act, g, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(g_r, b["g_router"], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(p, p1, rtol=1e-6, atol=1e-9)  # fp32 master values
    np.testing.assert_array_equal(res[0][2], res[1][2])  # identical replicas


def _dense_grad(inp, x, dy):
    logits = oracle.router_logits(x, inp["w_router"])
    idx, w = oracle.route_topk(logits, CFG.k)
    b = oracle.moe_backward(x, inp["w_router"], inp["w_gate_up"], inp["w_down"], idx, w, logits,
                            dy, dense_wgrad=True)
    return np.concatenate([b["dW_gate_up"].reshape(-1), b["dW_down"].reshape(-1)])


def _shard_reselect(rank):
    """One rank: the dense gradient of its half of the tokens, exchanged with the trainer's
    reduction, then both reselection rules (RigL drop/grow and the full re-rank)."""
    inp = synth.moe_inputs(CFG, seed=4)
    act = synth.uniform_mask(CFG.N, CFG.K, seed=4)
    sl = slice(rank * CFG.T // WORLD, (rank + 1) * CFG.T // WORLD)
    # fp64 shards: their sum is the whole batch's gradient up to fp64 rounding, so after the
    # fp32 cast the ranking is the whole batch's
    g64 = torch.from_numpy(np.ascontiguousarray(_dense_grad(inp, inp["x"][sl], inp["dy"][sl])))
    local = g64.numpy().astype(np.float32)
    allreduce_dense_grad(g64)
    g = g64.float()
    w = np.concatenate([inp["w_gate_up"].reshape(-1), inp["w_down"].reshape(-1)])
    p = w[act].copy()
    m, v = synth.adam_state(act.size, seed=4)
    D = int(0.3 * act.size)
    rig = oracle.rigl_swap(act, p, m, v, g.numpy(), D, lambda i: w[i])
    full = oracle.reselect_full(act, p, m, v, g.numpy(), act.size, lambda i: w[i])
    # without the exchange the replicas would rank different gradients
    alone = oracle.rigl_swap(act, p, m, v, local, D, lambda i: w[i])[0]
    return rig[0].copy(), rig[1].copy(), full[0].copy(), alone.copy(), g.numpy().copy()


def test_reselection_after_the_dense_exchange_agrees_across_ranks():
    res = _spawn(_shard_reselect)
    inp = synth.moe_inputs(CFG, seed=4)
    act = synth.uniform_mask(CFG.N, CFG.K, seed=4)
    g_all = _dense_grad(inp, inp["x"], inp["dy"])
    w = np.concatenate([inp["w_gate_up"].reshape(-1), inp["w_down"].reshape(-1)])
    p = w[act].copy()
    m, v = synth.adam_state(act.size, seed=4)
    D = int(0.3 * act.size)
    # the exchanged gradient is the whole batch's
    for *_, g in res:
        np.testing.assert_array_equal(g, g_all.astype(np.float32))
    np.testing.assert_array_equal(res[0][4], res[1][4])
    ref_rig = oracle.rigl_swap(act, p, m, v, res[0][4], D, lambda i: w[i])
    ref_full = oracle.reselect_full(act, p, m, v, res[0][4], act.size, lambda i: w[i])
    for rig_idx, rig_p, full_idx, _, _ in res:
        np.testing.assert_array_equal(rig_idx, ref_rig[0])
        np.testing.assert_array_equal(rig_p, ref_rig[1])
        np.testing.assert_array_equal(full_idx, ref_full[0])
    # the sets from the exchanged gradient are the whole batch's
    g32 = g_all.astype(np.float32)
    np.testing.assert_array_equal(
        ref_rig[0], oracle.rigl_swap(act, p, m, v, g32, D, lambda i: w[i])[0])
    np.testing.assert_array_equal(
        ref_full[0], oracle.reselect_full(act, p, m, v, g32, act.size, lambda i: w[i])[0])
    # and each rank alone would have installed a different set
    assert not np.array_equal(res[0][3], res[1][3])


@pytest.mark.skipif(torch.cuda.is_available(), reason="the GPU arm would use NCCL; CPU check")
def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched as two ranks: rank 0 alone runs the oracle and prints
    one JSON line; the other rank exits 0 without output."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--cpu-tokens", "8"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["n_gpus"] == 2 and d["config"]["parallelism"].startswith("dp2")
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    # the time of what ran: one 8-token step, its own rate; the full-batch figure apart
    assert d["ms_per_step"] == pytest.approx(1e3 * 8 / d["value"], rel=1e-9)
    assert d["est_ms_per_full_batch"] == pytest.approx(d["ms_per_step"] * 4096 / 8, rel=1e-9)
    assert d["cpu_baseline"]["value"] == d["value"]
