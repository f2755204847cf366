"""The benchmark's roofline arithmetic, checked on the host: the per-step algorithmic FLOPs and
bytes, and each main kernel's per-launch bytes, against the same quantities summed term by term
from the tensor sizes of the Qwen3-30B-A3B-shaped layer (T 4096, H 2048, E 128, top-8, I 768,
K = 3,019,899 active entries)."""
import importlib.util
import os

import pytest

from sparse_moe_fine_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)  # defines functions only; main() is not run
    return mod


CFG = synth.CONFIGS["qwen3_30b_a3b"]
MB = 1e6


def test_workload_sizes():
    assert (CFG.T, CFG.H, CFG.E, CFG.k, CFG.I) == (4096, 2048, 128, 8, 768)
    assert CFG.N == 603_979_776 and CFG.K == 3_019_899


def test_step_flops_by_term(bench):
    fl, _ = bench.algorithmic(CFG)
    R = 32_768  # routed rows, T * k
    terms_gf = {
        "forward: gate_up 2*R*2I*H + down 2*R*I*H": 206.158 + 103.079,
        "dgrad through down": 103.079,
        "dx through gate_up": 206.158,
        "router: logits, its gradient, the dx term": 3 * 2 * 4096 * 128 * 2048 / 1e9,
        "masked dW: 2 flops per (entry, routed token), R/E tokens per expert":
            2 * 3_019_899 * (R / 128) / 1e9,
    }
    assert fl / 1e9 == pytest.approx(sum(terms_gf.values()), rel=1e-4)
    assert fl / 1e9 == pytest.approx(626.46, abs=0.01)


def test_step_bytes_by_term(bench):
    _, by = bench.algorithmic(CFG)
    terms_mb = {
        "expert weights read in the forward and again in the backward": 2 * 1207.96,
        "x read twice (router, gather)": 33.55,
        "h written and read (bf16 [R, 2I])": 201.33,
        "A written and read (bf16 [R, I])": 100.66,
        "y, dy, dx once each": 50.33,
        "dh written and read": 201.33,
        "logits written and read (fp32 [T, E])": 4.19,
        "gradients written and read (K + E*H fp32)": 26.26,
        "SparseAdam: 8 idx + 4 g + 3 x 4 read + 3 x 4 written + 2 weight per entry":
            34 * (3_019_899 + 262_144) / MB,
    }
    assert by / MB == pytest.approx(sum(terms_mb.values()), rel=2e-4)
    assert by / 1e9 == pytest.approx(3.145, abs=0.001)


def test_kernel_bytes_match_the_operands(bench):
    u = bench.kernel_units(CFG)
    w_gu, w_d = 805.31, 402.65  # bf16 [E, 2I, H] and [E, H, I]
    x_perm, h, wa = 134.22, 100.66, 50.33  # bf16 [R, H], [R, 2I], [R, I]
    expect = {
        "tc_gate_up_swiglu": w_gu + x_perm + h + wa,
        "tc_down_combine": w_d + wa,
        "tc_gvec_swiglu_bwd": w_d + x_perm + h + h,  # dy_perm [R, H], h read, dh written
        "tc_dx": w_gu + h,                           # dh [R, 2I]
        "gather_x": 16.78 + x_perm,
        "wgrad_sddmm": h + x_perm + x_perm + wa + 3_019_899 * 12 / MB,
    }
    for name, mb in expect.items():
        assert u[name][1] / MB == pytest.approx(mb, rel=2e-4), name
    assert u["tc_gate_up_swiglu"][0] == u["tc_dx"][0] == 2 * 32_768 * 1536 * 2048
    assert u["tc_down_combine"][0] == u["tc_gvec_swiglu_bwd"][0] == 2 * 32_768 * 768 * 2048


def test_masked_gradient_units_split_between_the_two_kernels(bench):
    """With the plan listing some experts, the masked-gradient kernel counts only the others'
    pairs and operands; the dense-tile kernels count the listed experts' whole gradients."""
    import numpy as np
    E = CFG.E
    rows = np.full(E, CFG.T * CFG.k // E, np.int64)
    kgu = np.full(E, 10, np.int64)
    kd = np.full(E, 5, np.int64)
    dense = np.zeros(E, bool)
    dense[:3] = True
    kgu[:3] = 100_000
    kd[:3] = 50_000
    split = {"rows": rows, "k_gu": kgu, "k_down": kd, "dense": dense}
    u = bench.kernel_units(CFG, int((rows * (kgu + kd)).sum()), split)
    n = 256
    I, H = CFG.I, CFG.H
    assert u["wgrad_sddmm"][0] == 2 * n * 15 * (E - 3)
    assert u["wgrad_sddmm"][1] == n * (E - 3) * (2 * I + H + H + I) * 2 + 15 * (E - 3) * 12
    assert u["tc_wgrad_gather_gate_up"][0] == 2 * 3 * n * 2 * I * H
    assert u["tc_wgrad_gather_down"][0] == 2 * 3 * n * H * I
    assert u["tc_wgrad_gather_gate_up"][1] == 3 * n * (2 * I + H) * 2 + 300_000 * 12
    # no listed expert: the masked-gradient kernel counts everything, as without a split
    split["dense"] = np.zeros(E, bool)
    assert bench.kernel_units(CFG, 7, split) == bench.kernel_units(CFG, 7)


def test_traffic_is_reported_only_for_captured_kernels(bench):
    assert bench.ncu_traffic("gather_x") is None
    # a capture's bytes belong to its workload only
    assert bench.ncu_traffic("tc_dx", "mixtral_8x7b") is None
    assert set(bench.NCU_TRAFFIC) <= set(bench.kernel_units(CFG))


def test_clock_summary_parses_throttle_reasons(bench):
    clk = bench.ClockSampler(0)
    clk.lines = ["2070, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active",
                 "2055, 2070, 910.0, 0x0, Not Active, Not Active, Not Active, Not Active",
                 "[N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
                 "2070, 2070, 905.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    s = clk.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                 "samples": 3}


def test_json_line_carries_every_contract_key(bench):
    import argparse
    args = argparse.Namespace(steps=200, warmup=5, workload="qwen3_30b_a3b")
    clk = bench.ClockSampler(0)
    clk.lines = ["2070, 2070, 900, 0x0, Not Active, Not Active, Not Active, Not Active"]
    fl, by = bench.algorithmic(CFG)
    units = bench.kernel_units(CFG)
    trace = [("tc_dx", 200, 48.7), ("wgrad_sddmm", 200, 41.1), ("route_topk", 200, 2.4),
             ("router_grad", 200, 52.0)]
    nbytes = CFG.T * CFG.H * 2
    roof = {"bound": "hbm", "achieved": 3700.0, "peak": 6779.0, "unit": "GB/s", "frac": 0.55,
            "traffic": None}
    line = bench.make_line(args, CFG, 1, 1.31, 3.1e6, 0.464, fl, by, roof, trace, 92.2, None,
                           1.36, nbytes, 22, clk, units, 6779.0, 1918.6)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in line, key
    assert line["config"] == bench.workload_config("qwen3_30b_a3b", CFG, 1)
    assert line["config"]["workload"] == "qwen3_30b_a3b layer step"
    assert line["gpu_launches"] == 22 * 200
    assert line["e2e"]["h2d_bytes_per_step"] == 2 * nbytes  # x and dy in
    assert line["e2e"]["d2h_bytes_per_step"] == 2 * nbytes  # y and dx out
    assert line["e2e"]["value"] == pytest.approx(CFG.T / 1.36e-3)
    dx = next(k for k in line["kernels"] if k["name"] == "tc_dx")
    assert dx["gbs"] == pytest.approx(units["tc_dx"][1] / (48.7 / 200 / 1e3) / 1e9)
    assert "gbs" not in next(k for k in line["kernels"] if k["name"] == "route_topk")
    # a side-stream scope spans the kernels it runs beside: flagged, no share of the step
    rg = next(k for k in line["kernels"] if k["name"] == "router_grad")
    assert rg["overlapped"] and rg["share"] is None
    skipped = bench.make_line(args, CFG, 1, 1.31, 3.1e6, 0.464, fl, by, roof, trace, 92.2, None,
                              None, nbytes, 22, clk, units, 6779.0, 1918.6)
    assert skipped["e2e"] is None


def test_other_workloads_configs_and_active_sets(bench):
    """The skewed and Mixtral-shaped workloads: their JSON config names them, and the skewed
    layer's drawn active set puts 80% of K on the 16 experts with the largest logit offsets."""
    import numpy as np
    sk = synth.CONFIGS["qwen3_skewed"]
    c = bench.workload_config("qwen3_skewed", sk, 1)
    assert c["workload"] == "qwen3_skewed layer step" and c["T"] == 16384
    assert "Zipf" in c["routing"] and "16 most loaded" in c["active_set"]
    act = bench.fixed_active_set("qwen3_skewed", sk)
    assert act.size == sk.K and (np.diff(act) > 0).all()
    hot = set(np.argsort(-bench.skew_bias(sk), kind="stable")[:16].tolist())
    gu = act < sk.N_gu
    e = np.where(gu, act // (2 * sk.I * sk.H), (act - sk.N_gu) // (sk.H * sk.I))
    assert np.isin(e, list(hot)).sum() == int(0.8 * sk.K)
    mx = synth.CONFIGS["mixtral_8x7b"]
    assert bench.workload_config("mixtral_8x7b", mx, 1)["active_set"] == "uniform"
    assert mx.K == 7_046_431
    # the masked-gradient term of the step counts the live routing when given
    fl_u, _ = bench.algorithmic(sk)
    fl_l, _ = bench.algorithmic(sk, sddmm_pairs=10**10)
    assert fl_l - fl_u == pytest.approx(2 * (10**10 - sk.K * sk.T * sk.k / sk.E))
