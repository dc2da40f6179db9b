"""Host logic of bench.py (no GPU): the roofline denominators, the clock record of the timed
steps, the per-kernel roofline classification, and the algorithmic work of the headline workload
against its closed forms."""
import math

import pytest

import bench
from moe_inputs import WORKLOADS

PK = dict(hbm_gbs=6000.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="test")


def test_tensor_peak_is_the_burst_figure():
    # every kernel is timed inside millisecond-scale steps: the burst peak applies
    peak, name = bench.tensor_peak(PK)
    assert peak == 1800.0 and "burst" in name


def test_stage_roofline_binds_the_slower_roof():
    # 1.8e12 FLOP and 6e9 bytes: 1.0 ms at the burst tensor peak, 1.0 ms at HBM -> tensor
    r = bench.stage_roofline(1.8e12, 6e9, 2.0, PK)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(900.0)
    assert r["frac"] == pytest.approx(0.5) and r["peak"] == 1800.0
    # bandwidth work only
    r = bench.stage_roofline(0.0, 6e9, 2.0, PK)
    assert r["bound"] == "hbm" and r["achieved"] == pytest.approx(3000.0)
    assert r["frac"] == pytest.approx(0.5)


def test_cpu_sample_grows_until_half_the_target():
    # a fixed per-call cost: 16 tokens in 2.4 s extrapolates to 80 tokens for a 15 s target
    assert bench.grow_sample(16, 2.4, 4096, 15.0) == 80
    # a sample that still took 2.25 s grows again, at least doubling
    assert bench.grow_sample(80, 2.25, 4096, 15.0) == 426
    assert bench.grow_sample(80, 7.0, 4096, 15.0) == 160
    assert bench.grow_sample(80, 5.0, 4096, 15.0) == 192
    # long enough, or already the whole batch
    assert bench.grow_sample(426, 7.5, 4096, 15.0) is None
    assert bench.grow_sample(4096, 1.0, 4096, 15.0) is None
    assert bench.grow_sample(3000, 1.0, 4096, 15.0) == 4096


def _row(sm, mx, pw, cap="Not Active", hw="Not Active"):
    return [str(sm), str(mx), str(pw), "0x0", hw, "Not Active", "Not Active", cap]


def test_clock_summary_takes_the_samples_around_the_timed_steps():
    c = bench.ClockSampler(0)
    c.rows = [_row(2032, 2032, 120), _row(1300, 2032, 1050, cap="Active"),
              _row("[N/A]", 2032, 900), _row(1400, 2032, 1000), _row(1350, 2032, 1090),
              _row(2032, 2032, 150)]
    c.times = [0.0, 10.0, 10.2, 10.4, 10.6, 20.0]
    # the window 10.1 .. 10.5 s, widened by 0.2 s on each side: the samples at 10.0 .. 10.6
    s = c.summary(window=(10.1, 10.5))
    assert s["sm_mhz"] == 1350.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 4
    assert s["power_w_max"] == 1090.0
    # a window with no sample in reach has no clock record
    assert c.summary(window=(15.0, 15.1))["samples"] == 0
    # no window: every sample
    assert c.summary()["samples"] == 6


def test_clock_summary_reports_slowdowns_and_empty_records():
    c = bench.ClockSampler(0)
    c.rows = [_row(1000, 2032, 200, hw="Active")]
    c.times = [1.0]
    s = c.summary()
    assert s["sm_mhz"] == 1000.0 and s["reasons"] == ["hw_slowdown"]
    c.rows, c.times = [], []
    assert bench.ClockSampler.summary(c) == dict(sm_mhz=None, sm_max_mhz=None, reasons=[],
                                                  samples=0)


def test_traffic_is_read_only_while_the_kernel_source_is_unchanged(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "mixture_experts_layer_92_b300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("// kernel\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.source_sha(str(csrc / "k.cu"))
    prof = tmp_path / "profiles" / "gemm_x__wl.txt"
    prof.write_text(f"source_file: k.cu\nsource_sha256_16: {sha}\n"
                    "dram_bytes_per_launch: 1.5e9 (read + write)\n")
    assert bench.traffic_from_profile("wl", "gemm_x") == 1.5e9
    (csrc / "k.cu").write_text("// kernel, changed\n")
    assert bench.traffic_from_profile("wl", "gemm_x") is None      # stale capture
    assert bench.traffic_from_profile("other", "gemm_x") is None   # no capture


def test_reference_step_size_from_a_two_point_fit():
    # 2.4 s of fixed cost and 1 ms per token: a step of max(3, 4.8) s holds 2400 tokens
    t = lambda n: 2.4 + 1e-3 * n
    assert bench.step_tokens(8, t(8), 72, t(72), 4096) == 2400
    # no fixed cost: 3 s of tokens
    t = lambda n: 2e-3 * n
    assert bench.step_tokens(8, t(8), 72, t(72), 4096) == 1500
    # clamped to the batch, and never below the first sample
    assert bench.step_tokens(8, 0.01, 72, 0.02, 256) == 256
    # 4.5 s fixed, 62.5 ms per token: a 9 s step holds 72 tokens
    assert bench.step_tokens(8, 5.0, 72, 9.0, 4096) == 72
    # timing noise that makes the second sample faster: never below the first sample
    assert bench.step_tokens(8, 2.0, 72, 1.9, 4096) >= 8


def test_algorithmic_work_of_the_prefill_layer():
    """Mixtral prefill, no drop: R = T k kept rows, every expert touched."""
    w = WORKLOADS["mixtral_prefill"]
    T, d, E, F, k = w.T, w.d, w.E, w.d_ff, w.k
    R = T * k
    work = bench.algorithmic_work(w, R, E)
    assert work["flops"] == pytest.approx(2 * T * d * E + 6 * d * F * R)
    # x, W_r, all experts' three matrices and y, in bf16
    assert work["bytes"] == pytest.approx((T * d + E * d + 3 * E * d * F + T * d) * 2)
    st = work["per_stage"]
    assert st["gemm_gateup_swiglu"][0] == pytest.approx(4 * R * d * F)
    assert st["gemm_down_scale"][0] == pytest.approx(2 * R * d * F)
    assert math.isclose(sum(v[0] for v in st.values()), work["flops"])
    # the gather copies R rows in and out
    assert st["gather"][1] == pytest.approx(2 * R * d * 2)


def test_algorithmic_work_of_8bit_weights_counts_codes_and_scales():
    w = WORKLOADS["mixtral_decode"]
    R, E = w.T * w.k, w.E
    b16 = bench.algorithmic_work(w, R, E)["bytes"]
    b8 = bench.algorithmic_work(w, R, E, wb=1)["bytes"]
    weights16 = 3 * E * w.d * w.d_ff * 2
    weights8 = 3 * E * w.d * w.d_ff + E * (2 * w.d_ff + w.d) * 4
    assert b16 - b8 == pytest.approx(weights16 - weights8)


def test_routing_report_on_the_oracle_itself():
    """The bench's routing report (run in its CPU-baseline leg) on a small drop workload,
    fed the oracle's own routing and outputs: no difference, both rel L2 near 0; then one
    token's expert set changed by hand is counted."""
    import numpy as np
    import torch
    import oracle as O
    from moe_inputs import make_inputs
    w = WORKLOADS["tiny_fp32"]
    inp = make_inputs(w, device="cpu")
    ih = bench.host_inputs(inp)
    C = O.capacity(w.cf, w.T, w.k, w.E)
    ref = O.forward(ih["x"], ih["w_router"], ih["w1"], ih["w3"], ih["w2"], k=w.k, mode=w.gate,
                    C=C, alpha=w.alpha, beta=w.beta)
    y = torch.from_numpy(ref["y"])
    rep = bench.routing_report(w, ih, ref["idx"].copy(), y, C)
    assert rep["routed_differently"] == 0 and rep["all_differences_among_near_ties"]
    assert rep["rel_l2_direct"] < 1e-6 and rep["rel_l2_gpu_routing"] < 1e-6
    assert rep["near_ties"] == len(O.near_tie_tokens(ref["logits"], w.k))
    idx = ref["idx"].copy()
    t = 5
    idx[t] = [e for e in range(w.E) if e not in idx[t]][:w.k]
    rep = bench.routing_report(w, ih, idx, y, C)
    assert rep["routed_differently"] == 1


def test_launches_per_forward_follow_the_layer_structure():
    """The kernel count a forward launches (the bench line's gpu_launches per step): fused
    router, dispatch (with the statistics and losses), gather, two GEMMs, and a combine except
    for top-1 bf16 layers without a shared expert; the unfused router adds the top-k kernel;
    fp32 shared experts run two more GEMMs; expert choice runs its selection, an unrouted
    count and the statistics kernel in place of the dispatch."""
    W = WORKLOADS
    assert bench.launches_per_forward(W["mixtral_prefill"]) == 6
    assert bench.launches_per_forward(W["mixtral_decode"]) == 6
    assert bench.launches_per_forward(W["switch_top1"]) == 5                    # no combine
    assert bench.launches_per_forward(W["switch_top1"], quantized=True) == 6    # 8-bit: combine
    assert bench.launches_per_forward(W["deepseek_fine"]) == 6
    assert bench.launches_per_forward(W["switch_top1"].scaled(d_ff_shared=256)) == 6
    assert bench.launches_per_forward(W["switch_top1"].scaled(E=512)) == 6     # router + top-k
    assert bench.launches_per_forward(W["tiny_fp32"]) == 7                      # fp32 router pair
    assert bench.launches_per_forward(W["tiny_fp32"].scaled(d_ff_shared=64)) == 9
    ec = W["mixtral_prefill"].scaled(gate="expert_choice", cf=1.0)
    assert bench.launches_per_forward(ec) == 8
