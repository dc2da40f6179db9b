"""Host logic of bench.py (no GPU): the roofline denominators chosen from the clock record,
the per-kernel roofline classification, and the algorithmic work of the headline workload
against its closed forms."""
import math

import pytest

import bench
from moe_inputs import WORKLOADS

PK = dict(hbm_gbs=6000.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="test")


@pytest.mark.parametrize("clk,capped", [
    (dict(sm_mhz=1300.0, sm_max_mhz=2032.0, reasons=["sw_power_cap"]), True),
    (dict(sm_mhz=1800.0, sm_max_mhz=2032.0, reasons=[]), True),          # below 90 % of max
    (dict(sm_mhz=2032.0, sm_max_mhz=2032.0, reasons=["sw_power_cap"]), False),  # a momentary flag
    (dict(sm_mhz=1900.0, sm_max_mhz=2032.0, reasons=[]), False),
    (dict(sm_mhz=None, sm_max_mhz=None, reasons=[]), False),
    (None, False),
])
def test_power_capped(clk, capped):
    assert bench.power_capped(clk) is capped


def test_tensor_peak_follows_the_clock_record():
    peak, name = bench.tensor_peak(PK, dict(sm_mhz=1200.0, sm_max_mhz=2032.0, reasons=[]))
    assert peak == 1400.0 and "sustained" in name
    peak, name = bench.tensor_peak(PK, dict(sm_mhz=2032.0, sm_max_mhz=2032.0, reasons=[]))
    assert peak == 1800.0 and "burst" in name
    no_sustained = dict(PK, bf16_tflops_sustained=None)
    assert bench.tensor_peak(no_sustained, dict(sm_mhz=1200.0, sm_max_mhz=2032.0))[0] == 1800.0


def test_stage_roofline_binds_the_slower_roof():
    capped = dict(sm_mhz=1200.0, sm_max_mhz=2032.0, reasons=[])
    # 1.4e12 FLOP and 6e9 bytes: 1.0 ms at the sustained tensor peak, 1.0 ms at HBM -> tensor
    r = bench.stage_roofline(1.4e12, 6e9, 2.0, PK, capped)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(700.0)
    assert r["frac"] == pytest.approx(0.5) and r["frac_burst"] == pytest.approx(700.0 / 1800.0)
    # bandwidth work only
    r = bench.stage_roofline(0.0, 6e9, 2.0, PK, capped)
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


def test_clock_summary_takes_the_median_under_load():
    c = bench.ClockSampler(0)
    c.rows = [_row(2032, 2032, 120), _row(1300, 2032, 1050, cap="Active"),
              _row("[N/A]", 2032, 900), _row(1400, 2032, 1000), _row(1350, 2032, 1090)]
    s = c.summary()
    # rows above 300 W with a readable clock: 1300, 1400, 1350 (the idle 2032 MHz sample and
    # the unreadable one are left out, without shifting the clock/power pairing)
    assert s["sm_mhz"] == 1350.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 5
    assert s["power_w_max"] == 1090.0


def test_clock_summary_reports_slowdowns_and_empty_records():
    c = bench.ClockSampler(0)
    c.rows = [_row(1000, 2032, 200, hw="Active")]
    s = c.summary()
    assert s["sm_mhz"] == 1000.0 and s["reasons"] == ["hw_slowdown"]
    c.rows = []
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
