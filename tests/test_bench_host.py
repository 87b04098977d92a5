"""Host-side logic of bench.py that needs no GPU: the clock-sample summary
that decides whether a timed region is measured again."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _summary(lines):
    c = bench.ClockSampler(0)
    c.lines = lines
    return c.summary()


def test_clock_summary_median_and_reasons():
    # index, clocks.sm, clocks.max.sm, power.draw, active, hw, hw_thermal, sw_thermal, sw_power_cap
    lines = ["0, 1800, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 1900, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 2000, 2070, 980.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    s = _summary(lines)
    assert s["sm_mhz"] == 1900 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    assert not (bench.THROTTLE_REASONS & set(s["reasons"]))  # power cap alone: no re-measure


def test_clock_summary_flags_thermal_slowdown():
    lines = ["0, 1500, 2070, 1000.0, 0x20, Not Active, Not Active, Active, Not Active",
             "garbled line", "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    s = _summary(lines)
    assert s["samples"] == 1 and s["reasons"] == ["sw_thermal_slowdown"]
    assert bench.THROTTLE_REASONS & set(s["reasons"])  # would be measured again


def test_clock_summary_without_samples():
    s = _summary([])
    assert s["sm_mhz"] is None and s["samples"] == 0 and s["reasons"] == []


def test_oracle_sample_of_the_fp32_master_layer():
    """The secondary lines' CPU leg: the 256x256 fp32-master configuration is
    sampled whole (3 steps of dX + dW + AdamW), its flops counted like the GPU
    line (4NKT per step)."""
    dt, flops, desc = bench.oracle_sample_workload("single_256")
    assert dt > 0 and flops == 3 * 4.0 * 256 * 256 * 512
    assert "3 step(s)" in desc and "fp32 weights" in desc


def test_peak_follows_the_timed_region_length():
    """A region shorter than the sustained threshold is compared with the burst
    peak, a longer one with the sustained peak, and the line says which."""
    p, kind = bench.applicable_peak(0.17, 1931.0, 1747.4, "measured")
    assert p == 1931.0 and kind.startswith("bf16 burst")
    p, kind = bench.applicable_peak(bench.SUSTAINED_REGION_S, 1931.0, 1747.4, "measured")
    assert p == 1747.4 and kind.startswith("bf16 sustained")


def test_cpu_model_is_a_nonempty_string():
    m = bench.cpu_model()
    assert isinstance(m, str) and m
    assert bench.host_cores() >= 1
