"""The bench's clock record, from fabricated samples (no GPU, no NVML):
the window, the median clock and the throttle reasons it reports decide
whether a measurement is kept."""
from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_nvml_reason_bits():
    assert bench.nvml_reason_names(0) == []
    assert bench.nvml_reason_names(0x4 | 0x40) == ["sw_power_cap", "hw_thermal_slowdown"]
    assert bench.nvml_reason_names(0x1 | 0x2 | 0x10) == []      # idle, app clocks, sync boost
    assert bench.nvml_reason_names(0x8 | 0x20) == ["hw_slowdown", "sw_thermal_slowdown"]


def _samples():
    # one sample a second: clock, power, reasons
    return [(float(t), 2070.0 - 10 * t, 100.0 + t, ["sw_power_cap"] if t == 5 else [])
            for t in range(1, 11)]


def test_summary_keeps_the_samples_inside_the_timed_region():
    s = bench.summarize_clocks(_samples(), 3.0, 7.0, 2070.0)
    assert s["window"] == "timed region" and s["samples"] == 5
    assert s["sm_mhz"] == 2070.0 - 50                              # median of t = 3..7
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 107.0
    assert s["sm_max_mhz"] == 2070.0


def test_summary_of_a_region_shorter_than_the_sampling_period():
    s = bench.summarize_clocks(_samples(), 8.4, 8.45, 2070.0)
    assert s["window"] == "nearest to the timed region" and s["samples"] == 2
    assert s["sm_mhz"] == (2070.0 - 80 + 2070.0 - 90) / 2        # t = 8 and 9
    assert s["reasons"] == []


def test_summary_without_samples():
    s = bench.summarize_clocks([], 1.0, 2.0, 2070.0)
    assert s["sm_mhz"] is None and s["reasons"] == ["no samples"]


def test_nvidia_smi_rows():
    text = "\n".join([
        "2026/12/02 10:00:00.100, 0, 1965, 2070, 800.50, 0x0000000000000004, Not Active, "
        "Not Active, Not Active, Active",
        "2026/12/02 10:00:00.120, 0, 1410, 2070, 1390.00, 0x0000000000000048, Active, "
        "Active, Not Active, Not Active",
        "garbled line",
        "",
    ])
    rows = bench.ClockSampler.parse_rows(text)
    assert len(rows) == 2
    t0, mhz, mx, w, reasons = rows[0]
    assert (mhz, mx, w, reasons) == (1965.0, 2070.0, 800.5, ["sw_power_cap"])
    assert rows[1][4] == ["hw_slowdown", "hw_thermal_slowdown"]
    assert abs(rows[1][0] - t0 - 0.02) < 1e-6
