"""Host logic of bench.py that needs no GPU: the clock-record summary that
decides whether a timed run saw a throttle reason (CPU only)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _summary(lines):
    c = bench.ClockSampler(0)
    c.lines = list(lines)
    return c.summary()


def test_clock_summary_median_max_and_power_cap():
    rows = ["0, 2032, 2070, 1100.50, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
            "0, 2040, 2070, 1180.25, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
            "0, 1995, 2070, 1390.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"]
    s = _summary(rows)
    assert s["sm_mhz"] == 2032.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3


def test_clock_summary_reports_rejecting_reasons_and_skips_bad_lines():
    rows = ["0, 1500, 2070, 900.0, 0x08, Active, Not Active, Not Active, Not Active",
            "0, 1400, 2070, 900.0, 0x40, Not Active, Active, Active, Not Active",
            "garbage",
            "0, [N/A], 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            ""]
    s = _summary(rows)
    assert s["samples"] == 2 and s["sm_mhz"] == 1450.0
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples():
    s = _summary([])
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == ["unsampled"]
