"""Host-side logic of bench.py that needs no GPU: the summary of the clock
samples (nvidia-smi CSV lines, here written by hand in its format) that goes
into the bench line's "clocks" object, overall and per timed region."""
import datetime
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(t, sm, reasons=("Not Active",) * 4):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([stamp, "0", str(sm), "2032", "900.00", "0x0000000000000004", *reasons]) + "\n"


def test_clock_summary_overall_and_by_region():
    t0 = 1_800_000_000.0
    lines = [_line(t0 + 0.1 * i, sm) for i, sm in enumerate([1900, 1800, 1700, 1600, 1500, 1400])]
    lines.append(_line(t0 + 0.7, 1300, ("Not Active", "Not Active", "Not Active", "Active")))
    lines.append("garbage line\n")
    out = bench.ClockSampler.summarize(
        lines, {"device_timed": (t0 - 0.01, t0 + 0.25), "e2e": (t0 + 0.35, t0 + 0.75), "none": (t0 + 5, t0 + 6)})
    assert out["samples"] == 7
    assert out["sm_mhz"] == 1600
    assert out["sm_max_mhz"] == 2032
    assert out["reasons"] == ["sw_power_cap"]
    assert out["by_region"]["device_timed"] == {"sm_mhz": 1800, "samples": 3}
    assert out["by_region"]["e2e"] == {"sm_mhz": 1400, "samples": 3}
    assert out["by_region"]["none"] == {"sm_mhz": None, "samples": 0}


def test_clock_summary_throttle_reasons_and_no_regions():
    lines = [_line(1_800_000_000.0, 1500, ("Active", "Not Active", "Active", "Not Active"))]
    out = bench.ClockSampler.summarize(lines)
    assert out["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert "by_region" not in out
    assert bench.ClockSampler.summarize(["\n"]) is None
