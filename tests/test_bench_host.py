"""Host-side logic of bench.py that needs no GPU: the summary of the clock
samples (nvidia-smi CSV lines, here written by hand in its format) that goes
into the bench line's "clocks" object, overall and per timed region; the
choice of the tensor peak from those clocks; the DRAM/algorithmic traffic
ratio, valid only for the kernel source it was captured on; and the reference
arm's JSON line (the oracle timed on the host)."""
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


def test_tensor_peak_follows_the_clock():
    peaks = dict(hbm=6000.0, bf16=1800.0, bf16_sus=1400.0, max_mhz=2032.0, source="measured")
    p, why = bench.tensor_peak(peaks, {"sm_mhz": 2010.0, "sm_max_mhz": 2032.0})
    assert p == 1800.0 and "at the maximum" in why
    p, why = bench.tensor_peak(peaks, {"sm_mhz": 1524.0, "sm_max_mhz": 2032.0})
    assert abs(p - 1800.0 * 1524.0 / 2032.0) < 1e-9 and "1524" in why
    p, _ = bench.tensor_peak(peaks, None)          # no clock record: the burst figure
    assert p == 1800.0


def test_traffic_ratio_is_tied_to_the_kernel_source(tmp_path):
    src = os.path.join(ROOT, "decoder_only_transformer_06_b300", "csrc", "k_gemm_tc.cu")
    r = bench.traffic_ratio_from_profiles(src)
    # the committed capture names the current source's hash, so its ratio applies
    assert r is not None and 0.0 < r < 2.0
    other = tmp_path / "k_gemm_tc.cu"
    other.write_bytes(open(src, "rb").read() + b"\n// changed\n")
    assert bench.traffic_ratio_from_profiles(str(other)) is None
    assert bench.traffic_ratio_from_profiles(str(tmp_path / "missing.cu")) is None


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference times the oracle on the host (no GPU needed):
    one JSON line with the contract's keys, on the small character workload."""
    import json
    import subprocess
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "char", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    d = json.loads(out.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    for k in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config"):
        assert k in d, k
    assert d["config"]["workload"] == "char"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
