"""The benchmark's command-line contract on CPU: the reference arm (the float64 oracle on
the host cores) prints one JSON line with the keys the contract names, and our arm fails
loudly, with a non-zero exit status and no JSON line, when there is no GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=300):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                          text=True, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    r = _run("--impl", "reference", "--steps", "1", "--warmup", "1")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] >= 3  # the contract's minimum warm-up is enforced
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["vs_baseline"] is None and d["data"] == "synthetic"


def test_our_arm_fails_loudly_without_a_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = _run("--steps", "1", "--warmup", "3", timeout=120)
    assert r.returncode != 0
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_roofline_peak_rule():
    """The roofline fraction divides by the burst peak for a short timed region or one held at
    the maximum SM clock, by the sustained peak for a long region below it."""
    import bench
    assert bench.roofline_peak(57.0, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0})[0] == "burst"
    assert bench.roofline_peak(57.0, {"unavailable": "no samples"})[0] == "burst"
    assert bench.roofline_peak(1500.0, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0})[0] == "burst"
    assert bench.roofline_peak(1500.0, {"sm_mhz": 1942.0, "sm_max_mhz": 2070.0})[0] == "sustained"
    assert bench.roofline_peak(1500.0, {"unavailable": "no samples"})[0] == "sustained"


def test_clock_samples_are_taken_from_inside_the_timed_region():
    """Only the nvidia-smi samples stamped inside the timed region describe it: a sample
    before or after (an idle GPU at full clock) is left out, the stamps' time zone is
    recovered from when the samples arrived, and a region shorter than the sampling
    interval reports no clock rather than the idle one."""
    import datetime
    import bench

    zone = 3600.0  # the stamps are an hour ahead of the host's epoch time
    t_begin, t_end = 1_000_000.0, 1_000_000.1

    def line(t, sm, power, cap="Not Active"):
        stamp = datetime.datetime.fromtimestamp(t + zone).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return (t + 0.002, f"{stamp}, 0, {sm}, 2070, {power}, 0x0, Not Active, Not Active, Not Active, {cap}")

    s = bench.ClockSampler("0", start=False)
    s.lines = [line(t_begin - 0.05, 2070, 150.0), line(t_begin + 0.01, 1900, 900.0, "Active"),
               line(t_begin + 0.05, 1800, 1300.0, "Active"), line(t_begin + 0.09, 1850, 1200.0),
               line(t_end + 0.03, 2070, 1000.0), (t_end, "not, a, sample")]
    s.t_begin, s.t_end = t_begin, t_end
    r = s.summary()
    assert r["samples"] == 3 and r["samples_total"] == 5
    assert r["sm_mhz"] == 1850 and r["sm_min_mhz"] == 1800 and r["sm_max_mhz"] == 2070
    assert r["power_w_max"] == 1300.0 and r["reasons"] == ["sw_power_cap"]
    assert bench.roofline_peak(1500.0, r)[0] == "sustained"

    s.t_begin, s.t_end = t_begin + 0.06, t_begin + 0.08  # between two samples
    r = s.summary()
    assert r["samples"] == 0 and r["sm_mhz"] is None and "note" in r
    assert bench.roofline_peak(20.0, r)[0] == "burst"
