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
