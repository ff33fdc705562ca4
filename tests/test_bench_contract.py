"""The benchmark's one-line JSON contract, on a small workload (GPU)."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.gpu
def test_bench_line_has_the_contract_keys():
    d = run_bench("--workload", "plummer_16384", "--steps", "3", "--warmup", "3", "--cpu-seconds", "0.5")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "gpu_launches", "clocks", "roofline", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "plummer_16384" and "model" not in d["config"]
    assert d["gpu_launches"] >= 3 * 12  # every phase of every timed step is one of ours
    r = d["roofline"]
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s" and 0 < r["frac"] < 1.5
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert r["peak_measured_fma"]["scalar"] > 0 and r["peak_measured_fma"]["packed"] > 0
    assert r["peak_measured_fma"]["sm_mhz"] > 0
    assert 0 < r["frac_of_measured_fma"] < 1.5
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == 16 * 16384 and e["d2h_bytes_per_step"] == 24 * 16384
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}


@pytest.mark.gpu
def test_reference_arm_line():
    d = run_bench("--impl", "reference", "--workload", "plummer_16384", "--steps", "1", "--warmup", "0",
                  "--cpu-seconds", "0.5")
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
