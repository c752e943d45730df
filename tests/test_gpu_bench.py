"""bench.py's own arm on a small workload: one JSON line carrying the
contract's keys (metric, value, roofline with the measured peak, e2e with its
host<->device bytes, clocks, launch count, CPU baseline, per-workload
records), with value equal to the fold's algorithmic bytes over its time."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_on_the_toy_group():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "toy", "--steps", "6", "--warmup", "3",
           "--no-variants", "--no-baseline", "--no-interference", "--no-per-config", "--e2e-steps", "3",
           "--cpu-seconds", "1"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-3000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks",
              "step", "parts"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 6 and d["warmup"] >= 3 and d["unit"] == "GB/s"
    assert d["config"]["workload"] == "toy"
    assert d["gpu_launches"] == 2 * 6  # one fold and one placement per timed step
    fold = d["parts"]["rs_fold"]
    assert abs(d["value"] - fold["alg_bytes"] / (fold["ms"] * 1e-3) / 1e9) <= 0.01 * d["value"] + 0.1
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["peak"] > 0 and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["readback_matches_device"] is True and e["staged"]["readback_matches_device"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
