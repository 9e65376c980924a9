"""bench.py's decode arm on the GPU: one short run checked against the JSON
line contract (keys, units, timed-step count, the roofline fraction's
consistency with the timed region).  37 steps over 4 working sets leave a
remainder after the graph replays, so both parts of the timed region run."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_decode_bench_line_contract():
    cmd = [sys.executable, "bench.py", "--workload", "b1_l3297", "--steps", "37", "--warmup", "3",
           "--working-sets", "4", "--e2e-steps", "2", "--no-cpu-baseline", "--roofline-launches", "16"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks", "timing",
              "direct", "graph"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 37 and d["warmup"] == 3
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["data"] == "synthetic"
    assert d["gpu_launches"] == 37
    assert "9 replays of a CUDA graph of 4 calls" in d["timing"] and "+ 1 direct calls" in d["timing"]
    roof = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in roof, k
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["timed_launches"] == 37
    # every launch of the timed region is the decode kernel: the achieved rate is the line's value
    assert abs(roof["achieved"] - d["value"]) <= 1e-6 * d["value"]
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert abs(d["ms_per_step"] * 1e3 - roof["kernel_avg_us"]) < 1e-6 * roof["kernel_avg_us"]
    assert d["direct"]["us_per_call"] > 0 and d["graph"]["us_per_call"] > 0
    assert len(d["graph"]["samples_us"]) == 5
    e2e = d["e2e"]
    assert e2e["unit"] == "GB/s" and e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["clocks"]["sm_mhz"] is not None
