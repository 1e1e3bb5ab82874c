"""bench.py's JSON line on a GB300: every key of the benchmark contract is
there, and the numbers in it are consistent with one another.

A short run on the 5-row fp32 workload (a few seconds, most of them the
oracle's timed sample and the clock sampler's start and stop).
"""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
from paged_kv_decode_nsv_gb300 import workloads as W  # noqa: E402


@pytest.mark.gpu
def test_bench_line_carries_the_contract():
    steps = 3
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny_f32",
           "--steps", str(steps), "--warmup", "3", "--e2e-steps", str(steps),
           "--cpu-seconds", "0.5"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] >= 3
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["dtype"] == "f32" and d["config"]["workload"] == "tiny_f32"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # value: the step's algorithmic bytes over the step's time
    wl = W.WORKLOADS["tiny_f32"]()
    assert d["value"] == pytest.approx(wl.step_bytes() / (d["ms_per_step"] * 1e-3) / 1e9,
                                       rel=1e-6)
    assert d["roofline"]["bytes_per_launch"] == wl.read_bytes()
    # roofline: the read's algorithmic bytes over its own launch time, against the peak
    rl = d["roofline"]
    assert rl["bound"] == "hbm" and rl["unit"] == "GB/s" and rl["peak"] > 0
    assert rl["achieved"] == pytest.approx(
        rl["bytes_per_launch"] / (rl["us_per_launch"] * 1e-6) / 1e9, rel=1e-6)
    assert rl["frac"] == pytest.approx(rl["achieved"] / rl["peak"], rel=1e-9)
    assert "traffic" in rl
    # e2e: the same metric with the step's host copies inside the timed region
    e2e = d["e2e"]
    assert e2e["unit"] == "GB/s" and e2e["value"] > 0
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["ms_per_step"] >= d["ms_per_step"] * 0.5
    # two launches per timed step: the append (which zeroes the arrival
    # counters) and the read
    assert d["gpu_launches"] == 2 * steps
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s" and cb["value"] > 0
    assert cb["cores"] >= 1 and cb["sample"]
    clocks = d["clocks"]
    assert "sm_mhz" in clocks and "reasons" in clocks
