"""bench.py end to end on the GPU: a short run of one workload prints one JSON
line with the keys of the benchmark contract, a roofline consistent with its
own timing, and an end-to-end figure that moved bytes over the host link."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_contract():
    cmd = [sys.executable, "bench.py", "--workload", "fp8", "--slots", "65536", "--steps", "20",
           "--warmup", "3", "--suite", "none", "--no-cpu-baseline", "--long-ms", "1",
           "--e2e-steps", "3"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks", "timing", "per_config"):
        assert key in line, key
    assert (line["steps"], line["warmup"], line["n_gpus"]) == (20, 3, 1)
    assert line["gpu_launches"] == 20 and line["higher_is_better"] is True
    cfg = line["config"]
    assert cfg["tokens_per_step"] == 8192 and cfg["bytes_per_step"] == 50397184
    assert line["value"] == pytest.approx(cfg["tokens_per_step"] / (line["ms_per_step"] / 1e3))
    r = line["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert r["achieved"] == pytest.approx(cfg["bytes_per_step"] / (line["ms_per_step"] / 1e3) / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"]) and 0.2 < r["frac"] < 1.3
    head = line["timing"]["headline"]
    assert head["calls"] == 20 and head["us_per_call_long"] > 0
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["mode"] in ("staged", "zero_copy")
