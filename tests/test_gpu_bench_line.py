"""bench.py end to end on the GPU, on the small 128^3 workload with short
legs: it exits 0 and prints one JSON line with every key the benchmark
contract asks for, the roofline and e2e objects filled in, and the launch
count the library reports."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_bench_prints_one_complete_line():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "square_128_f16",
           "--steps", "20", "--warmup", "3", "--e2e-steps", "3", "--no-cpu-baseline",
           "--sustained-seconds", "0.2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks", "sustained"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "square_128_f16"
    assert d["config"]["kernel"] == "tile16"
    roof = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    e2e = d["e2e"]
    assert e2e["value"] > 0
    assert e2e["h2d_bytes_per_step"] == (128 * 128 + 128 * 128) * 2   # A and B, FP16
    assert e2e["d2h_bytes_per_step"] == 128 * 128 * 4
    assert e2e["link"]["h2d_gbs"] > 0 and e2e["link"]["d2h_gbs"] > 0
    assert d["gpu_launches"] == 20          # one single-tile launch per step
    assert d["sustained"]["value"] > 0
