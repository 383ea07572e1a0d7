"""bench.py's GPU arm on the tiny workload: one JSON line carrying every key of the benchmark
contract -- the metric and its value, the roofline of the dominant kernel, the end-to-end figure
with its host<->device bytes, the kernel launch count, the clocks sampled during the timed region
and the CPU oracle baseline."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_carries_the_contract():
    r = subprocess.run([sys.executable, "bench.py", "--workload", "tiny_decode", "--steps", "5", "--warmup", "3",
                        "--no-configs", "--cpu-seconds", "1"], cwd=ROOT, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["config"]["workload"] == "tiny_decode"
    rf = d["roofline"]
    assert rf["bound"] in ("hbm", "tensor", "alu") and rf["peak"] > 0 and rf["achieved"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    c = d["clocks"]
    assert c["sm_max_mhz"] > 0 and isinstance(c["reasons"], list)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
