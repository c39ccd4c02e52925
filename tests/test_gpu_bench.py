"""The benchmark's own arm on the GPU: one JSON line with the keys of the contract.

Runs `bench.py` on the smallest workload (a few steps) and checks the line's shape:
the metric, the roofline of the dominant kernel with its measured peak, the end-to-end
figure with the bytes its copies move, the launch count and the clock record.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_carries_the_contract_keys():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--config", "0", "--steps", "3",
                          "--warmup", "3", "--no-cpu-baseline"], cwd=ROOT, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks",
                "kernels"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["steps"] == 3 and d["n_gpus"] == 1
    roof = d["roofline"]
    assert roof["bound"] in ("hbm", "tensor") and roof["peak"] > 0 and roof["achieved"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    assert "plan" in d["kernels"] and "gemm_wgrad13" in d["kernels"]
