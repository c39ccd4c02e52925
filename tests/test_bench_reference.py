"""The benchmark's reference arm on CPU: one JSON line with the keys of the contract.

`bench.py --impl reference` times the CPU oracle on the chosen workload's metric and
unit; it needs no GPU, so the shape of its line is checked here on the smallest
workload.  (The GPU arm's line is exercised by the GPU runs.)
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_arm_prints_one_contract_line():
    d = _run("--impl", "reference", "--config", "0", "--steps", "1", "--warmup", "3")
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["data"] == "synthetic"
    assert d["config"]["T"] == 256 and d["config"]["E"] == 8
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_raises_short_warmup_to_three():
    d = _run("--impl", "reference", "--config", "0", "--steps", "1", "--warmup", "1")
    assert d["warmup"] == 3
