"""bench.py --impl reference: the oracle timed on the host cores prints one JSON
line with the same metric and unit as the GPU arm, its own cpu_baseline and an
e2e entry with no host/device copies. Runs on the CPU in a few seconds."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*extra):
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", *extra], cwd=ROOT, capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_line_contract():
    d = _run("--steps", "1", "--warmup", "3")
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] >= 3
    assert d["unit"] == "us" and d["higher_is_better"] is False
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["dtype"] == "f64" and d["data"] == "synthetic"
    assert "qwen_decode" in d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_keeps_three_warmup_steps():
    assert _run("--steps", "1", "--warmup", "0")["warmup"] >= 3
