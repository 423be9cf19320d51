"""The bench's JSON line for the reference arm (the oracle on the host cores), on the tiny workload: the keys
and units the contract names, as one parseable line, without a GPU.  The GPU arm's line carries the same
keys plus roofline, clocks, e2e and gpu_launches (checked on the GPU machine by running the bench itself)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "1", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["unit"] == "us/layer-step" and d["higher_is_better"] is False
    assert d["value"] > 0 and abs(d["ms_per_step"] * 1e3 - d["value"]) <= 1e-6 * d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "1", "--steps", "1",
                        "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr
