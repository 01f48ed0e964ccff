"""bench.py's CPU legs, run as a user runs them (no GPU): the reference arm's
JSON line and the oracle leg that the GPU arm starts as a child process."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*argv):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv], capture_output=True, text=True,
                       timeout=300, env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_reference_arm_line():
    d = _run("--impl", "reference", "--workload", "tiny-decode", "--steps", "2", "--warmup", "3",
             "--ref-seconds", "1")
    assert d["impl"] == "reference"
    assert d["unit"] == "GB/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"] == {"workload": "tiny-decode"}
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_oracle_leg_line():
    d = _run("--oracle-leg", "--workload", "t5-small-decode", "--cpu-seconds", "1")
    assert d["unit"] == "GB/s" and d["value"] > 0 and d["kind"] == "oracle"
    assert "drawn on the host" in d["sample"]
