"""The bench's reference arm runs on the CPU: check its JSON line against the
contract (one line, the metric and units of our arm, the cpu_baseline and e2e
objects) on the small fp32 workload, and that the arm refuses a warm-up
below three steps."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_json_line():
    r = _run("--impl", "reference", "--workload", "tiny_fp32", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    assert j["unit"] == "tokens/s" and j["higher_is_better"] is True
    assert j["steps"] == 3 and j["warmup"] == 3 and j["n_gpus"] == 1
    assert j["value"] > 0 and j["ms_per_step"] > 0
    assert j["config"]["workload"].startswith("tiny_fp32")
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == j["value"] and cb["cores"] >= 1 and cb["sample"]
    assert j["e2e"] == {"value": j["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_warmup_below_three_is_rejected():
    r = _run("--impl", "reference", "--workload", "tiny_fp32", "--steps", "2", "--warmup", "1")
    assert r.returncode != 0
    assert "warmup" in r.stderr
