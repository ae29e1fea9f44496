"""Our arm of the benchmark on a GPU: one JSON line with the keys the
benchmark contract names (metric, value, roofline with its peak and
fraction, cpu_baseline, e2e with the copied bytes, gpu_launches, clocks),
on the small workloads so the run takes seconds."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("workload,cpu", [("tiny_fp32", True), ("gptoss_decode", False)])
def test_our_arm_json_line(workload, cpu):
    args = ["--steps", "3", "--warmup", "3", "--workload", workload, "--no-all-workloads"]
    if not cpu:
        args.append("--no-cpu-baseline")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "roofline",
                "cpu_baseline", "e2e", "gpu_launches", "clocks", "layer_roofline", "kernels"):
        assert key in j, key
    assert j["n_gpus"] == 1 and j["steps"] == 3 and j["warmup"] == 3
    assert j["value"] > 0 and j["ms_per_step"] > 0
    rf = j["roofline"]
    assert rf["bound"] in ("tensor", "hbm") and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    e2e = j["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert j["gpu_launches"] > 0 and j["gpu_launches"] % 3 == 0  # the same launches each step
    if cpu:
        assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["value"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(j["clocks"])
    assert j["kernels"]["same_output_as_moe_forward"] is True
