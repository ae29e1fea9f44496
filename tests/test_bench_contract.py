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


def test_gemm_peak_follows_the_sampled_clocks():
    """Burst peak unless the power cap actually held the SM clock down."""
    import bench
    pk = {"hbm_gbs": 6777.0, "bf16_tflops": 1919.4, "bf16_tflops_sustained": 1711.7}
    assert bench.gemm_peak(pk, {"reasons": [], "sm_mhz": 2070.0, "sm_max_mhz": 2070.0})[0] == 1919.4
    assert bench.gemm_peak(pk, {"reasons": ["sw_power_cap"], "sm_mhz": 2070.0,
                                "sm_max_mhz": 2070.0})[0] == 1919.4
    assert bench.gemm_peak(pk, {"reasons": ["sw_power_cap"], "sm_mhz": 1500.0,
                                "sm_max_mhz": 2070.0})[0] == 1711.7


def test_layer_roofline_is_the_slower_bound():
    """FLOPs 2TdE + 6Pdf at the tensor peak against the touched experts'
    weights + x + out + Wr at the HBM peak; the slower decides."""
    import bench
    from token_dispatch_grouped_fp32_gb300 import synth
    pk = {"hbm_gbs": 6777.0}
    w = synth.WORKLOADS["mixtral"]
    r = bench.layer_roofline(w, 8, 1.8, pk, 1919.4)
    flops = 2 * 4096 * 4096 * 8 + 6 * 8192 * 4096 * 14336
    assert r["flops"] == flops and r["bound"] == "tensor"
    assert abs(r["frac"] - flops / 1919.4e12 / 1.8e-3) < 1e-12
    d = synth.WORKLOADS["gptoss_decode"]
    r = bench.layer_roofline(d, 111, 0.85, pk, 1919.4)
    nbytes = 111 * 3 * 2880 * 2880 * 2 + 2 * 64 * 2880 * 2 + 4 * 128 * 2880
    assert r["bytes"] == nbytes and r["bound"] == "hbm"
    assert abs(r["frac"] - nbytes / 6777e9 / 0.85e-3) < 1e-12


def test_forward_path_follows_the_workspace_layout():
    """The bench's description of how moe_forward moves the rows comes from
    the library's layout query (no x_perm region: no permuted copy)."""
    import bench
    from token_dispatch_grouped_fp32_gb300 import moe, synth

    def path(name, **kw):
        w = synth.WORKLOADS[name].with_(**kw)
        cfg = moe.config(w.T, w.d, w.E, w.k, w.f, w.dtype, w.renorm, scale_inputs=w.scale_inputs)
        return bench.forward_path(moe, cfg, w)

    assert path("mixtral").startswith("rows copied into x_perm")
    assert "scaled by their weights" in path("mixtral", scale_inputs=True)
    assert path("qwen3_zipf").startswith("the first grouped GEMM gathers")
    assert "bit-identical" in path("deepseek")
    assert path("gptoss_prefill").startswith("the first grouped GEMM gathers")
    assert "inside the first grouped GEMM" in path("qwen3_zipf", scale_inputs=True)
    assert path("mixtral_dense").startswith("every expert reads x itself")
    assert path("tiny_fp32").startswith("rows copied")  # fp32: no gather
