"""Benchmark: MoE-layer forward tokens/s on GB300 through libmoe's C ABI.

Default workload: the Mixtral-8x7B-shaped layer (T=4096 tokens, d=4096, E=8,
k=2, f=14336, bf16 activations and experts, fp32 router and accumulation),
seeded synthetic inputs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

One JSON line is printed by rank 0.  `value` is whole-job tokens/s with the
inputs resident in HBM (device-timed with CUDA events, per step, L2 flushed
between steps); `e2e` is the same metric through moe_forward_host with the
activations in pinned host memory (copies inside the timed region).
For N > 1 (torchrun) every rank runs its own batch of T tokens on its own GPU
(no data-path collective: tokens are independent), timing is the max over
ranks, and `scaling` is "weak".

The line also carries: `roofline` (the grouped GEMM against the bf16 tensor
peak: the burst figure, or the sustained one when the clocks sampled in the
timed region show sw_power_cap), `layer_roofline` (the slower of the layer's
FLOPs at that peak and its minimal HBM bytes at the HBM peak, against the
step time), a per-kernel breakdown, and `all_workloads`: the other
workloads timed the same way (K steps each, L2 flushed between steps).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s on 1 GB300; GEMM % tensor peak, permute/combine % HBM BW"
# every bf16 workload of the benchmark; the one named by --workload (default
# mixtral) is the headline line, the others go in its all_workloads block
ALL_WORKLOADS = ["mixtral", "gptoss_decode", "gptoss_prefill", "qwen3_zipf", "deepseek",
                 "mixtral_norenorm", "mixtral_dense"]
L2_FLUSH_BYTES = 256 << 20


# --------------------------------------------------------------------------
# multi-rank helpers (also exercised by the CPU gloo tests)
# --------------------------------------------------------------------------
def dist_env():
    """(rank, local_rank, world_size) from the torchrun environment."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate_throughput(units_per_rank: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    return units_per_rank * world / max_seconds


# --------------------------------------------------------------------------
# measurement helpers
# --------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]),
                             "power": float(parts[3]) if parts[3] not in ("[N/A]", "") else None,
                             "hw": parts[5], "hw_thermal": parts[6], "sw_thermal": parts[7],
                             "sw_power": parts[8]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm_max = max(r["max"] for r in rows)
        # "under load": samples whose power is within 30% of the run's peak power
        pw = [r["power"] for r in rows if r["power"] is not None]
        pmax = max(pw) if pw else None
        loaded = [r for r in rows if pmax is None or (r["power"] or 0) >= 0.7 * pmax] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": sm_max,
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": pmax}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# --------------------------------------------------------------------------
# the CPU oracle (reference arm and the cpu_baseline field)
# --------------------------------------------------------------------------
def oracle_sample_tokens_per_s(inp, w, budget_s: float, max_tokens: int):
    """Time the oracle's whole-layer forward on the first n tokens of the
    workload, n sized to about `budget_s` seconds of host work.
    Returns (tokens_per_s, n, seconds, threads)."""
    import numpy as np
    from oracle import oracle

    x = inp["x"].float().cpu().numpy()
    Wr = inp["Wr"].float().cpu().numpy()
    Wgu = inp["Wgu"].float().cpu().numpy()
    Wd = inp["Wd"].float().cpu().numpy()
    bias = None if inp["bias"] is None else inp["bias"].float().cpu().numpy()
    oracle.build()
    n = min(max_tokens, 8)
    t0 = time.perf_counter()
    oracle.moe_forward(x[:n], Wr, Wgu, Wd, w.k, renorm=w.renorm, bias=bias,
                       scale_inputs=w.scale_inputs)
    dt = time.perf_counter() - t0
    n = int(max(1, min(max_tokens, n * budget_s / max(dt, 1e-6))))
    t0 = time.perf_counter()
    oracle.moe_forward(np.ascontiguousarray(x[:n]), Wr, Wgu, Wd, w.k, renorm=w.renorm, bias=bias,
                       scale_inputs=w.scale_inputs)
    dt = time.perf_counter() - t0
    return n / dt, n, dt, oracle.num_threads()


def run_reference(args, w):
    import torch
    from oracle import oracle
    from token_dispatch_grouped_fp32_gb300 import synth

    rank, _, world = dist_env()
    if rank != 0:
        return
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = synth.make_inputs(w, device=gen_dev)
    x = inp["x"].float().cpu().numpy()
    Wr = inp["Wr"].float().cpu().numpy()
    Wgu = inp["Wgu"].float().cpu().numpy()
    Wd = inp["Wd"].float().cpu().numpy()
    del inp["Wgu"], inp["Wd"]
    bias = None if inp["bias"] is None else inp["bias"].float().cpu().numpy()
    oracle.build()
    # size each step to ~ step_s seconds of host work, so that the whole run
    # (K steps) stays near two minutes: 4 s per step for a few steps, down to
    # 0.25 s per step for long runs
    step_s = args.ref_step_s
    if step_s is None:
        step_s = min(4.0, max(0.25, 120.0 / max(1, args.steps)))
    n = min(w.T, 4)
    t0 = time.perf_counter()
    oracle.moe_forward(x[:n], Wr, Wgu, Wd, w.k, renorm=w.renorm, bias=bias,
                       scale_inputs=w.scale_inputs)
    dt = time.perf_counter() - t0
    n = int(max(1, min(w.T, n * step_s / max(dt, 1e-6))))
    for _ in range(args.warmup if args.ref_warmup else 0):
        oracle.moe_forward(x[:n], Wr, Wgu, Wd, w.k, renorm=w.renorm, bias=bias,
                       scale_inputs=w.scale_inputs)
    times = []
    for s in range(args.steps):
        lo = (s * n) % max(1, w.T - n + 1)
        xs = x[lo:lo + n]
        t0 = time.perf_counter()
        oracle.moe_forward(xs, Wr, Wgu, Wd, w.k, renorm=w.renorm, bias=bias,
                       scale_inputs=w.scale_inputs)
        times.append(time.perf_counter() - t0)
    value = n * len(times) / sum(times)
    threads = oracle.num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n} consecutive tokens of the workload per step "
                                   f"(whole layer: route, dispatch, experts, combine)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w):
    weights = "renormalised top-k weights" if w.renorm else "top-k softmax weights (not renormalised)"
    return {"workload": f"{w.name}: T={w.T} d={w.d} E={w.E} k={w.k} f={w.f} {w.dtype}, {weights}"
                        f"{', Zipf-skewed routing' if w.zipf else ''}"
                        f"{', routing weights on the expert inputs' if w.scale_inputs else ''}",
            "T": w.T, "d": w.d, "E": w.E, "k": w.k, "f": w.f, "seed": w.seed,
            "l2": "256 MiB L2 flush between timed steps (per-step working set "
                  "also exceeds L2)"}


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------
def gemm_peak(peaks, clocks):
    """The bf16 tensor peak the timed GEMM is held to: the sustained
    (power-capped) figure when the power cap actually held the clock down in
    the timed region (sw_power_cap active under load and the median SM clock
    below 97 % of its maximum), else the burst figure.  (nvidia-smi can show
    sw_power_cap active while the clock stays at its maximum.)"""
    reasons = clocks.get("reasons") or []
    sm, sm_max = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    held = sm is not None and sm_max and sm < 0.97 * sm_max
    if "sw_power_cap" in reasons and held and peaks.get("bf16_tflops_sustained"):
        return (peaks["bf16_tflops_sustained"],
                f"bf16_tflops_sustained (sw_power_cap held the clock at {sm:.0f} MHz)")
    note = "sw_power_cap shown, clock at maximum" if "sw_power_cap" in reasons else "no power cap"
    return peaks["bf16_tflops"], f"bf16_tflops (burst: {note})"


def layer_roofline(w, touched, ms, peaks, tflops_peak):
    """The layer's roofline: the slower of its FLOPs at the tensor peak and
    its minimal HBM bytes at the HBM peak, against the measured step time.
    FLOPs: 2*T*d*E (router) + 6*P*d*f (experts).  Bytes: the weights of the
    experts that received rows, x, out and the router weight."""
    es = 2 if w.dtype == "bf16" else 4
    P = w.T * w.k
    flops = 2.0 * w.T * w.d * w.E + 6.0 * P * w.d * w.f
    nbytes = touched * 3.0 * w.d * w.f * es + 2.0 * w.T * w.d * es + 4.0 * w.E * w.d
    t_flops = flops / (tflops_peak * 1e12)
    t_bytes = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_min = max(t_flops, t_bytes)
    return {"bound": "tensor" if t_flops >= t_bytes else "hbm", "frac": t_min / (ms * 1e-3),
            "t_roofline_ms": 1e3 * t_min, "ms": ms, "flops": flops, "bytes": nbytes,
            "touched_experts": int(touched), "peak_tflops": tflops_peak,
            "peak_hbm_gbs": peaks["hbm_gbs"]}


def measure_workload(moe, w, args, dev, rank, world, flush, with_e2e):
    """Times moe_forward on workload w (K steps, L2 flushed between steps),
    then the same launch sequence through the component entry points for the
    per-kernel breakdown, and (with_e2e) the host-buffer path."""
    import torch
    from token_dispatch_grouped_fp32_gb300 import synth

    wr = w.with_(seed=w.seed + 100 * rank) if world > 1 else w
    inp = synth.make_inputs(wr, device=dev)
    x, Wr, Wgu, Wd = inp["x"], inp["Wr"], inp["Wgu"], inp["Wd"]
    bias = inp["bias"]
    layer = moe.MoELayer(Wr, Wgu, Wd, w.k, bias, w.renorm, w.scale_inputs)
    T = w.T
    cfg = layer.config(T)
    ws = layer.workspace(T)
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream()

    def step():
        moe.moe_forward(cfg, x, Wr, bias, Wgu, Wd, out, ws, stream=stream)

    # warm-up: the layer and the L2 flush both run before the timed region
    for i in range(args.warmup):
        flush.fill_(float(-i))
        step()
    torch.cuda.synchronize()
    moe.moe_last_device_error()

    # ---- timed region: K steps of moe_forward, per-step events ----
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    with ClockSampler(dev.index) as clocks:
        barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        barrier()
        t_wall = time.perf_counter() - t_wall
    step_ms = [a.elapsed_time(b) for a, b in evs]
    moe.moe_last_device_error()
    ms = max_over_ranks(sum(step_ms) / len(step_ms), dev)
    clk = clocks.summary()
    L = moe.moe_workspace_layout(cfg)
    counts = ws[L.counts:L.counts + 4 * w.E].view(torch.int32).cpu()
    touched = int((counts > 0).sum())

    # ---- per-kernel breakdown: the same launch sequence through the
    # component entry points, events between the calls ----
    P = T * w.k
    logits = torch.empty(T, w.E, dtype=torch.float32, device=dev)
    idx = torch.empty(T, w.k, dtype=torch.int32, device=dev)
    wt = torch.empty(T, w.k, dtype=torch.float32, device=dev)
    cnt = torch.empty(w.E, dtype=torch.int32, device=dev)
    offsets = torch.empty(w.E + 1, dtype=torch.int32, device=dev)
    pos = torch.empty(P, dtype=torch.int32, device=dev)
    src = torch.empty(P, dtype=torch.int32, device=dev)
    x_perm = torch.empty(P, w.d, dtype=x.dtype, device=dev)
    h_perm = torch.empty(P, w.f, dtype=x.dtype, device=dev)
    y_perm = torch.empty(P, w.d, dtype=x.dtype, device=dev)
    out2 = torch.empty_like(x)
    dws = torch.empty(max(256, moe.moe_dispatch_workspace_size(cfg)), dtype=torch.uint8, device=dev)
    rws = torch.empty(max(256, moe.moe_route_workspace_size(cfg)), dtype=torch.uint8, device=dev)
    names = ["route", "dispatch", "grouped_swiglu", "combine"]

    def parts(ev=None):
        if ev: ev[0].record(stream)
        moe.moe_route(cfg, x, Wr, bias, logits, idx, wt, rws, stream=stream)
        if ev: ev[1].record(stream)
        moe.moe_dispatch(cfg, idx, wt, x, cnt, offsets, pos, src, x_perm, dws, stream=stream)
        if ev: ev[2].record(stream)
        moe.moe_grouped_swiglu(cfg, x_perm, offsets, Wgu, Wd, h_perm, y_perm, stream=stream)
        if ev: ev[3].record(stream)
        moe.moe_combine(cfg, y_perm, pos, None if w.scale_inputs else wt, out2, stream=stream)
        if ev: ev[4].record(stream)

    for _ in range(args.warmup):
        parts()
    torch.cuda.synchronize()
    per = {n: [] for n in names}
    for i in range(args.steps):
        flush.fill_(float(i))
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        parts(ev)
        torch.cuda.synchronize()
        for j, n in enumerate(names):
            per[n].append(ev[j].elapsed_time(ev[j + 1]))
    same_as_fused = bool(torch.equal(out, out2))
    kms = {n: sum(v) / len(v) for n, v in per.items()}

    peaks = measured_peaks()
    peak, peak_name = gemm_peak(peaks, clk)
    es = 2 if w.dtype == "bf16" else 4
    gemm_flops = 6.0 * P * w.d * w.f
    gemm_tflops = gemm_flops / (kms["grouped_swiglu"] * 1e-3) / 1e12
    weight_bytes = touched * 3.0 * w.d * w.f * es
    # minimal HBM bytes of the bandwidth kernels: dispatch reads each token row
    # once and writes each permuted row once (+ four int32 arrays of P);
    # combine reads the permuted rows and the (pos, weight) pairs and writes
    # the token rows; route reads x and writes the logits twice (partial sums
    # and the final logits) plus the selection
    disp_bytes = T * w.d * es + P * w.d * es + P * 4 * 4
    comb_bytes = P * w.d * es + P * 8 + T * w.d * es
    route_bytes = T * w.d * es + T * w.E * 4 * 2 + P * 8
    hbm = peaks["hbm_gbs"]
    kernels = {
        "route": {"ms": kms["route"], "GB/s": route_bytes / kms["route"] / 1e6},
        "dispatch": {"ms": kms["dispatch"], "GB/s": disp_bytes / kms["dispatch"] / 1e6,
                     "frac_hbm": disp_bytes / kms["dispatch"] / 1e6 / hbm},
        "grouped_swiglu": {"ms": kms["grouped_swiglu"], "TFLOP/s": gemm_tflops,
                           "frac_tensor": gemm_tflops / peak,
                           "frac_of_burst_peak": gemm_tflops / peaks["bf16_tflops"],
                           "weight_stream_GB/s": weight_bytes / kms["grouped_swiglu"] / 1e6,
                           "frac_hbm_weight_stream":
                               weight_bytes / kms["grouped_swiglu"] / 1e6 / hbm},
        "combine": {"ms": kms["combine"], "GB/s": comb_bytes / kms["combine"] / 1e6,
                    "frac_hbm": comb_bytes / kms["combine"] / 1e6 / hbm},
        "sum_ms": sum(kms.values()), "same_output_as_moe_forward": same_as_fused,
        "breakdown": "the component entry points (route, dispatch with its row copy, grouped "
                     "GEMMs, combine), timed one by one",
        "forward_path": forward_path(moe, cfg, w),
    }
    roofline = {"bound": "tensor", "achieved": gemm_tflops, "peak": peak,
                "unit": "TFLOP/s", "frac": gemm_tflops / peak,
                "frac_of_burst_peak": gemm_tflops / peaks["bf16_tflops"],
                "traffic": recorded_traffic(w), "kernel": "grouped_gemm_tc_kernel (G1 gate/up "
                "+ SwiGLU, G2 down) via moe_grouped_swiglu",
                "algorithmic": f"6*P*d*f = {gemm_flops:.4g} FLOP per call (P=T*k={P})",
                "peak_source": f"{peaks['source']} {peak_name}"}
    res = {"w": w, "ms": ms, "value": aggregate_throughput(T, world, ms / 1e3), "kernels": kernels,
           "roofline": roofline, "clocks": clk, "t_wall": t_wall,
           "layer_roofline": layer_roofline(w, touched, ms, peaks, peak),
           "launches_per_step": moe.moe_forward_kernel_launches(cfg), "inp": inp}
    if not with_e2e:
        return res

    # ---- e2e: activations in pinned host memory, copies inside the region ----
    # Each step copies its x from pinned host memory, runs the layer and copies
    # its output back, all through moe_forward_host.  Steps alternate between
    # two streams with their own staging buffers and workspaces, as a serving
    # loop would: one step's copies run on the copy engines while the other
    # stream computes.  The single-stream (serialised) figure is reported too.
    x_host = [x.cpu().pin_memory() for _ in range(2)]
    out_host = [torch.empty_like(x_host[0]).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    out_dev = [torch.empty_like(x) for _ in range(2)]
    wss = [ws, torch.empty_like(ws)]
    streams = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]

    def e2e_step(i, st):
        b = i % 2
        moe.moe_forward_host(cfg, x_host[b], Wr, bias, Wgu, Wd, out_host[b], x_dev[b], out_dev[b],
                             wss[b], stream=st)

    for i in range(args.warmup):
        e2e_step(i, stream)
    torch.cuda.synchronize()
    # serialised: one stream, per-step events (copies + layer + copy back)
    e2e_ms = []
    for i in range(args.steps):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step(i, stream)
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    e2e_serial = max_over_ranks(sum(e2e_ms) / len(e2e_ms), dev)
    # pipelined: two streams, the whole run timed between events on both
    torch.cuda.synchronize()
    barrier()
    start = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for st in streams:
        st.wait_stream(stream)
    for i in range(args.steps):
        st = streams[i % 2]
        e2e_step(i, st)
    ends = []
    for st in streams:
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(st)
        ends.append(ev)
    torch.cuda.synchronize()
    e2e_pipe = max_over_ranks(max(start.elapsed_time(ev) for ev in ends) / args.steps, dev)
    moe.moe_last_device_error()
    res["e2e"] = {"value": aggregate_throughput(T, world, e2e_pipe / 1e3), "unit": "tokens/s",
                  "h2d_bytes_per_step": T * w.d * es, "d2h_bytes_per_step": T * w.d * es,
                  "mode": "moe_forward_host, steps alternating on two streams (copies of one "
                          "step overlap the other's layer)",
                  "serial_value": aggregate_throughput(T, world, e2e_serial / 1e3)}
    return res


def workload_summary(r):
    """The per-workload entry of the all_workloads block."""
    k = r["kernels"]
    return {"config": workload_config(r["w"]), "value": r["value"], "unit": "tokens/s",
            "ms_per_step": r["ms"], "layer_roofline": r["layer_roofline"],
            "gemm": {"ms": k["grouped_swiglu"]["ms"], "TFLOP/s": k["grouped_swiglu"]["TFLOP/s"],
                     "frac_tensor": k["grouped_swiglu"]["frac_tensor"],
                     "frac_of_burst_peak": k["grouped_swiglu"]["frac_of_burst_peak"],
                     "frac_hbm_weight_stream": k["grouped_swiglu"]["frac_hbm_weight_stream"],
                     "peak_source": r["roofline"]["peak_source"]},
            "route_ms": k["route"]["ms"],
            "dispatch": {"ms": k["dispatch"]["ms"], "frac_hbm": k["dispatch"]["frac_hbm"]},
            "combine": {"ms": k["combine"]["ms"], "frac_hbm": k["combine"]["frac_hbm"]},
            "same_output_as_moe_forward": k["same_output_as_moe_forward"],
            "forward_path": k["forward_path"],
            "gpu_launches_per_step": r["launches_per_step"], "clocks": r["clocks"]}


def run_ours(args, w):
    import torch
    import torch.distributed as dist
    from token_dispatch_grouped_fp32_gb300 import build as _build
    from token_dispatch_grouped_fp32_gb300 import synth

    rank, local_rank, world = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    if rank == 0 or world == 1:
        _build.build()
    barrier()
    from token_dispatch_grouped_fp32_gb300 import moe

    dev = torch.device("cuda", local_rank)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    r = measure_workload(moe, w, args, dev, rank, world, flush, with_e2e=True)

    line = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            tps, n, secs, thr = oracle_sample_tokens_per_s(r["inp"], w, args.cpu_budget_s, w.T)
            cpu = {"value": tps, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                   "sample": f"first {n} tokens of the workload, whole layer "
                             f"(route, dispatch, experts, combine), {secs:.1f} s"}
        line = {
            "metric": METRIC, "value": r["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic", "config": workload_config(w),
            "roofline": r["roofline"], "layer_roofline": r["layer_roofline"],
            "kernels": r["kernels"], "cpu_baseline": cpu, "e2e": r["e2e"],
            "gpu_launches": r["launches_per_step"] * args.steps,
            "clocks": r["clocks"], "wall_s_timed_region": r["t_wall"],
        }
    del r
    torch.cuda.empty_cache()

    # the other workloads, each timed the same way (no e2e, no CPU baseline):
    # parity-test configurations that the headline line does not cover
    if not args.no_all_workloads and args.tokens is None and not args.scale_inputs:
        extra = {}
        for name in ALL_WORKLOADS:
            if name == w.name:
                continue
            rr = measure_workload(moe, synth.WORKLOADS[name], args, dev, rank, world, flush,
                                  with_e2e=False)
            extra[name] = workload_summary(rr)
            del rr
            torch.cuda.empty_cache()
        if line is not None:
            line["all_workloads"] = extra
    if line is not None:
        print(json.dumps(line), flush=True)
    barrier()
    if world > 1 and dist.is_initialized():
        dist.destroy_process_group()
    return line


def forward_path(moe, cfg, w):
    """How moe_forward moves the rows for this config, from the library's own
    workspace layout (an absent x_perm region: no permuted copy of x)."""
    copied = moe.moe_workspace_layout(cfg).x_perm != moe.MOE_WS_ABSENT
    if copied:
        return ("rows copied into x_perm" +
                (", scaled by their weights" if w.scale_inputs else "") +
                "; the same arithmetic as the component entry points")
    how = ("every expert reads x itself (k = E)" if w.k == w.E
           else "the first grouped GEMM gathers its rows from x through src_token")
    if w.scale_inputs:
        return how + "; the weights scale each row's gate and up products in fp32 inside the " \
                     "first grouped GEMM (the component path rounds w*x to bf16 first, so the " \
                     "outputs differ within the rounding)"
    return how + "; bit-identical to the component entry points"


def recorded_traffic(w):
    """DRAM bytes (read + write) per moe_grouped_swiglu call (G1 + G2) from
    the committed ncu summary, if it was taken on this workload with the
    current kernel source; else None."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "grouped_gemm_tc_traffic.json")
    src = os.path.join(ROOT, "token_dispatch_grouped_fp32_gb300", "csrc", "gemm_tc.cu")
    if not (os.path.exists(p) and os.path.exists(src)):
        return None
    with open(p) as fh:
        rec = json.load(fh)
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if rec.get("gemm_tc_sha256") != digest:
        return None
    return rec.get("per_call_bytes", {}).get(w.name)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixtral")
    ap.add_argument("--tokens", type=int, default=None, help="override T")
    ap.add_argument("--scale-inputs", action="store_true",
                    help="routing weights on the expert inputs (the dispatch scales the rows; "
                         "the combine sums unweighted)")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-all-workloads", action="store_true",
                    help="time only --workload (no all_workloads block)")
    ap.add_argument("--ref-step-s", type=float, default=None,
                    help="host seconds per reference step (default: 120 s / steps, within 0.25-4 s)")
    ap.add_argument("--ref-warmup", action="store_true",
                    help="run the warm-up steps in the reference arm too")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from token_dispatch_grouped_fp32_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.tokens:
        w = w.with_tokens(args.tokens)
    if args.scale_inputs:
        w = w.with_(scale_inputs=True)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
