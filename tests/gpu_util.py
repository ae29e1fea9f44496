"""Shared helpers of the GPU parity tests: library fixture, tolerances and
host copies.  Imported only by tests marked ``gpu``."""
from __future__ import annotations

import numpy as np
import torch

from token_dispatch_grouped_fp32_gb300 import synth

EPS32 = 2.0 ** -23


def load_moe():
    from token_dispatch_grouped_fp32_gb300 import build
    build.build()
    from token_dispatch_grouped_fp32_gb300 import moe
    return moe


def f32(t: torch.Tensor) -> np.ndarray:
    """Exact float32 image of a (bf16 or fp32) tensor, on the host."""
    return t.detach().float().cpu().numpy()


def layer_tolerance(ref: np.ndarray) -> float:
    """Output tolerance of the layer: max|err| <= 2e-2 * max|ref| + 1e-3."""
    return 2e-2 * float(np.max(np.abs(ref))) + 1e-3 if ref.size else 1e-3


def fp32_tolerance(ref: np.ndarray, *lengths: int) -> float:
    """Tolerance of an fp32 result against the oracle's double result.

    Probabilistic rounding-error model (Higham, "Accuracy and Stability of
    Numerical Algorithms", 2nd ed., section 2.8): an fp32 sum of n products of
    random sign carries an error of about u * sqrt(n) relative to the scale of
    its result (u = 2^-24); dot products in series (lengths d for gate and up,
    then f for the down projection) add their terms.  The factor 8 is a safety
    margin.  For the tiny workload (d = 128, f = 256) this is about 1.8e-5 of
    max|ref|: roughly 10x the errors the fp32 path shows, and 200x below an
    error of bf16 rounding size (2^-8 relative), which it is there to catch.
    """
    u = 2.0 ** -24
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    return 8.0 * u * sum(np.sqrt(n) for n in lengths) * scale + 1e-30


def output_tolerance(ref: np.ndarray, dtype: str, d: int, f: int, k: int = 1, E: int = 0) -> float:
    """The layer-output tolerance for the path's activation dtype: the
    stated bound 2e-2 * max|ref| + 1e-3 for bf16; for fp32 the rounding model
    of fp32_tolerance over the three dot products (d, d, f), plus k routing
    weights each within weight_tolerance(E) of the oracle's."""
    if dtype in ("bf16", torch.bfloat16):
        return layer_tolerance(ref)
    tol = fp32_tolerance(ref, d, d, f)
    if E:
        tol += k * weight_tolerance(E) * float(np.max(np.abs(ref)) if ref.size else 0.0)
    return tol


def weight_tolerance(E: int) -> float:
    """Bound on |w_gpu - w_oracle| for the routing weights.

    The GPU forms p = expf(L - m) / Z in fp32: each expf carries <= 2 ulp, the
    sum Z adds ceil(E/32) sequential terms per lane then 5 butterfly levels,
    the division and the renormalising sum over <= 32 slots add a few more
    roundings.  Weights are <= 1, so the absolute error stays below
    (ceil(E/32) + 16) ulp(1); the oracle's double result is exact to that
    order.
    """
    return (int(np.ceil(E / 32)) + 16) * EPS32


def logit_tolerance(x: np.ndarray, Wr: np.ndarray, bias=None) -> np.ndarray:
    """Per-entry bound on |L_gpu - L_oracle|: 32 * eps32 * sum_i |x_i W_ei|
    (+ one rounding of the bias add).  The GPU sums d products in fp32 in
    blocks of 32; the oracle's double sum rounded once is exact to that
    order."""
    mag = np.abs(x.astype(np.float64)) @ np.abs(Wr.astype(np.float64)).T
    tol = 32 * EPS32 * mag
    if bias is not None:
        tol = tol + 2 * EPS32 * (np.abs(bias.astype(np.float64))[None, :] + mag)
    return tol + 1e-30


def near_tie(L: np.ndarray, k: int, tol: np.ndarray) -> bool:
    """True when the k-th and (k+1)-th largest entries of the row L are
    within tol of each other (a selection that rounding may flip)."""
    if k >= L.shape[0]:
        return False
    s = np.sort(L.astype(np.float64))[::-1]
    return (s[k - 1] - s[k]) <= 2 * float(np.max(tol))


def _pick_tokens(idx_ref, T, sample, max_experts, seed):
    if sample is None:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    cand = [0, T - 1] + rng.permutation(T).tolist()
    chosen, experts = [], set()
    for t in cand:
        if t in chosen:
            continue
        new = experts | set(idx_ref(t))
        if len(new) > max_experts:
            continue
        chosen.append(t)
        experts = new
        if len(chosen) >= sample:
            break
    return np.array(sorted(chosen))


def check_layer(moe, oracle, w, device="cuda", sample=None, max_experts=48, bias=None):
    inp = synth.make_inputs(w, device=device)
    x, Wr, Wgu, Wd = (inp[n].cuda() for n in ("x", "Wr", "Wgu", "Wd"))
    if bias is None and inp["bias"] is not None:
        bias = inp["bias"]
    bias_d = None if bias is None else bias.cuda()
    layer = moe.MoELayer(Wr, Wgu, Wd, w.k, bias_d, w.renorm, w.scale_inputs)
    out = layer(x)
    torch.cuda.synchronize()
    assert moe.moe_last_device_error() == moe.MOE_OK

    # the GPU's own routing, from the same kernels moe_forward runs
    cfg = layer.config(w.T)
    g_idx = torch.empty(w.T, w.k, dtype=torch.int32, device="cuda")
    g_w = torch.empty(w.T, w.k, dtype=torch.float32, device="cuda")
    g_L = torch.empty(w.T, w.E, dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, x, Wr, bias_d, g_L, g_idx, g_w, layer.workspace(w.T))
    g_idx = g_idx.cpu().numpy()

    Wrs = f32(Wr)
    bs = None if bias is None else f32(bias)
    xs_all = None
    if sample is None:
        xs_all = f32(x)
        tokens = np.arange(w.T)
    else:
        # oracle routing of candidate tokens, computed lazily per token
        cache = {}

        def idx_ref(t):
            if t not in cache:
                L = oracle.router_logits(f32(x[t:t + 1]), Wrs, bs)
                cache[t] = oracle.topk(L, w.k, w.renorm)[0][0].tolist()
            return cache[t]
        tokens = _pick_tokens(idx_ref, w.T, sample, max_experts, w.seed)

    xs = xs_all[tokens] if xs_all is not None else f32(x[torch.from_numpy(tokens).cuda()])
    L_ref = oracle.router_logits(xs, Wrs, bs)
    idx_ref, w_ref = oracle.topk(L_ref, w.k, w.renorm)
    tol_L = logit_tolerance(xs, Wrs, bs)
    same = (g_idx[tokens] == idx_ref).all(1)
    for i in np.nonzero(~same)[0]:
        assert near_tie(L_ref[i], w.k, tol_L[i]) or \
            sorted(g_idx[tokens[i]].tolist()) == sorted(idx_ref[i].tolist()), tokens[i]
    assert same.sum() >= max(1, int(0.9 * len(tokens)))
    keep = np.nonzero(same)[0]

    experts = np.unique(idx_ref[keep])
    remap = np.full(w.E, -1, np.int32)
    remap[experts] = np.arange(len(experts), dtype=np.int32)
    sel = torch.from_numpy(experts).long().cuda()
    Wgu_c, Wd_c = f32(Wgu[sel]), f32(Wd[sel])
    ref = oracle.token_outputs(np.arange(len(keep)), xs[keep], Wgu_c, Wd_c,
                               remap[idx_ref[keep]], w_ref[keep], scale_inputs=w.scale_inputs)
    got = f32(out[torch.from_numpy(tokens[keep]).cuda()]).astype(np.float64)
    err = np.abs(got - ref).max()
    assert np.isfinite(got).all()
    tol = output_tolerance(ref, w.dtype, w.d, w.f, w.k, w.E)
    assert err <= tol, (err, tol)
    return len(keep)
