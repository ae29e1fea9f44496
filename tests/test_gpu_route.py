"""Router parity: top-k indices bit-exact and weights within the fp32 bound
against the oracle on the same fp32 logit buffer; router logits within the
fp32 summation bound, on both logit paths (CUDA-core FMAs for fp32 x and
small batches with E <= 32; tensor cores with the three-term bf16 split of
Wr for bf16 x, 8 <= E <= 256, E % 8 == 0)."""
import numpy as np
import pytest
import torch

from token_dispatch_grouped_fp32_gb300 import synth
from tests.gpu_util import f32, load_moe, logit_tolerance, near_tie, weight_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return load_moe()


ROUTE_CASES = [
    # T, E, k, ties
    (1, 8, 2, None),
    (37, 8, 2, None),
    (4096, 8, 2, None),
    (4096, 8, 2, "coarse"),
    (513, 128, 4, None),
    (777, 128, 8, "coarse"),
    (300, 256, 8, None),
    (300, 256, 8, "coarse"),
    (100, 33, 5, None),
    (64, 1024, 32, None),
    (200, 3, 3, None),
    (50, 64, 6, "all_equal"),
    (8192, 256, 8, None),
    # T >= 1024 with E <= 256 takes the sorted-heads selection: ties there too
    (2048, 128, 8, "coarse"),
    (1024, 256, 8, "coarse"),
    (1536, 48, 5, "coarse"),
    (1500, 64, 6, "all_equal"),
    (1024, 200, 7, None),
]


@pytest.mark.parametrize("renorm", [True, False])
@pytest.mark.parametrize("T,E,k,ties", ROUTE_CASES)
def test_route_from_logits_matches_oracle(moe, oracle, T, E, k, ties, renorm):
    L = synth.make_logits(T, E, 1000 + T + E, ties=ties)
    cfg = moe.config(T, 8, E, k, 8, "f32", renorm)
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), -7.0, dtype=torch.float32, device="cuda")
    moe.moe_route_from_logits(cfg, L.cuda(), idx, w)
    torch.cuda.synchronize()
    ref_idx, ref_w = oracle.topk(L.numpy(), k, renorm)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    err = np.abs(w.cpu().numpy().astype(np.float64) - ref_w).max()
    assert err <= weight_tolerance(E), err


@pytest.mark.parametrize("name,T", [("tiny_fp32", 64), ("mixtral", 512), ("gptoss_prefill", 700),
                                    ("qwen3_zipf", 1500), ("deepseek", 300), ("gptoss_decode", 64),
                                    ("deepseek", 8192), ("mixtral", 4096), ("mixtral", 1500)])
def test_route_logits_and_selection(moe, oracle, name, T):
    w = synth.WORKLOADS[name].with_tokens(T)
    inp = synth.make_inputs(w, weights=False)
    x, Wr, bias = inp["x"], inp["Wr"], inp["bias"]
    cfg = moe.config(T, w.d, w.E, w.k, w.f, w.torch_dtype, w.renorm)
    logits = torch.empty(T, w.E, dtype=torch.float32, device="cuda")
    idx = torch.empty(T, w.k, dtype=torch.int32, device="cuda")
    wt = torch.empty(T, w.k, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(256, moe.moe_route_workspace_size(cfg)), dtype=torch.uint8, device="cuda")
    moe.moe_route(cfg, x.cuda(), Wr.cuda(), None if bias is None else bias.cuda(), logits, idx, wt,
                  ws)
    torch.cuda.synchronize()
    xs, Wrs = f32(x), f32(Wr)
    bs = None if bias is None else f32(bias)
    ref_L = oracle.router_logits(xs, Wrs, bs)
    tol = logit_tolerance(xs, Wrs, bs)
    gL = logits.cpu().numpy()
    assert (np.abs(gL.astype(np.float64) - ref_L) <= tol).all()

    # moe_route selects on exactly the logits it wrote
    idx2 = torch.empty_like(idx)
    w2 = torch.empty_like(wt)
    moe.moe_route_from_logits(cfg, logits, idx2, w2)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2) and torch.equal(wt, w2)

    # against the oracle's own routing: equal except where a near tie may flip
    ref_idx, ref_w = oracle.topk(ref_L, w.k, w.renorm)
    g_idx = idx.cpu().numpy()
    differ = np.nonzero((g_idx != ref_idx).any(1))[0]
    for t in differ:
        assert near_tie(ref_L[t], w.k, tol[t]) or \
            sorted(g_idx[t].tolist()) == sorted(ref_idx[t].tolist()), t
    assert len(differ) <= max(2, T // 200)


# Tensor-core logit shapes: N = E rounded up to 16.  Single CTAs (E < 64 or
# T < 512): three W' tiles per stage for N <= 128 (x read once), one per
# stage above.  CTA pairs (E >= 64, T >= 512): 256-token tiles, each CTA with
# half of the N rows of every W' term; N = 64 ... 256, ragged token tiles
# (the peer CTA's rows past T), W' rows past E, one or several K splits.
TC_SHAPES = [
    # T, d, E, k
    (1024, 256, 8, 2),
    (1024, 4160, 8, 2),     # E = 8, d = 65 K steps
    (16400, 256, 8, 2),     # E = 8, 129 token tiles (the last of 16 tokens)
    (1100, 512, 24, 3),
    (2000, 128, 40, 4),
    (1500, 320, 48, 6),
    (1024, 64, 64, 8),
    (1030, 192, 136, 4),
    (1024, 64, 256, 8),
    (513, 256, 128, 8),     # pairs: 3 tiles, the last with one token; 2 K splits
    (777, 256, 128, 4),
    (1300, 192, 96, 4),     # N = 96: 48 W' rows per CTA
    (600, 128, 200, 8),     # N = 208: the peer's rows 200..207 read zeros
    (2048, 2048, 128, 8),   # 8 K splits
    (4096, 512, 256, 8),    # N = 256, 4 K splits
    (300, 448, 256, 8),     # T < 512: single CTAs, one W' tile per stage
]


# CUDA-core logit shapes outside the tensor-core router: fp32 x with E > 32
# (tiled FFMA kernel for T >= 2048, 32-expert groups below), bf16 x with
# E > 256 or E not a multiple of 8, and E <= 32 with the selection in the
# logits launch.
SIMT_SHAPES = [
    # T, d, E, k, dtype
    (2048, 256, 64, 6, "f32"),     # tiled kernel, 64 x 64 blocks
    (3000, 192, 128, 8, "f32"),    # tiled kernel, 64 x 128 blocks, ragged row tile
    (2500, 128, 36, 4, "bf16"),    # E % 8 != 0: tiled kernel
    (2048, 64, 520, 8, "bf16"),    # E > 256: tiled kernel, ragged column tile
    (1000, 320, 100, 5, "f32"),    # T < 2048: 32-expert groups, top-k launch
    (777, 96, 24, 3, "f32"),       # E <= 32: selection in the logits launch
    (1024, 264, 8, 2, "bf16"),     # E = 8 with d % 64 != 0: the same
]


@pytest.mark.parametrize("T,d,E,k,dtype", SIMT_SHAPES)
def test_route_cuda_core_shapes(moe, oracle, T, d, E, k, dtype):
    w = synth.Workload("simt_shape", T, d, E, k, 8, dtype, 57 + E)
    inp = synth.make_inputs(w, weights=False)
    x, Wr = inp["x"], inp["Wr"]
    bias = torch.linspace(-0.5, 0.5, E)
    cfg = moe.config(T, d, E, k, 8, w.torch_dtype, True)
    assert moe.moe_route_workspace_size(cfg) == 0  # not the tensor-core router
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    wt = torch.empty(T, k, dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, x.cuda(), Wr.cuda(), bias.cuda(), logits, idx, wt, None)
    torch.cuda.synchronize()
    xs, Wrs, bs = f32(x), f32(Wr), bias.numpy()
    ref_L = oracle.router_logits(xs, Wrs, bs)
    assert (np.abs(logits.cpu().numpy().astype(np.float64) - ref_L)
            <= logit_tolerance(xs, Wrs, bs)).all()
    ref_idx, ref_w = oracle.topk(logits.cpu().numpy(), k, True)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    assert np.abs(wt.cpu().numpy().astype(np.float64) - ref_w).max() <= weight_tolerance(E)


@pytest.mark.parametrize("T,d,E,k", TC_SHAPES)
def test_route_tensor_core_shapes(moe, oracle, T, d, E, k):
    w = synth.Workload("tc_shape", T, d, E, k, 8, "bf16", 31 + E)
    inp = synth.make_inputs(w, weights=False)
    x, Wr = inp["x"], inp["Wr"]
    cfg = moe.config(T, d, E, k, 8, torch.bfloat16, True)
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    wt = torch.empty(T, k, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(256, moe.moe_route_workspace_size(cfg)), dtype=torch.uint8, device="cuda")
    moe.moe_route(cfg, x.cuda(), Wr.cuda(), None, logits, idx, wt, ws)
    torch.cuda.synchronize()
    xs, Wrs = f32(x), f32(Wr)
    ref_L = oracle.router_logits(xs, Wrs, None)
    tol = logit_tolerance(xs, Wrs, None)
    assert (np.abs(logits.cpu().numpy().astype(np.float64) - ref_L) <= tol).all()
    ref_idx, ref_w = oracle.topk(logits.cpu().numpy(), k, True)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    assert np.abs(wt.cpu().numpy().astype(np.float64) - ref_w).max() <= weight_tolerance(E)


@pytest.mark.parametrize("T", [37, 1100])  # the plain selection; the sorted-heads one
@pytest.mark.parametrize("E,k", [(8, 6), (64, 24), (128, 32), (256, 32)])
def test_route_special_values_match_oracle(moe, oracle, T, E, k):
    """Signed zeros tie (the lower id wins), -inf ranks below every finite
    value and a NaN below everything, a later NaN losing to an earlier one.
    About half of each row's k picks are finite, so the selection reaches
    into the -inf and (on half the rows) the NaN entries.  Indices bit for
    bit against the oracle on the same buffer; weights too on the rows
    without a NaN and with a finite logit."""
    g = np.random.default_rng(4000 + T + E)
    L = np.round(g.standard_normal((T, E)) * 2.0) / 2.0  # many exact ties
    L[g.random((T, E)) < 0.15] = 0.0
    L[g.random((T, E)) < 0.15] = -0.0
    special = g.random((T, E)) < 1.0 - k / (2.0 * E)
    nan_rows = g.random(T) < 0.5
    as_nan = special & nan_rows[:, None] & (g.random((T, E)) < 0.85)
    L[special] = -np.inf
    L[as_nan] = np.nan
    L = L.astype(np.float32)
    cfg = moe.config(T, 8, E, k, 8, "f32", True)
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), -7.0, dtype=torch.float32, device="cuda")
    moe.moe_route_from_logits(cfg, torch.from_numpy(L).cuda(), idx, w)
    torch.cuda.synchronize()
    ref_idx, ref_w = oracle.topk(L, k, True)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    # weights are defined where no logit is NaN and some logit is finite
    clean = ~np.isnan(L).any(axis=1) & np.isfinite(L).any(axis=1)
    assert clean.any() and (~clean).any()
    got_w = w.cpu().numpy().astype(np.float64)[clean]
    assert np.abs(got_w - ref_w[clean]).max() <= weight_tolerance(E)
