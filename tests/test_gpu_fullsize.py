"""Full-size parity of moe_forward's own intermediates against the oracle.

Each benchmark workload runs once at its full size through moe_forward, in
the launch configuration the benchmark times (for ~256 rows per expert: the
CTA-pair launch and the single-CTA launch of each product, the second
overlapping the first).  The call's intermediates are then read from its
workspace (moe_workspace_layout) and checked:

- routing: the oracle's top-k on the GPU's own fp32 logit buffer gives the
  same expert ids bit for bit, and weights within the fp32 bound; the logits
  themselves within the fp32 summation bound of the oracle's;
- dispatch: the oracle's counts, offsets, pos and src_token for those ids,
  bit for bit; every x_perm row a byte copy of its token's row (where
  moe_forward forms x_perm; where its first grouped GEMM gathers the rows
  through src_token, the expert checks below cover the gather);
- experts: for EVERY expert that received rows, its first row, its last row
  (in the ragged last row tile) and the rows on each side of its tile
  boundaries, h_perm and y_perm against the oracle's FFN of that token's row,
  within the stated bf16 bound.

The oracle's inputs are the seeded inputs and, for the selection, the GPU's
logit buffer (the selection is defined on a given fp32 logit buffer); its
dispatch, hence which token each row holds, is its own."""
import numpy as np
import pytest
import torch

from token_dispatch_grouped_fp32_gb300 import synth
from tests.gpu_util import f32, layer_tolerance, load_moe, logit_tolerance, weight_tolerance

pytestmark = pytest.mark.gpu

WORKLOADS = ["mixtral", "gptoss_decode", "gptoss_prefill", "qwen3_zipf", "deepseek",
             "mixtral_norenorm", "mixtral_dense"]


@pytest.fixture(scope="module")
def moe():
    return load_moe()


def _region(ws, offset, count, dtype):
    nbytes = count * torch.empty((), dtype=dtype).element_size()
    return ws[offset:offset + nbytes].view(dtype)


@pytest.fixture(scope="module", params=WORKLOADS)
def run(moe, request):
    """One full-size moe_forward of a workload (a module-scoped parametrized
    fixture, so pytest runs every test of one workload before the next
    workload's inputs are drawn)."""
    torch.cuda.empty_cache()
    w = synth.WORKLOADS[request.param]
    inp = synth.make_inputs(w, device="cuda")
    layer = moe.MoELayer(inp["Wr"], inp["Wgu"], inp["Wd"], w.k, inp["bias"], w.renorm)
    out = layer(inp["x"])
    torch.cuda.synchronize()
    assert moe.moe_last_device_error() == moe.MOE_OK
    cfg = layer.config(w.T)
    L = moe.moe_workspace_layout(cfg)
    ws = layer.workspace(w.T)
    P, dt = w.T * w.k, w.torch_dtype
    yield {
        "w": w, "inp": inp, "out": out,
        "logits": _region(ws, L.logits, w.T * w.E, torch.float32).view(w.T, w.E),
        "idx": _region(ws, L.topk_idx, P, torch.int32).view(w.T, w.k),
        "wt": _region(ws, L.topk_w, P, torch.float32).view(w.T, w.k),
        "counts": _region(ws, L.counts, w.E, torch.int32),
        "offsets": _region(ws, L.offsets, w.E + 1, torch.int32),
        "pos": _region(ws, L.pos, P, torch.int32),
        "src": _region(ws, L.src_token, P, torch.int32),
        # absent where moe_forward forms no permuted copy of x (k == E, or
        # the first grouped GEMM gathers its rows through src_token)
        "x_perm": (None if L.x_perm == moe.MOE_WS_ABSENT
                   else _region(ws, L.x_perm, P * w.d, dt).view(P, w.d)),
        "h_perm": _region(ws, L.h_perm, P * w.f, dt).view(P, w.f),
        "y_perm": _region(ws, L.y_perm, P * w.d, dt).view(P, w.d),
    }
    del layer, inp, out, ws
    torch.cuda.empty_cache()


def test_full_size_routing_and_dispatch(oracle, run):
    r = run
    w = r["w"]
    g_logits = r["logits"].cpu().numpy()
    g_idx = r["idx"].cpu().numpy()
    g_w = r["wt"].cpu().numpy().astype(np.float64)

    # selection on the GPU's own logit buffer: bit-exact ids, weights in bound
    ref_idx, ref_w = oracle.topk(g_logits, w.k, w.renorm)
    np.testing.assert_array_equal(g_idx, ref_idx)
    assert np.abs(g_w - ref_w).max() <= weight_tolerance(w.E)

    # the logits themselves: within the fp32 summation bound, every token
    x = f32(r["inp"]["x"])
    Wr = f32(r["inp"]["Wr"])
    bias = None if r["inp"]["bias"] is None else f32(r["inp"]["bias"])
    ref_L = oracle.router_logits(x, Wr, bias)
    assert (np.abs(g_logits.astype(np.float64) - ref_L) <= logit_tolerance(x, Wr, bias)).all()

    # dispatch of those ids: bit-exact
    rc, ro, rp, rs = oracle.dispatch(ref_idx, w.E)
    np.testing.assert_array_equal(r["counts"].cpu().numpy(), rc)
    np.testing.assert_array_equal(r["offsets"].cpu().numpy(), ro)
    np.testing.assert_array_equal(r["pos"].cpu().numpy(), rp)
    np.testing.assert_array_equal(r["src"].cpu().numpy(), rs)
    assert rc.sum() == w.T * w.k
    # permuted rows are byte copies of the token rows (k == E: the experts
    # read x itself, and each segment holds the tokens in order)
    if w.k == w.E:
        np.testing.assert_array_equal(rs, np.tile(np.arange(w.T), w.E))
        assert r["x_perm"] is None
    elif r["x_perm"] is not None:
        src = torch.from_numpy(rs).long().cuda()
        assert torch.equal(r["x_perm"], r["inp"]["x"][src])


def _rows_to_check(count, rng):
    """Row indices (within an expert's segment) to compare: the first and the
    last, the rows on each side of every 128-row tile boundary, and two
    random interior rows."""
    rows = {0, count - 1}
    for b in range(128, count, 128):
        rows.update((b - 1, b))
    if count > 2:
        rows.update(rng.integers(1, count - 1, size=2).tolist())
    return sorted(rows)


def test_full_size_every_expert(oracle, run):
    r = run
    w = r["w"]
    # the oracle's own dispatch of the (already checked) selection
    ref_idx, _ = oracle.topk(r["logits"].cpu().numpy(), w.k, w.renorm)
    _, offs, _, src = oracle.dispatch(ref_idx, w.E)
    x = r["inp"]["x"]
    Wgu, Wd = r["inp"]["Wgu"], r["inp"]["Wd"]
    rng = np.random.default_rng(w.seed)
    # experts in batches, so the float images of their weights stay small
    batch = max(1, int(3e9 // (4 * 3 * w.d * w.f)))
    experts = [e for e in range(w.E) if offs[e + 1] > offs[e]]
    checked = 0
    for b0 in range(0, len(experts), batch):
        sel = experts[b0:b0 + batch]
        rows, local = [], []
        for i, e in enumerate(sel):
            for rr in _rows_to_check(int(offs[e + 1] - offs[e]), rng):
                rows.append(int(offs[e]) + rr)
                local.append(i)
        rows_t = torch.tensor(rows, dtype=torch.long, device="cuda")
        sel_t = torch.tensor(sel, dtype=torch.long, device="cuda")
        x_rows = f32(x[torch.from_numpy(src[rows]).long().cuda()])
        ref_h, ref_y = oracle.expert_ffn_rows(x_rows, np.array(local, np.int32),
                                              f32(Wgu[sel_t]), f32(Wd[sel_t]))
        got_h = f32(r["h_perm"][rows_t]).astype(np.float64)
        got_y = f32(r["y_perm"][rows_t]).astype(np.float64)
        assert np.isfinite(got_h).all() and np.isfinite(got_y).all()
        err_h, err_y = np.abs(got_h - ref_h).max(), np.abs(got_y - ref_y).max()
        assert err_h <= layer_tolerance(ref_h), (w.name, sel, err_h)
        assert err_y <= layer_tolerance(ref_y), (w.name, sel, err_y)
        checked += len(sel)
    assert checked == len(experts) and checked >= min(w.E, 40)
