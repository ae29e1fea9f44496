"""The gathered-row path of moe_forward against the copying path.

For bf16 activations with the weights on the outputs, d a multiple of 64 and
f <= 3072, moe_forward forms no permuted copy of x: the dispatch writes only
counts, offsets, pos and src_token, and the first grouped GEMM's extra warps
copy each A row of a stage from x[src_token[row]] into the swizzled shared
memory layout the tensor memory access (TMA) unit would have written
(Transformers docs "Expert parallelism", section "Token dispatch": only the
routed rows move).  The operand bytes the tensor cores read are the same as
on the copying path, so every intermediate and the output must match the
component calls (route, dispatch with its row copy, grouped GEMMs through
TMA, combine) bit for bit.

Cases cover the three tile modes (CTA pairs when experts average >= 512
rows, pairs plus single CTAs in between, single CTAs below 64), ragged
segments (skewed routing), an expert that receives no rows, a long K (d =
2048: 32 K steps per tile) and short ones, and an expert with so few rows
that the second CTA of its only pair tile gathers none."""
import pytest
import torch

from token_dispatch_grouped_fp32_gb300 import synth
from tests.gpu_util import check_layer, load_moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return load_moe()


def _bias(E, seed, dead=None, rare=None):
    g = torch.Generator().manual_seed(seed)
    b = 2.0 * torch.rand(E, generator=g)  # skewed loads: ragged segments
    if dead is not None:
        b[dead] = -1e4  # never selected
    if rare is not None:  # (expert, offset): selected by a few dozen tokens
        b[rare[0]] = rare[1]
    return b


CASES = [  # name, T, d, E, k, f, dead expert, rare expert and its logit offset
    ("pairs", 2048, 256, 8, 2, 512, None, (5, -0.5)),       # 512 rows per expert on average
    ("pairs_long_k", 1024, 2048, 4, 2, 256, 1, (3, -2.0)),  # 32 K steps, one empty expert
    ("hybrid", 1024, 512, 16, 2, 384, 7, None),     # 128 rows per expert on average
    ("singles", 64, 192, 32, 4, 256, None, None),   # 8 rows per expert on average
    ("pairs_k8", 4096, 128, 64, 8, 2048, 0, None),  # f at the gather's limit
    ("one_k_step", 1536, 64, 4, 2, 192, None, None),  # d = 64: one K step per tile
    ("two_experts", 1400, 128, 2, 1, 256, None, None),  # E = 2, k = 1: pairs, two segments
    ("one_token", 1, 256, 16, 4, 512, None, None),    # T = 1: four rows, one per expert
    ("many_experts", 2048, 128, 1024, 2, 64, None, None),  # E = 1024, about 4 rows each
]


@pytest.mark.parametrize("name,T,d,E,k,f,dead,rare", CASES, ids=[c[0] for c in CASES])
def test_gathered_rows_equal_copied_rows(moe, name, T, d, E, k, f, dead, rare):
    w = synth.Workload("gather_" + name, T, d, E, k, f, "bf16", 300 + T + d)
    inp = synth.make_inputs(w, device="cuda")
    bias = _bias(E, w.seed, dead, rare).cuda()
    layer = moe.MoELayer(inp["Wr"], inp["Wgu"], inp["Wd"], k, bias, True)
    x = inp["x"]
    out = layer(x)
    torch.cuda.synchronize()
    assert moe.moe_last_device_error() == moe.MOE_OK
    cfg = layer.config(T)
    L = moe.moe_workspace_layout(cfg)
    assert L.x_perm == moe.MOE_WS_ABSENT  # this config takes the gathered-row path
    ws = layer.workspace(T)
    P = T * k

    def region(off, n, dt):
        return ws[off:off + n * torch.empty((), dtype=dt).element_size()].view(dt)

    counts = region(L.counts, E, torch.int32)
    if dead is not None:
        assert int(counts[dead]) == 0
    if rare is not None:  # a CTA-pair tile whose second CTA gathers no row
        assert 0 < int(counts[rare[0]]) <= 128
    # the copying path through the component entry points
    wt = torch.empty(T, k, dtype=torch.float32, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    rws = torch.empty(max(256, moe.moe_route_workspace_size(cfg)), dtype=torch.uint8,
                      device="cuda")
    moe.moe_route(cfg, x, inp["Wr"], bias, logits, idx, wt, rws)
    cnt = torch.empty(E, dtype=torch.int32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pos = torch.empty(P, dtype=torch.int32, device="cuda")
    src = torch.empty(P, dtype=torch.int32, device="cuda")
    x_perm = torch.empty(P, d, dtype=x.dtype, device="cuda")
    h_perm = torch.empty(P, f, dtype=x.dtype, device="cuda")
    y_perm = torch.empty(P, d, dtype=x.dtype, device="cuda")
    dws = torch.empty(max(256, moe.moe_dispatch_workspace_size(cfg)), dtype=torch.uint8,
                      device="cuda")
    moe.moe_dispatch(cfg, idx, wt, x, cnt, off, pos, src, x_perm, dws)
    moe.moe_grouped_swiglu(cfg, x_perm, off, inp["Wgu"], inp["Wd"], h_perm, y_perm)
    out2 = torch.empty_like(x)
    moe.moe_combine(cfg, y_perm, pos, wt, out2)
    torch.cuda.synchronize()
    assert moe.moe_last_device_error() == moe.MOE_OK
    assert torch.equal(region(L.src_token, P, torch.int32), src)
    assert torch.equal(region(L.offsets, E + 1, torch.int32), off)
    assert torch.equal(region(L.h_perm, P * f, x.dtype).view(P, f), h_perm)
    assert torch.equal(region(L.y_perm, P * d, x.dtype).view(P, d), y_perm)
    assert torch.equal(out, out2)


@pytest.mark.parametrize("name", ["pairs", "hybrid", "singles"])
def test_gathered_rows_against_oracle(moe, oracle, name):
    """The gathered-row path against the oracle directly (sampled tokens,
    the layer tolerance)."""
    _, T, d, E, k, f, dead, rare = next(c for c in CASES if c[0] == name)
    w = synth.Workload("gather_" + name, T, d, E, k, f, "bf16", 700 + T)
    check_layer(moe, oracle, w, device="cpu", bias=_bias(E, w.seed, dead, rare))


SCALED = [  # name, T, d, E, k, f: weights on the inputs, no permuted copy of x
    ("gathered_pairs", 2048, 256, 8, 2, 512),     # rows gathered, CTA pairs
    ("gathered_hybrid", 1024, 512, 16, 2, 384),   # rows gathered, pairs and single CTAs
    ("dense_pairs", 1024, 256, 8, 8, 256),        # k = E: x itself, 1024 rows per expert
    ("dense_singles", 40, 192, 4, 4, 320),        # k = E, 40 rows per expert
]


@pytest.mark.parametrize("name,T,d,E,k,f", SCALED, ids=[c[0] for c in SCALED])
def test_weights_on_inputs_scaled_in_first_gemm(moe, oracle, name, T, d, E, k, f):
    """Weights on the inputs (the experts receive tokens already scaled by the
    router score; Transformers docs "Expert parallelism", introduction, the
    Llama 4 note) where moe_forward forms no permuted copy of x: the dispatch
    records each row's weight and the first grouped GEMM multiplies the row's
    gate and up accumulators by it before the SwiGLU, since (w x) W = w (x W)
    (the oracle forms (w x) W in fp64).  Checked against the oracle; the
    layout shows no x_perm region."""
    w = synth.Workload("scaled_" + name, T, d, E, k, f, "bf16", 500 + T + d, renorm=False,
                       scale_inputs=True)
    cfg = moe.config(T, d, E, k, f, "bf16", False, scale_inputs=True)
    assert moe.moe_workspace_layout(cfg).x_perm == moe.MOE_WS_ABSENT
    check_layer(moe, oracle, w, device="cpu")
