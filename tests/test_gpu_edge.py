"""Edge cases and properties of the layer on the GPU: a single token, one
expert, k = E without renormalisation, every token on one expert, layers
chained on one stream, an empty batch, determinism, CUDA-graph capture, and
the host-buffer entry point."""
import pytest
import torch

from token_dispatch_grouped_fp32_gb300 import synth
from tests.gpu_util import check_layer, load_moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return load_moe()


def test_single_token_decode(moe, oracle):
    w = synth.WORKLOADS["gptoss_decode"].with_tokens(1)
    check_layer(moe, oracle, w)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_one_expert(moe, oracle, dtype):
    w = synth.Workload("one", 300, 128, 1, 1, 264, dtype, 21)
    check_layer(moe, oracle, w, device="cpu")


@pytest.mark.parametrize("scale", [False, True])
@pytest.mark.parametrize("renorm", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_k_equals_E(moe, oracle, dtype, renorm, scale):
    """k = E: the path with nothing to permute (the experts read x itself);
    with the weights on the inputs, bf16 scales each row's products in the
    first GEMM and fp32 copies scaled rows."""
    w = synth.Workload("dense", 200, 96, 4, 4, 136, dtype, 22, renorm=renorm, scale_inputs=scale)
    check_layer(moe, oracle, w, device="cpu")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T,E", [(300, 8), (1000, 16), (77, 2)])
def test_all_experts_path_equals_routed_components(moe, dtype, T, E):
    """k = E: moe_forward's path without the permutation gives the same bits
    as the component calls (route, the general dispatch with its row copy,
    grouped GEMMs, combine), and its dispatch arrays are the identity order:
    expert e's segment is the T tokens in order."""
    w = synth.Workload("allexp", T, 128, E, E, 200, dtype, 40 + E, renorm=False)
    inp = synth.make_inputs(w, device="cuda")
    layer = moe.MoELayer(inp["Wr"], inp["Wgu"], inp["Wd"], E, None, False)
    x = inp["x"]
    out = layer(x)
    cfg = layer.config(T)
    L = moe.moe_workspace_layout(cfg)
    ws = layer.workspace(T)
    P = T * E
    idx = ws[L.topk_idx:L.topk_idx + 4 * P].view(torch.int32).view(T, E).clone()
    pos = ws[L.pos:L.pos + 4 * P].view(torch.int32).clone()
    src = ws[L.src_token:L.src_token + 4 * P].view(torch.int32).clone()
    counts = ws[L.counts:L.counts + 4 * E].view(torch.int32).clone()
    t_of = torch.arange(T, device="cuda", dtype=torch.int32)[:, None]
    assert torch.equal(pos.view(T, E), idx * T + t_of)
    assert torch.equal(src, torch.arange(T, device="cuda", dtype=torch.int32).repeat(E))
    assert (counts == T).all()
    # the general path through the component entry points
    wt = torch.empty(T, E, dtype=torch.float32, device="cuda")
    idx2 = torch.empty(T, E, dtype=torch.int32, device="cuda")
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    rws = torch.empty(max(256, moe.moe_route_workspace_size(cfg)), dtype=torch.uint8, device="cuda")
    moe.moe_route(cfg, x, inp["Wr"], None, logits, idx2, wt, rws)
    cnt = torch.empty(E, dtype=torch.int32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pos2 = torch.empty(P, dtype=torch.int32, device="cuda")
    src2 = torch.empty(P, dtype=torch.int32, device="cuda")
    x_perm = torch.empty(P, w.d, dtype=x.dtype, device="cuda")
    h_perm = torch.empty(P, w.f, dtype=x.dtype, device="cuda")
    y_perm = torch.empty(P, w.d, dtype=x.dtype, device="cuda")
    dws = torch.empty(max(256, moe.moe_dispatch_workspace_size(cfg)), dtype=torch.uint8,
                      device="cuda")
    moe.moe_dispatch(cfg, idx2, wt, x, cnt, off, pos2, src2, x_perm, dws)
    moe.moe_grouped_swiglu(cfg, x_perm, off, inp["Wgu"], inp["Wd"], h_perm, y_perm)
    out2 = torch.empty_like(x)
    moe.moe_combine(cfg, y_perm, pos2, wt, out2)
    torch.cuda.synchronize()
    assert moe.moe_last_device_error() == moe.MOE_OK
    assert torch.equal(pos, pos2) and torch.equal(src, src2)
    assert torch.equal(out, out2)


def test_every_token_on_one_expert(moe, oracle):
    w = synth.Workload("hot", 700, 128, 16, 2, 256, "bf16", 23)
    bias = torch.zeros(16)
    bias[5] = 100.0
    check_layer(moe, oracle, w, device="cpu", bias=bias)


def _layer(moe, name, T):
    w = synth.WORKLOADS[name].with_tokens(T)
    inp = synth.make_inputs(w, device="cuda")
    layer = moe.MoELayer(inp["Wr"], inp["Wgu"], inp["Wd"], w.k,
                         None if inp["bias"] is None else inp["bias"], w.renorm)
    return layer, inp["x"]


@pytest.mark.parametrize("name,T,f", [("mixtral", 4096, 3584),     # rows copied: one-launch dispatch
                                      ("qwen3_zipf", 4096, 768)])  # rows gathered in G1
def test_layers_chained_on_one_stream(moe, name, T, f):
    """Each call takes as its x the output that the previous call's combine
    has just written on the same stream.  The layer's kernels are scheduled
    before their predecessors finish (programmatic dependent launch) but
    read nothing before their wait, so four calls of two alternating layers
    queued with no synchronisation equal, bit for bit, the same chain with a
    device synchronisation after every call."""
    ws = [synth.WORKLOADS[name].with_(T=T, f=f, seed=s) for s in (11, 12)]
    layers = []
    for w in ws:
        inp = synth.make_inputs(w, device="cuda")
        layers.append(moe.MoELayer(inp["Wr"], inp["Wgu"], inp["Wd"], w.k, inp["bias"], w.renorm))
    x0 = synth.make_inputs(ws[0], device="cuda", weights=False)["x"]
    ref = x0
    for i in range(4):
        ref = layers[i % 2](ref).clone()
        torch.cuda.synchronize()
    outs = [torch.empty_like(x0) for _ in range(4)]
    cur = x0
    for i in range(4):
        layers[i % 2](cur, out=outs[i])
        cur = outs[i]
    torch.cuda.synchronize()
    assert torch.equal(outs[-1], ref)
    assert moe.moe_last_device_error(raise_on_error=False) == moe.MOE_OK


def test_empty_batch(moe):
    layer, x = _layer(moe, "qwen3_zipf", 16)
    out = layer(x[:0])
    assert out.shape == (0, x.shape[1])


def test_deterministic(moe):
    layer, x = _layer(moe, "qwen3_zipf", 3000)
    a = layer(x).clone()
    b = layer(x).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("name,T", [("gptoss_prefill", 1000),  # rows gathered in G1
                                    ("mixtral", 512),           # rows copied into x_perm
                                    ("mixtral_dense", 128)])    # k = E: x itself
def test_cuda_graph_capture(moe, name, T):
    """moe_forward needs no host synchronisation, so a captured graph replays
    it with the same result, on each of the ways it moves the rows."""
    layer, x = _layer(moe, name, T)
    ref = layer(x).clone()
    out = torch.empty_like(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer(x, out=out)  # warm up on the capture stream (allocates its workspace)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g, stream=s):
        layer(x, out=out)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_forward_host_buffers(moe):
    layer, x = _layer(moe, "mixtral", 256)
    ref = layer(x).clone()
    cfg = layer.config(x.shape[0])
    x_host = x.cpu().pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    x_dev = torch.empty_like(x)
    out_dev = torch.empty_like(x)
    moe.moe_forward_host(cfg, x_host, layer.Wr, layer.logit_bias, layer.W_gate_up, layer.W_down,
                         out_host, x_dev, out_dev, layer.workspace(x.shape[0]))
    torch.cuda.synchronize()
    assert torch.equal(out_host, ref.cpu())


def test_concurrent_streams_have_their_own_workspace(moe):
    """Two calls in flight on two streams: each stream gets its own workspace
    from MoELayer, and both outputs equal the serial result."""
    layer, x = _layer(moe, "qwen3_zipf", 2048)
    ref = layer(x).clone()
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    T = x.shape[0]
    assert layer.workspace(T, streams[0]).data_ptr() != layer.workspace(T, streams[1]).data_ptr()
    outs = [torch.empty_like(x) for _ in streams]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    for _ in range(4):  # interleaved, so the two streams' kernels overlap
        for st, o in zip(streams, outs):
            layer(x, out=o, stream=st)
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, ref)
