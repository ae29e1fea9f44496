"""Dispatch parity: counts, offsets, the permutation and its inverse bit-exact
against the oracle; the permuted rows are byte copies of the token rows."""
import numpy as np
import pytest
import torch

from token_dispatch_grouped_fp32_gb300 import synth
from tests.gpu_util import load_moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return load_moe()


def _routing(oracle, T, E, k, seed, skew=0.0):
    L = synth.make_logits(T, E, seed).numpy()
    if skew:
        L = L + skew * (np.arange(E, dtype=np.float32) == 3)[None, :]
    idx, _ = oracle.topk(L, k, True)
    return idx


def _run_dispatch(moe, idx, x, E):
    T, k = idx.shape
    d = x.shape[1]
    cfg = moe.config(T, d, E, k, 8, x.dtype)
    P = T * k
    dev = "cuda"
    counts = torch.full((E,), -1, dtype=torch.int32, device=dev)
    offsets = torch.full((E + 1,), -1, dtype=torch.int32, device=dev)
    pos = torch.full((P,), -1, dtype=torch.int32, device=dev)
    src = torch.full((P,), -1, dtype=torch.int32, device=dev)
    x_perm = torch.zeros(P, d, dtype=x.dtype, device=dev)
    ws = torch.empty(max(256, moe.moe_dispatch_workspace_size(cfg)), dtype=torch.uint8, device=dev)
    moe.moe_dispatch(cfg, torch.from_numpy(idx).cuda(), None, x.cuda(), counts, offsets, pos, src,
                     x_perm, ws)
    torch.cuda.synchronize()
    return counts.cpu().numpy(), offsets.cpu().numpy(), pos.cpu().numpy(), src.cpu().numpy(), \
        x_perm.cpu()


DISPATCH_CASES = [
    # T, E, k, d, dtype, skew
    (1, 8, 2, 64, torch.bfloat16, 0.0),
    (100, 8, 2, 64, torch.bfloat16, 0.0),
    (3000, 8, 2, 64, torch.float32, 0.0),      # 24 chunks, ragged tail
    (8192, 32, 2, 64, torch.bfloat16, 0.0),    # 64 chunks of 256 (2048 counts)
    (3, 1024, 8, 16, torch.bfloat16, 0.0),     # a single chunk, E = 1024
    (1500, 33, 4, 64, torch.bfloat16, 0.0),    # 24 chunks, E not a multiple of 8
    (8193, 32, 2, 64, torch.bfloat16, 0.0),    # 65 chunks, the last of 2 pairs
    (5000, 128, 8, 32, torch.bfloat16, 0.0),   # 20 chunks
    (2049, 1, 1, 16, torch.bfloat16, 0.0),     # single expert
    (1000, 64, 6, 24, torch.bfloat16, 0.0),
    (4000, 16, 2, 8, torch.bfloat16, 50.0),    # one expert takes every token
    (6000, 1024, 8, 8, torch.bfloat16, 0.0),   # many experts, most empty per chunk
    (300000, 16, 8, 8, torch.bfloat16, 0.0),   # 2.4M pairs: chunks grow past 2048
    # rows of at least k KB and at most 16 KB: a warp per token stages its row
    # in shared memory before the ranking ends and writes it k times
    (700, 8, 2, 1024, torch.bfloat16, 0.0),    # 2 KB rows, 175 blocks of 4 tokens
    (301, 64, 1, 512, torch.bfloat16, 0.0),    # k = 1 at 1 KB, last block of 1 token
    (513, 16, 4, 4096, torch.float32, 0.0),    # 16 KB fp32 rows (the largest staged)
    (257, 8, 2, 8192, torch.bfloat16, 50.0),   # 16 KB bf16 rows, one expert takes most
    (130, 8, 2, 8200, torch.bfloat16, 0.0),    # 16,400-byte rows: a warp per pair again
    (64, 32, 8, 2048, torch.bfloat16, 0.0),    # 4 KB rows with k = 8: a warp per pair
    # E <= 16 and P <= 16384 with staged rows: one launch, each block counting
    # every id itself (the cases above with E <= 16 and rows of k KB to 16 KB
    # take it too)
    (4096, 8, 2, 4096, torch.bfloat16, 0.0),   # the Mixtral layer's shape: 152 blocks
    (4096, 8, 2, 4096, torch.float32, 0.0),    # 16 KB fp32 rows: 8 warps a block
    (4096, 8, 2, 4096, torch.bfloat16, 50.0),  # one expert takes every token
    (8192, 16, 2, 4096, torch.bfloat16, 0.0),  # P = 16384, the largest; experts 8-15
    (8193, 16, 2, 4096, torch.bfloat16, 0.0),  # P = 16386: two launches again
    (2047, 16, 8, 8192, torch.bfloat16, 0.0),  # k = 8, 16 KB rows, ragged blocks
    (5, 16, 16, 8192, torch.bfloat16, 0.0),    # k = E = 16, one block of 5 tokens
    (2433, 8, 2, 1024, torch.bfloat16, 0.0),   # just past 152 blocks of 16 tokens
    (1000, 3, 2, 2048, torch.bfloat16, 0.0),   # three experts
    (1, 8, 2, 4096, torch.bfloat16, 0.0),      # a single token
    (64, 8, 2, 4096, torch.bfloat16, 0.0),     # 64 blocks of one token and one warp
    (1024, 8, 8, 4096, torch.bfloat16, 0.0),   # k = E = 8: each row written 8 times
    (16384, 16, 1, 1024, torch.bfloat16, 0.0), # k = 1 at P = 16384: 108 tokens a block
]


@pytest.mark.parametrize("T,E,k,d,dtype,skew", DISPATCH_CASES)
def test_dispatch_matches_oracle(moe, oracle, T, E, k, d, dtype, skew):
    idx = _routing(oracle, T, E, k, 77 + T + E, skew)
    g = torch.Generator().manual_seed(T)
    x = torch.randn(T, d, generator=g).to(dtype)
    counts, offsets, pos, src, x_perm = _run_dispatch(moe, idx, x, E)
    rc, ro, rp, rs = oracle.dispatch(idx, E)
    np.testing.assert_array_equal(counts, rc)
    np.testing.assert_array_equal(offsets, ro)
    np.testing.assert_array_equal(pos, rp)
    np.testing.assert_array_equal(src, rs)
    # rows are byte copies of the token rows
    assert torch.equal(x_perm, x[torch.from_numpy(rs).long()])


@pytest.mark.parametrize("T,d,E", [(50, 16, 8),     # one chunk
                                   (20000, 16, 8),  # 157 chunks
                                   (50, 2048, 32),  # rows staged, two launches
                                   (50, 2048, 8),   # one launch
                                   (3000, 4096, 8)])  # one launch, many blocks
def test_dispatch_flags_out_of_range_expert(moe, oracle, T, d, E):
    k = 2
    idx = _routing(oracle, T, E, k, 5)
    idx[7, 1] = E + 3
    x = torch.randn(T, d).to(torch.bfloat16)
    moe.moe_last_device_error(raise_on_error=False)  # clear
    counts, offsets, pos, src, x_perm = _run_dispatch(moe, idx, x, E)
    assert moe.moe_last_device_error(raise_on_error=False) == moe.MOE_ERR_BAD_ROUTING
    assert counts.sum() == T * k - 1 and offsets[-1] == T * k - 1
    assert pos[7 * k + 1] == -1
    # every placed row is its token's row; the dropped pair's token still has
    # its other pair placed
    keep = pos >= 0
    rows = torch.from_numpy(pos[keep]).long()
    toks = torch.from_numpy(np.nonzero(keep)[0] // k).long()
    assert torch.equal(x_perm[rows], x[toks])
    assert x_perm.shape[0] == T * k and int(keep.sum()) == T * k - 1
    assert moe.moe_last_device_error(raise_on_error=False) == moe.MOE_OK  # cleared


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_dispatch_scales_rows_when_weights_act_on_inputs(moe, oracle, dtype):
    """scale_inputs: row r of x_perm is w[q] * x[t] formed in fp32 and rounded
    once to the activation dtype (q the pair of row r, t its token)."""
    T, E, k, d = 1500, 16, 4, 136
    L = synth.make_logits(T, E, 41).numpy()
    idx, w = oracle.topk(L, k, True)
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(3)).to(dtype)
    wt = torch.from_numpy(w.astype(np.float32))
    cfg = moe.config(T, d, E, k, 8, dtype, True, scale_inputs=True)
    P = T * k
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pos = torch.empty(P, dtype=torch.int32, device="cuda")
    src = torch.empty(P, dtype=torch.int32, device="cuda")
    x_perm = torch.zeros(P, d, dtype=dtype, device="cuda")
    ws = torch.empty(max(256, moe.moe_dispatch_workspace_size(cfg)), dtype=torch.uint8, device="cuda")
    moe.moe_dispatch(cfg, torch.from_numpy(idx).cuda(), wt.cuda(), x.cuda(), counts, offsets, pos,
                     src, x_perm, ws)
    torch.cuda.synchronize()
    rc, ro, rp, rs = oracle.dispatch(idx, E)
    np.testing.assert_array_equal(pos.cpu().numpy(), rp)
    pair_of_row = np.empty(P, np.int64)
    pair_of_row[rp] = np.arange(P)
    expect = (x.float()[torch.from_numpy(rs).long()] *
              wt.reshape(-1)[torch.from_numpy(pair_of_row)][:, None]).to(dtype)
    assert torch.equal(x_perm.cpu(), expect)


@pytest.mark.parametrize("E", [8, 32])  # one launch / two launches
def test_dispatch_reads_x_written_just_before(moe, oracle, E):
    """The row copy of a standalone dispatch reads x before the ranking is
    done; x written by the kernel just before the call, on the same stream,
    must still be what it copies.  Each round overwrites x on the device and
    dispatches at once; every row of x_perm is checked."""
    T, k, d = 700, 2, 1024  # rows staged per token (2 KB, k = 2)
    idx = _routing(oracle, T, E, k, 19)
    _, _, _, rs = oracle.dispatch(idx, E)
    cfg = moe.config(T, d, E, k, 8, torch.bfloat16)
    P = T * k
    dev = "cuda"
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    pos = torch.empty(P, dtype=torch.int32, device=dev)
    src = torch.empty(P, dtype=torch.int32, device=dev)
    x_perm = torch.empty(P, d, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(256, moe.moe_dispatch_workspace_size(cfg)), dtype=torch.uint8, device=dev)
    idx_d = torch.from_numpy(idx).cuda()
    x_d = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    g = torch.Generator(device=dev).manual_seed(5)
    for _ in range(4):
        x_d.normal_(generator=g)  # a kernel writing x just before the dispatch
        moe.moe_dispatch(cfg, idx_d, None, x_d, counts, offsets, pos, src, x_perm, ws)
        assert torch.equal(x_perm, x_d[torch.from_numpy(rs).long().cuda()])


@pytest.mark.parametrize("E", [8, 32])
def test_dispatch_in_a_cuda_graph(moe, oracle, E):
    """A standalone dispatch captured in a CUDA graph (E = 8: its one launch;
    E = 32: its memset, the rank launch and the row copy) and replayed on new
    routing and rows gives the oracle's result each time."""
    T, k, d = 513, 2, 2048
    cfg = moe.config(T, d, E, k, 8, torch.bfloat16)
    P = T * k
    dev = "cuda"
    idx_d = torch.empty(T, k, dtype=torch.int32, device=dev)
    x_d = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    pos = torch.empty(P, dtype=torch.int32, device=dev)
    src = torch.empty(P, dtype=torch.int32, device=dev)
    x_perm = torch.empty(P, d, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(256, moe.moe_dispatch_workspace_size(cfg)), dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream()
    idx0 = _routing(oracle, T, E, k, 1)
    idx_d.copy_(torch.from_numpy(idx0))
    x_d.normal_()
    torch.cuda.synchronize()
    with torch.cuda.stream(st):  # one eager call first: the library's set-up
        moe.moe_dispatch(cfg, idx_d, None, x_d, counts, offsets, pos, src, x_perm, ws, stream=st)
    st.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        moe.moe_dispatch(cfg, idx_d, None, x_d, counts, offsets, pos, src, x_perm, ws, stream=st)
    for seed in (2, 3):
        idx = _routing(oracle, T, E, k, seed)
        idx_d.copy_(torch.from_numpy(idx))
        x = torch.randn(T, d, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
        x_d.copy_(x)
        graph.replay()
        torch.cuda.synchronize()
        rc, ro, rp, rs = oracle.dispatch(idx, E)
        np.testing.assert_array_equal(counts.cpu().numpy(), rc)
        np.testing.assert_array_equal(offsets.cpu().numpy(), ro)
        np.testing.assert_array_equal(pos.cpu().numpy(), rp)
        np.testing.assert_array_equal(src.cpu().numpy(), rs)
        assert torch.equal(x_perm.cpu(), x[torch.from_numpy(rs).long()])
