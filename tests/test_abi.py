"""The C ABI library loads and exports what include/moe.h declares; host-side
argument checks and workspace queries behave as documented (no GPU needed:
every call here returns before touching the device)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    from token_dispatch_grouped_fp32_gb300 import build
    build.build()
    from token_dispatch_grouped_fp32_gb300 import moe as _moe
    return _moe


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(moe):
    names = _declared_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(moe):
    for code, name in [(0, "MOE_OK"), (-1, "MOE_ERR_INVALID_ARG"), (-2, "MOE_ERR_UNSUPPORTED"),
                       (-3, "MOE_ERR_WORKSPACE"), (-4, "MOE_ERR_CUDA"),
                       (-5, "MOE_ERR_DEVICE_TIMEOUT"), (-6, "MOE_ERR_BAD_ROUTING")]:
        assert moe.moe_status_string(code) == name


def test_workspace_sizes(moe):
    cfg = moe.config(4096, 4096, 8, 2, 14336, "bf16")
    ws = moe.moe_workspace_size(cfg)
    P = 4096 * 2
    perm = 2 * P * (4096 + 14336 + 4096)
    # + logits, routing and dispatch arrays, and the tensor-core router's scratch:
    # the three-term split weight (E x 3d bf16) and its K-split partial logits
    router = 3 * 8 * 4096 * 2 + 32 * 4096 * 8 * 4
    assert perm <= ws <= perm + 4096 * 8 * 4 + 10 * P * 4 + router + 64 * 1024
    assert moe.moe_workspace_size(moe.config(0, 4096, 8, 2, 14336)) == 0
    # P = 8192 pairs in chunks of 256 (the smallest chunk that keeps <= 256 chunks):
    # the [E][chunks] count matrix, then the rank kernel's ticket (16 bytes)
    assert moe.moe_dispatch_workspace_size(cfg) == 4 * 8 * (P // 256) + 16
    # 40,000 pairs: 128 experts x 157 chunks of 256 would exceed 4096 entries,
    # so chunks of 2048: a [128][20] count matrix
    mid = moe.config(5000, 64, 128, 8, 64)
    assert moe.moe_dispatch_workspace_size(mid) == 4 * 128 * 20 + 16
    big = moe.config(70000, 8, 1024, 8, 8)  # 560,000 pairs: chunks of 2048
    assert moe.moe_dispatch_workspace_size(big) == 4 * 1024 * ((560000 + 2047) // 2048) + 16
    # invalid config -> 0
    assert moe.moe_workspace_size(moe.config(4, 4096, 8, 9, 14336)) == 0


@pytest.mark.parametrize("bad", [
    dict(T=-1), dict(d=0), dict(f=0), dict(E=0), dict(k=0), dict(k=9), dict(d=12), dict(f=20),
    dict(T=2 ** 29, k=8),
])
def test_bad_config_rejected_before_launch(moe, bad):
    base = dict(T=16, d=64, E=8, k=2, f=64)
    base.update(bad)
    cfg = moe.config(base["T"], base["d"], base["E"], base["k"], base["f"])
    st = moe.moe_combine(cfg, 16, 16, 16, 16, stream=0, raise_on_error=False)
    assert st == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_last_error_message()


def test_unsupported_shapes(moe):
    cfg = moe.config(16, 64, 2048, 2, 64)
    assert moe.moe_combine(cfg, 16, 16, 16, 16, stream=0, raise_on_error=False) == \
        moe.MOE_ERR_UNSUPPORTED
    cfg = moe.config(16, 64, 8, 2, 64, dtype=7)
    assert moe.moe_combine(cfg, 16, 16, 16, 16, stream=0, raise_on_error=False) == \
        moe.MOE_ERR_UNSUPPORTED


def test_null_and_misaligned_pointers(moe):
    cfg = moe.config(16, 64, 8, 2, 64)
    assert moe.moe_combine(cfg, None, 16, 16, 16, stream=0, raise_on_error=False) == \
        moe.MOE_ERR_INVALID_ARG
    assert moe.moe_combine(cfg, 16, 16, 16, 24, stream=0, raise_on_error=False) == \
        moe.MOE_ERR_INVALID_ARG
    assert moe.moe_forward(cfg, 16, 16, None, 16, 16, None, 16, 1 << 30, stream=0,
                           raise_on_error=False) == moe.MOE_ERR_INVALID_ARG


def test_route_workspace_size(moe):
    # CUDA-core logits (fp32 activations, or E <= 32 with a small batch) need no workspace
    assert moe.moe_route_workspace_size(moe.config(512, 4096, 8, 2, 14336, "bf16")) == 0
    assert moe.moe_route_workspace_size(moe.config(64, 128, 128, 2, 256, "f32")) == 0
    assert moe.moe_route_workspace_size(moe.config(4096, 4096, 33, 2, 14336, "bf16")) == 0
    # E = 8 at T = 4096 runs on the tensor cores (N padded to 16)
    n8 = moe.moe_route_workspace_size(moe.config(4096, 4096, 8, 2, 14336, "bf16"))
    assert 8 * 3 * 4096 * 2 + 4096 * 8 * 4 <= n8 <= 8 * 3 * 4096 * 2 + 256 + 64 * 4096 * 8 * 4
    # tensor-core logits: split weight (E*3d bf16) + fp32 partial logits
    T, d, E = 8192, 7168, 256
    n = moe.moe_route_workspace_size(moe.config(T, d, E, 8, 2048, "bf16"))
    assert n >= E * 3 * d * 2 + T * E * 4
    assert n <= E * 3 * d * 2 + 256 + 64 * T * E * 4
    cfg = moe.config(T, d, E, 8, 2048, "bf16")
    st = moe.moe_route(cfg, 16, 16, None, 16, 16, 16, 16, n - 1, stream=0, raise_on_error=False)
    assert st == moe.MOE_ERR_WORKSPACE
    # moe_forward's workspace also holds h_perm and y_perm (this shape gathers
    # its rows through src_token, so it holds no x_perm)
    assert moe.moe_workspace_size(cfg) >= n + 2 * T * 8 * (2048 + d)


def test_workspace_too_small(moe):
    cfg = moe.config(16, 64, 8, 2, 64)
    need = moe.moe_workspace_size(cfg)
    st = moe.moe_forward(cfg, 16, 16, None, 16, 16, 16, 16, need - 1, stream=0,
                         raise_on_error=False)
    assert st == moe.MOE_ERR_WORKSPACE
    st = moe.moe_dispatch(cfg, 16, None, 16, 16, 16, 16, 16, 16, 16, 3, stream=0,
                          raise_on_error=False)
    assert st == moe.MOE_ERR_WORKSPACE


def test_empty_batch_is_a_no_op(moe):
    cfg = moe.config(0, 64, 8, 2, 64)
    assert moe.moe_forward(cfg, 16, 16, None, 16, 16, 16, 16, 0, stream=0) == moe.MOE_OK
    assert moe.moe_route(cfg, 16, 16, None, 16, 16, 16, None, 0, stream=0) == moe.MOE_OK
    assert moe.moe_dispatch(cfg, 16, None, 16, 16, 16, 16, 16, 16, 16, 0, stream=0) == moe.MOE_OK
    assert moe.moe_grouped_swiglu(cfg, 16, 16, 16, 16, 16, 16, stream=0) == moe.MOE_OK
    assert moe.moe_combine(cfg, 16, 16, 16, 16, stream=0) == moe.MOE_OK


def test_raises_with_detail(moe):
    cfg = moe.config(16, 64, 8, 2, 64)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_combine(cfg, None, 16, 16, 16, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    assert "NULL" in str(ei.value)


def test_input_scaling_needs_weights_at_dispatch_only(moe):
    cfg = moe.config(16, 64, 8, 2, 64, scale_inputs=True)
    ws = 1 << 20
    st = moe.moe_dispatch(cfg, 16, None, 16, 16, 16, 16, 16, 16, 16, ws, stream=0,
                          raise_on_error=False)
    assert st == moe.MOE_ERR_INVALID_ARG  # scale_inputs without topk_w
    assert "NULL" in moe.moe_last_error_message()


def test_forward_kernel_launches(moe):
    """The bench's gpu_launches claim comes from the library's own launch plan."""
    # Mixtral-shaped, bf16, E = 8, T = 4096: tensor-core router (weight split,
    # logits, top-k) + dispatch (one launch: E <= 16, P <= 16384, 8 KB rows)
    # + G1, G2 + combine
    assert moe.moe_forward_kernel_launches(moe.config(4096, 4096, 8, 2, 14336, "bf16")) == 7
    # the dispatch in two launches (rank, place rows): P > 16384, E > 16,
    # rows under k KB, or rows scaled by the weights (fp32 copies them)
    assert moe.moe_forward_kernel_launches(moe.config(8193, 4096, 16, 2, 14336, "bf16")) == 8
    # (E = 17: CUDA-core logits with the selection in the same launch)
    assert moe.moe_forward_kernel_launches(moe.config(8192, 4096, 17, 2, 14336, "bf16")) == 6
    assert moe.moe_forward_kernel_launches(moe.config(4096, 512, 8, 2, 14336, "bf16")) == 8
    # fp32 (CUDA-core logits and selection in one launch): 5, and 6 when the
    # dispatch copies rows scaled by the weights
    assert moe.moe_forward_kernel_launches(moe.config(4096, 4096, 8, 2, 14336, "f32")) == 5
    assert moe.moe_forward_kernel_launches(
        moe.config(4096, 4096, 8, 2, 14336, "f32", scale_inputs=True)) == 6
    # about 256 rows per expert: G1 and G2 each as a CTA-pair launch and a
    # single-CTA launch, the experts split between them
    assert moe.moe_forward_kernel_launches(moe.config(8192, 2880, 128, 4, 2880, "bf16")) == 10
    # small batch, E <= 32: logits and selection in one CUDA-core launch
    assert moe.moe_forward_kernel_launches(moe.config(64, 128, 8, 2, 256, "f32")) == 6
    # fp32 activations, E > 32: CUDA-core logits, then the top-k kernel
    assert moe.moe_forward_kernel_launches(moe.config(4096, 128, 64, 2, 256, "f32")) == 7
    # k = E: one dispatch launch, no permutation (bf16 with the weights on
    # the inputs too: the first GEMM scales the rows' products); fp32 with
    # the weights on the inputs copies scaled rows (two dispatch launches)
    assert moe.moe_forward_kernel_launches(moe.config(1024, 4096, 8, 8, 14336, "bf16", False)) == 7
    assert moe.moe_forward_kernel_launches(
        moe.config(1024, 4096, 8, 8, 14336, "bf16", False, scale_inputs=True)) == 7
    assert moe.moe_forward_kernel_launches(
        moe.config(64, 128, 8, 8, 256, "f32", False, scale_inputs=True)) == 6
    assert moe.moe_forward_kernel_launches(moe.config(0, 128, 8, 2, 256, "bf16")) == 0
    assert moe.moe_forward_kernel_launches(moe.config(4, 4096, 8, 9, 14336)) == -1


def test_wait_limit_has_a_floor_outside_the_test_hook(moe):
    """A limit below one pipeline stage could let one CTA of a pair abort with
    a copy in flight that its pair never armed, so limits below 10 ms are
    raised to 10 ms; only the failure-path test hook may go lower."""
    try:
        moe.moe_set_wait_limit_ns(1_000)
        assert moe.moe_wait_limit_ns() == 10_000_000
        moe.moe_set_wait_limit_ns(50_000_000)
        assert moe.moe_wait_limit_ns() == 50_000_000
        moe.moe_set_wait_limit_ns(1_000_000)
        moe.moe_debug_inject_wait_timeout(True)
        assert moe.moe_wait_limit_ns() == 1_000_000
        moe.moe_debug_inject_wait_timeout(False)
        assert moe.moe_wait_limit_ns() == 10_000_000
    finally:
        moe.moe_debug_inject_wait_timeout(False)
        moe.moe_set_wait_limit_ns(0)
    assert moe.moe_wait_limit_ns() == 2_000_000_000


@pytest.mark.parametrize("T,d,E,k,f,dtype,scale,x_perm", [
    (4096, 4096, 8, 2, 14336, "bf16", False, True),   # f > 2048: the permuted copy
    (8192, 7168, 256, 8, 2048, "bf16", False, False),  # gathered rows
    (8192, 2880, 128, 4, 2880, "bf16", False, False),  # gathered rows, f at 2880
    (8192, 2880, 128, 4, 3136, "bf16", False, True),   # f above the gather's limit: copied
    (8192, 7168, 256, 8, 2048, "bf16", True, False),   # weights on the inputs: still gathered
    (4096, 4096, 8, 2, 14336, "bf16", True, True),     # weights on the inputs, f > 2048: scaled copy
    (8192, 7200, 256, 8, 2048, "bf16", False, True),   # d not a multiple of 64
    (64, 128, 8, 2, 256, "f32", False, True),          # fp32 path
    (1, 64, 3, 3, 8, "bf16", False, False),           # k == E: x itself
    (1, 64, 3, 3, 8, "bf16", True, False),           # k == E, weights on the inputs: x itself
    (64, 128, 8, 8, 256, "f32", True, True)])          # the same in fp32: scaled copy
def test_workspace_layout(moe, T, d, E, k, f, dtype, scale, x_perm):
    """The documented regions of moe_forward's workspace are 256-byte
    aligned, in order, large enough for their arrays, and inside the total;
    x_perm is absent exactly where moe_forward forms no permuted copy of x
    (k == E, except fp32 with the weights on the inputs; or the gathered-row
    path: bf16, d a multiple of 64, f <= 3072), and the total is then that
    much smaller."""
    cfg = moe.config(T, d, E, k, f, dtype, scale_inputs=scale)
    L = moe.moe_workspace_layout(cfg)
    es = 2 if dtype == "bf16" else 4
    P = T * k
    regions = [("logits", 4 * T * E), ("topk_idx", 4 * P), ("topk_w", 4 * P), ("counts", 4 * E),
               ("offsets", 4 * (E + 1)), ("pos", 4 * P), ("src_token", 4 * P),
               ("h_perm", es * P * f), ("y_perm", es * P * d)]
    assert (L.x_perm != moe.MOE_WS_ABSENT) == x_perm
    if x_perm:
        regions.append(("x_perm", es * P * d))
    spans = sorted((getattr(L, n), getattr(L, n) + size, n) for n, size in regions)
    for (a0, a1, n), (b0, _, m) in zip(spans, spans[1:]):
        assert a1 <= b0, (n, m)  # no overlap
    for a0, a1, n in spans:
        assert a0 % 256 == 0, n
        assert a1 <= L.total, n
    assert L.total == moe.moe_workspace_size(cfg)
    z = moe.moe_workspace_layout(moe.config(0, d, E, k, f, dtype))
    assert z.total == 0 and z.x_perm == 0
    with pytest.raises(moe.MoEError):
        moe.moe_workspace_layout(moe.config(4, 64, 8, 9, 8))
