"""moe_dispatch_noalloc: the dispatch for callers that cannot allocate device
memory for scratch (a plugin whose host framework owns every device buffer,
or a service that must not call cudaMalloc after start-up).  Its histogram
scratch lives in a fixed array inside the library.

Called straight through the C ABI (ctypes), twice in a row with different
routings, and compared with moe_dispatch on a torch-allocated workspace.
Dispatch results are integers and byte copies, so the tolerance the other
dispatch tests use -- bit-exact -- applies.  This file is collected last on
purpose; it needs no state from the other tests."""
import ctypes

import numpy as np
import pytest
import torch

from token_dispatch_grouped_fp32_gb300 import synth
from tests.gpu_util import load_moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    moe = load_moe()
    lib = ctypes.CDLL(moe.LIB_PATH)
    vp = ctypes.c_void_p
    lib.moe_dispatch_noalloc.argtypes = [ctypes.POINTER(moe.moe_config_t)] + [vp] * 9
    lib.moe_dispatch_noalloc.restype = ctypes.c_int
    return moe, lib


def _outputs(T, E, k, d, dtype):
    P = T * k
    return [torch.full((E,), -1, dtype=torch.int32, device="cuda"),
            torch.full((E + 1,), -1, dtype=torch.int32, device="cuda"),
            torch.full((P,), -1, dtype=torch.int32, device="cuda"),
            torch.full((P,), -1, dtype=torch.int32, device="cuda"),
            torch.zeros(P, d, dtype=dtype, device="cuda")]


def _noalloc(lib, cfg, idx, x, outs):
    moe, so = lib
    p = [ctypes.c_void_p(idx.data_ptr()), None] + [ctypes.c_void_p(t.data_ptr()) for t in [x] + outs]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return so.moe_dispatch_noalloc(ctypes.byref(cfg), *p, stream)


@pytest.mark.parametrize("T,E,k,d", [(3000, 8, 2, 64), (5000, 128, 8, 32), (300000, 16, 8, 8),
                                     (777, 1024, 8, 16)])
def test_noalloc_matches_dispatch_twice(lib, oracle, T, E, k, d):
    moe, _ = lib
    dtype = torch.bfloat16
    cfg = moe.config(T, d, E, k, 8, dtype)
    for call in range(2):  # second call reuses the array with a different routing
        L = synth.make_logits(T, E, 500 + call + T).numpy()
        idx_np, _ = oracle.topk(L, k, True)
        idx = torch.from_numpy(idx_np).cuda()
        x = torch.randn(T, d, generator=torch.Generator().manual_seed(call)).to(dtype).cuda()
        ref = _outputs(T, E, k, d, dtype)
        ws = torch.empty(max(256, moe.moe_dispatch_workspace_size(cfg)), dtype=torch.uint8,
                         device="cuda")
        moe.moe_dispatch(cfg, idx, None, x, *ref, ws)
        got = _outputs(T, E, k, d, dtype)
        assert _noalloc(lib, cfg, idx, x, got) == moe.MOE_OK
        torch.cuda.synchronize()
        assert moe.moe_last_device_error() == moe.MOE_OK
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_noalloc_rejects_sizes_beyond_the_array(lib):
    moe, _ = lib
    T, E, k, d = 70000, 1024, 8, 8  # 274 chunks x 1024 experts > 262,144 entries
    cfg = moe.config(T, d, E, k, 8, torch.bfloat16)
    assert moe.moe_dispatch_workspace_size(cfg) > (1 << 20)
    idx = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    x = torch.zeros(T, d, dtype=torch.bfloat16, device="cuda")
    outs = _outputs(T, E, k, d, torch.bfloat16)
    assert _noalloc(lib, cfg, idx, x, outs) == moe.MOE_ERR_UNSUPPORTED
    assert "static array" in moe.moe_last_error_message()
    torch.cuda.synchronize()
    assert (outs[0] == -1).all()  # nothing launched


def test_noalloc_empty_batch(lib):
    moe, so = lib
    cfg = moe.config(0, 8, 8, 2, 8, torch.bfloat16)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert so.moe_dispatch_noalloc(ctypes.byref(cfg), *([None] * 8), stream) == moe.MOE_OK
