"""Failure detection without a GPU fault: the grouped GEMM's bounded waits.

The test hook moe_debug_inject_wait_timeout makes the GEMM's MMA issuer wait
on a barrier that nothing signals before it issues any MMA.  With the wait
limit at 1 ms that wait runs out: the kernel records MOE_ERR_DEVICE_TIMEOUT in
the device error word, the other roles give up at their next wait, the
producers wait for the copies they issued (a 1 s floor), the tensor memory is
freed and the kernel returns.  The host reads the status; the context stays
usable and the next call (hook off, default limit) is bit-identical to one
made before.  No trap, fault or hang is involved.  Every tile mode is
covered: CTA pairs (Mixtral-shaped, >= 512 rows per expert), single CTAs, and
the experts split between the two (about 128 rows per expert); and each of
them again on the Qwen3 shape, whose first grouped GEMM gathers its rows (its
copying and reporting warps give up at their next wait as well, and every
copy they issued lands before the kernel returns)."""
import pytest
import torch

from token_dispatch_grouped_fp32_gb300 import synth
from tests.gpu_util import load_moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return load_moe()


@pytest.mark.parametrize("name,T", [("mixtral", 4096), ("gptoss_prefill", 512),
                                    ("gptoss_prefill", 4096),  # pairs; single CTAs; both
                                    ("qwen3_zipf", 8192), ("qwen3_zipf", 512),
                                    ("qwen3_zipf", 2048)])  # the same, rows gathered
def test_wait_timeout_is_reported_and_recoverable(moe, name, T):
    w = synth.WORKLOADS[name].with_tokens(T)
    inp = synth.make_inputs(w, device="cuda")
    layer = moe.MoELayer(inp["Wr"], inp["Wgu"], inp["Wd"], w.k, inp["bias"], w.renorm)
    x = inp["x"]
    ref = layer(x).clone()
    torch.cuda.synchronize()
    assert moe.moe_last_device_error() == moe.MOE_OK
    try:
        moe.moe_set_wait_limit_ns(1_000_000)
        moe.moe_debug_inject_wait_timeout(True)
        layer(x)
        st = moe.moe_last_device_error(raise_on_error=False)
    finally:
        moe.moe_debug_inject_wait_timeout(False)
        moe.moe_set_wait_limit_ns(0)  # back to the default
    assert st == moe.MOE_ERR_DEVICE_TIMEOUT
    out = layer(x)
    torch.cuda.synchronize()
    assert moe.moe_last_device_error() == moe.MOE_OK
    assert torch.equal(out, ref)
