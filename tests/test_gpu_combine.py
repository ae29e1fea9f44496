"""Combine parity: moe_combine alone against the oracle's combine.

- One-hot expert rows (row r of y_perm is the unit vector of column r): then
  out[t] holds exactly w[t, j] (rounded once to the activation dtype) at
  column pos[t*k + j] and zeros elsewhere, so the GPU result must equal the
  oracle's exactly.  Distinct weights per slot catch a weight taken from the
  wrong slot; columns tell the rows apart.
- Random expert rows: elementwise within the rounding of k fused
  multiply-adds in fp32 (each off by at most 2^-24 of the running sum, itself
  at most S = sum_j |w_j y_j|), plus the final rounding to bf16 (2^-8
  relative) for bf16 activations.

The routing (pos, w) comes from the oracle's top-k and dispatch on seeded
logits; the expert rows are seeded random values."""
import numpy as np
import pytest
import torch

from token_dispatch_grouped_fp32_gb300 import synth
from tests.gpu_util import f32, load_moe

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24


@pytest.fixture(scope="module")
def moe():
    return load_moe()


def _routing(oracle, T, E, k, seed, renorm=True):
    L = synth.make_logits(T, E, seed).numpy()
    idx, w = oracle.topk(L, k, renorm)
    _, _, pos, _ = oracle.dispatch(idx, E)
    return pos, w.astype(np.float32)


def _combine(moe, T, d, k, y_perm, pos, w, dtype, scale_inputs=False):
    cfg = moe.config(T, d, 16, k, 8, dtype, scale_inputs=scale_inputs)
    out = torch.full((T, d), float("nan"), dtype=dtype, device="cuda")
    moe.moe_combine(cfg, y_perm.cuda(), torch.from_numpy(pos).cuda(),
                    None if scale_inputs else torch.from_numpy(w).cuda(), out)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("scale_inputs", [False, True])
@pytest.mark.parametrize("T,k", [(37, 2), (64, 8), (200, 1)])
def test_combine_one_hot_rows_exact(moe, oracle, dtype, scale_inputs, T, k):
    P = T * k
    d = (P + 7) // 8 * 8 + 8  # every row its own column, d a multiple of 8
    pos, w = _routing(oracle, T, 16, k, 900 + T + k)
    y_perm = torch.zeros(P, d, dtype=dtype)
    y_perm[torch.arange(P), torch.arange(P)] = 1.0
    got = _combine(moe, T, d, k, y_perm, pos, w, dtype, scale_inputs)
    ref = oracle.combine(f32(y_perm), pos, w.astype(np.float64), k, scale_inputs=scale_inputs)
    # each entry of ref is one weight (or 1, or 0): round it once like the GPU
    ref_t = torch.from_numpy(ref).to(torch.float32).to(dtype)
    assert torch.equal(got, ref_t)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("scale_inputs", [False, True])
@pytest.mark.parametrize("T,d,k", [(1000, 136, 2), (333, 4096, 8), (8, 64, 4), (4099, 520, 1)])
def test_combine_random_rows(moe, oracle, dtype, scale_inputs, T, d, k):
    P = T * k
    pos, w = _routing(oracle, T, 32, k, 950 + T + d, renorm=bool(k % 2))
    y_perm = torch.randn(P, d, generator=torch.Generator().manual_seed(T + d)).to(dtype)
    got = f32(_combine(moe, T, d, k, y_perm, pos, w, dtype, scale_inputs)).astype(np.float64)
    ys = f32(y_perm).astype(np.float64)
    wd = np.ones((T, k)) if scale_inputs else w.astype(np.float64)
    ref = oracle.combine(ys, pos, wd, k)
    S = oracle.combine(np.abs(ys), pos, np.abs(wd), k)  # sum_j |w_j y_j|
    tol = k * U32 * S
    if dtype == torch.bfloat16:
        tol = tol + 2.0 ** -8 * (np.abs(ref) + tol)
    assert np.isfinite(got).all()
    assert (np.abs(got - ref) <= tol + 1e-30).all()
