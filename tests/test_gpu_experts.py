"""Grouped SwiGLU parity: h_perm and y_perm of every row against the oracle's
expert FFN, for ragged segments (empty experts, partial row tiles, partial
column tiles and a partial K step), with both tile shapes: 128-row tiles on
one CTA (small per-expert batches), 256-row tiles on a CTA pair (batches
averaging >= 512 rows per expert), and in between each expert on the shape
that pads it less."""
import numpy as np
import pytest
import torch

from tests.gpu_util import f32, fp32_tolerance, layer_tolerance, load_moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return load_moe()


EXPERT_CASES = [
    # counts per expert, d, f
    ([0, 300, 1, 129, 0, 700, 128, 2], 256, 384),
    ([5, 0, 260], 264, 200),            # ragged K (264 = 4*64 + 8), ragged N tiles
    ([1], 128, 2880 // 8),              # one row
    ([513], 64, 1024),                  # one expert, 5 row tiles
    ([40] * 16, 320, 136),
    ([0, 0, 0, 9], 72, 8),              # tiny f: one partial column vector
    # >= 512 rows per expert on average: CTA-pair tiles (256 rows)
    ([0, 700, 1030, 5, 1500], 264, 200),
    ([600, 0, 900], 128, 384),
    ([2049], 64, 136),
    # K above 3072: the per-row epilogue store (shorter K uses transposed stores)
    ([3, 130, 0, 70], 3136, 136),       # gate/up K = 3136, down K = 136
    ([1, 90, 40], 96, 3136),            # down K = 3136
    ([520, 0, 530], 3136, 72),          # CTA pairs, gate/up K = 3136
    ([520, 530], 64, 3200),             # CTA pairs, down K = 3200
    # CTA pairs whose experts end in short row tiles (76, 108, 176 rows; 128, 129, 1)
    ([1100, 620, 1200, 0], 200, 328),
    ([128, 129, 1, 1800], 72, 136),
    # 64..511 rows per expert on average: each expert on the tile shape that pads
    # it less (256-row pairs for 129..256 rows, 128-row single CTAs for 300)
    ([200, 256, 129, 250], 128, 256),   # every expert on pairs: the single-CTA launch is empty
    ([300, 129, 64, 256, 1], 192, 136), # both launches busy
    # segment ends on both sides of every tile boundary, in both launches
    ([128, 129, 256, 257, 384, 385, 0, 1, 511, 512, 640], 136, 200),
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("counts,d,f", EXPERT_CASES)
def test_grouped_swiglu_matches_oracle(moe, oracle, counts, d, f, dtype):
    E = len(counts)
    P = int(sum(counts))
    g = torch.Generator().manual_seed(P + d + f)
    x_perm = torch.randn(P, d, generator=g).to(dtype)
    Wgu = (torch.randn(E, d, 2 * f, generator=g) * d ** -0.5).to(dtype)
    Wd = (torch.randn(E, f, d, generator=g) * d ** -0.5).to(dtype)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    # T*k must equal P for the call's sizes; use k = 1
    cfg = moe.config(P, d, E, 1, f, dtype)
    h = torch.full((P, f), float("nan"), dtype=dtype, device="cuda")
    y = torch.full((P, d), float("nan"), dtype=dtype, device="cuda")
    moe.moe_grouped_swiglu(cfg, x_perm.cuda(), torch.from_numpy(offsets).cuda(), Wgu.cuda(),
                           Wd.cuda(), h, y)
    torch.cuda.synchronize()
    xs, gus, ds = f32(x_perm), f32(Wgu), f32(Wd)
    ref_h = np.empty((P, f))
    ref_y = np.empty((P, d))
    for e in range(E):
        for r in range(offsets[e], offsets[e + 1]):
            ref_h[r], ref_y[r] = oracle.expert_ffn_row(xs[r], gus[e], ds[e])
    gh, gy = f32(h).astype(np.float64), f32(y).astype(np.float64)
    assert np.isfinite(gh).all() and np.isfinite(gy).all()
    if dtype == torch.float32:  # fp32 path: the fp32 rounding bound
        tol_h, tol_y = fp32_tolerance(ref_h, d, d), fp32_tolerance(ref_y, d, d, f)
    else:  # bf16 operands, h and y rounded to bf16: the stated layer bound
        tol_h, tol_y = layer_tolerance(ref_h), layer_tolerance(ref_y)
    assert np.abs(gh - ref_h).max() <= tol_h
    assert np.abs(gy - ref_y).max() <= tol_y
