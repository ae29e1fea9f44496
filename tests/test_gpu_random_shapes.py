"""A seeded sweep of layer shapes through moe_forward against the oracle.

Each case draws T, d, E, k, f, the activation dtype, renormalisation and
where the routing weights act (outputs or inputs), so the sweep crosses the
paths moe_forward chooses among: rows copied into x_perm or gathered inside
the first grouped GEMM (bf16, d a multiple of 64, f <= 3072), k = E with no
permutation, weights applied at dispatch or inside the first GEMM, and the
three tile modes (CTA pairs, pairs and single CTAs, single CTAs).  Every
token is compared with the oracle within the stated tolerance.  The list is
fixed by its seed; a few targeted cases make sure each path appears."""
import numpy as np
import pytest

from token_dispatch_grouped_fp32_gb300 import synth
from tests.gpu_util import check_layer, load_moe

pytestmark = pytest.mark.gpu


def _cases(n=64, seed=2024):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        dtype = "bf16" if g.random() < 0.75 else "f32"
        d = int(g.choice([64, 128, 192, 200, 256, 320, 448]))
        f = int(g.choice([64, 96, 128, 200, 256, 384]))
        E = int(g.choice([1, 2, 3, 8, 16, 33, 64]))
        k = int(g.integers(1, min(E, 8) + 1))
        T = int(g.choice([1, 7, 64, 200, 513, 1024, 2048, 4096]))
        renorm = bool(g.random() < 0.6)
        scale = bool(g.random() < 0.3)
        out.append((f"r{i}", T, d, E, k, f, dtype, renorm, scale))
    out += [  # targeted: each path at least once
        ("pairs_gather", 2048, 128, 2, 1, 128, "bf16", True, False),   # P/E = 1024
        ("pairs_gather_scaled", 2048, 128, 2, 1, 128, "bf16", True, True),
        ("pairs_copy_d200", 2048, 200, 2, 1, 128, "bf16", True, False),  # d % 64 != 0
        ("hybrid_gather", 1024, 192, 8, 2, 96, "bf16", False, False),   # P/E = 256
        ("dense_scaled", 300, 128, 4, 4, 128, "bf16", False, True),     # k = E, weights in G1
        ("dense_f32_scaled", 100, 64, 3, 3, 64, "f32", False, True),    # k = E, fp32 copies
    ]
    return out


CASES = _cases()


@pytest.fixture(scope="module")
def moe():
    return load_moe()


@pytest.mark.parametrize("name,T,d,E,k,f,dtype,renorm,scale", CASES, ids=[c[0] for c in CASES])
def test_random_shape_layer(moe, oracle, name, T, d, E, k, f, dtype, renorm, scale):
    w = synth.Workload("sweep_" + name, T, d, E, k, f, dtype, 800 + T + d + E + f,
                       renorm=renorm, scale_inputs=scale)
    assert check_layer(moe, oracle, w, device="cpu") >= max(1, int(0.9 * T))
