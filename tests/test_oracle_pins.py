"""Pins for the CPU oracle: each check comes from outside the oracle itself.

- hand-worked fixtures under tests/golden/ (routing and SwiGLU arithmetic);
- closed forms (two-expert softmax = sigmoid, all-equal logits);
- library routines for special cases (numpy lexsort top-k, stable argsort
  permutation, bincount/cumsum offsets, float64 matmuls for the dense SwiGLU
  MLP when E = 1, k = 1, scipy softmax for the dense soft mixture when k = E
  without renormalisation);
- brute force on tiny inputs (every expert evaluated densely per token).

A plausible slip in the oracle (swapped gate/up, transposed down projection,
wrong tie rule, dropped renormalisation, unstable permutation, wrong weight
index in the combine) fails at least one test here.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from token_dispatch_grouped_fp32_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np_silu(z):
    return z / (1.0 + np.exp(-z))


def _sort_topk(L, k):
    """Top-k by a library sort: key (-logit, expert id), ascending."""
    T, E = L.shape
    idx = np.empty((T, k), np.int32)
    ids = np.arange(E)
    for t in range(T):
        order = np.lexsort((ids, -L[t].astype(np.float64)))
        idx[t] = order[:k]
    return idx


def _np_expert(x, Wgu_e, Wd_e):
    f = Wd_e.shape[0]
    gu = x.astype(np.float64) @ Wgu_e.astype(np.float64)
    return (_np_silu(gu[..., :f]) * gu[..., f:]) @ Wd_e.astype(np.float64)


def test_routing_golden_cases(oracle):
    cases = json.load(open(os.path.join(GOLDEN, "routing_hand.json")))["cases"]
    for c in cases:
        L = np.array([c["logits"]], np.float32)
        idx, w = oracle.topk(L, c["k"], c["renorm"])
        assert idx[0].tolist() == c["idx"], c
        np.testing.assert_allclose(w[0], c["w"], rtol=1e-14, atol=0)


@pytest.mark.parametrize("renorm", [True, False])
def test_all_equal_logits_closed_form(oracle, renorm):
    T, E, k = 5, 16, 4
    L = synth.make_logits(T, E, 0, ties="all_equal").numpy()
    idx, w = oracle.topk(L, k, renorm)
    assert (idx == np.arange(k)[None, :]).all()
    np.testing.assert_allclose(w, (1.0 / k if renorm else 1.0 / E), rtol=1e-14)


def test_two_expert_sigmoid_closed_form(oracle):
    rng = np.random.default_rng(3)
    L = rng.normal(size=(200, 2)).astype(np.float32)
    idx, w = oracle.topk(L, 2, False)
    for t in range(200):
        a, b = float(L[t, 0]), float(L[t, 1])
        first = 0 if a >= b else 1
        assert idx[t].tolist() == [first, 1 - first]
        hi, lo = max(a, b), min(a, b)
        assert w[t, 0] == pytest.approx(1.0 / (1.0 + math.exp(lo - hi)), rel=1e-13)
        assert w[t, 1] == pytest.approx(1.0 / (1.0 + math.exp(hi - lo)), rel=1e-13)


def test_nan_ranks_last(oracle):
    L = np.array([[np.nan, 1.0, -np.inf, 0.0]], np.float32)
    idx, _ = oracle.topk(L, 4, False)
    assert idx[0].tolist() == [1, 3, 2, 0]


@pytest.mark.parametrize("ties", [None, "coarse"])
@pytest.mark.parametrize("E,k", [(8, 2), (64, 6), (128, 8), (3, 3)])
def test_topk_matches_library_sort_and_softmax(oracle, ties, E, k):
    T = 300
    L = synth.make_logits(T, E, 11 + E, ties=ties).numpy()
    idx, w = oracle.topk(L, k, True)
    np.testing.assert_array_equal(idx, _sort_topk(L, k))
    p = scipy.special.softmax(L.astype(np.float64), axis=1)
    sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-12)
    _, w0 = oracle.topk(L, k, False)
    np.testing.assert_allclose(w0, sel, rtol=1e-12)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (7, 4, 2), (100, 8, 2), (333, 64, 6), (50, 128, 8)])
def test_dispatch_matches_stable_argsort(oracle, T, E, k):
    L = synth.make_logits(T, E, 5 + T).numpy()
    idx, _ = oracle.topk(L, k, True)
    counts, offsets, pos, src = oracle.dispatch(idx, E)
    flat = idx.reshape(-1)
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    order = np.argsort(flat, kind="stable")  # pair ids in expert-contiguous order
    expect_pos = np.empty_like(order)
    expect_pos[order] = np.arange(order.size)
    np.testing.assert_array_equal(pos, expect_pos)
    np.testing.assert_array_equal(src, order // k)
    # invariants the method fixes
    assert counts.sum() == T * k
    for t in range(T):
        assert len(set(idx[t].tolist())) == k
    assert sorted(pos.tolist()) == list(range(T * k))  # bijection
    np.testing.assert_array_equal(src[pos], np.repeat(np.arange(T), k))  # inverse restores order
    for e in range(E):
        seg = src[offsets[e]:offsets[e + 1]]
        assert (np.diff(seg) > 0).all()  # ascending token id within an expert


def test_swiglu_golden(oracle):
    g = json.load(open(os.path.join(GOLDEN, "swiglu_hand.json")))
    h, y = oracle.expert_ffn_row(np.array(g["x"]), np.array(g["Wgu"]), np.array(g["Wd"]))
    np.testing.assert_allclose(h, g["h"], rtol=1e-15, atol=0)
    np.testing.assert_allclose(y, g["y"], rtol=1e-15, atol=0)


def test_logits_match_float64_matmul(oracle):
    w = synth.WORKLOADS["tiny_fp32"]
    inp = synth.make_inputs(w, weights=False)
    bias = torch.linspace(-1, 2, w.E)
    x, Wr = inp["x"].numpy(), inp["Wr"].numpy()
    L = oracle.router_logits(x, Wr, bias.numpy())
    ref = (x.astype(np.float64) @ Wr.astype(np.float64).T + bias.numpy().astype(np.float64))
    ulp = np.spacing(np.abs(ref).astype(np.float32))
    assert (np.abs(L.astype(np.float64) - ref) <= ulp).all()


def test_dense_mlp_when_one_expert(oracle):
    """E = 1, k = 1: the layer is a plain SwiGLU MLP with weight 1."""
    w = synth.Workload("e1", 37, 24, 1, 1, 40, "f32", 7)
    inp = synth.make_inputs(w)
    x, Wr, Wgu, Wd = (inp[n].numpy() for n in ("x", "Wr", "Wgu", "Wd"))
    r = oracle.moe_forward(x, Wr, Wgu, Wd, 1, renorm=False)
    assert (r["idx"] == 0).all() and np.all(r["w"] == 1.0)
    ref = _np_expert(x, Wgu[0], Wd[0])
    np.testing.assert_allclose(r["out"], ref, rtol=1e-12, atol=1e-12)


def test_soft_mixture_when_k_equals_E(oracle):
    """k = E without renormalisation: sum_e softmax(L)_e * FFN_e(x)."""
    w = synth.Workload("mix", 19, 32, 6, 6, 16, "f32", 8)
    inp = synth.make_inputs(w)
    x, Wr, Wgu, Wd = (inp[n].numpy() for n in ("x", "Wr", "Wgu", "Wd"))
    r = oracle.moe_forward(x, Wr, Wgu, Wd, w.E, renorm=False)
    L = (x.astype(np.float64) @ Wr.astype(np.float64).T).astype(np.float32)
    p = scipy.special.softmax(L.astype(np.float64), axis=1)
    ref = sum(p[:, e:e + 1] * _np_expert(x, Wgu[e], Wd[e]) for e in range(w.E))
    np.testing.assert_allclose(r["out"], ref, rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("bias", [False, True])
def test_brute_force_tiny_layer(oracle, bias):
    """Every expert evaluated densely for every token, then selected."""
    w = synth.WORKLOADS["tiny_fp32"].with_(zipf=bias)
    inp = synth.make_inputs(w)
    x, Wr, Wgu, Wd = (inp[n].numpy() for n in ("x", "Wr", "Wgu", "Wd"))
    b = inp["bias"].numpy() if bias else None
    r = oracle.moe_forward(x, Wr, Wgu, Wd, w.k, renorm=True, bias=b)
    L = x.astype(np.float64) @ Wr.astype(np.float64).T
    if bias:
        L = L + b.astype(np.float64)
    L = L.astype(np.float32)
    idx = _sort_topk(L, w.k)
    np.testing.assert_array_equal(r["idx"], idx)
    p = scipy.special.softmax(L.astype(np.float64), axis=1)
    sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    wt = sel / sel.sum(1, keepdims=True)
    dense = np.stack([_np_expert(x, Wgu[e], Wd[e]) for e in range(w.E)], 1)  # [T, E, d]
    ref = np.einsum("tk,tkd->td", wt, np.take_along_axis(dense, idx[:, :, None].astype(np.int64), 1))
    np.testing.assert_allclose(r["out"], ref, rtol=1e-10, atol=1e-12)


def test_token_outputs_equal_forward_rows(oracle):
    w = synth.WORKLOADS["tiny_fp32"]
    inp = synth.make_inputs(w)
    x, Wr, Wgu, Wd = (inp[n].numpy() for n in ("x", "Wr", "Wgu", "Wd"))
    r = oracle.moe_forward(x, Wr, Wgu, Wd, w.k)
    toks = np.array([0, 5, 63, 17])
    out = oracle.token_outputs(toks, x, Wgu, Wd, r["idx"], r["w"])
    np.testing.assert_array_equal(out, r["out"][toks])


def test_empty_batch(oracle):
    w = synth.WORKLOADS["tiny_fp32"].with_tokens(0)
    inp = synth.make_inputs(w)
    x, Wr, Wgu, Wd = (inp[n].numpy() for n in ("x", "Wr", "Wgu", "Wd"))
    r = oracle.moe_forward(x, Wr, Wgu, Wd, w.k)
    assert r["out"].shape == (0, w.d)
    assert (r["counts"] == 0).all() and (r["offsets"] == 0).all()


@pytest.mark.parametrize("E,k,renorm", [(6, 2, True), (6, 6, False), (4, 1, True)])
def test_input_scaled_equals_dense_no_dispatch(oracle, E, k, renorm):
    """Routing weights on the expert inputs: the layer equals the form with
    nothing to dispatch, in which every expert receives every token already
    scaled by its router score (0 for experts the token did not pick, and
    SwiGLU(0) = 0 without biases).  Computed here densely with matmuls."""
    w = synth.Workload("in", 23, 40, E, k, 24, "f32", 31)
    inp = synth.make_inputs(w)
    x, Wr, Wgu, Wd = (inp[n].numpy() for n in ("x", "Wr", "Wgu", "Wd"))
    r = oracle.moe_forward(x, Wr, Wgu, Wd, k, renorm=renorm, scale_inputs=True)
    s = np.zeros((w.T, E))
    np.put_along_axis(s, r["idx"].astype(np.int64), r["w"], axis=1)
    dense = sum(_np_expert(s[:, e:e + 1] * x.astype(np.float64), Wgu[e], Wd[e]) for e in range(E))
    np.testing.assert_allclose(r["out"], dense, rtol=1e-9, atol=1e-12)
    # and the weights really do act on the inputs: unless every weight is 1
    # (k = 1 renormalised), the output-weighted layer differs
    r_out = oracle.moe_forward(x, Wr, Wgu, Wd, k, renorm=renorm, scale_inputs=False)
    if np.all(r["w"] == 1.0):
        np.testing.assert_array_equal(r_out["out"], r["out"])
    else:
        assert np.abs(r_out["out"] - r["out"]).max() > 1e-3


def test_input_scaled_single_expert_is_plain_mlp(oracle):
    w = synth.Workload("in1", 17, 32, 1, 1, 16, "f32", 32)
    inp = synth.make_inputs(w)
    x, Wr, Wgu, Wd = (inp[n].numpy() for n in ("x", "Wr", "Wgu", "Wd"))
    a = oracle.moe_forward(x, Wr, Wgu, Wd, 1, scale_inputs=True)["out"]
    b = oracle.moe_forward(x, Wr, Wgu, Wd, 1, scale_inputs=False)["out"]
    np.testing.assert_array_equal(a, b)
    toks = np.array([0, 3, 16])
    c = oracle.token_outputs(toks, x, Wgu, Wd, np.zeros((17, 1), np.int32), np.ones((17, 1)),
                             scale_inputs=True)
    np.testing.assert_array_equal(c, a[toks])


@pytest.mark.parametrize("scale_inputs", [False, True])
def test_combine_one_hot_rows(oracle, scale_inputs):
    """Combine on one-hot expert rows: row r of y_perm is the unit vector of
    column r, so out[t] holds w[t, j] exactly at column pos[t*k + j] (1 when
    the weights scaled the inputs) and 0 elsewhere -- no rounding anywhere, so
    the comparison is exact.  Distinct random weights per slot catch a weight
    taken from the wrong slot."""
    T, E, k = 40, 8, 3
    L = synth.make_logits(T, E, 71).numpy()
    idx, w = oracle.topk(L, k, True)
    _, _, pos, _ = oracle.dispatch(idx, E)
    P = T * k
    y_perm = np.eye(P)
    out = oracle.combine(y_perm, pos, w, k, scale_inputs=scale_inputs)
    expect = np.zeros((T, P))
    for t in range(T):
        for j in range(k):
            expect[t, pos[t * k + j]] = 1.0 if scale_inputs else w[t, j]
    np.testing.assert_array_equal(out, expect)


def test_combine_matches_einsum_on_random_rows(oracle):
    """Random expert rows: the combine equals a float64 gather-and-weigh with
    numpy (a library routine), to rounding."""
    T, E, k, d = 57, 16, 4, 24
    L = synth.make_logits(T, E, 72).numpy()
    idx, w = oracle.topk(L, k, False)
    _, _, pos, _ = oracle.dispatch(idx, E)
    y_perm = np.random.default_rng(4).normal(size=(T * k, d))
    out = oracle.combine(y_perm, pos, w, k)
    ref = np.einsum("tk,tkd->td", w, y_perm[pos.reshape(T, k)])
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-15)


def test_expert_ffn_rows_equal_single_rows(oracle):
    """The batched expert FFN is the single-row FFN on every row (bit-equal),
    each row through its own expert of the block."""
    rng = np.random.default_rng(5)
    ne, d, f, n = 3, 24, 16, 11
    x = rng.normal(size=(n, d)).astype(np.float32)
    Wgu = (rng.normal(size=(ne, d, 2 * f)) / np.sqrt(d)).astype(np.float32)
    Wd = (rng.normal(size=(ne, f, d)) / np.sqrt(f)).astype(np.float32)
    expert = rng.integers(0, ne, size=n).astype(np.int32)
    h, y = oracle.expert_ffn_rows(x, expert, Wgu, Wd)
    for r in range(n):
        h1, y1 = oracle.expert_ffn_row(x[r], Wgu[expert[r]], Wd[expert[r]])
        np.testing.assert_array_equal(h[r], h1)
        np.testing.assert_array_equal(y[r], y1)
    # and against the library form of the FFN
    for r in range(n):
        np.testing.assert_allclose(y[r], _np_expert(x[r], Wgu[expert[r]], Wd[expert[r]]),
                                   rtol=1e-12, atol=1e-13)
