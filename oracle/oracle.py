"""CPU oracle for one MoE layer forward: numpy front end over ``moe_oracle.c``.

TEST INFRASTRUCTURE ONLY.  The test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  Nothing in the product
path imports this module; it imports nothing from the product package.

Every function takes numpy arrays holding the exact float values the GPU
reads (bf16 tensors are passed as their float32 images) and returns numpy
arrays.  The arithmetic lives in ``moe_oracle.c`` (double precision, plain
loops); see that file's header for the definitions and their sources.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_moe.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``moe_oracle.c`` into a shared library (gcc, OpenMP, IEEE math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    i64, i32 = ctypes.c_int64, ctypes.c_int32
    vp = ctypes.c_void_p
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_router_logits.argtypes = [i64, i32, i32, vp, vp, vp, vp]
    lib.oracle_topk.argtypes = [i64, i32, i32, i32, vp, vp, vp]
    lib.oracle_dispatch.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp]
    lib.oracle_expert_ffn_row.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp]
    lib.oracle_expert_ffn_rows.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp, vp]
    lib.oracle_combine.argtypes = [i64, i32, i32, vp, vp, vp, i32, vp]
    lib.oracle_token_outputs.argtypes = [i64, vp, i32, i32, i32, vp, vp, vp, vp, vp, i32, vp]
    lib.oracle_moe_forward.argtypes = [i64, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                       vp, vp, vp, vp, vp, vp, vp, vp]
    for fn in ("oracle_router_logits", "oracle_topk", "oracle_dispatch",
               "oracle_expert_ffn_row", "oracle_expert_ffn_rows", "oracle_combine",
               "oracle_token_outputs", "oracle_moe_forward"):
        getattr(lib, fn).restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def build_from_source(source: str, tag: str) -> str:
    """Compile a (test-modified) copy of the oracle source; returns the .so path.
    Used only by the mutation test, which plants mistakes in the oracle."""
    d = os.path.join(_BUILD_DIR, "variants")
    os.makedirs(d, exist_ok=True)
    src = os.path.join(d, f"{tag}.c")
    out = os.path.join(d, f"lib{tag}.so")
    with open(src, "w") as fh:
        fh.write(source)
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    "-fno-fast-math", src, "-o", out, "-lm"], check=True)
    return out


def source() -> str:
    with open(_SRC) as fh:
        return fh.read()


class Oracle:
    """The functions below, bound to a given oracle library (for the
    mutation test); the module-level functions use the built-in library."""

    def __init__(self, lib_path: str):
        self._lib = _bind(ctypes.CDLL(lib_path))

    def _use(self):
        return _Scoped(self._lib)


class _Scoped:
    def __init__(self, lib):
        self.lib = lib

    def __enter__(self):
        global _lib_override
        self.prev = _lib_override
        _lib_override = self.lib

    def __exit__(self, *exc):
        global _lib_override
        _lib_override = self.prev


_lib_override = None


def _L():
    return _lib_override if _lib_override is not None else _load()


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_L().oracle_num_threads())


def router_logits(x, Wr, bias=None):
    """fp32 logits [T, E] of x [T, d] against the router weight Wr [E, d]."""
    x, Wr = _f32(x), _f32(Wr)
    T, d = x.shape
    E = Wr.shape[0]
    b = None if bias is None else _f32(bias)
    out = np.empty((T, E), np.float32)
    _L().oracle_router_logits(T, d, E, _p(x), _p(Wr), _p(b), _p(out))
    return out


def topk(logits, k, renorm=True):
    """(idx [T, k] int32, w [T, k] float64) from a given fp32 logit buffer."""
    L = _f32(logits)
    T, E = L.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _L().oracle_topk(T, E, k, int(bool(renorm)), _p(L), _p(idx), _p(w))
    return idx, w


def dispatch(idx, E):
    """(counts [E], offsets [E+1], pos [T*k], src_token [T*k]) from idx [T, k]."""
    idx = _i32(idx)
    T, k = idx.shape
    P = T * k
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    pos = np.empty(P, np.int32)
    src = np.empty(P, np.int32)
    _L().oracle_dispatch(T, E, k, _p(idx), _p(counts), _p(offsets), _p(pos), _p(src))
    return counts, offsets, pos, src


def expert_ffn_row(xrow, Wgu_e, Wd_e):
    """One expert's SwiGLU FFN on one row: returns (h [f], y [d]) in float64."""
    xrow, Wgu_e, Wd_e = _f32(xrow), _f32(Wgu_e), _f32(Wd_e)
    d = xrow.shape[0]
    f = Wd_e.shape[0]
    gu = np.empty(2 * f, np.float64)
    h = np.empty(f, np.float64)
    y = np.empty(d, np.float64)
    _L().oracle_expert_ffn_row(d, f, _p(xrow), _p(Wgu_e), _p(Wd_e), _p(gu), _p(h), _p(y))
    return h, y


def expert_ffn_rows(x_rows, expert, Wgu, Wd):
    """The expert FFN on many rows at once: row r of x_rows [n, d] through
    expert expert[r] of the weight block Wgu [ne, d, 2f], Wd [ne, f, d].
    Returns (h [n, f], y [n, d]) in float64, each row exactly expert_ffn_row."""
    x_rows, Wgu, Wd, expert = _f32(x_rows), _f32(Wgu), _f32(Wd), _i32(expert)
    n, d = x_rows.shape
    f = Wd.shape[1]
    assert expert.shape == (n,) and (n == 0 or (expert.min() >= 0 and expert.max() < Wgu.shape[0]))
    h = np.empty((n, f), np.float64)
    y = np.empty((n, d), np.float64)
    _L().oracle_expert_ffn_rows(n, d, f, _p(x_rows), _p(expert), _p(Wgu), _p(Wd), _p(h), _p(y))
    return h, y


def combine(y_perm, pos, w, k, scale_inputs=False):
    """Combine [T, d] (float64) of the expert rows y_perm [P, d]: token t sums
    w[t, j] * y_perm[pos[t*k + j]] over its slots j in order (unweighted with
    scale_inputs)."""
    y_perm = np.ascontiguousarray(y_perm, dtype=np.float64)
    pos = _i32(pos).reshape(-1)
    P, d = y_perm.shape
    T = pos.shape[0] // k
    assert pos.shape[0] == T * k and (P == 0 or (pos.min() >= 0 and pos.max() < P))
    wd = np.ascontiguousarray(np.zeros((T, k)) if w is None else w, dtype=np.float64)
    out = np.empty((T, d), np.float64)
    _L().oracle_combine(T, k, d, _p(y_perm), _p(pos), _p(wd), int(bool(scale_inputs)), _p(out))
    return out


def token_outputs(tokens, x, Wgu, Wd, idx, w, scale_inputs=False):
    """Layer output rows [len(tokens), d] (float64) for the listed tokens.
    scale_inputs: the routing weights scale each expert's input instead of
    its output."""
    x, Wgu, Wd, idx = _f32(x), _f32(Wgu), _f32(Wd), _i32(idx)
    w = np.ascontiguousarray(w, dtype=np.float64)
    tokens = np.ascontiguousarray(tokens, dtype=np.int64)
    d = x.shape[1]
    k = idx.shape[1]
    f = Wd.shape[1]
    out = np.empty((tokens.shape[0], d), np.float64)
    _L().oracle_token_outputs(tokens.shape[0], _p(tokens), d, k, f, _p(x), _p(Wgu),
                              _p(Wd), _p(idx), _p(w), int(bool(scale_inputs)), _p(out))
    return out


def moe_forward(x, Wr, Wgu, Wd, k, renorm=True, bias=None, scale_inputs=False):
    """Whole layer.  Returns a dict with logits, idx, w, counts, offsets, pos,
    src_token and out (float64 [T, d]).  scale_inputs: the routing weights
    scale each expert's input instead of its output."""
    x, Wr, Wgu, Wd = _f32(x), _f32(Wr), _f32(Wgu), _f32(Wd)
    T, d = x.shape
    E = Wr.shape[0]
    f = Wd.shape[1]
    b = None if bias is None else _f32(bias)
    P = T * k
    r = {
        "logits": np.empty((T, E), np.float32),
        "idx": np.empty((T, k), np.int32),
        "w": np.empty((T, k), np.float64),
        "counts": np.empty(E, np.int32),
        "offsets": np.empty(E + 1, np.int32),
        "pos": np.empty(P, np.int32),
        "src_token": np.empty(P, np.int32),
        "out": np.empty((T, d), np.float64),
    }
    _L().oracle_moe_forward(T, d, E, k, f, int(bool(renorm)), int(bool(scale_inputs)), _p(x),
                            _p(Wr), _p(b),
                               _p(Wgu), _p(Wd), _p(r["logits"]), _p(r["idx"]), _p(r["w"]),
                               _p(r["counts"]), _p(r["offsets"]), _p(r["pos"]),
                               _p(r["src_token"]), _p(r["out"]))
    return r


def _method(fn):
    def m(self, *a, **k):
        with self._use():
            return fn(*a, **k)
    m.__name__ = fn.__name__
    m.__doc__ = fn.__doc__
    return m


for _fn in (num_threads, router_logits, topk, dispatch, expert_ffn_row, expert_ffn_rows, combine,
            token_outputs, moe_forward):
    setattr(Oracle, _fn.__name__, _method(_fn))
