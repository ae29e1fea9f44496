"""Python binding of libmoe (include/moe.h): argument marshalling only.

Every function below has the name of the C entry point it calls and takes
torch tensors (or None for a NULL pointer, or an int address) in the C
argument order.  All arithmetic runs in libmoe's CUDA kernels; if the library
is missing this module raises at import time instead of falling back to
anything else.

``MoELayer`` is a small convenience holder: it keeps the weights and one
workspace per stream (allocated with torch) and calls ``moe_forward``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_CUDA = -4
MOE_ERR_DEVICE_TIMEOUT = -5
MOE_ERR_BAD_ROUTING = -6
MOE_F32 = 0
MOE_BF16 = 1


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: {_status_name(status)} ({detail})")
        self.status = status


class moe_config_t(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("f", ctypes.c_int32), ("act_dtype", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("scale_inputs", ctypes.c_int32)]


# moe_workspace_layout: offset of a region moe_forward does not use
MOE_WS_ABSENT = (1 << (8 * ctypes.sizeof(ctypes.c_size_t))) - 1


class moe_workspace_layout_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("logits", "topk_idx", "topk_w", "counts", "offsets",
                                               "pos", "src_token", "x_perm", "h_perm", "y_perm",
                                               "total")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run token_dispatch_grouped_fp32_gb300.build.build() "
            "(nvcc, sm_103a). There is no fallback path.")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    cfgp = ctypes.POINTER(moe_config_t)
    sig = {
        "moe_status_string": ([st], ctypes.c_char_p),
        "moe_last_error_message": ([], ctypes.c_char_p),
        "moe_workspace_size": ([cfgp], sz),
        "moe_dispatch_workspace_size": ([cfgp], sz),
        "moe_forward_kernel_launches": ([cfgp], st),
        "moe_route": ([cfgp, vp, vp, vp, vp, vp, vp, vp, sz, vp], st),
        "moe_route_workspace_size": ([cfgp], sz),
        "moe_route_from_logits": ([cfgp, vp, vp, vp, vp], st),
        "moe_dispatch": ([cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], st),
        "moe_grouped_swiglu": ([cfgp, vp, vp, vp, vp, vp, vp, vp], st),
        "moe_combine": ([cfgp, vp, vp, vp, vp, vp], st),
        "moe_forward": ([cfgp, vp, vp, vp, vp, vp, vp, vp, sz, vp], st),
        "moe_forward_host": ([cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], st),
        "moe_last_device_error": ([vp], st),
        "moe_set_wait_limit_ns": ([ctypes.c_uint64], None),
        "moe_wait_limit_ns": ([], ctypes.c_uint64),
        "moe_workspace_layout": ([cfgp, ctypes.POINTER(moe_workspace_layout_t)], st),
        "moe_debug_inject_wait_timeout": ([ctypes.c_int], None),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def _status_name(status: int) -> str:
    return _lib.moe_status_string(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"expected a torch.Tensor, an int address or None, got {type(t)}")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libmoe must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(status: int, where: str, raise_on_error: bool):
    if status != MOE_OK and raise_on_error:
        raise MoEError(status, where, _lib.moe_last_error_message().decode())
    return status


def config(T: int, d: int, E: int, k: int, f: int, dtype=torch.bfloat16,
           renormalize: bool = True, scale_inputs: bool = False) -> moe_config_t:
    if dtype in (torch.bfloat16, "bf16", MOE_BF16):
        act = MOE_BF16
    elif dtype in (torch.float32, "f32", MOE_F32):
        act = MOE_F32
    else:
        act = int(dtype)
    return moe_config_t(int(T), int(d), int(E), int(k), int(f), act, int(bool(renormalize)),
                        int(bool(scale_inputs)))


def moe_status_string(status: int) -> str:
    return _status_name(status)


def moe_last_error_message() -> str:
    return _lib.moe_last_error_message().decode()


def moe_workspace_size(cfg: moe_config_t) -> int:
    return int(_lib.moe_workspace_size(ctypes.byref(cfg)))


def moe_dispatch_workspace_size(cfg: moe_config_t) -> int:
    return int(_lib.moe_dispatch_workspace_size(ctypes.byref(cfg)))


def moe_forward_kernel_launches(cfg: moe_config_t) -> int:
    return int(_lib.moe_forward_kernel_launches(ctypes.byref(cfg)))


def moe_set_wait_limit_ns(ns: int) -> None:
    _lib.moe_set_wait_limit_ns(int(ns))


def moe_wait_limit_ns() -> int:
    return int(_lib.moe_wait_limit_ns())


def moe_workspace_layout(cfg: moe_config_t, raise_on_error=True) -> moe_workspace_layout_t:
    layout = moe_workspace_layout_t()
    _check(_lib.moe_workspace_layout(ctypes.byref(cfg), ctypes.byref(layout)),
           "moe_workspace_layout", raise_on_error)
    return layout


def moe_debug_inject_wait_timeout(enable: bool) -> None:
    _lib.moe_debug_inject_wait_timeout(int(bool(enable)))


def moe_route_workspace_size(cfg: moe_config_t) -> int:
    return int(_lib.moe_route_workspace_size(ctypes.byref(cfg)))


def moe_route(cfg, x, Wr, logit_bias, logits, topk_idx, topk_w, ws=None, ws_bytes=None,
              stream=None, raise_on_error=True):
    if ws_bytes is None:
        ws_bytes = 0 if ws is None or isinstance(ws, int) else ws.numel() * ws.element_size()
    s = _lib.moe_route(ctypes.byref(cfg), _ptr(x), _ptr(Wr), _ptr(logit_bias), _ptr(logits),
                       _ptr(topk_idx), _ptr(topk_w), _ptr(ws), int(ws_bytes), _stream(stream))
    return _check(s, "moe_route", raise_on_error)


def moe_route_from_logits(cfg, logits, topk_idx, topk_w, stream=None, raise_on_error=True):
    s = _lib.moe_route_from_logits(ctypes.byref(cfg), _ptr(logits), _ptr(topk_idx), _ptr(topk_w),
                                   _stream(stream))
    return _check(s, "moe_route_from_logits", raise_on_error)


def moe_dispatch(cfg, topk_idx, topk_w, x, counts, offsets, pos, src_token, x_perm, ws,
                 ws_bytes=None, stream=None, raise_on_error=True):
    if ws_bytes is None:
        ws_bytes = 0 if ws is None or isinstance(ws, int) else ws.numel() * ws.element_size()
    s = _lib.moe_dispatch(ctypes.byref(cfg), _ptr(topk_idx), _ptr(topk_w), _ptr(x), _ptr(counts),
                          _ptr(offsets), _ptr(pos), _ptr(src_token), _ptr(x_perm), _ptr(ws),
                          int(ws_bytes), _stream(stream))
    return _check(s, "moe_dispatch", raise_on_error)


def moe_grouped_swiglu(cfg, x_perm, offsets, W_gate_up, W_down, h_perm, y_perm, stream=None,
                       raise_on_error=True):
    s = _lib.moe_grouped_swiglu(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(W_gate_up),
                                _ptr(W_down), _ptr(h_perm), _ptr(y_perm), _stream(stream))
    return _check(s, "moe_grouped_swiglu", raise_on_error)


def moe_combine(cfg, y_perm, pos, topk_w, out, stream=None, raise_on_error=True):
    s = _lib.moe_combine(ctypes.byref(cfg), _ptr(y_perm), _ptr(pos), _ptr(topk_w), _ptr(out),
                         _stream(stream))
    return _check(s, "moe_combine", raise_on_error)


def moe_forward(cfg, x, Wr, logit_bias, W_gate_up, W_down, out, ws, ws_bytes=None, stream=None,
                raise_on_error=True):
    if ws_bytes is None:
        ws_bytes = 0 if ws is None or isinstance(ws, int) else ws.numel() * ws.element_size()
    s = _lib.moe_forward(ctypes.byref(cfg), _ptr(x), _ptr(Wr), _ptr(logit_bias), _ptr(W_gate_up),
                         _ptr(W_down), _ptr(out), _ptr(ws), int(ws_bytes), _stream(stream))
    return _check(s, "moe_forward", raise_on_error)


def moe_forward_host(cfg, x_host, Wr, logit_bias, W_gate_up, W_down, out_host, x_dev, out_dev, ws,
                     ws_bytes=None, stream=None, raise_on_error=True):
    if ws_bytes is None:
        ws_bytes = 0 if ws is None or isinstance(ws, int) else ws.numel() * ws.element_size()
    s = _lib.moe_forward_host(ctypes.byref(cfg), _ptr(x_host), _ptr(Wr), _ptr(logit_bias),
                              _ptr(W_gate_up), _ptr(W_down), _ptr(out_host), _ptr(x_dev),
                              _ptr(out_dev), _ptr(ws), int(ws_bytes), _stream(stream))
    return _check(s, "moe_forward_host", raise_on_error)


def moe_last_device_error(stream=None, raise_on_error=True):
    s = _lib.moe_last_device_error(_stream(stream))
    return _check(s, "moe_last_device_error", raise_on_error)


class MoELayer:
    """Weights of one MoE layer plus reusable workspaces; ``forward`` runs
    ``moe_forward`` on the given (default: current) stream.  Weights: Wr [E, d]
    fp32, W_gate_up [E, d, 2f] and W_down [E, f, d] in the activation dtype,
    optional per-expert logit bias [E] fp32.

    The workspace holds a call's intermediates (logits, routing, permuted
    rows), so two calls in flight at once must not share one: the layer keeps
    a separate workspace for each stream it is called on."""

    def __init__(self, Wr, W_gate_up, W_down, k, logit_bias=None, renormalize=True,
                 scale_inputs=False):
        self.Wr, self.W_gate_up, self.W_down = Wr, W_gate_up, W_down
        self.logit_bias = logit_bias
        self.E, self.d = Wr.shape
        self.f = W_down.shape[1]
        self.k = int(k)
        self.dtype = W_gate_up.dtype
        self.renormalize = renormalize
        self.scale_inputs = scale_inputs
        self._ws = {}  # stream handle -> workspace

    def config(self, T: int) -> moe_config_t:
        return config(T, self.d, self.E, self.k, self.f, self.dtype, self.renormalize,
                      self.scale_inputs)

    def workspace(self, T: int, stream=None):
        """The workspace for calls on `stream` (default: the current stream),
        grown to moe_workspace_size for T tokens when needed."""
        key = _stream(stream).value or 0
        need = moe_workspace_size(self.config(T))
        ws = self._ws.get(key)
        if ws is None or ws.numel() < need:
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.Wr.device)
            self._ws[key] = ws
        return ws

    def forward(self, x, out=None, stream=None):
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        cfg = self.config(T)
        moe_forward(cfg, x, self.Wr, self.logit_bias, self.W_gate_up, self.W_down, out,
                    self.workspace(T, stream), stream=stream)
        return out

    __call__ = forward
