"""ctypes binding of libmoe's C ABI (include/moe.h).

Argument marshalling only: torch tensors are turned into device pointers and
the current CUDA stream into a cudaStream_t; every step of the layer runs in
the library's CUDA kernels.  Importing works without a GPU; calling the
compute entry points needs the built library and a CUDA device, and raises
when either is missing.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_BF16 = 0
MOE_MXFP8 = 1
# moe_config.flags bits (include/moe.h)
MOE_FLAG_REPLAY = 1
MOE_FLAG_WGRAD_FP32 = 2

EXPORTED = ["moe_workspace_size", "moe_mxfp8_weights_size", "moe_quantize_weights_mxfp8",
            "moe_route_topk", "moe_route_topk_noalloc", "moe_forward",
            "moe_backward", "moe_read_device_status", "moe_profile_enable", "moe_profile_report",
            "moe_status_string"]


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int64), ("I", ctypes.c_int64),
                ("E", ctypes.c_int64), ("top_k", ctypes.c_int64), ("n_shared", ctypes.c_int64),
                ("I_shared", ctypes.c_int64), ("precision", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class MoeWeights(ctypes.Structure):
    _fields_ = [("W_router", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("W_gate", ctypes.c_void_p), ("W_up", ctypes.c_void_p), ("W_down", ctypes.c_void_p),
                ("Ws_gate", ctypes.c_void_p), ("Ws_up", ctypes.c_void_p), ("Ws_down", ctypes.c_void_p),
                ("mxfp8", ctypes.c_void_p)]


class MoeGrads(ctypes.Structure):
    _fields_ = [("dW_router", ctypes.c_void_p), ("dW_gate", ctypes.c_void_p), ("dW_up", ctypes.c_void_p),
                ("dW_down", ctypes.c_void_p), ("dWs_gate", ctypes.c_void_p), ("dWs_up", ctypes.c_void_p),
                ("dWs_down", ctypes.c_void_p), ("d_topk_w", ctypes.c_void_p), ("dx_ready", ctypes.c_void_p)]


class MoeError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


_lib = None


def load():
    """Loads libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with moe_layer_gb300.build_ext.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    cfgp = ctypes.POINTER(MoeConfig)
    sz = ctypes.POINTER(ctypes.c_size_t)
    lib.moe_workspace_size.argtypes = [cfgp, sz, sz, sz]
    lib.moe_mxfp8_weights_size.argtypes = [cfgp, sz]
    lib.moe_quantize_weights_mxfp8.argtypes = [cfgp, ctypes.POINTER(MoeWeights), P, P]
    lib.moe_route_topk.argtypes = [cfgp] + [P] * 13
    lib.moe_route_topk_noalloc.argtypes = [cfgp] + [P] * 12
    lib.moe_forward.argtypes = [cfgp, P, ctypes.POINTER(MoeWeights), P, P, P, P]
    lib.moe_backward.argtypes = [cfgp, P, ctypes.POINTER(MoeWeights), P, P, P,
                                 ctypes.POINTER(MoeGrads), P, P]
    lib.moe_read_device_status.argtypes = [P, P]
    lib.moe_profile_enable.argtypes = [ctypes.c_int]
    lib.moe_profile_report.argtypes = [ctypes.c_char_p, ctypes.c_size_t]
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_status_string.restype = ctypes.c_char_p
    for name in EXPORTED[:-1]:
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().moe_status_string(int(code)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code, where):
    if code != MOE_OK:
        raise MoeError(code, where)


def make_config(T, d, I, E, top_k, n_shared=0, I_shared=0, precision=MOE_BF16, flags=0):
    return MoeConfig(T, d, I, E, top_k, n_shared, I_shared if n_shared else 0, precision, flags)


def moe_workspace_size(cfg: MoeConfig):
    """Returns (fwd_ws_bytes, saved_bytes, bwd_ws_bytes)."""
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(a), ctypes.byref(b),
                                     ctypes.byref(c)), "moe_workspace_size")
    return a.value, b.value, c.value


def moe_mxfp8_weights_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t()
    _check(load().moe_mxfp8_weights_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_mxfp8_weights_size")
    return n.value


def moe_quantize_weights_mxfp8(cfg, weights: MoeWeights, mx, stream=None):
    _check(load().moe_quantize_weights_mxfp8(ctypes.byref(cfg), ctypes.byref(weights), _ptr(mx),
                                             _stream(stream)), "moe_quantize_weights_mxfp8")


def moe_route_topk(cfg, x, W_router, router_bias, logits_in, logits_out, topk_idx, topk_w,
                   counts, offsets, perm_token, route_row, ws, stream=None):
    _check(load().moe_route_topk(ctypes.byref(cfg), _ptr(x), _ptr(W_router), _ptr(router_bias),
                                 _ptr(logits_in), _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w),
                                 _ptr(counts), _ptr(offsets), _ptr(perm_token), _ptr(route_row),
                                 _ptr(ws), _stream(stream)), "moe_route_topk")


def moe_route_topk_noalloc(cfg, x, W_router, router_bias, logits_in, logits_out, topk_idx, topk_w,
                           counts, offsets, perm_token, route_row, stream=None):
    """moe_route_topk without a workspace: for callers that cannot allocate
    device memory (see include/moe.h)."""
    _check(load().moe_route_topk_noalloc(ctypes.byref(cfg), _ptr(x), _ptr(W_router), _ptr(router_bias),
                                         _ptr(logits_in), _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w),
                                         _ptr(counts), _ptr(offsets), _ptr(perm_token), _ptr(route_row),
                                         _stream(stream)), "moe_route_topk_noalloc")


def make_weights(W_router, W_gate, W_up, W_down, router_bias=None, Ws_gate=None, Ws_up=None,
                 Ws_down=None, mxfp8=None) -> MoeWeights:
    return MoeWeights(_ptr(W_router), _ptr(router_bias), _ptr(W_gate), _ptr(W_up), _ptr(W_down),
                      _ptr(Ws_gate), _ptr(Ws_up), _ptr(Ws_down), _ptr(mxfp8))


def make_grads(dW_router, dW_gate, dW_up, dW_down, dWs_gate=None, dWs_up=None, dWs_down=None,
               d_topk_w=None, dx_ready=None) -> MoeGrads:
    """dx_ready: optional torch.cuda.Event (recorded by moe_backward once dx is
    complete, before the weight gradients)."""
    ev = None
    if dx_ready is not None:
        ev = dx_ready.cuda_event if hasattr(dx_ready, "cuda_event") else int(dx_ready)
        if not ev:
            raise ValueError("dx_ready event has no CUDA event yet: record it once before passing it")
    return MoeGrads(_ptr(dW_router), _ptr(dW_gate), _ptr(dW_up), _ptr(dW_down), _ptr(dWs_gate),
                    _ptr(dWs_up), _ptr(dWs_down), _ptr(d_topk_w), ev)


def moe_forward(cfg, x, weights: MoeWeights, y, saved, ws, stream=None):
    _check(load().moe_forward(ctypes.byref(cfg), _ptr(x), ctypes.byref(weights), _ptr(y), _ptr(saved),
                              _ptr(ws), _stream(stream)), "moe_forward")


def moe_backward(cfg, x, weights: MoeWeights, dy, saved, dx, grads: MoeGrads, ws, stream=None):
    _check(load().moe_backward(ctypes.byref(cfg), _ptr(x), ctypes.byref(weights), _ptr(dy),
                               _ptr(saved), _ptr(dx), ctypes.byref(grads), _ptr(ws),
                               _stream(stream)), "moe_backward")


def moe_read_device_status(ws, stream=None) -> int:
    return int(load().moe_read_device_status(_ptr(ws), _stream(stream)))


def moe_profile_enable(enable: bool = True):
    _check(load().moe_profile_enable(1 if enable else 0), "moe_profile_enable")


def moe_profile_report() -> dict:
    """{step name: (calls, kernels, total_ms)} for the calls recorded since the last report."""
    buf = ctypes.create_string_buffer(1 << 16)
    _check(load().moe_profile_report(buf, len(buf)), "moe_profile_report")
    out = {}
    for line in buf.value.decode().splitlines():
        name, n, nk, ms = line.split()
        out[name] = (int(n), int(nk), float(ms))
    return out
