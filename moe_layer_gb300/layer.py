"""Thin convenience layer over the C ABI: allocates the caller-owned buffers
with torch and forwards the calls.  No arithmetic happens here."""
from __future__ import annotations

import torch

from . import _abi


class MoEBuffers:
    """Workspace, saved-state and output buffers for one configuration."""

    def __init__(self, cfg: _abi.MoeConfig, device="cuda", training: bool = True):
        self.cfg = cfg
        f, s, b = _abi.moe_workspace_size(cfg)
        dev = torch.device(device)
        self.fwd_ws = torch.zeros(max(f, 256), dtype=torch.uint8, device=dev)
        self.saved = torch.zeros(max(s, 256), dtype=torch.uint8, device=dev) if training else None
        self.bwd_ws = torch.zeros(max(b, 256), dtype=torch.uint8, device=dev) if training else None


def weights_from(inp: dict) -> _abi.MoeWeights:
    return _abi.make_weights(inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"],
                             inp.get("router_bias"), inp.get("Ws_gate"), inp.get("Ws_up"),
                             inp.get("Ws_down"), inp.get("mxfp8"))


def quantize_weights(cfg, inp: dict, stream=None):
    """MXFP8 mode: allocates the pre-quantized weight buffer, fills it from the
    bf16 expert weights and stores it as inp["mxfp8"] (redo after a weight
    update)."""
    if cfg.precision != _abi.MOE_MXFP8:
        raise ValueError("quantize_weights needs an MXFP8 configuration")
    n = _abi.moe_mxfp8_weights_size(cfg)
    mx = inp.get("mxfp8")
    if mx is None or mx.numel() < n:
        mx = torch.empty(n, dtype=torch.uint8, device=inp["W_gate"].device)
    _abi.moe_quantize_weights_mxfp8(cfg, weights_from(inp), mx, stream)
    inp["mxfp8"] = mx
    return mx


def alloc_grads(cfg: _abi.MoeConfig, device="cuda", with_topk: bool = True) -> dict:
    dev = torch.device(device)
    T, d, I, E, k = cfg.T, cfg.d, cfg.I, cfg.E, cfg.top_k
    wdt = torch.float32 if cfg.flags & _abi.MOE_FLAG_WGRAD_FP32 else torch.bfloat16
    g = {
        "dW_router": torch.empty(E, d, dtype=torch.float32, device=dev),
        "dW_gate": torch.empty(E, I, d, dtype=wdt, device=dev),
        "dW_up": torch.empty(E, I, d, dtype=wdt, device=dev),
        "dW_down": torch.empty(E, d, I, dtype=wdt, device=dev),
        "d_topk_w": torch.empty(T, k, dtype=torch.float32, device=dev) if with_topk else None,
    }
    if cfg.n_shared:
        Is = cfg.I_shared
        g["dWs_gate"] = torch.empty(Is, d, dtype=wdt, device=dev)
        g["dWs_up"] = torch.empty(Is, d, dtype=wdt, device=dev)
        g["dWs_down"] = torch.empty(d, Is, dtype=wdt, device=dev)
    else:
        g["dWs_gate"] = g["dWs_up"] = g["dWs_down"] = None
    return g


def grads_struct(g: dict) -> _abi.MoeGrads:
    return _abi.make_grads(g["dW_router"], g["dW_gate"], g["dW_up"], g["dW_down"], g["dWs_gate"],
                           g["dWs_up"], g["dWs_down"], g["d_topk_w"], g.get("dx_ready"))


def forward(cfg, inp: dict, bufs: MoEBuffers, y=None, stream=None):
    if y is None:
        y = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device=inp["x"].device)
    _abi.moe_forward(cfg, inp["x"], weights_from(inp), y, bufs.saved, bufs.fwd_ws, stream)
    return y


def backward(cfg, inp: dict, dy, bufs: MoEBuffers, grads: dict, dx=None, stream=None):
    if dx is None:
        dx = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device=dy.device)
    _abi.moe_backward(cfg, inp["x"], weights_from(inp), dy, bufs.saved, dx, grads_struct(grads),
                      bufs.bwd_ws, stream)
    return dx


class MoEFunction(torch.autograd.Function):
    """torch.autograd wrapper: y = MoE(x) with moe_forward, and in the backward
    dx and every weight gradient from one moe_backward call.  Argument
    marshalling only.  `bufs` holds this call's saved state, so each layer (and
    each call whose backward is still pending) needs its own MoEBuffers.
    Gradients come back in the parameters' dtypes (dW_router is computed in
    fp32).  MXFP8 mode: pass the pre-quantized weight buffer as `mxfp8`.

        y = MoEFunction.apply(cfg, bufs, x, W_router, W_gate, W_up, W_down,
                              Ws_gate, Ws_up, Ws_down, router_bias, mxfp8)
    """

    _NAMES = ("x", "W_router", "W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down", "router_bias", "mxfp8")

    @staticmethod
    def forward(ctx, cfg, bufs, x, W_router, W_gate, W_up, W_down, Ws_gate=None, Ws_up=None, Ws_down=None,
                router_bias=None, mxfp8=None):
        x = x.contiguous()
        inp = dict(zip(MoEFunction._NAMES, (x, W_router, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down,
                                            router_bias, mxfp8)))
        y = forward(cfg, inp, bufs)
        ctx.save_for_backward(x, W_router, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, router_bias, mxfp8)
        ctx.cfg, ctx.bufs = cfg, bufs
        return y

    @staticmethod
    def backward(ctx, dy):
        cfg, bufs = ctx.cfg, ctx.bufs
        inp = dict(zip(MoEFunction._NAMES, ctx.saved_tensors))
        g = alloc_grads(cfg, device=dy.device, with_topk=False)
        dx = backward(cfg, inp, dy.contiguous(), bufs, g)
        return (None, None, dx, g["dW_router"], g["dW_gate"], g["dW_up"], g["dW_down"], g["dWs_gate"],
                g["dWs_up"], g["dWs_down"], None, None)
