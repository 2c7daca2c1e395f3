"""Shared helpers for the GPU parity tests: building the library, running the
layer through the C ABI, and running the oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O


def ensure_lib():
    from moe_layer_gb300 import _abi, build_ext
    build_ext.build()
    _abi.load()


def f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def rel_err(gpu, ref):
    """max |gpu - ref| / max |ref| (inputs: tensor or array)."""
    g = f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    return float(np.abs(g - r).max() / max(np.abs(r).max(), 1e-300))


class LazyExperts:
    """Indexable view of an [E, ...] bf16 tensor that upcasts one expert at a time."""

    def __init__(self, t):
        self.t = t
        self.cache = {}

    def __len__(self):
        return self.t.shape[0]

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = f64(self.t[e])
        return self.cache[e]


def oracle_forward(inp, k, logits=None, tokens=None, mxfp8=False):
    """Oracle forward on the CPU copies of the inputs (optionally a token subset)."""
    x = f64(inp["x"]) if tokens is None else f64(inp["x"][tokens])
    bias = None if inp.get("router_bias") is None else f64(inp["router_bias"])
    sh = inp.get("Ws_gate") is not None
    return O.moe_forward(x, f64(inp["W_router"]), LazyExperts(inp["W_gate"]), LazyExperts(inp["W_up"]),
                         LazyExperts(inp["W_down"]), k, router_bias=bias,
                         ws_gate=f64(inp["Ws_gate"]) if sh else None,
                         ws_up=f64(inp["Ws_up"]) if sh else None,
                         ws_down=f64(inp["Ws_down"]) if sh else None, logits=logits, mxfp8=mxfp8)


def oracle_backward(inp, fwd, tokens=None):
    x = f64(inp["x"]) if tokens is None else f64(inp["x"][tokens])
    dy = f64(inp["dy"]) if tokens is None else f64(inp["dy"][tokens])
    sh = inp.get("Ws_gate") is not None
    return O.moe_backward(x, f64(inp["W_router"]), LazyExperts(inp["W_gate"]), LazyExperts(inp["W_up"]),
                          LazyExperts(inp["W_down"]), dy, fwd,
                          ws_gate=f64(inp["Ws_gate"]) if sh else None,
                          ws_up=f64(inp["Ws_up"]) if sh else None,
                          ws_down=f64(inp["Ws_down"]) if sh else None)


def topk_gap(logits, k):
    """Gap between the k-th and (k+1)-th largest logit per token (inf if k == E)."""
    s = -np.sort(-np.asarray(logits, np.float64), axis=1)
    if s.shape[1] == k:
        return np.full(s.shape[0], np.inf)
    return s[:, k - 1] - s[:, k]


def order_gap(logits, k):
    """Smallest gap between consecutive values among the k+1 largest logits per
    token: below it, float error could swap two slots or the k-th choice."""
    s = -np.sort(-np.asarray(logits, np.float64), axis=1)
    kk = min(k + 1, s.shape[1])
    if kk < 2:
        return np.full(s.shape[0], np.inf)
    d = s[:, :kk - 1] - s[:, 1:kk]
    d = np.where(np.isfinite(d), d, np.inf)
    return d.min(axis=1)


def full_router_grad_err(inp, topk_idx, topk_w, d_topk_w, dW_router):
    """max|err| / max|ref| of the GPU's dW_router against the oracle's router
    backward run on the GPU's own routing (ids, weights) and router-weight
    gradient: the whole [E, d] gradient, at any size."""
    _, ref, _ = O.router_backward(np.asarray(topk_idx.cpu(), np.int64), f64(topk_w), f64(d_topk_w),
                                  f64(inp["x"]), f64(inp["W_router"]))
    return rel_err(dW_router, ref)


def shared_rows_err(inp, grads, cols):
    """The shared expert's weight gradients restricted to intermediate columns
    `cols` (rows of dWs_gate and dWs_up, columns of dWs_down), from the oracle's
    SwiGLU expert with weight 1 (R1) on every token: those rows and columns
    depend only on the same columns of the shared weights.  Returns the three
    max|err| / max|ref|."""
    c = torch.as_tensor(np.asarray(cols), device=inp["Ws_gate"].device)
    x, dy = f64(inp["x"]), f64(inp["dy"])
    wg, wu, wd = f64(inp["Ws_gate"][c]), f64(inp["Ws_up"][c]), f64(inp["Ws_down"][:, c])
    a, b, h, _ = O.expert_forward(x, wg, wu, wd)
    dWg, dWu, dWd, _, _ = O.expert_backward(x, dy, np.ones(x.shape[0]), a, b, h, wg, wu, wd)
    return (rel_err(grads["dWs_gate"][c], dWg), rel_err(grads["dWs_up"][c], dWu),
            rel_err(grads["dWs_down"][:, c], dWd))
