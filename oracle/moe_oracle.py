"""CPU oracle for the DeepSeek-V3-style MoE layer.  TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
legs may import or run this module.  The product path (moe_layer_gb300) never
touches it, and the two share no code.

It is the plain definition of the layer, written out in float64 numpy: every
input is upcast to float64, every intermediate stays float64.  Library
primitives (matrix products, a sort) are used as single steps; nothing is
fused, blocked or reordered beyond the definitions cited below.

Sources (titles and sections of the pages that define the method):
  [Blog]  Mixture-of-Kittens blog post (full text), section "Overlapping
          computation and communication in MoE": each token gets a router
          projection, the top-k routed experts with one router weight each; each
          selected expert runs up and gate projections, a SwiGLU activation and a
          down projection; the shared and routed expert outputs are summed with
          the router weights.  Section "Choosing the right communication
          direction / Scheduling" gives the two-pass counting schedule.  Section
          "Router weight gradient computation" gives the router-weight gradient
          as the inner product of the SwiGLU activation and the down-projection
          dgrad.  Section "Determinism" fixes the order of floating-point work.
  [Paper] "Mixture-of-Kittens: MoE Megakernel for NVL72s", section 2.1: outputs
          are summed using normalized router weights.

Readings taken where the pages are silent:
  R1  the shared expert enters the sum with weight 1;
  R2  router weights: softmax over all E logits, restricted to the k selected
      experts and renormalized (equal to a softmax over the selected logits);
  R3  SwiGLU(a, b) = SiLU(a) * b with a = gate projection, b = up projection,
      SiLU(z) = z * sigmoid(z);
  R4  top-k order: logits descending, ties broken towards the lower expert index;
  R5  the backward propagates through the router weights into the logits (and
      so into W_router and x); an optional router bias is a constant.

Parity pins: every function here is checked by tests/test_oracle_pins.py
against brute force, closed forms, library routines or finite differences;
the MXFP8 composition (which GEMM operand is quantized along which axis, the
token blocks of the weight gradients, the router and shared expert left in
full precision) by tests/test_oracle_mx_composition.py, with operands exactly
representable along one axis only, and planted mistakes that those pins catch.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "router_logits", "topk_route", "expert_schedule", "silu", "swiglu",
    "moe_forward", "moe_backward", "expert_forward", "expert_backward", "router_backward",
    "e4m3_decode", "e4m3_quantize", "mx_quantize", "mx_dequantize", "mx_round", "E4M3_TABLE",
    "bf16_round",
]


def _f64(a):
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------- routing
def router_logits(x, w_router, bias=None):
    """Router projection l[t, e] = sum_i x[t, i] * W_r[e, i] (+ bias[e]).  [Blog]"""
    logits = _f64(x) @ _f64(w_router).T
    if bias is not None:
        logits = logits + _f64(bias)[None, :]
    return logits


def topk_route(logits, k):
    """Top-k routed experts per token and their normalized router weights.

    Selection (R4): experts ordered by logit descending, equal logits by
    ascending expert index; the first k form the token's slots 0..k-1.
    Weights (R2): p = softmax over all E logits; g_j = p[e_j] / sum_i p[e_i].
    The comparisons are made on the values as given (float32 logits compare
    exactly as float32 because the upcast to float64 is exact).  [Blog], [Paper §2.1]
    """
    logits = _f64(logits)
    T, E = logits.shape
    # lexsort: the last key is the primary key
    tie = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((tie, -logits), axis=-1)
    idx = order[:, :k].copy()
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    p = p / p.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, idx, axis=1)
    w = sel / sel.sum(axis=1, keepdims=True)
    return idx.astype(np.int64), w


def expert_schedule(topk_idx, E):
    """Per-expert counts, offsets and the stable permutation of routes.

    The one-rank form of the pages' two-pass schedule [Blog, "Scheduling"]:
    pass 1 walks the routes (token ascending, slot ascending) and counts per
    expert; the region offsets are the exclusive prefix sum of the counts;
    pass 2 walks the routes in the same order and hands each one the next row
    of its expert's region.  Returns counts[E], offsets[E+1],
    perm_token[R] (row -> token), perm_slot[R] (row -> slot) and
    route_row[T, k] ((token, slot) -> row).
    """
    idx = np.asarray(topk_idx).tolist()
    T = len(idx)
    k = len(idx[0]) if T else 0
    counts = [0] * E
    for t in range(T):
        for j in range(k):
            counts[idx[t][j]] += 1
    offsets = [0] * (E + 1)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    cursor = offsets[:E]
    perm_token = [0] * (T * k)
    perm_slot = [0] * (T * k)
    route_row = [[0] * k for _ in range(T)]
    for t in range(T):
        for j in range(k):
            e = idx[t][j]
            r = cursor[e]
            cursor[e] = r + 1
            perm_token[r] = t
            perm_slot[r] = j
            route_row[t][j] = r
    return (np.array(counts, np.int64), np.array(offsets, np.int64),
            np.array(perm_token, np.int64), np.array(perm_slot, np.int64),
            np.array(route_row, np.int64).reshape(T, k))


# ---------------------------------------------------------------- expert FFN
def silu(z):
    """SiLU(z) = z * sigmoid(z)  (R3)."""
    z = _f64(z)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def dsilu(z):
    """d/dz SiLU(z) = sigmoid(z) * (1 + z * (1 - sigmoid(z)))."""
    z = _f64(z)
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def swiglu(a, b):
    """SwiGLU(a, b) = SiLU(a) * b  (R3).  [Blog]"""
    return silu(a) * _f64(b)


def expert_forward(x_rows, w_gate, w_up, w_down, mxfp8=False):
    """One SwiGLU expert FFN on a batch of rows: returns a, b, h, o with
    a = x W_gate^T, b = x W_up^T, h = SiLU(a) * b, o = h W_down^T.  [Blog]
    With mxfp8=True every operand of the two GEMMs goes through an MXFP8
    round trip along that GEMM's reduction axis first: x and W_gate/W_up along
    d, h and W_down along I [Blog, "MXFP8 support"]; the returned h is the
    unquantized one."""
    return _ffn(_f64(x_rows), w_gate, w_up, w_down, mxfp8)


def _ffn(x_rows, w_gate, w_up, w_down, mxfp8=False):
    """One SwiGLU expert on a batch of rows: returns a, b, h, o."""
    q = mx_round if mxfp8 else (lambda v, axis=-1: _f64(v))
    xq = q(x_rows, axis=-1)
    a = xq @ q(w_gate, axis=-1).T
    b = xq @ q(w_up, axis=-1).T
    h = swiglu(a, b)
    o = q(h, axis=-1) @ q(w_down, axis=-1).T
    return a, b, h, o


# ---------------------------------------------------------------- MXFP8
# The MX block format (MXFP8 with E4M3 elements and E8M0 shared scales) that
# the pages' MXFP8 mode uses [Blog, "MXFP8 support"; the MX format reference
# the pages cite].  Reading taken here:
#   * a block is 32 consecutive elements along the reduction axis of the GEMM
#     the operand feeds;
#   * shared scale X = 2^(floor(log2(amax)) - 8), 8 being the largest exponent
#     of E4M3; X is stored as the biased exponent E8M0 (bias 127); an all-zero
#     block gets the smallest scale code 0;
#   * each element is v / X rounded to the nearest E4M3 value (ties to even
#     mantissa), saturating at +-448.
E4M3_MAX = 448.0


def e4m3_decode(code):
    """Value of an E4M3 byte: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
    bits; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN (no inf)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_decode(c) for c in range(256)])


def e4m3_quantize(v):
    """Round float64 values to E4M3 codes: nearest value, ties to the even
    mantissa (even code), magnitudes beyond 448 saturate to 448.

    Written out from the format: the non-negative values of binade k
    (2^k <= a < 2^(k+1), k = -6..8) are 2^k (1 + j/8), j = 0..7, code
    8 (k + 7) + j; below 2^-6 the subnormals j 2^-9, code j.  So in every
    binade (the subnormals counted with k = -6) the values are the multiples
    m 2^(k-3) with m in [8, 16) (m in [0, 8) for the subnormals), code
    8 (k + 7) + m - 8, and the nearest one is the magnitude rounded to a
    multiple of 2^(k-3), ties to the even multiple (np.rint) -- the even code,
    as m and the code have the same parity.  m = 16 is 2^(k+1), the first value
    of the next binade, and the same formula gives its code."""
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    _, ex = np.frexp(a)                      # a = f 2^ex, f in [0.5, 1): binade k = ex - 1
    k = np.where(a < 2.0 ** -6, -6, ex.astype(np.int64) - 1)  # zero and subnormals: k = -6
    m = np.rint(np.ldexp(a, 3 - k))          # a / 2^(k-3), exact scaling by a power of two
    code = (8 * (k + 7) + m.astype(np.int64) - 8).astype(np.uint8)
    neg = (v < 0) & (code != 0)
    return np.where(neg, code | 0x80, code).astype(np.uint8)


def mx_quantize(v, axis=-1):
    """MXFP8 quantization of v along `axis` in blocks of 32 (the axis length
    must be a multiple of 32).  Returns (codes uint8, same shape as v; scale
    exponents uint8 (E8M0 codes) with that axis divided by 32)."""
    v = np.moveaxis(np.asarray(v, np.float64), axis, -1)
    shp = v.shape
    blk = v.reshape(shp[:-1] + (shp[-1] // 32, 32))
    amax = np.abs(blk).max(axis=-1)
    with np.errstate(divide="ignore"):
        e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 8, -127)
    e = np.minimum(np.maximum(e, -127), 127)
    scale = np.ldexp(1.0, e.astype(np.int64))
    codes = e4m3_quantize(blk / scale[..., None]).reshape(shp)
    return np.moveaxis(codes, -1, axis), np.moveaxis((e + 127).astype(np.uint8), -1, axis)


def mx_dequantize(codes, scale_codes, axis=-1):
    """Float64 values of MXFP8 codes with their E8M0 block scales."""
    c = np.moveaxis(np.asarray(codes), axis, -1)
    s = np.moveaxis(np.asarray(scale_codes), axis, -1).astype(np.int64) - 127
    vals = E4M3_TABLE[c.astype(np.int64)]
    return np.moveaxis(vals * np.ldexp(1.0, np.repeat(s, 32, axis=-1)), -1, axis)


def mx_round(v, axis=-1):
    """v after an MXFP8 round trip along `axis` (the value the GEMM sees)."""
    return mx_dequantize(*mx_quantize(v, axis), axis=axis)


def bf16_round(v):
    """v as a bfloat16 value (float64 result): rounded to float32 first, then to
    the nearest bfloat16 (8-bit significand), ties to the even significand --
    the value a float32 computation leaves after a bfloat16 store.  Used only
    where an MXFP8 quantization decision is taken on a stored bf16 tensor
    (reading R12: the saved a and b of the MXFP8 backward)."""
    f = np.ascontiguousarray(np.asarray(v, np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- forward
def moe_forward(x, w_router, w_gate, w_up, w_down, top_k, router_bias=None,
                ws_gate=None, ws_up=None, ws_down=None, logits=None, mxfp8=False):
    """The MoE layer forward, per token t:

        y_t = FFN_shared(x_t) + sum_j g_tj * FFN_{e_tj}(x_t)

    with FFN(v) = W_down (SiLU(W_gate v) * (W_up v)).  [Blog], [Paper §2.1]

    w_gate/w_up/w_down are indexable by expert (w_gate[e] is [I, d],
    w_down[e] is [d, I]).  `logits` may be given to route on precomputed
    values (e.g. float32 values for an exact comparison of the routing);
    otherwise they are computed in float64 from x and w_router.  mxfp8=True
    runs the routed experts' GEMMs on MXFP8 operands (expert_forward); the
    router and the shared expert stay in full precision [Blog, "MXFP8 support"].
    Returns a dict with y [T, d] and everything the backward needs.
    """
    x = _f64(x)
    T = x.shape[0]
    E = len(w_gate)
    if logits is None:
        logits = router_logits(x, w_router, router_bias)
    idx, w = topk_route(logits, top_k)
    counts, offsets, perm_token, perm_slot, route_row = expert_schedule(idx, E)
    d = x.shape[1]
    y = np.zeros((T, d))
    cache = {"a": {}, "b": {}, "h": {}, "o": {}}
    # routed experts, one expert's rows at a time
    for e in range(E):
        rows = np.arange(offsets[e], offsets[e + 1])
        if rows.size == 0:
            continue
        toks = perm_token[rows]
        a, b, h, o = _ffn(x[toks], w_gate[e], w_up[e], w_down[e], mxfp8)
        cache["a"][e], cache["b"][e], cache["h"][e], cache["o"][e] = a, b, h, o
        g = w[toks, perm_slot[rows]]
        np.add.at(y, toks, g[:, None] * o)
    shared = None
    if ws_gate is not None:
        a_s, b_s, h_s, o_s = _ffn(x, ws_gate, ws_up, ws_down)
        y += o_s  # R1: weight 1
        shared = {"a": a_s, "b": b_s, "h": h_s}
    return {
        "y": y, "logits": logits, "topk_idx": idx, "topk_w": w, "counts": counts,
        "offsets": offsets, "perm_token": perm_token, "perm_slot": perm_slot,
        "route_row": route_row, "cache": cache, "shared": shared, "mxfp8": mxfp8,
    }


# ---------------------------------------------------------------- backward
def _mx_rows(v):
    """MXFP8 round trip along the token axis (axis 0) in blocks of 32 rows, the
    rows padded with zeros to a multiple of 32 (the padding is dropped)."""
    v = _f64(v)
    n = v.shape[0]
    pad = (-n) % 32
    vp = np.concatenate([v, np.zeros((pad,) + v.shape[1:])], axis=0) if pad else v
    return mx_round(vp, axis=0)[:n]


def expert_backward(x_rows, dy_rows, g, a, b, h, w_gate_e, w_up_e, w_down_e, mxfp8=False):
    """Backward of one routed expert over its rows (tokens routed to it).

    x_rows, dy_rows [n, d]; g [n] router weights; a, b, h [n, I] from the
    forward.  Per row, with dh = W_down^T dy:
      dg = <h, dh>                                 [Blog, "Router weight gradient computation"]
      dW_down = sum dy (g h)^T;  da = g dh * b * SiLU'(a);  db = g dh * SiLU(a)
      dW_gate = sum da x^T;  dW_up = sum db x^T;  dx_row = W_gate^T da + W_up^T db
    Returns (dW_gate, dW_up, dW_down, dg [n], dx_rows [n, d]).
    With mxfp8=True every operand of the five GEMMs goes through an MXFP8 round
    trip along that GEMM's reduction axis: dy and W_down along d for dh;
    [da | db] and [W_gate; W_up] along 2I for dx; the token axis (blocks of 32
    rows of this expert, zero-padded) for the three weight gradients.  dg uses
    the unquantized h and dh [Blog, "MXFP8 support", "Router weight gradient
    computation"].  Each quantization decision is taken on the value the
    layer holds at that point (reading R12): a and b as saved in bf16 (h is
    recomputed from them); da, db and g*h unrounded, both for the dx operand
    and for the weight-gradient operands.
    """
    x_rows, dy_rows = _f64(x_rows), _f64(dy_rows)
    wg, wu, wd = _f64(w_gate_e), _f64(w_up_e), _f64(w_down_e)
    g = _f64(g)[:, None]
    if mxfp8:
        a, b = bf16_round(a), bf16_round(b)
        h = swiglu(a, b)
        dh = mx_round(dy_rows, axis=-1) @ mx_round(wd, axis=0)
    else:
        dh = dy_rows @ wd
    dg = np.sum(dh * h, axis=1)
    da = g * dh * _f64(b) * dsilu(a)
    db = g * dh * silu(a)
    hg = g * h
    if not mxfp8:
        return da.T @ x_rows, db.T @ x_rows, dy_rows.T @ hg, dg, da @ wg + db @ wu
    dadb = mx_round(np.concatenate([da, db], axis=1), axis=-1)
    wgu = mx_round(np.concatenate([wg, wu], axis=0), axis=0)
    xr = _mx_rows(x_rows)
    return (_mx_rows(da).T @ xr, _mx_rows(db).T @ xr, _mx_rows(dy_rows).T @ _mx_rows(hg), dg,
            dadb @ wgu)


def router_backward(topk_idx, topk_w, dg, x, w_router):
    """Backward of the router given dL/dg (R2, R5): g = softmax over the
    selected logits, so for a selected expert e of token t
      dl_te = g_te (dg_te - sum_i g_ti dg_ti), and 0 for the others;
    dW_router = dl^T x and the router's share of dx is dl W_router.
    Returns (dlogits [T, E], dW_router [E, d], dx_router [T, d])."""
    x, w, dg = _f64(x), _f64(topk_w), _f64(dg)
    w_router = _f64(w_router)
    s = np.sum(w * dg, axis=1, keepdims=True)
    dlogits = np.zeros((x.shape[0], w_router.shape[0]))
    np.put_along_axis(dlogits, np.asarray(topk_idx, np.int64), w * (dg - s), axis=1)
    return dlogits, dlogits.T @ x, dlogits @ w_router


def moe_backward(x, w_router, w_gate, w_up, w_down, dy, fwd,
                 ws_gate=None, ws_up=None, ws_down=None, dense_expert_grads=True):
    """Gradients of L = sum(dy * y) for the forward `fwd` (from moe_forward).

    Per route (t, j) with expert e and weight g, o = W_down h, h = SiLU(a)*b:
      dh      = W_down^T dy_t                       (down-projection dgrad)
      dg_tj   = <h, dh>                             [Blog, "Router weight gradient computation"]
      dW_down += dy_t (g h)^T
      da      = g dh * b * SiLU'(a);  db = g dh * SiLU(a)
      dW_gate += da x_t^T;  dW_up += db x_t^T;  dx_t += W_gate^T da + W_up^T db
    Router (R2, R5): g = softmax over the selected logits, so for selected e
      dl_te = g_te (dg_te - sum_i g_ti dg_ti), and 0 elsewhere;
      dW_router = dl^T x;  dx += dl W_router.
    Shared expert: the same SwiGLU backward with g = 1.
    Returns a dict of float64 arrays.  With dense_expert_grads=False the
    expert weight gradients are dicts {expert: array} holding only experts
    that received tokens (the others are zero), which keeps large layers in
    memory.
    """
    x = _f64(x)
    dy = _f64(dy)
    T, d = x.shape
    E = len(w_gate)
    idx, w = fwd["topk_idx"], fwd["topk_w"]
    k = idx.shape[1]
    offsets, perm_token, perm_slot = fwd["offsets"], fwd["perm_token"], fwd["perm_slot"]
    dx = np.zeros((T, d))
    dWg, dWu, dWd = {}, {}, {}
    dg = np.zeros((T, k))
    for e in range(E):
        rows = np.arange(offsets[e], offsets[e + 1])
        if rows.size == 0:
            continue
        toks, slots = perm_token[rows], perm_slot[rows]
        c = fwd["cache"]
        dWg[e], dWu[e], dWd[e], dg_e, dx_rows = expert_backward(
            x[toks], dy[toks], w[toks, slots], c["a"][e], c["b"][e], c["h"][e],
            w_gate[e], w_up[e], w_down[e], fwd.get("mxfp8", False))
        dg[toks, slots] = dg_e
        np.add.at(dx, toks, dx_rows)
    dlogits, dW_router, dx_router = router_backward(idx, w, dg, x, w_router)
    dx += dx_router
    if dense_expert_grads:
        I = np.shape(w_gate[0])[0]
        dense = {"dW_gate": np.zeros((E, I, d)), "dW_up": np.zeros((E, I, d)),
                 "dW_down": np.zeros((E, d, I))}
        for name, part in (("dW_gate", dWg), ("dW_up", dWu), ("dW_down", dWd)):
            for e, v in part.items():
                dense[name][e] = v
        dWg, dWu, dWd = dense["dW_gate"], dense["dW_up"], dense["dW_down"]
    out = {"dx": dx, "dW_gate": dWg, "dW_up": dWu, "dW_down": dWd, "dW_router": dW_router,
           "d_topk_w": dg, "dlogits": dlogits}
    if ws_gate is not None:
        sh = fwd["shared"]
        wsg, wsu, wsd = _f64(ws_gate), _f64(ws_up), _f64(ws_down)
        dh_s = dy @ wsd
        da_s = dh_s * sh["b"] * dsilu(sh["a"])
        db_s = dh_s * silu(sh["a"])
        out["dWs_down"] = dy.T @ sh["h"]
        out["dWs_gate"] = da_s.T @ x
        out["dWs_up"] = db_s.T @ x
        dx += da_s @ wsg + db_s @ wsu
    return out
