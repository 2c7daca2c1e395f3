"""Pins for the oracle's MXFP8 composition: which operand of which GEMM is
quantized, along which axis, in blocks of 32 counted from where, and that the
router and the shared expert stay in full precision (MoK blog post, "MXFP8
support": every routed-expert GEMM runs on MX-quantized operands, blocks along
that GEMM's reduction axis; the shared expert stays BF16).  CPU only.

The pins rest on one property of the MX format, not on the oracle's code: an
operand whose 32-element blocks along an axis are each E4M3 values times one
power of two passes an MXFP8 round trip along that axis unchanged (the shared
scale is a power of two and the scaled elements are E4M3 values again).  So

  * P1: when every operand of a GEMM is built that way along the GEMM's
    reduction axis, and deliberately NOT along the other axis (neighbouring
    blocks carry powers of two 2^12 apart, so a block taken across them
    loses the small elements), the MXFP8 result equals the full-precision one
    to float64 rounding: quantizing along the wrong axis, with other block
    boundaries, or quantizing an operand that is not quantized in the layer,
    would change it;
  * P2: with one operand made of ordinary values instead, the MXFP8 result
    differs from the full-precision one: that operand is quantized at all.

test_pins_catch_planted_mistakes plants each plausible mistake in the oracle
(one quantization along the other axis, one left out, the token blocks
counted from the other end) and checks that some pin fails.

Intermediate operands (h, [da | db], g h) are steered through their inputs:
with a >= 64, SiLU(a) = a, SiLU'(a) = 1 exactly in float64, so h = a b,
da = g dh b and db = g dh a are products of values chosen here; a one-hot
dy row makes dh a row of W_down times a power of two.
"""
import numpy as np
import pytest

from oracle import moe_oracle as O

SP = 12  # exponent gap between neighbouring blocks


def _rng(seed):
    return np.random.default_rng(seed)


def _safe(rng, shape):
    """E4M3 normal values with significand 1.0 .. 1.75 and exponents -3 .. 5:
    any arrangement of them passes an MXFP8 round trip along any axis (the
    block scale is 2^(e_max - 8), and the scaled elements stay E4M3 values no
    larger than 448)."""
    m = rng.integers(0, 7, size=shape)
    e = rng.integers(-3, 6, size=shape)
    sgn = np.where(rng.random(shape) < 0.5, -1.0, 1.0)
    return sgn * (1.0 + m / 8.0) * np.exp2(e)


def _blocky(rng, shape, axis):
    """Values exactly MXFP8-representable in 32-blocks along `axis` only: safe
    E4M3 values times 2^0 or 2^SP, constant on each 32-block along `axis` and
    alternating between neighbouring blocks and between neighbouring positions
    along the other axis."""
    r = np.arange(shape[0])[:, None]
    c = np.arange(shape[1])[None, :]
    blk, other = (c // 32, r) if axis in (1, -1) else (r // 32, c)
    return _safe(rng, shape) * np.exp2(SP * ((blk + other) % 2))


def _ordinary(rng, shape):
    return rng.normal(size=shape)


def _same(u, v):
    u, v = np.asarray(u, np.float64), np.asarray(v, np.float64)
    return float(np.abs(u - v).max() / max(np.abs(v).max(), 1e-300)) <= 1e-12


def _differs(u, v):
    u, v = np.asarray(u, np.float64), np.asarray(v, np.float64)
    return float(np.abs(u - v).max() / max(np.abs(v).max(), 1e-300)) > 1e-6


def test_construction_is_representable_along_one_axis_only():
    """The building blocks do what the pins assume (checked with the codec,
    which is pinned on its own against brute force and torch)."""
    rng = _rng(1)
    s = _safe(rng, (64, 96))
    np.testing.assert_array_equal(O.mx_round(s, axis=1), s)
    np.testing.assert_array_equal(O.mx_round(s, axis=0), s)
    for axis in (0, 1):
        b = _blocky(rng, (64, 96), axis)
        np.testing.assert_array_equal(O.mx_round(b, axis=axis), b)
        assert not np.array_equal(O.mx_round(b, axis=1 - axis), b)


# ------------------------------------------------------------------ forward
def _chk(out, name, fn):
    """Records (name, fn()); a check that raises (a planted mistake may break a
    shape) counts as failed."""
    try:
        ok = bool(fn())
    except Exception as exc:
        name, ok = f"{name} (raised {type(exc).__name__})", False
    out.append((name, ok))


def _fwd(k, x, wg, wu, wd):
    """Output k (a, b, h, o) of the expert forward, MXFP8 and full precision."""
    return O.expert_forward(x, wg, wu, wd, mxfp8=True)[k], O.expert_forward(x, wg, wu, wd)[k]


def _scenarios_forward(rng):
    """[(name, ok)] for the forward pins (gate/up GEMM and down GEMM)."""
    out = []
    T, d, I = 64, 64, 64
    # gate/up: x, W_gate, W_up along d (their last axis)
    x, wg, wu, wd = _blocky(rng, (T, d), 1), _blocky(rng, (I, d), 1), _blocky(rng, (I, d), 1), _safe(rng, (d, I))
    _chk(out, "P1 gate/up: a", lambda: _same(*_fwd(0, x, wg, wu, wd)))
    _chk(out, "P1 gate/up: b", lambda: _same(*_fwd(1, x, wg, wu, wd)))
    xo, wgo, wuo = _ordinary(rng, (T, d)), _ordinary(rng, (I, d)), _ordinary(rng, (I, d))
    _chk(out, "P2 gate/up: x quantized", lambda: _differs(*_fwd(0, xo, wg, wu, wd)))
    _chk(out, "P2 gate/up: W_gate quantized", lambda: _differs(*_fwd(0, x, wgo, wu, wd)))
    _chk(out, "P2 gate/up: W_up quantized", lambda: _differs(*_fwd(1, x, wg, wuo, wd)))
    # down: h along I (per token), W_down along I.  x one-hot (token t at
    # column t, 2^(10 (t % 2))), W_gate rows 2^(6 + 12 (i // 32 % 2)), W_up safe:
    # a = 2^(p_t + 6 + 12 q_i) >= 64, h = a b = 2^(2 p_t + 6 + 12 q_i) W_up[i, t]:
    # exact along I in 32-blocks, not along the tokens (2 p_t alternates 0, 20)
    p = 10 * (np.arange(T) % 2)
    x1 = np.zeros((T, d))
    x1[np.arange(T), np.arange(T)] = np.exp2(p)
    qi = (np.arange(I) // 32) % 2
    wg1 = np.repeat(np.exp2(6 + SP * qi)[:, None], d, axis=1)
    wu1 = _safe(rng, (I, d))
    wd1 = _blocky(rng, (d, I), 1)
    a, b, h, _ = O.expert_forward(x1, wg1, wu1, wd1)
    assert np.array_equal(h, a * b)  # SiLU(a) = a exactly here
    assert not np.array_equal(O.mx_round(h, axis=0), h)
    wdo = _ordinary(rng, (d, I))
    _chk(out, "P1 down: o", lambda: _same(*_fwd(3, x1, wg1, wu1, wd1)))
    _chk(out, "P2 down: W_down quantized", lambda: _differs(*_fwd(3, x1, wg1, wu1, wdo)))
    # 1.5 W_gate: h = 1.5 a b holds products of two 3-bit significands
    _chk(out, "P2 down: h quantized", lambda: _differs(*_fwd(3, x1, 1.5 * wg1, wu1, wd1)))
    return out


# ------------------------------------------------------------------ backward
def _bwd(k, x, dy, g, a, b, wg, wu, wd):
    """Output k (dW_gate, dW_up, dW_down, dg, dx) of the expert backward,
    MXFP8 and full precision."""
    h = O.swiglu(a, b)
    return (O.expert_backward(x, dy, g, a, b, h, wg, wu, wd, mxfp8=True)[k],
            O.expert_backward(x, dy, g, a, b, h, wg, wu, wd)[k])


def _onehot(n, d, scale):
    v = np.zeros((n, d))
    v[np.arange(n), np.arange(n) % d] = scale
    return v


def _scenarios_backward(rng):
    """[(name, ok)] for the backward pins: dh (dgrad of down), dx (dgrad of
    gate/up) and the three weight gradients."""
    out = []
    n, d, I = 64, 64, 64
    DWG, DWU, DWD, DG, DX = range(5)
    # ---- dh = dy W_down: dy along d, W_down along d (its first axis); seen through dg
    a = np.exp2(6 + rng.integers(0, 4, size=(n, I)))
    b = _safe(rng, (n, I))
    g = np.full(n, 0.5)
    x = _safe(rng, (n, d))
    wg, wu = _safe(rng, (I, d)), _safe(rng, (I, d))
    dy, wd = _blocky(rng, (n, d), 1), _blocky(rng, (d, I), 0)
    dyo, wdo = _ordinary(rng, (n, d)), _ordinary(rng, (d, I))
    _chk(out, "P1 dgrad down: dg", lambda: _same(*_bwd(DG, x, dy, g, a, b, wg, wu, wd)))
    _chk(out, "P2 dgrad down: dy quantized", lambda: _differs(*_bwd(DG, x, dyo, g, a, b, wg, wu, wd)))
    _chk(out, "P2 dgrad down: W_down quantized", lambda: _differs(*_bwd(DG, x, dy, g, a, b, wg, wu, wdo)))

    # ---- dx = [da | db] [W_gate; W_up]: both along 2I.  dy one-hot, W_down
    # safe, so dh[t] = W_down[t % d] (exact); a = 2^(6 + 12 s), b = 2^(12 s)
    # with s = (t + i // 32) % 2: da = g dh b and db = g dh a are exact along I
    # in 32-blocks and not along the tokens
    t_ = np.arange(n)[:, None]
    s = (t_ + np.arange(I)[None, :] // 32) % 2
    a2, b2 = np.exp2(6 + SP * s), np.exp2(SP * s)
    dy2, wd2 = _onehot(n, d, 1.0), _safe(rng, (d, I))
    g2 = np.exp2(-1 - (np.arange(n) % 2))
    wg2, wu2 = _blocky(rng, (I, d), 0), _blocky(rng, (I, d), 0)
    # ordinary weights as large as W_up's entries (da is 64x smaller than db here)
    wgo, wuo = _ordinary(rng, (I, d)) * np.abs(wu2).max(), _ordinary(rng, (I, d))
    _chk(out, "P1 dgrad gate/up: dx", lambda: _same(*_bwd(DX, x, dy2, g2, a2, b2, wg2, wu2, wd2)))
    # 1.5 b (1.5 a): da (db) holds products of two 3-bit significands
    _chk(out, "P2 dgrad gate/up: da quantized", lambda: _differs(*_bwd(DX, x, dy2, g2, a2, 1.5 * b2, wg2, wu2, wd2)))
    _chk(out, "P2 dgrad gate/up: db quantized", lambda: _differs(*_bwd(DX, x, dy2, g2, 1.5 * a2, b2, wg2, wu2, wd2)))
    _chk(out, "P2 dgrad gate/up: W_gate quantized", lambda: _differs(*_bwd(DX, x, dy2, g2, a2, b2, wgo, wu2, wd2)))
    _chk(out, "P2 dgrad gate/up: W_up quantized", lambda: _differs(*_bwd(DX, x, dy2, g2, a2, b2, wg2, wuo, wd2)))

    # ---- weight gradients: operands along the tokens, blocks of 32 rows from
    # the expert's first row, the last block zero-padded (n = 50 rows)
    n3 = 50
    tb = (np.arange(n3) // 32)[:, None]
    s3 = (tb + np.arange(I)[None, :]) % 2
    a3, b3 = np.exp2(6 + SP * s3), np.exp2(SP * s3)
    g3 = np.exp2(-1.0 - (np.arange(n3) // 32))
    dy3, wd3 = _onehot(n3, d, 1.0), _safe(rng, (d, I))
    x3 = _blocky(rng, (n3, d), 0)
    for arr in (x3, g3[:, None] * wd3[np.arange(n3) % d] * b3, g3[:, None] * wd3[np.arange(n3) % d] * a3):
        assert not np.array_equal(O.mx_round(arr, axis=1), arr)
    x3o = _ordinary(rng, (n3, d))
    _chk(out, "P1 wgrad: dW_gate", lambda: _same(*_bwd(DWG, x3, dy3, g3, a3, b3, wg, wu, wd3)))
    _chk(out, "P1 wgrad: dW_up", lambda: _same(*_bwd(DWU, x3, dy3, g3, a3, b3, wg, wu, wd3)))
    _chk(out, "P2 wgrad: x quantized for dW_gate", lambda: _differs(*_bwd(DWG, x3o, dy3, g3, a3, b3, wg, wu, wd3)))
    _chk(out, "P2 wgrad: x quantized for dW_up", lambda: _differs(*_bwd(DWU, x3o, dy3, g3, a3, b3, wg, wu, wd3)))
    _chk(out, "P2 wgrad: da quantized", lambda: _differs(*_bwd(DWG, x3, dy3, g3, a3, 1.5 * b3, wg, wu, wd3)))
    _chk(out, "P2 wgrad: db quantized", lambda: _differs(*_bwd(DWU, x3, dy3, g3, 1.5 * a3, b3, wg, wu, wd3)))
    # dW_down = dy^T (g h): dy along the tokens; g h = g a b with a = 2^(6 + 12 s3), b safe
    dy4 = _blocky(rng, (n3, d), 0)
    b4 = _safe(rng, (n3, I))
    dy4o = _ordinary(rng, (n3, d))
    _chk(out, "P1 wgrad: dW_down", lambda: _same(*_bwd(DWD, x3, dy4, g3, a3, b4, wg, wu, wd3)))
    _chk(out, "P2 wgrad: dy quantized", lambda: _differs(*_bwd(DWD, x3, dy4o, g3, a3, b4, wg, wu, wd3)))
    _chk(out, "P2 wgrad: g h quantized", lambda: _differs(*_bwd(DWD, x3, dy4, g3, 1.5 * a3, b4, wg, wu, wd3)))
    return out


def _failures(results):
    return [name for name, ok in results if not ok]


def test_mxfp8_expert_forward_composition():
    assert _failures(_scenarios_forward(_rng(2))) == []


def test_mxfp8_expert_backward_composition():
    assert _failures(_scenarios_backward(_rng(3))) == []


# ------------------------------------------------------------------ layer
def _layer_problem(rng, ordinary_wd=False):
    """A layer whose routed operands are all exactly representable along every
    axis (one-hot x and dy rows, constant W_gate = 64 and W_up = 1, safe
    W_down), two-way ties in the router so every weight is 1/2, and a shared
    expert and router with ordinary values."""
    T, d, I, E, k, Is = 40, 64, 64, 4, 2, 32
    x = _onehot(T, d, 1.0)
    wr = -np.ones((E, d))
    for c in range(d):
        e0 = c % 3
        wr[e0, c] = wr[e0 + 1, c] = 1.0  # experts e0, e0+1 tie for the top two
    wr = wr + 0.0
    wg = [np.full((I, d), 64.0) for _ in range(E)]
    wu = [np.ones((I, d)) for _ in range(E)]
    wd = [(_ordinary(rng, (d, I)) if ordinary_wd else _safe(rng, (d, I))) for _ in range(E)]
    sh = dict(ws_gate=_ordinary(rng, (Is, d)) * 0.3, ws_up=_ordinary(rng, (Is, d)) * 0.3,
              ws_down=_ordinary(rng, (d, Is)) * 0.3)
    dy = _onehot(T, d, 1.0)[::-1].copy()
    return x, wr, wg, wu, wd, k, sh, dy


def _layer_results(rng, ordinary_wd=False):
    x, wr, wg, wu, wd, k, sh, dy = _layer_problem(rng, ordinary_wd)
    fq = O.moe_forward(x, wr, wg, wu, wd, k, mxfp8=True, **sh)
    ff = O.moe_forward(x, wr, wg, wu, wd, k, **sh)
    assert np.all(ff["topk_w"] == 0.5)
    assert (ff["counts"] % 32 != 0).any()
    bq = O.moe_backward(x, wr, wg, wu, wd, dy, fq, **sh)
    bf = O.moe_backward(x, wr, wg, wu, wd, dy, ff, **sh)
    return fq, ff, bq, bf


def _scenarios_layer(rng):
    out = []
    try:
        fq, ff, bq, bf = _layer_results(rng)
    except Exception as exc:
        return [(f"P1 layer (raised {type(exc).__name__})", False)]
    _chk(out, "P1 layer: y", lambda: _same(fq["y"], ff["y"]))
    for key in ("dx", "dW_gate", "dW_up", "dW_down", "dW_router", "d_topk_w", "dWs_gate", "dWs_up", "dWs_down"):
        _chk(out, f"P1 layer: {key}", lambda key=key: _same(bq[key], bf[key]))
    _chk(out, "P2 layer: routed experts quantized",
         lambda: (lambda r: _differs(r[0]["y"], r[1]["y"]))(_layer_results(rng, ordinary_wd=True)))
    return out


def test_mxfp8_layer_composition_router_and_shared_stay_full_precision():
    """With every routed operand exactly representable, the MXFP8 layer equals
    the full-precision one in every output and gradient, although the router
    and the shared expert hold ordinary values: neither is quantized."""
    assert _failures(_scenarios_layer(_rng(4))) == []


# ------------------------------------------------------------------ planted mistakes
_REAL_MX_ROUND = O.mx_round


class _Planted:
    """Stands in for O.mx_round: while `active` (inside the expert function
    under test), its call number `which` is taken along the other axis
    ("flip") or left out ("skip"); every other call is the real one."""

    def __init__(self, which=-1, kind="flip"):
        self.which, self.kind, self.n, self.active = which, kind, 0, False

    def __call__(self, v, axis=-1):
        if self.active:
            i, self.n = self.n, self.n + 1
            if i == self.which:
                if self.kind == "skip":
                    return np.asarray(v, np.float64)
                axis = 0 if axis in (-1, 1) else 1
        return _REAL_MX_ROUND(v, axis=axis)


def _plant(monkeypatch, name, planted):
    """Routes O.<name> through `planted`: its counter restarts at each call."""
    real = getattr(O, name)

    def wrapped(*args, **kw):
        planted.n, planted.active = 0, True
        try:
            return real(*args, **kw)
        finally:
            planted.active = False
    monkeypatch.setattr(O, name, wrapped)
    monkeypatch.setattr(O, "mx_round", planted)


def _one_call_args(target):
    rng = _rng(9)
    n, d, I = 40, 64, 64
    if target == "_ffn":
        return (_safe(rng, (n, d)), _safe(rng, (I, d)), _safe(rng, (I, d)), _safe(rng, (d, I)), True)
    a, b = _safe(rng, (n, I)), _safe(rng, (n, I))
    return (_safe(rng, (n, d)), _safe(rng, (n, d)), np.ones(n), a, b, O.swiglu(a, b),
            _safe(rng, (I, d)), _safe(rng, (I, d)), _safe(rng, (d, I)), True)


def _run_all(seed=2):
    return (_scenarios_forward(_rng(seed)) + _scenarios_backward(_rng(seed + 1))
            + _scenarios_layer(_rng(seed + 2)))


def _pad_at_top(v):
    """Planted mistake: token blocks counted from the expert's last row."""
    v = np.asarray(v, np.float64)
    pad = (-v.shape[0]) % 32
    vp = np.concatenate([np.zeros((pad,) + v.shape[1:]), v], axis=0) if pad else v
    return O.mx_round(vp, axis=0)[pad:]


def test_pins_catch_planted_mistakes(monkeypatch):
    """Every planted mistake in the oracle's MXFP8 composition makes at least
    one pin fail: each quantization of the expert forward (reached through
    _ffn) and backward taken along the other axis or left out, the token
    blocks counted from the expert's last row, and the shared expert
    quantized like the routed ones."""
    assert _failures(_run_all()) == []
    missed = []
    n_mutants = 0
    for target in ("_ffn", "expert_backward"):
        counter = _Planted()
        _plant(monkeypatch, target, counter)
        getattr(O, target)(*_one_call_args(target))
        calls = counter.n
        monkeypatch.undo()
        assert calls == (5 if target == "_ffn" else 9)
        for which in range(calls):
            for kind in ("flip", "skip"):
                _plant(monkeypatch, target, _Planted(which, kind))
                # caught by a changed value, not only by a shape that breaks
                if not [f for f in _failures(_run_all()) if "raised" not in f]:
                    missed.append(f"{target} quantization #{which} {kind}")
                monkeypatch.undo()
                n_mutants += 1
    assert n_mutants == 28 and missed == [], missed

    monkeypatch.setattr(O, "_mx_rows", _pad_at_top)
    assert _failures(_run_all()) != []
    monkeypatch.undo()

    # the shared expert's FFN quantized whenever the layer runs in MXFP8 mode
    real_fwd, real_ffn, mode = O.moe_forward, O._ffn, {"mx": False}

    def fwd(*args, mxfp8=False, **kw):
        mode["mx"] = mxfp8
        try:
            return real_fwd(*args, mxfp8=mxfp8, **kw)
        finally:
            mode["mx"] = False
    monkeypatch.setattr(O, "moe_forward", fwd)
    monkeypatch.setattr(O, "_ffn", lambda xr, wg, wu, wd, mxfp8=False: real_ffn(xr, wg, wu, wd, mxfp8 or mode["mx"]))
    assert "P1 layer: y" in _failures(_scenarios_layer(_rng(4)))
    monkeypatch.undo()
