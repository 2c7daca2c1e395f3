"""Pins for the CPU oracle: checks against what the method and mathematics fix
(brute force, closed forms, library routines, finite differences), never
against the oracle's own formulas retyped.  CPU only."""
import itertools
import json
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ top-k
def _brute_topk_set(row, k):
    """Max-sum k-subset; among equal sums the lexicographically smallest."""
    best, best_key = None, None
    for comb in itertools.combinations(range(len(row)), k):
        key = (-sum(row[c] for c in comb), comb)
        if best_key is None or key < best_key:
            best, best_key = comb, key
    return best


@pytest.mark.parametrize("ties", [False, True])
def test_topk_matches_bruteforce_subsets(ties):
    rng = _rng(1 if ties else 2)
    T, E, k = 60, 7, 3
    logits = (rng.integers(-2, 3, (T, E)) * 0.5) if ties else rng.normal(size=(T, E))
    idx, w = O.topk_route(logits, k)
    for t in range(T):
        assert tuple(sorted(idx[t])) == _brute_topk_set(list(logits[t]), k)
        # slot order: non-increasing logits, ties in ascending expert index
        for j in range(k - 1):
            a, b = logits[t, idx[t, j]], logits[t, idx[t, j + 1]]
            assert a > b or (a == b and idx[t, j] < idx[t, j + 1])


def test_topk_weights_are_softmax_over_selected():
    rng = _rng(3)
    logits = rng.normal(size=(40, 16)) * 3
    idx, w = O.topk_route(logits, 5)
    sel = np.take_along_axis(logits, idx, axis=1)
    np.testing.assert_allclose(w, scipy.special.softmax(sel, axis=1), rtol=1e-13, atol=0)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)


def test_topk_uniform_logits_k_equals_E():
    E = 8
    idx, w = O.topk_route(np.zeros((5, E)), E)
    assert (idx == np.arange(E)).all()
    np.testing.assert_allclose(w, 1.0 / E, rtol=0, atol=1e-16)


def test_topk_golden_ties():
    g = json.load(open(os.path.join(GOLDEN, "topk_ties.json")))
    idx, w = O.topk_route(np.array(g["logits"]), g["k"])
    assert idx.tolist() == g["expected_idx"]
    np.testing.assert_allclose(w, np.array(g["expected_w"]), rtol=1e-14)


def test_topk_ignores_minus_inf_experts():
    logits = np.array([[0.1, -np.inf, 0.3, -np.inf, 0.2]])
    idx, w = O.topk_route(logits, 3)
    assert idx.tolist() == [[2, 4, 0]]
    assert np.isfinite(w).all()


# ------------------------------------------------------------------ schedule
@pytest.mark.parametrize("seed", [0, 1])
def test_schedule_bruteforce(seed):
    rng = _rng(seed)
    T, E, k = 37, 9, 3
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    counts, offsets, perm_token, perm_slot, route_row = O.expert_schedule(idx, E)
    # brute force: expert by expert, every (t, j) in ascending order
    rows = []
    for e in range(E):
        rows += [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
    assert list(zip(perm_token.tolist(), perm_slot.tolist())) == rows
    assert counts.sum() == T * k
    assert sorted(perm_token.tolist()) == sorted(np.repeat(np.arange(T), k).tolist())
    for t in range(T):
        for j in range(k):
            r = route_row[t, j]
            assert perm_token[r] == t and perm_slot[r] == j
            e = idx[t, j]
            assert offsets[e] <= r < offsets[e + 1]
    assert offsets[0] == 0 and (np.diff(offsets) == counts).all()


def test_schedule_empty_experts():
    idx = np.array([[0, 2], [2, 0]])
    counts, offsets, perm_token, _, _ = O.expert_schedule(idx, 4)
    assert counts.tolist() == [2, 0, 2, 0]
    assert offsets.tolist() == [0, 2, 2, 4, 4]
    assert perm_token.tolist() == [0, 1, 0, 1]


# ------------------------------------------------------------------ forward
def _weights(rng, E, d, I, I_s, std=0.3):
    wg = rng.normal(size=(E, I, d)) * std
    wu = rng.normal(size=(E, I, d)) * std
    wd = rng.normal(size=(E, d, I)) * std
    ws = (rng.normal(size=(I_s, d)) * std, rng.normal(size=(I_s, d)) * std,
          rng.normal(size=(d, I_s)) * std)
    return wg, wu, wd, ws


def test_silu_special_values():
    np.testing.assert_allclose(O.silu([0.0, 1.0, -1.0, 50.0, -800.0]),
                               [0.0, 1.0 / (1.0 + np.exp(-1.0)), -1.0 / (1.0 + np.e), 50.0, 0.0],
                               rtol=1e-15, atol=1e-300)
    # SiLU(z) = z * scipy.special.expit(z)
    z = np.linspace(-20, 20, 101)
    np.testing.assert_allclose(O.silu(z), z * scipy.special.expit(z), rtol=1e-14, atol=1e-300)


def test_forward_dense_reduction_k_equals_E():
    """k = E and W_router = 0: every expert gets weight 1/E, so
    y = shared(x) + mean_e FFN_e(x), computed here with einsum over all experts."""
    rng = _rng(4)
    T, d, I, E, I_s = 6, 10, 4, 5, 3
    x = rng.normal(size=(T, d))
    wg, wu, wd, (sg, su, sd) = _weights(rng, E, d, I, I_s)
    fwd = O.moe_forward(x, np.zeros((E, d)), wg, wu, wd, E, ws_gate=sg, ws_up=su, ws_down=sd)
    a = np.einsum("eid,td->eti", wg, x)
    b = np.einsum("eid,td->eti", wu, x)
    h = a * scipy.special.expit(a) * b
    routed = np.einsum("edi,eti->td", wd, h) / E
    a_s, b_s = x @ sg.T, x @ su.T
    shared = (a_s * scipy.special.expit(a_s) * b_s) @ sd.T
    np.testing.assert_allclose(fwd["y"], routed + shared, rtol=1e-12, atol=1e-12)


def test_forward_single_expert_closed_form():
    """E = 1, k = 1: g = 1, y = W_d (SiLU(W_g x) * W_u x) + shared(x), via torch float64."""
    rng = _rng(5)
    T, d, I, I_s = 7, 12, 5, 3
    x = rng.normal(size=(T, d))
    wg, wu, wd, (sg, su, sd) = _weights(rng, 1, d, I, I_s)
    wr = rng.normal(size=(1, d))
    fwd = O.moe_forward(x, wr, wg, wu, wd, 1, ws_gate=sg, ws_up=su, ws_down=sd)
    X = torch.from_numpy(x)
    F = torch.nn.functional
    ref = F.linear(F.silu(F.linear(X, torch.from_numpy(wg[0]))) * F.linear(X, torch.from_numpy(wu[0])),
                   torch.from_numpy(wd[0]))
    ref += F.linear(F.silu(F.linear(X, torch.from_numpy(sg))) * F.linear(X, torch.from_numpy(su)),
                    torch.from_numpy(sd))
    np.testing.assert_allclose(fwd["y"], ref.numpy(), rtol=1e-12, atol=1e-12)
    assert (fwd["topk_w"] == 1.0).all()


def test_forward_token_independence():
    """The forward of a token subset equals the matching rows of the full forward."""
    rng = _rng(6)
    T, d, I, E, k = 20, 8, 4, 6, 2
    x = rng.normal(size=(T, d))
    wg, wu, wd, _ = _weights(rng, E, d, I, 1)
    wr = rng.normal(size=(E, d))
    full = O.moe_forward(x, wr, wg, wu, wd, k)["y"]
    sub = [3, 11, 17]
    part = O.moe_forward(x[sub], wr, wg, wu, wd, k)["y"]
    np.testing.assert_allclose(part, full[sub], rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ backward
def _tiny_problem(seed=7):
    rng = _rng(seed)
    T, d, I, E, k, I_s = 3, 8, 4, 4, 2, 4
    x = rng.normal(size=(T, d))
    wr = rng.normal(size=(E, d)) * 0.7
    wg, wu, wd, (sg, su, sd) = _weights(rng, E, d, I, I_s, std=0.4)
    dy = rng.normal(size=(T, d))
    return dict(x=x, wr=wr, wg=wg, wu=wu, wd=wd, sg=sg, su=su, sd=sd, dy=dy, k=k)


def _loss(P):
    y = O.moe_forward(P["x"], P["wr"], P["wg"], P["wu"], P["wd"], P["k"],
                      ws_gate=P["sg"], ws_up=P["su"], ws_down=P["sd"])["y"]
    return float(np.sum(P["dy"] * y))


def test_backward_finite_differences():
    P = _tiny_problem()
    fwd = O.moe_forward(P["x"], P["wr"], P["wg"], P["wu"], P["wd"], P["k"],
                        ws_gate=P["sg"], ws_up=P["su"], ws_down=P["sd"])
    # no top-k boundary may sit within the step: gap between k-th and (k+1)-th logit
    srt = -np.sort(-fwd["logits"], axis=1)
    assert (srt[:, P["k"] - 1] - srt[:, P["k"]]).min() > 1e-3
    G = O.moe_backward(P["x"], P["wr"], P["wg"], P["wu"], P["wd"], P["dy"], fwd,
                       ws_gate=P["sg"], ws_up=P["su"], ws_down=P["sd"])
    eps = 1e-6
    pairs = [("x", "dx"), ("wr", "dW_router"), ("wg", "dW_gate"), ("wu", "dW_up"),
             ("wd", "dW_down"), ("sg", "dWs_gate"), ("su", "dWs_up"), ("sd", "dWs_down")]
    for pname, gname in pairs:
        base = P[pname]
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            orig = base[i]
            base[i] = orig + eps
            lp = _loss(P)
            base[i] = orig - eps
            lm = _loss(P)
            base[i] = orig
            num[i] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(G[gname], num, rtol=1e-6, atol=1e-7, err_msg=gname)


def test_router_weight_grad_is_output_inner_product():
    """dL/dg_tj = <dy_t, o_tj>, with o the expert's down-projection output:
    the oracle's <h, W_down^T dy> must equal it."""
    P = _tiny_problem(8)
    fwd = O.moe_forward(P["x"], P["wr"], P["wg"], P["wu"], P["wd"], P["k"])
    G = O.moe_backward(P["x"], P["wr"], P["wg"], P["wu"], P["wd"], P["dy"], fwd)
    for t in range(P["x"].shape[0]):
        for j in range(P["k"]):
            e = fwd["topk_idx"][t, j]
            xt = P["x"][t]
            a, b = P["wg"][e] @ xt, P["wu"][e] @ xt
            o = P["wd"][e] @ (a * scipy.special.expit(a) * b)
            assert G["d_topk_w"][t, j] == pytest.approx(float(P["dy"][t] @ o), rel=1e-12, abs=1e-12)


def test_backward_single_expert_router_grad_is_zero():
    """E = 1: g is the constant 1, so the logits (and W_router) get no gradient."""
    rng = _rng(9)
    T, d, I = 5, 6, 3
    x = rng.normal(size=(T, d))
    wg, wu, wd, _ = _weights(rng, 1, d, I, 1)
    wr = rng.normal(size=(1, d))
    dy = rng.normal(size=(T, d))
    fwd = O.moe_forward(x, wr, wg, wu, wd, 1)
    G = O.moe_backward(x, wr, wg, wu, wd, dy, fwd)
    assert (G["dlogits"] == 0).all() and (G["dW_router"] == 0).all()


def test_backward_empty_expert_gets_zero_grad():
    rng = _rng(10)
    T, d, I, E = 4, 6, 3, 3
    x = rng.normal(size=(T, d))
    wg, wu, wd, _ = _weights(rng, E, d, I, 1)
    wr = np.zeros((E, d))
    bias = np.array([0.0, 0.0, -np.inf])
    dy = rng.normal(size=(T, d))
    fwd = O.moe_forward(x, wr, wg, wu, wd, 2, router_bias=bias)
    assert fwd["counts"][2] == 0
    G = O.moe_backward(x, wr, wg, wu, wd, dy, fwd)
    assert (G["dW_gate"][2] == 0).all() and (G["dW_down"][2] == 0).all()


# ------------------------------------------------------------------ MXFP8
def test_e4m3_table_matches_torch_float8():
    """Every non-NaN E4M3 code decodes as torch's float8_e4m3fn does; the
    format's fixed points: max 448, smallest subnormal 2^-9, NaN at S.1111.111."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.tolist() == [c in (0x7F, 0xFF) for c in range(256)]
    assert np.isnan(O.E4M3_TABLE[nan]).all()
    np.testing.assert_array_equal(O.E4M3_TABLE[~nan], ref[~nan])
    assert O.E4M3_TABLE[0x7E] == 448.0 and O.E4M3_TABLE[1] == 2.0 ** -9


def _brute_e4m3(v):
    vals = O.E4M3_TABLE[:0x7F]  # non-negative codes
    a = min(abs(v), 448.0)
    d = np.abs(vals - a)
    best = np.nonzero(d == d.min())[0]
    code = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])  # tie: even mantissa
    return O.E4M3_TABLE[code] * (-1.0 if v < 0 else 1.0)


def test_e4m3_quantize_bruteforce_nearest_even():
    rng = _rng(11)
    vals = np.concatenate([rng.normal(size=300) * 50, rng.normal(size=100) * 1e-2,
                           O.E4M3_TABLE[:0x7E] + 1e-12, [0.0, 448.0, 464.0, 1000.0, -1000.0, 2.0 ** -10]])
    got = O.E4M3_TABLE[O.e4m3_quantize(vals)]
    want = np.array([_brute_e4m3(v) for v in vals])
    np.testing.assert_array_equal(got, want)
    # exact midpoints between neighbours go to the even-mantissa code
    pos = O.E4M3_TABLE[:0x7E]
    mids = (pos[:-1] + pos[1:]) / 2
    codes = O.e4m3_quantize(mids)
    assert (codes % 2 == 0).all()


def test_e4m3_quantize_matches_torch_cast_in_range():
    rng = _rng(12)
    v = np.clip(rng.normal(size=2000) * 60, -448, 448)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_quantize(v)
    np.testing.assert_array_equal(O.E4M3_TABLE[got], O.E4M3_TABLE[ref])


def test_mx_block_scale_definition():
    """amax / 2^(E-127) lies in [256, 512) for every non-zero block (the E8M0
    scale is 2^(floor(log2 amax) - 8)); an all-zero block gets code 0 and zero
    elements; every element is within half an E4M3 step of v / X, or saturated."""
    rng = _rng(13)
    v = rng.normal(size=(20, 96)) * np.exp(rng.normal(size=(20, 1)) * 4)
    v[3, 32:64] = 0.0
    codes, sc = O.mx_quantize(v, axis=1)
    X = np.ldexp(1.0, sc.astype(np.int64) - 127)
    amax = np.abs(v.reshape(20, 3, 32)).max(-1)
    nz = amax > 0
    r = amax[nz] / X[nz]
    assert (r >= 256).all() and (r < 512).all()
    assert sc[3, 1] == 0 and (codes[3, 32:64] == 0).all()
    y = O.mx_dequantize(codes, sc, axis=1)
    Xe = np.repeat(X, 32, axis=1)
    scaled = v / Xe
    sat = np.abs(scaled) > 448
    assert (np.abs(y[sat]) == 448 * Xe[sat]).all()
    # E4M3 step at magnitude m (normal range) is 2^(floor(log2 m) - 3)
    m = np.abs(scaled[~sat & (np.abs(scaled) >= 2 ** -6)])
    step = np.ldexp(1.0, np.floor(np.log2(m)).astype(np.int64) - 3)
    assert (np.abs(y[~sat & (np.abs(scaled) >= 2 ** -6)] / Xe[~sat & (np.abs(scaled) >= 2 ** -6)] - np.sign(scaled[~sat & (np.abs(scaled) >= 2 ** -6)]) * m) <= step / 2).all()


def test_mx_round_is_idempotent_and_axis_consistent():
    rng = _rng(14)
    v = rng.normal(size=(64, 96))
    r1 = O.mx_round(v, axis=1)
    np.testing.assert_array_equal(O.mx_round(r1, axis=1), r1)
    np.testing.assert_array_equal(O.mx_round(v.T, axis=0), r1.T)


def test_mxfp8_layer_stays_near_full_precision():
    """The MXFP8 layer differs from the full-precision one only by the
    quantization of the routed GEMM operands (a few percent at most)."""
    rng = _rng(15)
    T, d, I, E, k, I_s = 9, 64, 64, 4, 2, 32
    wg, wu, wd, (sg, su, sd) = _weights(rng, E, d, I, I_s, std=0.2)
    P = dict(x=rng.normal(size=(T, d)), wr=rng.normal(size=(E, d)) * 0.3, wg=wg, wu=wu, wd=wd,
             dy=rng.normal(size=(T, d)), k=k)
    kw = dict(ws_gate=sg, ws_up=su, ws_down=sd)
    f = O.moe_forward(P["x"], P["wr"], P["wg"], P["wu"], P["wd"], P["k"], **kw)
    fq = O.moe_forward(P["x"], P["wr"], P["wg"], P["wu"], P["wd"], P["k"], mxfp8=True, **kw)
    rel = np.abs(fq["y"] - f["y"]).max() / np.abs(f["y"]).max()
    assert 0 < rel < 0.1
    b = O.moe_backward(P["x"], P["wr"], P["wg"], P["wu"], P["wd"], P["dy"], f, **kw)
    bq = O.moe_backward(P["x"], P["wr"], P["wg"], P["wu"], P["wd"], P["dy"], fq, **kw)
    for key in ["dx", "dW_gate", "dW_up", "dW_down", "dW_router"]:
        r = np.abs(bq[key] - b[key]).max() / np.abs(b[key]).max()
        assert 0 < r < 0.15, key


def test_bf16_round_matches_torch_bfloat16_cast():
    """float32 values round to bfloat16 as torch's cast does (nearest, ties to
    the even significand), including exact ties, signed zero, subnormals and
    overflow to infinity."""
    rng = _rng(16)
    v32 = np.concatenate([rng.normal(size=3000) * np.exp(rng.normal(size=3000) * 6),
                          [0.0, -0.0, 1e-40, -3e-39, 3.4e38, -3.4e38, 1.0, 2.0 ** -126]]).astype(np.float32)
    # exact ties: low 16 bits 0x8000, even and odd upper halves
    ties = (np.array([0x3F808000, 0x3F818000, 0xC0A08000, 0x00018000], np.uint32)).view(np.float32)
    v32 = np.concatenate([v32, ties])
    ref = torch.from_numpy(v32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.bf16_round(v32.astype(np.float64)), ref)
    assert O.bf16_round(np.array([1.0 + 2.0 ** -8]))[0] == 1.0        # tie to even (down)
    assert O.bf16_round(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6  # tie to even (up)


def test_mxfp8_backward_takes_decisions_on_stored_values():
    """MXFP8 backward: a and b enter as their stored bf16 values, so moving
    them by less than half a bf16 step changes no output bit, and h is
    recomputed from them (the h argument does not matter)."""
    rng = _rng(17)
    n, d, I = 40, 64, 32
    x = rng.normal(size=(n, d))
    dy = rng.normal(size=(n, d))
    g = rng.uniform(0.1, 1.0, size=n)
    a0 = O.bf16_round(rng.normal(size=(n, I)))
    b0 = O.bf16_round(rng.normal(size=(n, I)))
    a1 = a0 * (1 + 1e-5 * rng.uniform(-1, 1, size=a0.shape))
    b1 = b0 * (1 + 1e-5 * rng.uniform(-1, 1, size=b0.shape))
    assert (a1 != a0).any()
    wg, wu, wd = rng.normal(size=(I, d)), rng.normal(size=(I, d)), rng.normal(size=(d, I))
    r0 = O.expert_backward(x, dy, g, a0, b0, O.swiglu(a0, b0), wg, wu, wd, mxfp8=True)
    r1 = O.expert_backward(x, dy, g, a1, b1, O.swiglu(a0, b0) + 1.0, wg, wu, wd, mxfp8=True)
    for u, v in zip(r0, r1):
        np.testing.assert_array_equal(u, v)
    # without MXFP8 the same perturbation is visible (the rounding is MXFP8-only)
    f0 = O.expert_backward(x, dy, g, a0, b0, O.swiglu(a0, b0), wg, wu, wd)
    f1 = O.expert_backward(x, dy, g, a1, b1, O.swiglu(a1, b1), wg, wu, wd)
    assert not np.array_equal(f0[4], f1[4])


def test_e4m3_quantize_matches_nearest_table_search_at_scale():
    """The closed-form rounding equals a search for the nearest of the 127
    non-negative code values (ties to the even code) on 200k values spanning
    every binade, the subnormals, exact midpoints and the saturation range."""
    rng = _rng(18)
    pos = O.E4M3_TABLE[:0x7F]  # ascending non-negative values, codes 0x00..0x7E
    mids = (pos[:-1] + pos[1:]) / 2
    v = np.concatenate([rng.uniform(-1, 1, 100_000) * np.exp2(rng.uniform(-12, 10, 100_000)),
                        mids, -mids, pos, np.nextafter(mids, 0), np.nextafter(mids, 1e9), [448.0, 460.0, 1e30]])
    a = np.minimum(np.abs(v), 448.0)
    hi = np.minimum(np.searchsorted(pos, a, side="left"), len(pos) - 1)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - pos[lo], pos[hi] - a
    want = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    got = O.e4m3_quantize(v) & 0x7F
    np.testing.assert_array_equal(got, want)
