"""GPU path vs the CPU oracle, through the C ABI, on seeded synthetic inputs.

Bars: routing integers (top-k ids, counts, offsets, permutation) bit-exact on
the same float32 logits; logits within 1e-5 of the float64 oracle relative to
max|logit|; bf16 outputs and gradients max|err| / max|ref| <= 1e-2; router
weights within 1e-6 relative."""
import numpy as np
import pytest
import torch

from moe_layer_gb300 import _abi, layer
from oracle import moe_oracle as O
from synth.inputs import MoEShape, make_inputs, random_logits

from .helpers import ensure_lib, f64, oracle_backward, oracle_forward, order_gap, rel_err, topk_gap

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ensure_lib()


def _cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _route_on_logits(logits_cpu, k, expect_status=0):
    T, E = logits_cpu.shape
    cfg = _abi.make_config(T, 64, 64, E, k)
    bufs = layer.MoEBuffers(cfg, training=False)
    dev = "cuda"
    out = dict(
        topk_idx=torch.empty(T, k, dtype=torch.int32, device=dev),
        topk_w=torch.empty(T, k, dtype=torch.float32, device=dev),
        counts=torch.empty(E, dtype=torch.int32, device=dev),
        offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
        perm_token=torch.empty(T * k, dtype=torch.int32, device=dev),
        route_row=torch.empty(T, k, dtype=torch.int32, device=dev),
    )
    lg = logits_cpu.cuda()
    _abi.moe_route_topk(cfg, None, None, None, lg, None, out["topk_idx"], out["topk_w"], out["counts"],
                        out["offsets"], out["perm_token"], out["route_row"], bufs.fwd_ws)
    torch.cuda.synchronize()
    assert _abi.moe_read_device_status(bufs.fwd_ws) == expect_status
    return {k_: v.cpu().numpy() for k_, v in out.items()}


@pytest.mark.parametrize("T,E,k,ties", [
    (1000, 8, 2, False), (1000, 8, 2, True), (777, 64, 8, False), (513, 256, 8, True),
    (130, 300, 5, False), (64, 32, 32, True), (1, 4, 1, False), (2049, 512, 8, False),
])
def test_routing_bit_exact_on_given_logits(T, E, k, ties):
    logits = random_logits(T, E, seed=T + E + k, ties=ties)
    if E >= 16:
        logits[:, E - 3:] = -float("inf")  # experts that never win
    g = _route_on_logits(logits, k)
    idx, w = O.topk_route(logits.numpy().astype(np.float64), k)
    counts, offsets, perm_token, perm_slot, route_row = O.expert_schedule(idx, E)
    assert (g["topk_idx"] == idx).all()
    assert (g["counts"] == counts).all()
    assert (g["offsets"] == offsets).all()
    assert (g["perm_token"] == perm_token).all()
    assert (g["route_row"] == route_row).all()
    np.testing.assert_allclose(g["topk_w"], w, rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("E", [64, 300])
def test_nan_logits_are_passed_over_and_an_all_nan_token_is_reported(E):
    """moe.h / the top-k kernel: a NaN logit loses to every real logit, so its token routes as if
    that logit were below all others; a token with nothing but NaN left to choose records
    MOE_ERR_DEVICE (5) in the status word.  E = 64 and 300 cover both register layouts."""
    T, k = 96, 6
    logits = random_logits(T, E, seed=11 + E, ties=True)
    nan_cols = [0, 7, 33, E - 1]
    ref = logits.clone()
    ref[5, nan_cols] = -float("inf")
    ref[6, 1::2] = -float("inf")
    logits[5, nan_cols] = float("nan")
    logits[6, 1::2] = float("nan")  # half the experts NaN, the rest still enough
    g = _route_on_logits(logits, k)
    idx, _ = O.topk_route(ref.numpy().astype(np.float64), k)
    assert (g["topk_idx"] == idx).all()
    bad = logits[:4].clone()
    bad[2, :] = float("nan")
    _route_on_logits(bad, k, expect_status=5)


def _run_layer(shape, seed=0, backward=True, flags=0):
    inp_cpu = make_inputs(shape, seed=seed, with_dy=backward)
    inp = _cuda(inp_cpu)
    cfg = _abi.make_config(shape.T, shape.d, shape.I, shape.E, shape.k, shape.n_shared, shape.I_shared,
                           flags=flags)
    bufs = layer.MoEBuffers(cfg, training=backward)
    y = layer.forward(cfg, inp, bufs)
    res = {"y": y, "inp_cpu": inp_cpu, "cfg": cfg, "bufs": bufs, "inp": inp}
    if backward:
        grads = layer.alloc_grads(cfg)
        dx = layer.backward(cfg, inp, inp["dy"], bufs, grads)
        res.update(dx=dx, grads=grads)
    torch.cuda.synchronize()
    assert _abi.moe_read_device_status(bufs.fwd_ws) == 0
    if backward:
        assert _abi.moe_read_device_status(bufs.bwd_ws) == 0
    return res


SHAPES = {
    "tiny": MoEShape(T=512, d=256, I=128, E=8, k=2, n_shared=1, I_shared=128, w_std=0.02),
    "ragged": MoEShape(T=333, d=192, I=192, E=5, k=3, n_shared=1, I_shared=64, w_std=0.05),
    "noshared": MoEShape(T=700, d=256, I=320, E=16, k=4, n_shared=0, I_shared=0, w_std=0.05),
    "wide": MoEShape(T=300, d=576, I=384, E=12, k=6, n_shared=1, I_shared=320, w_std=0.04),
    "k_equals_E": MoEShape(T=129, d=128, I=64, E=4, k=4, n_shared=1, I_shared=64, w_std=0.05),
    "single_expert": MoEShape(T=200, d=128, I=128, E=1, k=1, n_shared=0, I_shared=0, w_std=0.05),
    "zipf_zero": MoEShape(T=640, d=256, I=128, E=32, k=4, n_shared=1, I_shared=128, w_std=0.05,
                          zipf=True, zero_experts=8),
    # every expert and the shared expert have a single 64-row tile (the GEMMs' SM-pair pass has
    # no work, all tiles go through the one-SM pass); the weight gradients run on one SM with
    # eight epilogue warps (16 rows per expert)
    "small_T": MoEShape(T=64, d=384, I=128, E=8, k=2, n_shared=1, I_shared=128, w_std=0.05),
    "single_token": MoEShape(T=1, d=256, I=256, E=16, k=4, n_shared=1, I_shared=256, w_std=0.05),
    # four of eight experts with an odd m-tile count in 44 tiles: the even experts' tiles run in
    # pairs on SM pairs and every tile of the odd ones on one SM, so both passes of each grouped
    # GEMM have work; 640 rows per expert put the weight gradients on SM pairs
    "pairs_leftover": MoEShape(T=2560, d=512, I=256, E=8, k=2, n_shared=1, I_shared=128, w_std=0.05),
    # two experts take every token (the other six are never chosen): 2048 rows each, four row
    # chunks of the router weight gradient per expert (summed as partials in chunk order), and
    # six experts whose gradients must be exact zeros
    "two_hot": MoEShape(T=2048, d=256, I=128, E=8, k=2, n_shared=0, I_shared=0, w_std=0.05, zero_experts=6),
    # the open-weight model shapes the MoK blog benchmarks ("Speedups"), scaled down with their
    # E, top-k and d:I ratio kept: Kimi-K2.7 (384, 8, 3.5), GLM-5.2 (256, 8, 3), Qwen3.5-397B-A17B
    # (512, 10, 4), DeepSeek-V4-Pro (384, 6, 7:3); logits spread wider so that seeds without
    # near-ties exist at these E and k
    "kimi_k27_scaled": MoEShape(T=256, d=448, I=128, E=384, k=8, n_shared=1, I_shared=128, w_std=0.05,
                                wr_std=0.1),
    "glm52_scaled": MoEShape(T=256, d=384, I=128, E=256, k=8, n_shared=1, I_shared=128, w_std=0.05, wr_std=0.1),
    "qwen35_scaled": MoEShape(T=256, d=512, I=128, E=512, k=10, n_shared=1, I_shared=128, w_std=0.05,
                              wr_std=0.1),
    "dsv4pro_scaled": MoEShape(T=256, d=448, I=192, E=384, k=6, n_shared=1, I_shared=192, w_std=0.05,
                               wr_std=0.1),
}


# seeds chosen so that no token has a top-k boundary gap below 1e-4 (checked
# below on the oracle's float64 logits)
SEEDS = {"noshared": 2, "pairs_leftover": 2, "glm52_scaled": 1, "qwen35_scaled": 2}


def _check_against_oracle(shape, r):
    """y, dx and every gradient of the run `r` against the oracle on its inputs."""
    inp = r["inp_cpu"]
    fwd = oracle_forward(inp, shape.k)
    # routing of the GPU (fp32 logits) vs the oracle (fp64 logits): identical
    # except possibly at near-ties, which these seeds do not have
    gap = topk_gap(fwd["logits"], shape.k)
    assert gap.min() > 1e-4, "seeded input has a near-tie; pick another seed"
    # slot order too (d_topk_w is compared slot by slot); logit errors here are ~1e-6
    assert order_gap(fwd["logits"], shape.k).min() > 1e-5
    bwd = oracle_backward(inp, fwd)
    assert rel_err(r["y"], fwd["y"]) <= TOL
    assert rel_err(r["dx"], bwd["dx"]) <= TOL
    g = r["grads"]
    for key in ["dW_gate", "dW_up", "dW_down", "dW_router", "d_topk_w"]:
        assert rel_err(g[key], bwd[key]) <= TOL, key
    if shape.n_shared:
        for key in ["dWs_gate", "dWs_up", "dWs_down"]:
            assert rel_err(g[key], bwd[key]) <= TOL, key
    if shape.zero_experts:
        for e in range(shape.E - shape.zero_experts, shape.E):
            assert fwd["counts"][e] == 0
            for key in ["dW_gate", "dW_up", "dW_down", "dW_router"]:
                assert (g[key][e] == 0).all(), (key, e)


@pytest.mark.parametrize("name", list(SHAPES))
def test_forward_backward_parity(name):
    shape = SHAPES[name]
    _check_against_oracle(shape, _run_layer(shape, seed=SEEDS.get(name, 0)))


FLAGS = {"replay": "MOE_FLAG_REPLAY", "wgrad_fp32": "MOE_FLAG_WGRAD_FP32",
         "replay_wgrad_fp32": ("MOE_FLAG_REPLAY", "MOE_FLAG_WGRAD_FP32")}


@pytest.mark.parametrize("flag", list(FLAGS))
@pytest.mark.parametrize("name", ["ragged", "zipf_zero", "pairs_leftover", "qwen35_scaled"])
def test_flag_paths_against_oracle(name, flag):
    """Forward activation replay (the backward recomputes the routed x rows, a
    and b) and fp32 weight gradients, each compared with the oracle itself."""
    names = FLAGS[flag] if isinstance(FLAGS[flag], tuple) else (FLAGS[flag],)
    flags = 0
    for n in names:
        flags |= getattr(_abi, n)
    shape = SHAPES[name]
    r = _run_layer(shape, seed=SEEDS.get(name, 0), flags=flags)
    if flags & _abi.MOE_FLAG_WGRAD_FP32:
        assert r["grads"]["dW_gate"].dtype == torch.float32
    _check_against_oracle(shape, r)


def test_routing_outputs_of_forward_match_oracle_routing():
    """The forward's own routing (GPU logits) equals the oracle's on every token
    whose top-k boundary gap is above the logits' error bound."""
    shape = SHAPES["tiny"]
    inp_cpu = make_inputs(shape, seed=3, with_dy=False)
    inp = _cuda(inp_cpu)
    T, E, k = shape.T, shape.E, shape.k
    cfg = _abi.make_config(T, shape.d, shape.I, E, k, shape.n_shared, shape.I_shared)
    bufs = layer.MoEBuffers(cfg, training=False)
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pt = torch.empty(T * k, dtype=torch.int32, device="cuda")
    rr = torch.empty(T, k, dtype=torch.int32, device="cuda")
    _abi.moe_route_topk(cfg, inp["x"], inp["W_router"], None, None, logits, idx, w, counts, offs, pt, rr,
                        bufs.fwd_ws)
    torch.cuda.synchronize()
    ref = O.router_logits(f64(inp_cpu["x"]), f64(inp_cpu["W_router"]))
    lg = f64(logits)
    assert np.abs(lg - ref).max() <= 1e-5 * np.abs(ref).max()
    ridx, _ = O.topk_route(ref, k)
    gap = topk_gap(ref, k)
    safe = gap > 1e-4
    assert (idx.cpu().numpy()[safe] == ridx[safe]).all()


@pytest.mark.parametrize("grid_limit", [None, "3"])
def test_bitwise_determinism(grid_limit, monkeypatch):
    """Same input -> bitwise identical outputs, also with a different number of
    persistent GEMM CTAs."""
    shape = SHAPES["wide"]
    a = _run_layer(shape, seed=5)
    if grid_limit:
        monkeypatch.setenv("MOE_GRID_LIMIT", grid_limit)
    b = _run_layer(shape, seed=5)
    assert torch.equal(a["y"], b["y"])
    assert torch.equal(a["dx"], b["dx"])
    for key in a["grads"]:
        if a["grads"][key] is not None:
            assert torch.equal(a["grads"][key], b["grads"][key]), key


@pytest.mark.parametrize("name", ["ragged", "noshared", "zipf_zero"])
def test_replay_matches_saved_activations_bitwise(name):
    """MOE_FLAG_REPLAY (saved state = routing only, the backward recomputes the
    x rows, a and b) gives bitwise the outputs and gradients of the path that
    saves them, with a saved buffer that holds no activations."""
    shape = SHAPES[name]
    a = _run_layer(shape, seed=SEEDS.get(name, 0))
    b = _run_layer(shape, seed=SEEDS.get(name, 0), flags=_abi.MOE_FLAG_REPLAY)
    assert b["bufs"].saved.numel() < a["bufs"].saved.numel()
    assert torch.equal(a["y"], b["y"])
    assert torch.equal(a["dx"], b["dx"])
    for key in a["grads"]:
        if a["grads"][key] is not None:
            assert torch.equal(a["grads"][key], b["grads"][key]), key


@pytest.mark.parametrize("name", ["ragged", "wide", "small_T", "pairs_leftover"])
def test_fp32_weight_gradients_round_to_the_bf16_ones(name):
    """MOE_FLAG_WGRAD_FP32 writes the fp32 accumulators the bf16 path rounds: rounded to bf16
    (nearest even) they are bitwise the bf16 weight gradients, and nothing else changes.  The
    shapes cover the three weight-gradient schedules and output row counts that are not a
    multiple of the 128-row tile (I = 192, I_s = 320)."""
    b = _run_layer(SHAPES[name])
    f = _run_layer(SHAPES[name], flags=_abi.MOE_FLAG_WGRAD_FP32)
    for n in ("dW_gate", "dW_up", "dW_down", "dWs_gate", "dWs_up", "dWs_down"):
        if b["grads"][n] is None:
            continue
        assert f["grads"][n].dtype == torch.float32, n
        assert torch.equal(f["grads"][n].to(torch.bfloat16), b["grads"][n]), n
    assert torch.equal(f["dx"], b["dx"])
    assert torch.equal(f["grads"]["dW_router"], b["grads"]["dW_router"])


def test_inference_without_saved_state_matches_training_forward():
    shape = SHAPES["ragged"]
    a = _run_layer(shape, seed=2, backward=False)
    b = _run_layer(shape, seed=2, backward=True)
    assert torch.equal(a["y"], b["y"])


def test_empty_batch():
    shape = MoEShape(T=0, d=128, I=64, E=4, k=2, n_shared=0, I_shared=0)
    cfg = _abi.make_config(0, 128, 64, 4, 2)
    bufs = layer.MoEBuffers(cfg)
    x = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    w = _abi.MoeWeights()
    _abi.moe_forward(cfg, x, w, x, bufs.saved, bufs.fwd_ws)


def test_dx_ready_event_marks_complete_dx():
    """moe_backward records the optional dx_ready event once dx is final: a
    copy taken on another stream after that event equals dx after the whole
    backward (the weight gradients computed after it do not touch dx)."""
    shape = SHAPES["wide"]
    inp = _cuda(make_inputs(shape, seed=7, with_dy=True))
    cfg = _abi.make_config(shape.T, shape.d, shape.I, shape.E, shape.k, shape.n_shared, shape.I_shared)
    bufs = layer.MoEBuffers(cfg)
    layer.forward(cfg, inp, bufs)
    grads = layer.alloc_grads(cfg)
    ev = torch.cuda.Event()
    ev.record()
    grads["dx_ready"] = ev
    dx = torch.empty(shape.T, shape.d, dtype=torch.bfloat16, device="cuda")
    early = torch.empty_like(dx)
    side = torch.cuda.Stream()
    layer.backward(cfg, inp, inp["dy"], bufs, grads, dx)
    with torch.cuda.stream(side):
        side.wait_event(ev)
        early.copy_(dx)
    torch.cuda.synchronize()
    assert torch.equal(early, dx)
    assert _abi.moe_read_device_status(bufs.bwd_ws) == 0
