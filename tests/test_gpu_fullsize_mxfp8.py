"""The DSV3-shaped layer in MXFP8 mode at full size (T=16384, d=7168, I=2048,
E=256, top-8, one shared expert), in the launch configuration bench.py times,
checked against the oracle's MXFP8 emulation on sampled tokens and on one
expert's weight gradients (max|err| / max|ref| <= 5e-2), plus a bitwise rerun.

MXFP8 quantization of the forward and of dx is local to a token row (blocks
along d, I or 2I), so the oracle run on a token subset sees the same blocks as
the full batch; the weight gradients' token-axis blocks are an expert's rows in
(token, slot) order, which the oracle rebuilds from the routing."""
import numpy as np
import pytest
import torch

from moe_layer_gb300 import _abi, layer
from oracle import moe_oracle as O
from synth.inputs import CONFIGS, make_inputs

from .helpers import ensure_lib, f64, full_router_grad_err, order_gap, shared_rows_err, topk_gap

pytestmark = pytest.mark.gpu
TOL_MX = 5e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ensure_lib()


class Experts64:
    """Indexable [E, ...] bf16 device tensor, one expert copied to the host as
    float64 on first use."""

    def __init__(self, t):
        self.t, self.cache = t, {}

    def __len__(self):
        return self.t.shape[0]

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = f64(self.t[e])
        return self.cache[e]


def _run(shape, seed=0):
    inp = make_inputs(shape, seed=seed, device="cuda")
    cfg = _abi.make_config(shape.T, shape.d, shape.I, shape.E, shape.k, shape.n_shared, shape.I_shared,
                           precision=_abi.MOE_MXFP8)
    layer.quantize_weights(cfg, inp)
    bufs = layer.MoEBuffers(cfg)
    grads = layer.alloc_grads(cfg)
    y = layer.forward(cfg, inp, bufs)
    dx = layer.backward(cfg, inp, inp["dy"], bufs, grads)
    # the routing the forward used, through the routing entry point (the same
    # bf16 router kernels; ids and weights do not depend on the precision)
    T, E, k = shape.T, shape.E, shape.k
    rcfg = _abi.make_config(T, shape.d, shape.I, E, k, shape.n_shared, shape.I_shared)
    rbufs = layer.MoEBuffers(rcfg, training=False)
    rt = dict(idx=torch.empty(T, k, dtype=torch.int32, device="cuda"), w=torch.empty(T, k, device="cuda"))
    scratch = [torch.empty(n, dtype=torch.int32, device="cuda") for n in (E, E + 1, T * k, T * k)]
    _abi.moe_route_topk(rcfg, inp["x"], inp["W_router"], None, None, None, rt["idx"], rt["w"], scratch[0],
                        scratch[1], scratch[2], scratch[3].view(T, k), rbufs.fwd_ws)
    torch.cuda.synchronize()
    assert _abi.moe_read_device_status(bufs.fwd_ws) == 0
    assert _abi.moe_read_device_status(bufs.bwd_ws) == 0
    return dict(inp=inp, y=y, dx=dx, grads=grads, rt=rt)


@pytest.fixture(scope="module")
def run():
    shape = CONFIGS["dsv3"]
    r = _run(shape)
    inp = r["inp"]
    r["shape"] = shape
    r["ref_logits"] = O.router_logits(f64(inp["x"]), f64(inp["W_router"]))
    yield r
    del r
    torch.cuda.empty_cache()


def test_sampled_tokens_forward_backward(run):
    s, inp, ref = run["shape"], run["inp"], run["ref_logits"]
    rng = np.random.default_rng(1)
    cand = np.nonzero(order_gap(ref, s.k) > 1e-3)[0]
    tokens = np.sort(rng.choice(cand, size=2, replace=False))
    tt = torch.as_tensor(tokens, device="cuda")
    wg, wu, wd = Experts64(inp["W_gate"]), Experts64(inp["W_up"]), Experts64(inp["W_down"])
    sh = dict(ws_gate=f64(inp["Ws_gate"]), ws_up=f64(inp["Ws_up"]), ws_down=f64(inp["Ws_down"]))
    x, dy = f64(inp["x"][tt]), f64(inp["dy"][tt])
    fwd = O.moe_forward(x, f64(inp["W_router"]), wg, wu, wd, s.k, mxfp8=True, **sh)
    bwd = O.moe_backward(x, f64(inp["W_router"]), wg, wu, wd, dy, fwd, dense_expert_grads=False, **sh)
    rel = lambda a, b: np.abs(a - b).max() / np.abs(b).max()
    assert rel(f64(run["y"][tt]), fwd["y"]) <= TOL_MX
    assert rel(f64(run["dx"][tt]), bwd["dx"]) <= TOL_MX
    assert rel(f64(run["grads"]["d_topk_w"][tt]), bwd["d_topk_w"]) <= TOL_MX


def test_sampled_expert_weight_gradients(run):
    s, inp, ref = run["shape"], run["inp"], run["ref_logits"]
    ridx, rw = O.topk_route(ref, s.k)
    gap = topk_gap(ref, s.k)
    srt = np.argsort(-ref, axis=1, kind="stable")
    near = gap <= 1e-4
    touchy = set(srt[near, s.k - 1].tolist()) | set(srt[near, s.k].tolist())
    counts = np.bincount(ridx.ravel(), minlength=s.E)
    order = [e for e in np.argsort(-counts) if e not in touchy and counts[e] > 0]
    e = order[len(order) // 2]
    t, j = np.nonzero(ridx == e)  # (token, slot) order: the expert's row order on the GPU
    tt = torch.as_tensor(t, device="cuda")
    xs, dys = f64(inp["x"][tt]), f64(inp["dy"][tt])
    wg, wu, wd = f64(inp["W_gate"][e]), f64(inp["W_up"][e]), f64(inp["W_down"][e])
    a, b, h, _ = O.expert_forward(xs, wg, wu, wd, mxfp8=True)
    dWg, dWu, dWd, _, _ = O.expert_backward(xs, dys, rw[t, j], a, b, h, wg, wu, wd, mxfp8=True)
    g = run["grads"]
    for gpu, refw, name in ((g["dW_gate"][e], dWg, "dW_gate"), (g["dW_up"][e], dWu, "dW_up"),
                            (g["dW_down"][e], dWd, "dW_down")):
        assert np.abs(f64(gpu) - refw).max() / np.abs(refw).max() <= TOL_MX, (name, e)


def test_router_weight_gradient_whole(run):
    """dW_router [E, d] in full (the router stays bf16 in MXFP8 mode): the
    oracle's router backward on the GPU's routing and d_topk_w."""
    rt, g = run["rt"], run["grads"]
    assert full_router_grad_err(run["inp"], rt["idx"], rt["w"], g["d_topk_w"], g["dW_router"]) <= TOL_MX


def test_sampled_shared_expert_weight_gradients(run):
    """The shared expert stays bf16 in MXFP8 mode: sampled rows at the bf16 bound."""
    cols = np.sort(np.random.default_rng(3).choice(run["shape"].I_shared, size=4, replace=False))
    errs = shared_rows_err(run["inp"], run["grads"], cols)
    assert max(errs) <= 1e-2, errs


def test_rerun_is_bitwise_identical(run):
    r2 = _run(run["shape"])
    assert torch.equal(r2["y"], run["y"]) and torch.equal(r2["dx"], run["dx"])
    for key in ("dW_gate", "dW_up", "dW_down", "dW_router", "d_topk_w"):
        assert torch.equal(r2["grads"][key], run["grads"][key]), key
