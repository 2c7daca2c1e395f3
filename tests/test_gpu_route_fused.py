"""The fused persistent routing launch (router GEMM with the top-k in its
epilogue, scan and scatter in one cooperative launch, stages handing off
through bounded device barriers) against the separate kernels it
replaces (MOE_ROUTING_SEPARATE=1): bitwise the same routing, layer outputs and
gradients; the separate kernels are themselves checked against the oracle in
test_gpu_parity.py, and so is the fused path (the default) there.  Also the
barrier's failure path: a barrier that waits for an arrival that never comes
returns MOE_ERR_DEVICE_TIMEOUT, and the context stays usable."""
import time

import numpy as np
import pytest
import torch

from moe_layer_gb300 import _abi, layer
from oracle import moe_oracle as O
from synth.inputs import MoEShape, make_inputs

from .helpers import ensure_lib, f64, topk_gap

pytestmark = pytest.mark.gpu
MOE_ERR_DEVICE = 5
MOE_ERR_DEVICE_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ensure_lib()


def _cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _route(cfg, inp, T, E, k, with_logits=True):
    bufs = layer.MoEBuffers(cfg, training=False)
    out = dict(
        logits=torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda") if with_logits else None,
        idx=torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
        w=torch.full((T, k), -1.0, dtype=torch.float32, device="cuda"),
        counts=torch.full((E,), -7, dtype=torch.int32, device="cuda"),
        offsets=torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
        perm=torch.full((T * k,), -7, dtype=torch.int32, device="cuda"),
        route_row=torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
    )
    _abi.moe_route_topk(cfg, inp["x"], inp["W_router"], inp["router_bias"], None, out["logits"], out["idx"], out["w"],
                        out["counts"], out["offsets"], out["perm"], out["route_row"], bufs.fwd_ws)
    status = _abi.moe_read_device_status(bufs.fwd_ws)
    return out, status


def _same_bits(a, b):
    if a is None or b is None:
        return a is None and b is None
    if a.dtype == torch.float32:
        return torch.equal(a.view(torch.int32), b.view(torch.int32))
    return torch.equal(a, b)


ROUTE_SHAPES = [
    MoEShape(T=1000, d=256, I=64, E=64, k=8, n_shared=0, I_shared=0, zipf=True),
    MoEShape(T=4097, d=448, I=64, E=256, k=8, n_shared=0, I_shared=0, zero_experts=8, zipf=True),
    MoEShape(T=77, d=128, I=64, E=200, k=16, n_shared=0, I_shared=0),
    MoEShape(T=1, d=64, I=64, E=4, k=1, n_shared=0, I_shared=0),
]


@pytest.mark.parametrize("shape", ROUTE_SHAPES, ids=lambda s: f"T{s.T}_E{s.E}_k{s.k}")
def test_fused_routing_equals_separate_kernels_bitwise(shape, monkeypatch):
    inp = _cuda(make_inputs(shape, seed=3, with_dy=False))
    cfg = _abi.make_config(shape.T, shape.d, shape.I, shape.E, shape.k)
    fused, st_f = _route(cfg, inp, shape.T, shape.E, shape.k)
    monkeypatch.setenv("MOE_ROUTING_SEPARATE", "1")
    sep, st_s = _route(cfg, inp, shape.T, shape.E, shape.k)
    assert st_f == st_s == 0
    for key in fused:
        assert _same_bits(fused[key], sep[key]), key


def test_fused_routing_nan_logits_match_separate_kernels(monkeypatch):
    """A token whose x row is NaN: both paths flag MOE_ERR_DEVICE and pick the
    same (in-range) ids for every token."""
    shape = MoEShape(T=300, d=128, I=64, E=32, k=4, n_shared=0, I_shared=0)
    inp = _cuda(make_inputs(shape, seed=5, with_dy=False))
    inp["x"][17] = float("nan")
    cfg = _abi.make_config(shape.T, shape.d, shape.I, shape.E, shape.k)
    fused, st_f = _route(cfg, inp, shape.T, shape.E, shape.k)
    monkeypatch.setenv("MOE_ROUTING_SEPARATE", "1")
    sep, st_s = _route(cfg, inp, shape.T, shape.E, shape.k)
    assert st_f == st_s == MOE_ERR_DEVICE
    for key in ("idx", "counts", "offsets", "perm", "route_row"):
        assert torch.equal(fused[key], sep[key]), key
    ok = torch.arange(shape.T, device="cuda") != 17
    assert _same_bits(fused["w"][ok], sep["w"][ok])
    assert int(fused["idx"].min()) >= 0 and int(fused["idx"].max()) < shape.E


LAYER_SHAPES = {
    "tiny": MoEShape(T=512, d=256, I=128, E=8, k=2, n_shared=1, I_shared=128, w_std=0.02),
    "zipf_zero": MoEShape(T=640, d=256, I=128, E=32, k=4, n_shared=1, I_shared=128, w_std=0.05,
                          zipf=True, zero_experts=8),
    "pairs_leftover": MoEShape(T=2560, d=512, I=256, E=8, k=2, n_shared=1, I_shared=128, w_std=0.05),
}


def _layer(shape, flags=0, mx=False):
    inp = _cuda(make_inputs(shape, seed=2, with_dy=True))
    cfg = _abi.make_config(shape.T, shape.d, shape.I, shape.E, shape.k, shape.n_shared, shape.I_shared,
                           precision=_abi.MOE_MXFP8 if mx else _abi.MOE_BF16, flags=flags)
    if mx:
        layer.quantize_weights(cfg, inp)
    bufs = layer.MoEBuffers(cfg)
    grads = layer.alloc_grads(cfg)
    y = layer.forward(cfg, inp, bufs)
    dx = layer.backward(cfg, inp, inp["dy"], bufs, grads)
    torch.cuda.synchronize()
    assert _abi.moe_read_device_status(bufs.fwd_ws) == 0
    assert _abi.moe_read_device_status(bufs.bwd_ws) == 0
    out = {"y": y, "dx": dx}
    out.update({k: v for k, v in grads.items() if isinstance(v, torch.Tensor)})
    return out


@pytest.mark.parametrize("name,flags,mx", [("tiny", 0, False), ("zipf_zero", 0, False), ("pairs_leftover", 0, False),
                                           ("zipf_zero", "replay", False), ("tiny", 0, True)])
def test_layer_with_fused_routing_equals_separate_kernels_bitwise(name, flags, mx, monkeypatch):
    shape = LAYER_SHAPES[name]
    if mx:
        shape = MoEShape(T=512, d=256, I=256, E=8, k=2, n_shared=1, I_shared=128, w_std=0.05)
    fl = _abi.MOE_FLAG_REPLAY if flags == "replay" else 0
    a = _layer(shape, fl, mx)
    monkeypatch.setenv("MOE_ROUTING_SEPARATE", "1")
    b = _layer(shape, fl, mx)
    for key in a:
        assert torch.equal(a[key], b[key]), key


def test_stuck_grid_barrier_reports_timeout_and_the_context_stays_usable(monkeypatch):
    """MOE_DEBUG_STALL_COUNTER: the fused routing launch's first grid barrier
    waits for one arrival more than the grid has.  Every CTA's bounded wait
    runs out, the call returns with the timeout status, and the next call
    routes correctly (checked against the oracle)."""
    shape = MoEShape(T=512, d=256, I=64, E=64, k=4, n_shared=0, I_shared=0, w_std=0.05)
    inp_cpu = make_inputs(shape, seed=0, with_dy=False)
    inp = _cuda(inp_cpu)
    cfg = _abi.make_config(shape.T, shape.d, shape.I, shape.E, shape.k)
    monkeypatch.setenv("MOE_DEBUG_STALL_COUNTER", "1")
    t0 = time.monotonic()
    _, status = _route(cfg, inp, shape.T, shape.E, shape.k)
    elapsed = time.monotonic() - t0
    assert status == MOE_ERR_DEVICE_TIMEOUT
    assert 1.0 < elapsed < 60.0, elapsed
    monkeypatch.delenv("MOE_DEBUG_STALL_COUNTER")
    out, status = _route(cfg, inp, shape.T, shape.E, shape.k)
    assert status == 0
    ref = O.router_logits(f64(inp_cpu["x"]), f64(inp_cpu["W_router"]))
    ridx, _ = O.topk_route(ref, shape.k)
    safe = topk_gap(ref, shape.k) > 1e-4
    assert (out["idx"].cpu().numpy()[safe] == ridx[safe]).all()
    counts, offsets, _, _, _ = O.expert_schedule(out["idx"].cpu().numpy(), shape.E)
    assert np.array_equal(out["counts"].cpu().numpy(), counts)
    assert np.array_equal(out["offsets"].cpu().numpy(), offsets)
