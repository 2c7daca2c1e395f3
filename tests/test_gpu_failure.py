"""Device-side failure path: a bounded wait that runs out.

Every mbarrier wait of the tensor-core GEMM gives up after a time limit,
records MOE_ERR_DEVICE_TIMEOUT in the workspace status word, drains its
in-flight copies and lets the CTA exit, so that a stuck pipeline neither hangs
the GPU nor loses the context.  The library's test hook MOE_DEBUG_STALL_ROUTER
makes the router projection's first pipeline stage expect 16 bytes that no
copy brings: a wait that nothing completes.  No fault is raised on the GPU."""
import time

import numpy as np
import pytest
import torch

from moe_layer_gb300 import _abi, layer
from oracle import moe_oracle as O

from synth.inputs import MoEShape, make_inputs

from .helpers import ensure_lib, f64, oracle_forward, rel_err, topk_gap

pytestmark = pytest.mark.gpu
MOE_ERR_DEVICE_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ensure_lib()


def _route(shape, inp):
    T, E, k = shape.T, shape.E, shape.k
    cfg = _abi.make_config(T, shape.d, shape.I, E, k)
    bufs = layer.MoEBuffers(cfg, training=False)
    out = {
        "logits": torch.empty(T, E, dtype=torch.float32, device="cuda"),
        "idx": torch.empty(T, k, dtype=torch.int32, device="cuda"),
        "w": torch.empty(T, k, dtype=torch.float32, device="cuda"),
        "counts": torch.empty(E, dtype=torch.int32, device="cuda"),
        "offs": torch.empty(E + 1, dtype=torch.int32, device="cuda"),
        "pt": torch.empty(T * k, dtype=torch.int32, device="cuda"),
        "rr": torch.empty(T, k, dtype=torch.int32, device="cuda"),
    }
    _abi.moe_route_topk(cfg, inp["x"], inp["W_router"], None, None, out["logits"], out["idx"], out["w"],
                        out["counts"], out["offs"], out["pt"], out["rr"], bufs.fwd_ws)
    return bufs, out


def test_stuck_pipeline_reports_timeout_and_the_context_stays_usable(monkeypatch):
    # d = 512: eight K stages for four pipeline slots, so the producer also
    # blocks (on a slot the stuck MMA warp never frees) and takes the abort path
    shape = MoEShape(T=256, d=512, I=128, E=64, k=4, n_shared=0, I_shared=0, w_std=0.05)
    inp_cpu = make_inputs(shape, seed=0, with_dy=False)
    inp = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp_cpu.items()}

    monkeypatch.setenv("MOE_DEBUG_STALL_ROUTER", "1")
    t0 = time.monotonic()
    bufs, _ = _route(shape, inp)
    status = _abi.moe_read_device_status(bufs.fwd_ws)  # synchronizes the stream
    elapsed = time.monotonic() - t0
    assert status == MOE_ERR_DEVICE_TIMEOUT
    # the waits are bounded (a few seconds each), not a hang
    assert 1.0 < elapsed < 60.0, elapsed

    # the context survives: the same call without the hook routes correctly
    monkeypatch.delenv("MOE_DEBUG_STALL_ROUTER")
    bufs, out = _route(shape, inp)
    assert _abi.moe_read_device_status(bufs.fwd_ws) == 0
    ref = O.router_logits(f64(inp_cpu["x"]), f64(inp_cpu["W_router"]))
    assert np.abs(out["logits"].double().cpu().numpy() - ref).max() <= 1e-5 * np.abs(ref).max()
    ridx, _ = O.topk_route(ref, shape.k)
    safe = topk_gap(ref, shape.k) > 1e-4
    assert (out["idx"].cpu().numpy()[safe] == ridx[safe]).all()


def test_stuck_sm_pair_pipeline_reports_timeout_and_the_context_stays_usable(monkeypatch):
    """The same on the SM-pair GEMMs (cta_group::2): MOE_DEBUG_STALL_PAIR makes
    the even CTA of every pair of the shared expert's gate/up wait for bytes
    that never come.  Its MMA warp gives up, its producer drains, and the odd
    CTA, whose stage releases never arrive, gives up on its own bounded waits;
    both reach the final cluster barrier.  The forward returns with the
    timeout status, and the next forward on the context matches the oracle."""
    # T = 512: four 128-row m-tiles of the shared expert's dense rows, two
    # pairs; d = 512: eight K stages for six pipeline slots
    shape = MoEShape(T=512, d=512, I=128, E=8, k=2, n_shared=1, I_shared=128, w_std=0.05)
    inp_cpu = make_inputs(shape, seed=0, with_dy=False)
    inp = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp_cpu.items()}
    cfg = _abi.make_config(shape.T, shape.d, shape.I, shape.E, shape.k, shape.n_shared, shape.I_shared)

    monkeypatch.setenv("MOE_DEBUG_STALL_PAIR", "1")
    bufs = layer.MoEBuffers(cfg, training=False)
    t0 = time.monotonic()
    layer.forward(cfg, inp, bufs)
    status = _abi.moe_read_device_status(bufs.fwd_ws)  # synchronizes the stream
    elapsed = time.monotonic() - t0
    assert status == MOE_ERR_DEVICE_TIMEOUT
    assert 1.0 < elapsed < 60.0, elapsed

    monkeypatch.delenv("MOE_DEBUG_STALL_PAIR")
    bufs = layer.MoEBuffers(cfg, training=False)
    y = layer.forward(cfg, inp, bufs)
    assert _abi.moe_read_device_status(bufs.fwd_ws) == 0
    fwd = oracle_forward(inp_cpu, shape.k)
    assert topk_gap(fwd["logits"], shape.k).min() > 1e-4
    assert rel_err(y, fwd["y"]) <= 1e-2
