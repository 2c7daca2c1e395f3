"""moe_route_topk_noalloc: routing for callers that cannot allocate device
memory (a process whose device memory comes from a pool fixed at start-up,
code that must not create allocations while it runs).  It keeps its
intermediates in a static device array inside the library instead of a
caller workspace, and must return exactly what moe_route_topk returns.

Two calls in a row with different shapes and inputs check that what the
shared static array keeps from the previous call does not leak into the next.
"""
import pytest
import torch

from moe_layer_gb300 import _abi, layer
from synth.inputs import MoEShape, make_inputs, random_logits

from .helpers import ensure_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ensure_lib()


def _outputs(T, E, k):
    dev = "cuda"
    return dict(
        logits=torch.full((T, E), float("nan"), dtype=torch.float32, device=dev),
        topk_idx=torch.full((T, k), -7, dtype=torch.int32, device=dev),
        topk_w=torch.full((T, k), float("nan"), dtype=torch.float32, device=dev),
        counts=torch.full((E,), -7, dtype=torch.int32, device=dev),
        offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        perm_token=torch.full((T * k,), -7, dtype=torch.int32, device=dev),
        route_row=torch.full((T, k), -7, dtype=torch.int32, device=dev),
    )


def _route(noalloc, cfg, x, w_router, bias, logits_in, T, E, k):
    o = _outputs(T, E, k)
    args = (cfg, x, w_router, bias, logits_in, o["logits"] if logits_in is None else None,
            o["topk_idx"], o["topk_w"], o["counts"], o["offsets"], o["perm_token"], o["route_row"])
    if noalloc:
        _abi.moe_route_topk_noalloc(*args)
    else:
        bufs = layer.MoEBuffers(cfg, training=False)
        _abi.moe_route_topk(*args, bufs.fwd_ws)
        o["_bufs"] = bufs
    torch.cuda.synchronize()
    if not noalloc:
        assert _abi.moe_read_device_status(o.pop("_bufs").fwd_ws) == 0
    return o


def _compare(a, b, with_logits):
    """Both calls run the same kernels on the same inputs: every output,
    weights and logits included, is bitwise the same."""
    for key in ["topk_idx", "topk_w", "counts", "offsets", "perm_token", "route_row"]:
        assert torch.equal(a[key], b[key]), key
    if with_logits:
        assert torch.equal(a["logits"], b["logits"])


def test_noalloc_routing_matches_workspace_routing_on_two_calls_in_a_row():
    # call 1: logits computed from x and W_router (with a router bias)
    s1 = MoEShape(T=1000, d=256, I=64, E=64, k=8, n_shared=0, I_shared=0, zipf=True)
    inp = {k: (v.cuda() if v is not None else None) for k, v in make_inputs(s1, seed=4, with_dy=False).items()}
    cfg1 = _abi.make_config(s1.T, s1.d, s1.I, s1.E, s1.k)
    ref1 = _route(False, cfg1, inp["x"], inp["W_router"], inp["router_bias"], None, s1.T, s1.E, s1.k)
    got1 = _route(True, cfg1, inp["x"], inp["W_router"], inp["router_bias"], None, s1.T, s1.E, s1.k)
    _compare(got1, ref1, with_logits=True)

    # call 2: a different shape, routing given logits with many ties
    T2, E2, k2 = 513, 256, 8
    logits = random_logits(T2, E2, seed=11, ties=True).cuda()
    cfg2 = _abi.make_config(T2, 64, 64, E2, k2)
    ref2 = _route(False, cfg2, None, None, None, logits, T2, E2, k2)
    got2 = _route(True, cfg2, None, None, None, logits, T2, E2, k2)
    _compare(got2, ref2, with_logits=False)


def test_noalloc_takes_the_documented_largest_shape():
    """65536 tokens at top-8 with 256 experts fit in the static array."""
    T, E, k = 65536, 256, 8
    logits = random_logits(T, E, seed=12).cuda()
    cfg = _abi.make_config(T, 64, 64, E, k)
    _compare(_route(True, cfg, None, None, None, logits, T, E, k),
             _route(False, cfg, None, None, None, logits, T, E, k), with_logits=False)


@pytest.mark.parametrize("T", [73728, 1 << 20])
def test_noalloc_rejects_shapes_beyond_its_static_scratch(T):
    E, k = 256, 8  # intermediates larger than the static array
    cfg = _abi.make_config(T, 64, 64, E, k)
    i32 = lambda: torch.empty(1, dtype=torch.int32, device="cuda")
    f32 = lambda: torch.empty(1, dtype=torch.float32, device="cuda")
    with pytest.raises(_abi.MoeError) as e:
        _abi.moe_route_topk_noalloc(cfg, None, None, None, f32(), None, i32(), f32(), i32(), i32(), i32(), i32())
    assert e.value.code == 2  # MOE_ERR_UNSUPPORTED, returned before anything is launched


def test_noalloc_rejects_configs_the_workspace_routing_rejects():
    i32 = lambda: torch.empty(1, dtype=torch.int32, device="cuda")
    f32 = lambda: torch.empty(1, dtype=torch.float32, device="cuda")
    for cfg, code in ((_abi.make_config(64, 64, 64, 8, 2, n_shared=1, I_shared=0), 1),
                      (_abi.make_config(64, 64, 96, 8, 2), 2),
                      (_abi.make_config(64, 64, 64, 8, 2, flags=_abi.MOE_FLAG_REPLAY), 2)):
        with pytest.raises(_abi.MoeError) as e:
            _abi.moe_route_topk_noalloc(cfg, None, None, None, f32(), None, i32(), f32(), i32(), i32(), i32(), i32())
        assert e.value.code == code
