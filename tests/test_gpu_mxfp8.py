"""MXFP8 mode on the GPU vs the oracle's MXFP8 emulation.

Quantization of bf16 inputs is an exact decision taken the same way on both
sides (power-of-two scales, round to nearest even), so codes and scales must
match bit for bit."""
import numpy as np
import pytest
import torch

from moe_layer_gb300 import _abi, layer
from oracle import moe_oracle as O

from synth.inputs import MoEShape, make_inputs

from .helpers import ensure_lib, f64, oracle_backward, oracle_forward, order_gap, rel_err, topk_gap

pytestmark = pytest.mark.gpu
# MXFP8 outputs vs the oracle's MXFP8 emulation: max|err| / max|ref|
TOL_MX = 5e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ensure_lib()


def unpack_sf(sf, R, K):
    """[R, K/32] E8M0 codes from the 512-byte tcgen05.cp block layout."""
    sf = np.asarray(sf, np.uint8)
    r = np.arange(R)[:, None]
    b = np.arange(K // 32)[None, :]
    g, j = b // 4, b % 4
    off = (g * (R // 128) + r // 128) * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + j
    return sf[off]


def _mx_buffers(cfg, E, I, d, mx):
    """Views of the MXFP8 weight buffer (offsets as documented in moe.h)."""
    def al(x):
        return (x + 255) // 256 * 256
    sizes = [(E * I, d), (E * I, d), (E * d, I), (E * I, d), (E * d, 2 * I)]
    out, off = [], 0
    for R, K in sizes:
        q = mx[off:off + R * K].view(R, K)
        off = al(off + R * K)
        nsf = (R // 128) * (K // 128) * 512
        sf = mx[off:off + nsf]
        off = al(off + nsf + 512)  # one spare scale block
        out.append((q, sf, R, K))
    return out


def test_weight_quantization_bit_exact():
    E, I, d = 3, 256, 384
    g = torch.Generator().manual_seed(0)
    scale = torch.exp(torch.randn(E, 1, 1, generator=g) * 2)
    Wg = (torch.randn(E, I, d, generator=g) * 0.02 * scale).to(torch.bfloat16)
    Wu = (torch.randn(E, I, d, generator=g) * 0.02).to(torch.bfloat16)
    Wd = (torch.randn(E, d, I, generator=g) * 0.02).to(torch.bfloat16)
    Wg[1, 5, 32:64] = 0  # an all-zero block
    Wu[2, 7, :] = 1e-30  # subnormal-range values
    cfg = _abi.make_config(128, d, I, E, 2, precision=_abi.MOE_MXFP8)
    mx = torch.zeros(_abi.moe_mxfp8_weights_size(cfg), dtype=torch.uint8, device="cuda")
    w = _abi.make_weights(None, Wg.cuda(), Wu.cuda(), Wd.cuda())
    _abi.moe_quantize_weights_mxfp8(cfg, w, mx)
    torch.cuda.synchronize()
    bufs = _mx_buffers(cfg, E, I, d, mx)
    refs = [
        np.concatenate([f64(Wg[e]) for e in range(E)]),
        np.concatenate([f64(Wu[e]) for e in range(E)]),
        np.concatenate([f64(Wd[e]) for e in range(E)]),
        np.concatenate([f64(Wd[e]).T for e in range(E)]),
        np.concatenate([np.concatenate([f64(Wg[e]), f64(Wu[e])]).T for e in range(E)]),
    ]
    for (q, sf, R, K), ref, name in zip(bufs, refs, ["wg", "wu", "wd", "wd^T", "[wg;wu]^T"]):
        codes, sc = O.mx_quantize(ref, axis=-1)
        got_q = q.cpu().numpy()
        got_sc = unpack_sf(sf.cpu().numpy(), R, K)
        assert (got_sc == sc).all(), name
        # +0 and -0 encode the same value
        same = (got_q == codes) | ((got_q & 0x7F) == 0) & ((codes & 0x7F) == 0)
        assert same.all(), (name, np.argwhere(~same)[:5])


MX_SHAPES = {
    "mx_small": MoEShape(T=512, d=256, I=256, E=8, k=2, n_shared=1, I_shared=128, w_std=0.05),
    # d % 256 == 128: the last n-tile of every B operand has a 128-row second half
    "mx_ragged": MoEShape(T=333, d=384, I=128, E=5, k=3, n_shared=0, I_shared=0, w_std=0.05),
    "mx_zipf_zero": MoEShape(T=640, d=256, I=384, E=32, k=4, n_shared=1, I_shared=128, w_std=0.05,
                             zipf=True, zero_experts=8),
    # 603-690 rows per expert: four experts with an even number of 128-row tiles (their GEMM
    # tiles run on SM pairs) and four with an odd number (one SM per tile); d % 256 == 128
    "mx_pairs_leftover": MoEShape(T=2560, d=384, I=256, E=8, k=2, n_shared=1, I_shared=128, w_std=0.05),
    # model shapes of the MoK blog ("Speedups"), scaled down with E, top-k and d:I kept
    "mx_qwen35_scaled": MoEShape(T=256, d=512, I=128, E=512, k=10, n_shared=1, I_shared=128, w_std=0.05,
                                 wr_std=0.1),
    "mx_dsv4pro_scaled": MoEShape(T=256, d=896, I=384, E=384, k=6, n_shared=1, I_shared=384, w_std=0.03,
                                  wr_std=0.1),
}
MX_SEEDS = {"mx_qwen35_scaled": 2, "mx_pairs_leftover": 1}


def _cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _run_mx(shape, seed=0, backward=True, flags=0):
    inp_cpu = make_inputs(shape, seed=seed, with_dy=backward)
    inp = _cuda(inp_cpu)
    cfg = _abi.make_config(shape.T, shape.d, shape.I, shape.E, shape.k, shape.n_shared, shape.I_shared,
                           precision=_abi.MOE_MXFP8, flags=flags)
    layer.quantize_weights(cfg, inp)
    bufs = layer.MoEBuffers(cfg, training=backward)
    y = layer.forward(cfg, inp, bufs)
    res = {"y": y, "inp_cpu": inp_cpu}
    if backward:
        grads = layer.alloc_grads(cfg)
        dx = layer.backward(cfg, inp, inp["dy"], bufs, grads)
        res.update(dx=dx, grads=grads)
    torch.cuda.synchronize()
    assert _abi.moe_read_device_status(bufs.fwd_ws) == 0
    if backward:
        assert _abi.moe_read_device_status(bufs.bwd_ws) == 0
    return res


@pytest.mark.parametrize("name,flags", [(n, 0) for n in MX_SHAPES] + [("mx_zipf_zero", "replay")])
def test_mxfp8_forward_backward_parity(name, flags):
    """Forward and backward in MXFP8 mode vs the oracle's MXFP8 emulation
    (every operand of the routed experts' GEMMs rounded through MXFP8 along
    its reduction axis), and measurably farther from the full-precision
    oracle: the kernels do quantize.  Also with forward activation replay."""
    shape = MX_SHAPES[name]
    r = _run_mx(shape, seed=MX_SEEDS.get(name, 0), flags=_abi.MOE_FLAG_REPLAY if flags == "replay" else 0)
    inp = r["inp_cpu"]
    fwd = oracle_forward(inp, shape.k, mxfp8=True)
    assert topk_gap(fwd["logits"], shape.k).min() > 1e-4, "seeded input has a near-tie"
    assert order_gap(fwd["logits"], shape.k).min() > 1e-5
    bwd = oracle_backward(inp, fwd)
    e_y = rel_err(r["y"], fwd["y"])
    assert e_y <= TOL_MX, e_y
    assert rel_err(r["dx"], bwd["dx"]) <= TOL_MX
    g = r["grads"]
    for key in ["dW_gate", "dW_up", "dW_down", "dW_router", "d_topk_w"]:
        assert rel_err(g[key], bwd[key]) <= TOL_MX, key
    if shape.n_shared:
        for key in ["dWs_gate", "dWs_up", "dWs_down"]:
            assert rel_err(g[key], bwd[key]) <= TOL_MX, key
    if shape.zero_experts:
        for e in range(shape.E - shape.zero_experts, shape.E):
            assert fwd["counts"][e] == 0
            for key in ["dW_gate", "dW_up", "dW_down", "dW_router"]:
                assert (g[key][e] == 0).all(), (key, e)
    full = oracle_forward(inp, shape.k, mxfp8=False)
    assert e_y < 0.5 * rel_err(r["y"], full["y"])


def test_mxfp8_inference_matches_training_forward_and_is_deterministic(monkeypatch):
    shape = MX_SHAPES["mx_ragged"]
    a = _run_mx(shape, seed=4, backward=False)
    b = _run_mx(shape, seed=4, backward=True)
    assert torch.equal(a["y"], b["y"])
    monkeypatch.setenv("MOE_GRID_LIMIT", "3")
    c = _run_mx(shape, seed=4, backward=True)
    assert torch.equal(b["y"], c["y"])
    assert torch.equal(b["dx"], c["dx"])
    for key in b["grads"]:
        if b["grads"][key] is not None:
            assert torch.equal(b["grads"][key], c["grads"][key]), key


def test_mxfp8_replay_matches_saved_activations_bitwise():
    shape = MX_SHAPES["mx_zipf_zero"]
    a = _run_mx(shape, seed=1)
    b = _run_mx(shape, seed=1, flags=_abi.MOE_FLAG_REPLAY)
    assert torch.equal(a["y"], b["y"])
    assert torch.equal(a["dx"], b["dx"])
    for key in a["grads"]:
        if a["grads"][key] is not None:
            assert torch.equal(a["grads"][key], b["grads"][key]), key


def test_mxfp8_forward_requires_quantized_weights():
    shape = MX_SHAPES["mx_small"]
    inp = _cuda(make_inputs(shape, seed=0, with_dy=False))
    cfg = _abi.make_config(shape.T, shape.d, shape.I, shape.E, shape.k, shape.n_shared, shape.I_shared,
                           precision=_abi.MOE_MXFP8)
    bufs = layer.MoEBuffers(cfg, training=False)
    with pytest.raises(_abi.MoeError) as ei:
        layer.forward(cfg, inp, bufs)
    assert ei.value.code == 1


@pytest.mark.parametrize("name", ["mx_small", "mx_ragged", "mx_zipf_zero", "mx_qwen35_scaled"])
def test_stateless_forward_equals_training_forward_bitwise(name):
    """A forward that keeps no state quantizes the dispatched rows with its own
    kernel (a scatter of the token rows) instead of the gather that also
    writes the transposed copy for the weight gradients: the codes and scales
    are the same, so y is bitwise the training forward's (which the other
    tests check against the oracle)."""
    shape = MX_SHAPES[name]
    inp = _cuda(make_inputs(shape, seed=MX_SEEDS.get(name, 0), with_dy=False))
    cfg = _abi.make_config(shape.T, shape.d, shape.I, shape.E, shape.k, shape.n_shared, shape.I_shared,
                           precision=_abi.MOE_MXFP8)
    layer.quantize_weights(cfg, inp)
    y_train = layer.forward(cfg, inp, layer.MoEBuffers(cfg))
    ibufs = layer.MoEBuffers(cfg, training=False)
    y_inf = layer.forward(cfg, inp, ibufs)
    torch.cuda.synchronize()
    assert _abi.moe_read_device_status(ibufs.fwd_ws) == 0
    assert torch.equal(y_inf, y_train)
