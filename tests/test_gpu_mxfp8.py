"""MXFP8 mode on the GPU vs the oracle's MXFP8 emulation.

Quantization of bf16 inputs is an exact decision taken the same way on both
sides (power-of-two scales, round to nearest even), so codes and scales must
match bit for bit."""
import numpy as np
import pytest
import torch

from moe_layer_gb300 import _abi, layer
from oracle import moe_oracle as O

from .helpers import ensure_lib, f64

pytestmark = pytest.mark.gpu


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
        off = al(off + nsf)
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
