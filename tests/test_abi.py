"""The C-ABI library loads and exports every entry point include/moe.h
declares; host-only calls (sizes, argument checks) behave.  No GPU needed."""
import ctypes
import os
import re

import pytest

from moe_layer_gb300 import _abi, build_ext

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_ext.build()
    return _abi.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(moe_\w+)\s*\(", text, re.M)))


def test_header_declares_expected_api():
    syms = declared_symbols()
    for name in ["moe_workspace_size", "moe_route_topk", "moe_forward", "moe_backward",
                 "moe_read_device_status", "moe_status_string"]:
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert _abi.status_string(0) == "ok"
    assert "unsupported" in _abi.status_string(2)


def test_workspace_sizes_scale_with_shape(lib):
    small = _abi.moe_workspace_size(_abi.make_config(512, 256, 128, 8, 2, 1, 128))
    big = _abi.moe_workspace_size(_abi.make_config(16384, 7168, 2048, 256, 8, 1, 2048))
    assert all(s > 0 for s in small) and all(b > s for b, s in zip(big, small))
    # saved state holds at least a and b for every (padded) route row
    assert big[1] >= 16384 * 8 * 2 * 2048 * 2


def test_replay_flag_moves_the_activations_from_saved_to_the_backward_workspace(lib):
    """MOE_FLAG_REPLAY moves the routed experts' x rows, a and b out of the
    saved state into the backward workspace; the shared expert's a and b (T
    rows) stay saved."""
    T, d, I, E, k, Is = 4096, 1024, 512, 64, 6, 256
    base = _abi.moe_workspace_size(_abi.make_config(T, d, I, E, k, 1, Is))
    rep = _abi.moe_workspace_size(_abi.make_config(T, d, I, E, k, 1, Is, flags=_abi.MOE_FLAG_REPLAY))
    Rp = T * k + E * 63  # routes padded to 64 rows per expert (bf16 mode)
    acts = Rp * (2 * d + 4 * I)  # x rows, a and b of the routed experts
    slack = 4 * 256  # 256-byte alignment of each buffer
    assert rep[0] == base[0]
    assert abs((base[1] - rep[1]) - acts) <= slack
    assert abs((rep[2] - base[2]) - acts) <= slack
    # the routing (a few ints per route and per expert) and the shared expert's a and b
    assert 4 * T * Is <= rep[1] < 64 * T * k + 4 * T * Is


def test_unknown_flag_bits_rejected(lib):
    a = ctypes.c_size_t()
    for bit in (4, 1 << 31):  # bits 0 and 1 are MOE_FLAG_REPLAY and MOE_FLAG_WGRAD_FP32
        c = _abi.make_config(512, 256, 128, 8, 2, flags=bit)
        assert lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(a), None, None) == 2


@pytest.mark.parametrize("cfg,code", [
    ((512, 100, 128, 8, 2, 0, 0), 2),     # d not a multiple of 64
    ((512, 256, 96, 8, 2, 0, 0), 2),      # I not a multiple of 64
    ((512, 256, 128, 8, 9, 0, 0), 2),     # top_k > E
    ((512, 256, 128, 600, 2, 0, 0), 2),   # E > 512
    ((512, 256, 128, 64, 33, 0, 0), 2),   # top_k > 32
    ((-1, 256, 128, 8, 2, 0, 0), 1),      # negative T
    ((512, 256, 128, 8, 2, 1, 0), 1),     # shared expert without width
])
def test_invalid_configs_rejected(lib, cfg, code):
    c = _abi.make_config(*cfg)
    a = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(a), None, None) == code


def test_mxfp8_needs_dims_multiple_of_128(lib):
    a = ctypes.c_size_t()
    bad = _abi.make_config(512, 256, 192, 8, 2, precision=_abi.MOE_MXFP8)
    assert lib.moe_workspace_size(ctypes.byref(bad), ctypes.byref(a), None, None) == 2
    good = _abi.make_config(512, 256, 128, 8, 2, precision=_abi.MOE_MXFP8)
    assert lib.moe_workspace_size(ctypes.byref(good), ctypes.byref(a), None, None) == 0
    assert _abi.moe_mxfp8_weights_size(good) >= 3 * 8 * 128 * 256 * 2  # five fp8 weight copies


def test_null_arguments_rejected_before_launch(lib):
    c = _abi.make_config(64, 128, 64, 4, 2)
    w = _abi.MoeWeights()
    # no workspace
    assert lib.moe_forward(ctypes.byref(c), None, ctypes.byref(w), None, None, None, None) == 3
    # workspace given but weights missing: invalid argument, nothing launched
    assert lib.moe_forward(ctypes.byref(c), None, ctypes.byref(w), None, None, 256, None) == 1


def test_misaligned_workspace_or_saved_state_rejected(lib):
    """moe.h: the workspaces and the saved state are 256-byte aligned (their
    sub-buffers take 32-byte vector accesses); a misaligned one is an invalid
    argument, rejected before anything is launched (the placeholder addresses
    are never dereferenced)."""
    c = _abi.make_config(64, 128, 64, 4, 2)
    fake = 1 << 20
    w = _abi.MoeWeights(fake, 0, fake, fake, fake, 0, 0, 0, None)
    assert lib.moe_forward(ctypes.byref(c), fake, ctypes.byref(w), fake, None, fake + 16, None) == 1
    assert lib.moe_forward(ctypes.byref(c), fake, ctypes.byref(w), fake, fake + 32, fake, None) == 1
    i32 = ctypes.c_void_p(fake)
    assert lib.moe_route_topk(ctypes.byref(c), fake, fake, None, None, None, i32, i32, i32, i32, i32, i32,
                              fake + 128, None) == 1
    g = _abi.MoeGrads(fake, fake, fake, fake, 0, 0, 0, None, None)
    assert lib.moe_backward(ctypes.byref(c), fake, ctypes.byref(w), fake, fake + 64, fake, ctypes.byref(g),
                            fake, None) == 1


def test_fp32_weight_gradient_flag(lib):
    """moe.h: MOE_FLAG_WGRAD_FP32 is a bf16-mode option (MXFP8 gives MOE_ERR_UNSUPPORTED);
    gradient buffers, like every pointer, must be 16-byte aligned, checked before any launch
    (the placeholder addresses are never dereferenced)."""
    sz = ctypes.c_size_t()
    c = _abi.make_config(64, 128, 64, 4, 2, flags=_abi.MOE_FLAG_WGRAD_FP32)
    assert lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(sz), None, None) == 0
    m = _abi.make_config(64, 128, 128, 4, 2, precision=_abi.MOE_MXFP8, flags=_abi.MOE_FLAG_WGRAD_FP32)
    assert lib.moe_workspace_size(ctypes.byref(m), ctypes.byref(sz), None, None) == 2
    fake = 1 << 20
    w = _abi.MoeWeights(fake, 0, fake, fake, fake, 0, 0, 0, None)
    g = _abi.MoeGrads(fake, fake + 8, fake, fake, 0, 0, 0, None, None)
    assert lib.moe_backward(ctypes.byref(c), fake, ctypes.byref(w), fake, fake, fake, ctypes.byref(g),
                            fake, None) == 1


def test_empty_batch_is_a_no_op(lib):
    c = _abi.make_config(0, 128, 64, 4, 2)
    w = _abi.MoeWeights()
    assert lib.moe_forward(ctypes.byref(c), None, ctypes.byref(w), None, None, 256, None) == 0


def test_package_imports_without_gpu():
    import moe_layer_gb300
    assert moe_layer_gb300.moe_forward is _abi.moe_forward


def test_mxfp8_weight_buffer_size_matches_documented_layout(lib):
    """moe.h: W_gate and W_up [E*I, d], W_down [E*d, I], W_down^T [E*I, d] and
    [W_gate; W_up]^T [E*d, 2I], each followed by its scales (R/128 x K/128
    blocks of 512 bytes) and one spare block, every piece 256-byte aligned."""
    E, d, I = 5, 384, 256
    cfg = _abi.make_config(300, d, I, E, 2, precision=_abi.MOE_MXFP8)
    al = lambda x: (x + 255) // 256 * 256
    off = 0
    for R, K in ((E * I, d), (E * I, d), (E * d, I), (E * I, d), (E * d, 2 * I)):
        off = al(off) + R * K
        off = al(off) + (R // 128) * (K // 128) * 512 + 512
    assert _abi.moe_mxfp8_weights_size(cfg) == off
    # bf16 configurations have no such buffer
    assert lib.moe_mxfp8_weights_size(ctypes.byref(_abi.make_config(300, d, I, E, 2)),
                                      ctypes.byref(ctypes.c_size_t())) == 2


def test_mxfp8_forward_needs_the_quantized_weights(lib):
    """MXFP8 mode rejects a missing or misaligned pre-quantized weight buffer
    before launching anything (the pointers below are never dereferenced)."""
    c = _abi.make_config(64, 128, 128, 4, 2, precision=_abi.MOE_MXFP8)
    fake = 1 << 20  # 256-byte aligned placeholder address
    w = _abi.MoeWeights(fake, 0, fake, fake, fake, 0, 0, 0, None)
    assert lib.moe_forward(ctypes.byref(c), fake, ctypes.byref(w), fake, None, fake, None) == 1
    w.mxfp8 = fake + 16  # not 256-byte aligned
    assert lib.moe_forward(ctypes.byref(c), fake, ctypes.byref(w), fake, None, fake, None) == 1
