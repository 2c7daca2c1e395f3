"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws random numbers with fixed seeds and shapes; it holds
none of the layer's arithmetic.  Both the CUDA path (tests, bench) and the CPU
oracle's checks take their inputs from here.

Workloads (shapes of the DeepSeek-V3-style layers the Mixture-of-Kittens pages
benchmark; the value distributions are fixed here):

  tiny   T=512,   d=256,  I=128,  E=8,   k=2, one shared expert (I_s=128),
         x ~ N(0,1), every weight ~ N(0, 0.02)
  dsv3   T=16384, d=7168, I=2048, E=256, k=8, one shared expert (I_s=2048),
         x ~ N(0,1), expert and shared weights ~ N(0, 0.006), W_router ~ N(0, 0.02)
  qwen3  T=8192,  d=4096, I=1536, E=128, k=8, no shared expert, same
         distributions as dsv3 plus a per-expert router bias
         b_e = alpha * log(rank_e ** -1.2), rank_e a seeded permutation of 1..E
         (Zipf 1.2 skew, alpha fixed below so expert loads span roughly 10x)
  kimi_k27, glm52, qwen35, dsv4pro
         the open-weight model shapes the Mixture-of-Kittens blog benchmarks
         (E, d, I, top-k): (384, 7168, 2048, 8), (256, 6144, 2048, 8),
         (512, 4096, 1024, 10), (384, 7168, 3072, 6); the blog gives only those
         four numbers, the rest is as dsv3 (T=16384, one shared expert of
         width I, same distributions)
  sweep  dsv3 shapes at T in {512, 2048, 8192, 32768}; optional Zipf bias as
         qwen3; optionally 8 experts (ids E-8..E-1) get bias -inf so they
         receive no tokens
The upstream gradient dy ~ N(0, 1).
"""
from __future__ import annotations

import dataclasses
import math

import torch

# Fixed Zipf bias scale (see module docstring).
ZIPF_ALPHA = 0.35
ZIPF_S = 1.2


@dataclasses.dataclass(frozen=True)
class MoEShape:
    T: int
    d: int
    I: int
    E: int
    k: int
    n_shared: int
    I_shared: int
    w_std: float = 0.02
    wr_std: float = 0.02
    zipf: bool = False
    zero_experts: int = 0

    @property
    def R(self) -> int:
        return self.T * self.k


CONFIGS = {
    "tiny": MoEShape(T=512, d=256, I=128, E=8, k=2, n_shared=1, I_shared=128, w_std=0.02),
    "dsv3": MoEShape(T=16384, d=7168, I=2048, E=256, k=8, n_shared=1, I_shared=2048, w_std=0.006),
    "qwen3": MoEShape(T=8192, d=4096, I=1536, E=128, k=8, n_shared=0, I_shared=0, w_std=0.006, zipf=True),
    "kimi_k27": MoEShape(T=16384, d=7168, I=2048, E=384, k=8, n_shared=1, I_shared=2048, w_std=0.006),
    "glm52": MoEShape(T=16384, d=6144, I=2048, E=256, k=8, n_shared=1, I_shared=2048, w_std=0.006),
    "qwen35": MoEShape(T=16384, d=4096, I=1024, E=512, k=10, n_shared=1, I_shared=1024, w_std=0.006),
    "dsv4pro": MoEShape(T=16384, d=7168, I=3072, E=384, k=6, n_shared=1, I_shared=3072, w_std=0.006),
}


def sweep_shape(T: int, zipf: bool = False, zero_experts: int = 0) -> MoEShape:
    return MoEShape(T=T, d=7168, I=2048, E=256, k=8, n_shared=1, I_shared=2048, w_std=0.006,
                    zipf=zipf, zero_experts=zero_experts)


def _randn(shape, gen, device, std=1.0, dtype=torch.bfloat16):
    t = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _randn_stack(E, rows, cols, gen, device, std):
    """[E, rows, cols] bf16 drawn one expert at a time (bounded temporaries)."""
    out = torch.empty(E, rows, cols, dtype=torch.bfloat16, device=device)
    for e in range(E):
        out[e].copy_(_randn((rows, cols), gen, device, std))
    return out


def router_bias(shape: MoEShape, seed: int = 0):
    """Per-expert fp32 router bias, or None for unbiased routing."""
    if not shape.zipf and shape.zero_experts == 0:
        return None
    gen = torch.Generator(device="cpu").manual_seed(seed + 7919)
    bias = torch.zeros(shape.E, dtype=torch.float32)
    if shape.zipf:
        rank = torch.randperm(shape.E, generator=gen).to(torch.float64) + 1.0
        bias = (ZIPF_ALPHA * (-ZIPF_S) * torch.log(rank)).to(torch.float32)
    if shape.zero_experts:
        bias[shape.E - shape.zero_experts:] = -math.inf
    return bias


def make_inputs(shape: MoEShape, seed: int = 0, device="cpu", with_dy: bool = True):
    """All tensors of one layer call, deterministic in (shape, seed, device type).

    Returns a dict of torch tensors: x [T,d], W_router [E,d], W_gate/W_up
    [E,I,d], W_down [E,d,I], Ws_gate/Ws_up [I_s,d], Ws_down [d,I_s] (bf16),
    router_bias [E] fp32 or None, dy [T,d] bf16.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(seed)
    s = shape
    out = {}
    out["x"] = _randn((s.T, s.d), gen, device)
    out["W_router"] = _randn((s.E, s.d), gen, device, s.wr_std)
    out["W_gate"] = _randn_stack(s.E, s.I, s.d, gen, device, s.w_std)
    out["W_up"] = _randn_stack(s.E, s.I, s.d, gen, device, s.w_std)
    out["W_down"] = _randn_stack(s.E, s.d, s.I, gen, device, s.w_std)
    if s.n_shared:
        out["Ws_gate"] = _randn((s.I_shared, s.d), gen, device, s.w_std)
        out["Ws_up"] = _randn((s.I_shared, s.d), gen, device, s.w_std)
        out["Ws_down"] = _randn((s.d, s.I_shared), gen, device, s.w_std)
    else:
        out["Ws_gate"] = out["Ws_up"] = out["Ws_down"] = None
    b = router_bias(s, seed)
    out["router_bias"] = None if b is None else b.to(device)
    out["dy"] = _randn((s.T, s.d), gen, device) if with_dy else None
    return out


def random_logits(T: int, E: int, seed: int = 0, ties: bool = False):
    """fp32 logits [T,E] for routing-only tests.  With ties=True the values are
    drawn from a coarse grid so that equal logits occur often."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    if ties:
        return (torch.randint(-3, 4, (T, E), generator=gen).to(torch.float32) * 0.5)
    return torch.randn(T, E, generator=gen, dtype=torch.float32) * 2.0
