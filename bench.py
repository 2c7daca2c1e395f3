"""Benchmark of the MoE layer hot path (forward + backward) through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload dsv3|qwen3|tiny|dsv3_mxfp8|kimi_k27|glm52|qwen35|dsv4pro]

One step = forward + backward of the whole layer on one batch of seeded
synthetic input of the workload (default: the DeepSeek-V3-shaped layer,
T=16384 tokens, d=7168, I=2048, E=256 routed experts, top-8, one shared
expert).  Inputs and weights are resident in HBM before the timed region;
they are larger than L2 (x 235 MB, expert weights 22.6 GB), so no L2 flush is
done between steps.  With N > 1 (torchrun) every rank runs an independent
replica on its own tokens (weak scaling, no collective on the data path);
the timed region is bracketed by barriers and the slowest rank's time counts.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead
(bounded sample per step) and prints the same metric with "impl": "reference".

dsv3_mxfp8 runs the same layer with the routed experts in MXFP8.  Its weights
are quantized once per weight update (moe_quantize_weights_mxfp8); that pass is
timed on its own and reported as "weight_quant", together with the throughput
of a step that includes it.  Its tensor peak is measured in the same run
(measure_mxfp8_peak).

With the default workload the line also carries, under "workloads", the
DSV3-shaped MXFP8 layer and the Qwen3-235B-shaped layer (Zipf routing), each
timed the same way after the headline's buffers are freed (--no-extra skips
them); the headline value stays the DSV3 BF16 one.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s and TFLOPS (fwd, fwd+bwd) at 1 GB300, % of tensor peak"


# Nominal dense FP8 (and MXFP8) / BF16 tensor rate ratio (4.5 vs 2.25 PFLOP/s):
# the fallback when no block-scaled FP8 GEMM can be timed on the device.
FP8_OVER_BF16 = 2.0


def measure_mxfp8_peak(n=8192, sustain_s=4.0):
    """Tensor peak for the MXFP8 GEMMs, measured on this device the way the
    bf16 denominators are: a library GEMM of n^3 (2 n^3 flops) on E4M3 operands
    with E8M0 scales per 32 elements along K (torch._scaled_mm, cuBLASLt),
    best of 10 timed singly (burst) and back to back for sustain_s seconds
    (sustained).  Falls back to per-tensor-scaled E4M3 (the same tensor rate)
    where the block-scaled form is not available.  Returns a dict, or None."""
    import torch
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(0)
    a = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn).t()  # column-major [K, N]
    nsf = ((n + 127) // 128 * 128) * ((n // 32 + 3) // 4 * 4)
    forms = []
    if hasattr(torch, "float8_e8m0fnu"):
        sf = torch.full((nsf,), 127, dtype=torch.uint8, device=dev).view(torch.float8_e8m0fnu)
        forms.append(("mxfp8 (e4m3, e8m0 scales per 32 along K)", sf, sf))
    one = torch.ones((), dtype=torch.float32, device=dev)
    forms.append(("fp8 e4m3, per-tensor scale", one, one))
    for label, sa, sb in forms:
        try:
            fn = lambda: torch._scaled_mm(a, b, sa, sb, out_dtype=torch.bfloat16)
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
        except Exception:
            continue
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        reps, t_total = 0, 0.0
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        per = max(1, int(sustain_s * 1e3 / max(best, 1e-3) / 4))
        t0 = time.perf_counter()
        e0.record()
        while time.perf_counter() - t0 < sustain_s:
            for _ in range(per):
                fn()
            reps += per
            torch.cuda.synchronize()
        e1.record()
        torch.cuda.synchronize()
        t_total = e0.elapsed_time(e1)
        fl = 2.0 * n ** 3
        return {"form": label, "tflops": fl / (best * 1e-3) / 1e12,
                "tflops_sustained": fl * reps / (t_total * 1e-3) / 1e12,
                "how": f"torch._scaled_mm {n}^3 (2 n^3 flops), bf16 out: best of 10 (burst) and "
                       f"{reps} back to back in {t_total / 1e3:.1f} s (sustained)"}
    return None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm": p["hbm_gbs"], "bf16": p["bf16_tflops"],
                "bf16_sustained": p["bf16_tflops_sustained"], "src": "measured"}
    except Exception:
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "fallback"}


def _tensor_peaks(peaks, mxfp8, mx_peak=None):
    """(burst, sustained, label) tensor peaks for the routed GEMMs' dtype."""
    if not mxfp8:
        return peaks["bf16"], peaks["bf16_sustained"], peaks["src"] + " bf16"
    if mx_peak:
        return (mx_peak["tflops"], mx_peak["tflops_sustained"],
                f"measured in this run: {mx_peak['form']}, {mx_peak['how']}")
    return (peaks["bf16"] * FP8_OVER_BF16, peaks["bf16_sustained"] * FP8_OVER_BF16,
            peaks["src"] + f" bf16 x nominal mxfp8/bf16 ratio {FP8_OVER_BF16:g}")


def _workload(name, tokens=0, experts=0, zipf=False, zero_experts=0):
    """(shape, description, mxfp8) of a named workload."""
    import dataclasses

    from synth.inputs import CONFIGS
    s = CONFIGS["dsv3" if name == "dsv3_mxfp8" else name]
    desc = {
        "dsv3": "DSV3-shaped BF16 MoE layer forward+backward",
        "qwen3": "Qwen3-235B-shaped BF16 MoE layer forward+backward (Zipf-skewed routing)",
        "tiny": "tiny BF16 MoE layer forward+backward",
        "dsv3_mxfp8": "DSV3-shaped MXFP8 MoE layer forward+backward (routed experts MXFP8, "
                      "router and shared expert BF16, BF16 outputs)",
        "kimi_k27": "Kimi-K2.7-shaped BF16 MoE layer forward+backward (E=384, d=7168, I=2048, top-8)",
        "glm52": "GLM-5.2-shaped BF16 MoE layer forward+backward (E=256, d=6144, I=2048, top-8)",
        "qwen35": "Qwen3.5-397B-A17B-shaped BF16 MoE layer forward+backward (E=512, d=4096, I=1024, top-10)",
        "dsv4pro": "DeepSeek-V4-Pro-shaped BF16 MoE layer forward+backward (E=384, d=7168, I=3072, top-6)",
    }[name]
    if tokens or experts:  # scaled variant (token sweep, profiling captures)
        s = dataclasses.replace(s, T=tokens or s.T, E=experts or s.E)
        desc += f" (scaled: T={s.T}, E={s.E})"
    if zipf or zero_experts:  # the granularity sweep's skewed routing
        s = dataclasses.replace(s, zipf=zipf or s.zipf, zero_experts=zero_experts)
        desc += f" (Zipf {1.2 if s.zipf else 0} router bias, {zero_experts} experts never chosen)"
    return s, desc, name == "dsv3_mxfp8"


def _flops(s):
    """Algorithmic flops per token of the forward pass (backward = 2x)."""
    return 6 * s.d * s.I * s.k + 6 * s.d * s.I_shared * s.n_shared + 2 * s.d * s.E


def _kernel_flops(name, s):
    """Algorithmic flops of one launch of a tensor-core kernel."""
    R, T, d, I, Is, E = s.T * s.k, s.T, s.d, s.I, s.I_shared, s.E
    table = {
        "router_gemm": 2 * T * d * E,
        "gateup_routed": 4 * R * d * I, "down_routed": 2 * R * d * I,
        "dgrad_down_routed": 2 * R * d * I, "dgrad_gateup_routed": 4 * R * d * I,
        "wgrad_down": 2 * R * d * I, "wgrad_gate": 2 * R * d * I, "wgrad_up": 2 * R * d * I,
        "gateup_shared": 4 * T * d * Is, "down_shared": 2 * T * d * Is,
        "dgrad_down_shared": 2 * T * d * Is, "dgrad_gateup_shared": 4 * T * d * Is,
        "wgrad_shared_down": 2 * T * d * Is, "wgrad_shared_gate": 2 * T * d * Is,
        "wgrad_shared_up": 2 * T * d * Is,
    }
    return table.get(name)


# DRAM bytes per launch (read + write) of the dominant kernel, measured with
# ncu (dram__bytes_read.sum + dram__bytes_write.sum, one pass over the full
# workload, first timed step; summed over the kernels of the step).  An entry
# must be removed or re-measured when its kernel changes.
NCU_TRAFFIC = {
    # the 2-SM pass (even experts) and the 1-SM pass (odd experts), summed
    # (profiles/launches_dsv3_fwd_bwd.md, profiles/launches_dsv3_mxfp8_fwd_bwd.md)
    ("dsv3", "gateup_routed"): 8.937e9 + 0.804e9 + 9.243e9 + 0.881e9,
    ("dsv3_mxfp8", "gateup_routed"): 4.542e9 + 0.669e9 + 4.542e9 + 0.813e9,
}


class _Ranks:
    """The replicas' only cross-rank steps: a barrier around each timed region
    and the slowest rank's time (the job's time).  `device` holds the reduced
    value: "cuda" with NCCL, "cpu" with gloo."""

    def __init__(self, world, device):
        self.world, self.device = world, device

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max(self, v):
        if self.world == 1:
            return v
        import torch
        import torch.distributed as dist
        t = torch.tensor([v], dtype=torch.float64, device=self.device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        try:
            sm = [float(r[1]) for r in rows]
            smax = max(float(r[2]) for r in rows)
        except ValueError:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows)}


def _lazy_experts(t):
    import numpy as np
    import torch

    class Lazy:
        def __init__(self):
            self.cache = {}

        def __len__(self):
            return t.shape[0]

        def __getitem__(self, e):
            e = int(e)
            if e not in self.cache:
                self.cache[e] = t[e].to(torch.float64).cpu().numpy()
            return self.cache[e]
    return Lazy()


def _oracle_step(inp, s, tokens, mxfp8=False):
    """The CPU oracle's forward + backward on a token sample (test infrastructure,
    used only for the reported CPU baseline)."""
    import torch
    from oracle import moe_oracle as O
    f = lambda t: t.to(torch.float64).cpu().numpy()
    x = f(inp["x"][tokens])
    dy = f(inp["dy"][tokens])
    wr = f(inp["W_router"])
    bias = None if inp.get("router_bias") is None else f(inp["router_bias"])
    wg, wu, wd = _lazy_experts(inp["W_gate"]), _lazy_experts(inp["W_up"]), _lazy_experts(inp["W_down"])
    sh = {}
    if s.n_shared:
        sh = dict(ws_gate=f(inp["Ws_gate"]), ws_up=f(inp["Ws_up"]), ws_down=f(inp["Ws_down"]))
    fwd = O.moe_forward(x, wr, wg, wu, wd, s.k, router_bias=bias, mxfp8=mxfp8, **sh)
    O.moe_backward(x, wr, wg, wu, wd, dy, fwd, dense_expert_grads=False, **sh)


def _cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def cpu_baseline(inp, s, n_tokens, rounds, seed=1, mxfp8=False):
    """Oracle forward+backward on `rounds` independent random samples of
    `n_tokens` tokens each (each round upcasts only the experts its tokens
    touch, which bounds host memory)."""
    import torch
    g = torch.Generator().manual_seed(seed)
    dt = 0.0
    for _ in range(rounds):
        tokens = torch.randperm(s.T, generator=g)[:n_tokens].sort().values.to(inp["x"].device)
        t0 = time.perf_counter()
        _oracle_step(inp, s, tokens, mxfp8)
        dt += time.perf_counter() - t0
    n = n_tokens * rounds
    return {"value": n / dt, "unit": "tokens/s", "cores": _cpu_cores(), "cpu": _cpu_model(), "kind": "oracle",
            "extrapolated": True,
            "sample": f"float64 numpy oracle forward+backward{' (MXFP8 emulation)' if mxfp8 else ''}, "
                      f"{rounds} rounds of {n_tokens} random tokens "
                      f"of the same workload ({n} tokens, expert weights upcast on first use per round), "
                      f"{dt:.1f} s; tokens/s extrapolated linearly from that sample (per-token cost); "
                      f"numpy BLAS default threading"}


def run_reference(args):
    """The CPU oracle timed on the host cores, each step a bounded sample."""
    import torch
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from synth.inputs import make_inputs
    s, desc, mx = _workload(args.workload, args.tokens, args.experts, args.zipf, args.zero_experts)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = make_inputs(s, seed=0, device=dev)
    per_step = args.ref_tokens
    g = torch.Generator().manual_seed(1)
    for _ in range(args.warmup):
        _oracle_step(inp, s, torch.randperm(s.T, generator=g)[:per_step].sort().values.to(dev), mx)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(inp, s, torch.randperm(s.T, generator=g)[:per_step].sort().values.to(dev), mx)
    dt = (time.perf_counter() - t0) / args.steps
    value = per_step / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc, "T": s.T, "d": s.d, "I": s.I, "E": s.E, "top_k": s.k,
                   "n_shared": s.n_shared, "I_shared": s.I_shared, "tokens_per_step": per_step},
        "tflops": value * 3 * _flops(s) / 1e12,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _cpu_cores(), "cpu": _cpu_model(),
                         "kind": "oracle", "extrapolated": True,
                         "sample": f"{per_step} random tokens per step, oracle forward+backward; tokens/s "
                                   f"extrapolated linearly from that sample"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dsv3",
                    choices=["dsv3", "qwen3", "tiny", "dsv3_mxfp8", "kimi_k27", "glm52", "qwen35", "dsv4pro"])
    ap.add_argument("--tokens", type=int, default=0, help="override T (scaled-down profiling runs)")
    ap.add_argument("--experts", type=int, default=0, help="override E (scaled-down profiling runs)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="with the default workload, skip the MXFP8 and Qwen3-shaped workloads measured after it")
    ap.add_argument("--cpu-tokens", type=int, default=4, help="oracle tokens per cpu_baseline round (0 = skip)")
    ap.add_argument("--cpu-rounds", type=int, default=4, help="cpu_baseline rounds")
    ap.add_argument("--ref-tokens", type=int, default=4, help="oracle tokens per reference step")
    ap.add_argument("--cpu-mx", action="store_true",
                    help="also time the MXFP8 oracle for dsv3_mxfp8 (about 11 min per token)")
    ap.add_argument("--zipf", action="store_true", help="Zipf(1.2)-skewed router bias (the sweep's skewed routing)")
    ap.add_argument("--zero-experts", type=int, default=0, help="that many experts never chosen (bias -inf)")
    ap.add_argument("--replay", action="store_true",
                    help="MOE_FLAG_REPLAY: save the routing and the shared expert's a, b; recompute the routed "
                         "x rows, a and b in the backward")
    ap.add_argument("--wgrad-fp32", action="store_true",
                    help="MOE_FLAG_WGRAD_FP32: weight gradients written in fp32 (bf16 mode)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    from moe_layer_gb300 import _abi

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    ranks = _Ranks(world, "cuda")

    _abi.load()
    head = measure_workload(args, args.workload, world, rank, local, ranks, full=True)
    # The other workloads the layer is benchmarked on, measured in the same run
    # so that the printed line carries them too (the headline stays the first).
    extras = {}
    plain = not (args.tokens or args.experts or args.zipf or args.zero_experts or args.replay or args.wgrad_fp32)
    if plain and args.workload == "dsv3" and not args.no_extra:
        for name in ("dsv3_mxfp8", "qwen3"):
            torch.cuda.empty_cache()
            extras[name] = measure_workload(args, name, world, rank, local, ranks, full=False)

    if rank == 0:
        s = head.pop("_shape")
        line = {
            "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8" if head["mx"] else "bf16", "data": "synthetic",
            "config": {"workload": head["workload"], "T": s.T, "d": s.d, "I": s.I, "E": s.E, "top_k": s.k,
                       "n_shared": s.n_shared, "I_shared": s.I_shared, "tokens_per_gpu": s.T,
                       "parallelism": f"replicas x{world}",
                       "activations": "replayed in the backward" if args.replay else "saved",
                       "weight_grads": "fp32" if args.wgrad_fp32 else "bf16",
                       "l2": "inputs larger than L2 (x 235 MB, expert weights 22.6 GB at dsv3); no flush"},
        }
        for key in ("tflops", "pct_tensor_peak", "pct_tensor_peak_sustained", "tensor_peak_src", "weight_quant",
                    "fwd", "fwd_inference", "roofline", "kernels_ms_per_step", "kernel_share", "gpu_launches", "e2e",
                    "cpu_baseline", "clocks"):
            line[key] = head.get(key)
        if extras:
            line["workloads"] = {}
            for name, r in extras.items():
                r.pop("_shape", None)
                r.pop("mx", None)
                line["workloads"][name] = r
            line["gpu_launches_all_workloads"] = head["gpu_launches"] + sum(r["gpu_launches"] for r in extras.values())
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


_MX_PEAK = {}


def measure_workload(args, name, world, rank, local, ranks, full):
    """Times forward+backward steps of workload `name` (and the forward alone)
    through the C ABI on resident inputs; with `full`, also the end-to-end step
    with host copies and the CPU oracle baseline.  Returns a dict of results
    (the step's buffers are freed on return)."""
    import torch

    from moe_layer_gb300 import _abi, layer
    from synth.inputs import make_inputs

    barrier, max_over_ranks = ranks.barrier, ranks.max
    tok_override = (args.tokens, args.experts, args.zipf, args.zero_experts) if full else (0, 0, False, 0)
    s, desc, mx = _workload(name, *tok_override)
    inp = make_inputs(s, seed=rank, device="cuda")
    cfg = _abi.make_config(s.T, s.d, s.I, s.E, s.k, s.n_shared, s.I_shared,
                           precision=_abi.MOE_MXFP8 if mx else _abi.MOE_BF16,
                           flags=((_abi.MOE_FLAG_REPLAY if args.replay else 0)
                                  | (_abi.MOE_FLAG_WGRAD_FP32 if args.wgrad_fp32 else 0)) if full else 0)
    if mx:
        layer.quantize_weights(cfg, inp)
    bufs = layer.MoEBuffers(cfg)
    grads = layer.alloc_grads(cfg)
    y = torch.empty(s.T, s.d, dtype=torch.bfloat16, device="cuda")
    dx = torch.empty_like(y)
    stream = torch.cuda.current_stream()

    def step():
        layer.forward(cfg, inp, bufs, y)
        layer.backward(cfg, inp, inp["dy"], bufs, grads, dx)

    def timed(fn, n):
        torch.cuda.synchronize()
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        barrier()
        return a.elapsed_time(b) / n

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = _abi.moe_read_device_status(bufs.fwd_ws) or _abi.moe_read_device_status(bufs.bwd_ws)
    if st:
        raise RuntimeError(f"device status {st} after warm-up ({name})")

    # forward + backward: the headline, with per-kernel events and clock samples
    sampler = ClockSampler(local)
    sampler.start()
    _abi.moe_profile_enable(True)
    ms = timed(step, args.steps)
    _abi.moe_profile_enable(False)
    clocks = sampler.stop()
    prof = _abi.moe_profile_report()
    ms = max_over_ranks(ms)
    # forward alone
    for _ in range(2):
        layer.forward(cfg, inp, bufs, y)
    ms_fwd = max_over_ranks(timed(lambda: layer.forward(cfg, inp, bufs, y), args.steps))
    # forward for serving: no saved state (the routed experts' a, b and, in
    # MXFP8 mode, the transposed activation copies are not written)
    ibufs = layer.MoEBuffers(cfg, training=False)
    for _ in range(2):
        layer.forward(cfg, inp, ibufs, y)
    ms_inf = max_over_ranks(timed(lambda: layer.forward(cfg, inp, ibufs, y), args.steps))
    del ibufs

    wq = None
    if mx:  # the once-per-weight-update quantization pass, timed on its own
        ms_wq = max_over_ranks(timed(lambda: layer.quantize_weights(cfg, inp), args.steps))
        if "peak" not in _MX_PEAK:
            _MX_PEAK["peak"] = measure_mxfp8_peak()

    tokens = s.T * world
    flops_tok = _flops(s)
    peaks = _peaks()
    t_burst, t_sust, t_src = _tensor_peaks(peaks, mx, _MX_PEAK.get("peak") if mx else None)
    if mx:
        wq = {"ms": ms_wq, "per": "weight update",
              "value_incl": tokens / ((ms + ms_wq) * 1e-3), "unit": "tokens/s",
              "note": "fwd+bwd step plus one weight quantization pass"}
    value = tokens / (ms * 1e-3)
    tflops = value * 3 * flops_tok / 1e12
    fwd_value = tokens / (ms_fwd * 1e-3)

    # prof: {step: (calls, kernels, total ms)}; a grouped row GEMM step runs as
    # two kernels (its 2-SM pass and the pass over leftover tiles)
    launches = sum(nk for _, nk, _ in prof.values())
    kern_ms = {k: v[2] for k, v in prof.items()}
    total_kern = sum(kern_ms.values())
    top = max(kern_ms, key=kern_ms.get)
    n_top, nk_top, ms_top = prof[top]
    fl = _kernel_flops(top, s)
    roofline = None
    scaled = any(tok_override)
    if fl is not None:
        achieved = fl / (ms_top / n_top * 1e-3) / 1e12
        traffic = NCU_TRAFFIC.get((name, top)) if not scaled else None
        roofline = {"kernel": top, "bound": "tensor", "achieved": achieved,
                    "peak": t_sust, "unit": "TFLOP/s",
                    "frac": achieved / t_sust, "traffic": traffic,
                    "algorithmic_flops_per_launch": fl,
                    "kernels_per_launch": nk_top / n_top,
                    "peak_src": t_src + " sustained (kernel timed inside a long step)"}
        if mx:
            roofline["frac_of_burst"] = achieved / t_burst

    e2e = None
    if full and not args.no_e2e:
        xh = inp["x"].cpu().pin_memory()
        dyh = inp["dy"].cpu().pin_memory()
        yh = torch.empty(s.T, s.d, dtype=torch.bfloat16).pin_memory()
        dxh = torch.empty_like(yh).pin_memory()
        xd = torch.empty_like(inp["x"])
        dyd = torch.empty_like(inp["dy"])
        inp_e2e = dict(inp)
        inp_e2e["x"] = xd

        # Within a step, dy's upload overlaps the forward, y's download the
        # backward, and dx's download the weight gradients (moe_backward
        # records dx_ready once dx is complete), on a side stream; x goes up
        # before the forward, and dy after x (the two uploads would otherwise
        # share the host link, delaying x).  Every copy of the step is inside
        # it: the step ends when the side stream has finished too.
        side = torch.cuda.Stream()
        prev_done = torch.cuda.Event()
        prev_done.record(stream)
        dx_ready = torch.cuda.Event()
        dx_ready.record(stream)  # creates the CUDA event the library records
        grads_e2e = dict(grads)
        grads_e2e["dx_ready"] = dx_ready

        def e2e_step():
            xd.copy_(xh, non_blocking=True)
            x_up = torch.cuda.Event()
            x_up.record(stream)
            with torch.cuda.stream(side):
                side.wait_event(prev_done)  # the previous step no longer reads dyd or writes yh
                side.wait_event(x_up)
                dyd.copy_(dyh, non_blocking=True)
                dy_up = torch.cuda.Event()
                dy_up.record(side)
            layer.forward(cfg, inp_e2e, bufs, y)
            y_done = torch.cuda.Event()
            y_done.record(stream)
            with torch.cuda.stream(side):
                side.wait_event(y_done)
                yh.copy_(y, non_blocking=True)
            stream.wait_event(dy_up)
            layer.backward(cfg, inp_e2e, dyd, bufs, grads_e2e, dx)
            with torch.cuda.stream(side):
                side.wait_event(dx_ready)
                dxh.copy_(dx, non_blocking=True)
            stream.wait_stream(side)  # the downloads are part of the step
            prev_done.record(stream)

        e2e_step()
        ms_e2e = max_over_ranks(timed(e2e_step, args.steps))
        nb = s.T * s.d * 2
        e2e = {"value": tokens / (ms_e2e * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": 2 * nb,
               "d2h_bytes_per_step": 2 * nb, "ms_per_step": ms_e2e}

    cpu = None
    if full and rank == 0 and world == 1 and args.cpu_tokens > 0:
        if mx and not args.cpu_mx:
            # The MXFP8 oracle round-trips every expert weight it touches
            # (about 15 s per [2048, 7168] matrix on one core, 48 per token).
            cpu = {"value": None, "unit": "tokens/s", "cores": _cpu_cores(), "cpu": _cpu_model(), "kind": "oracle",
                   "sample": "not timed by default: the MXFP8 oracle takes about 11 min per token "
                             "(--cpu-mx --cpu-tokens 1 --cpu-rounds 1 times one token)"}
        else:
            cpu = cpu_baseline(inp, s, args.cpu_tokens, args.cpu_rounds, mxfp8=mx)

    out = {
        "_shape": s, "mx": mx, "workload": desc, "value": value, "unit": "tokens/s", "ms_per_step": ms,
        "dtype": "mxfp8" if mx else "bf16",
        "tflops": tflops, "pct_tensor_peak": tflops / t_burst,
        "pct_tensor_peak_sustained": tflops / t_sust, "tensor_peak_src": t_src,
        "weight_quant": wq,
        "fwd": {"value": fwd_value, "unit": "tokens/s", "ms": ms_fwd,
                "tflops": fwd_value * flops_tok / 1e12, "note": "the forward of a training step (state saved)"},
        "fwd_inference": {"value": tokens / (ms_inf * 1e-3), "unit": "tokens/s", "ms": ms_inf,
                          "tflops": tokens / (ms_inf * 1e-3) * flops_tok / 1e12, "note": "no saved state"},
        "roofline": roofline,
        "kernels_ms_per_step": {k: round(v / args.steps, 4) for k, v in
                                sorted(kern_ms.items(), key=lambda kv: -kv[1])},
        "kernel_share": {k: round(v / total_kern, 4) for k, v in kern_ms.items()},
        "gpu_launches": launches, "clocks": clocks,
    }
    if full:
        out["e2e"], out["cpu_baseline"] = e2e, cpu
    else:
        out["config"] = {"T": s.T, "d": s.d, "I": s.I, "E": s.E, "top_k": s.k, "n_shared": s.n_shared,
                         "I_shared": s.I_shared}
    if mx and _MX_PEAK.get("peak"):
        out["mxfp8_peak"] = _MX_PEAK["peak"]
    del inp, bufs, grads, y, dx
    torch.cuda.synchronize()
    return out


if __name__ == "__main__":
    sys.exit(main())
