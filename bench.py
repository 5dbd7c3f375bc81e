#!/usr/bin/env python3
"""Benchmark of the routed top-k expert layer's forward pass on GB300.

One step = one pass of the whole path over one batch: routing (histogram, scan, stable permute,
row gather), the gate/up grouped GEMM with SwiGLU, the down grouped GEMM with the score
weighting, and the combine -- through the C ABI, on inputs already resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--also NAMES]
                    [--impl ours|reference] [--precision bf16|mxfp8|nvfp4] [--pass fwd|bwd]
                    [--pipeline staged|mega]

The line's workload is --config (default: large, T=16384 D=7168 F=2048 E=256 K=8, the largest
single-GPU workload and the compute-bound target). The workloads named by --also (default: decode,
the weight-streaming target at T=64 on the same weights, and medium) are measured the same way after
it and reported in the same line, each as a sub-record under its own name with its own timing, stage
times, rooflines, end-to-end rate, clocks and CPU baseline.

--pipeline mega runs the bf16 forward with both grouped GEMMs fused into one grid
(dispatch, fused GEMMs, combine); the default runs them as separate kernels.

--precision mxfp8 / nvfp4 runs a block-scaled forward (E4M3 operands with UE8M0 scales per 32, or
E2M1 with UE4M3 scales per 16 and tensor scales; weights prepared once before the timed region,
activations quantized inside each step).

Prints ONE JSON line (rank 0). Under torchrun each rank runs its own replica of the workload
(tokens drawn with a rank-specific seed, the same weights): the path has no exchange step on one
GPU per replica, so scaling is weak and no collective touches the data path; the ranks only meet
at the barriers and the max-over-ranks reduction of the timings.

--impl reference times the CPU oracle (test infrastructure, a deliberately plain C loop) on the
box's host cores on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "routed-expert fwd tokens/s and TFLOP/s on 1 GB300; % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20  # > 2x the 129 MB L2
STAGES = ("dispatch", "gemm1_swiglu", "gemm2_score", "combine")
KERNELS_PER_STEP = 7  # hist, scan, permute, gather, gemm1, gemm2, combine
MEGA_STAGES = ("dispatch", "fused_gemms", "combine")
MEGA_KERNELS_PER_STEP = 6  # hist, scan, permute, gather, the fused GEMMs, combine
# backward: hist, scan, permute, pad tiles, pad rows, gather; recompute, two dgrads, two wgrads; dscores, dx
BWD_KERNELS_PER_STEP = 13

# Operand formats of the forward: bytes per quantized element (codes + scales), the tensor peak as
# a multiple of the measured bf16 peak (nominal dense ratios: fp8 4.5 / 2.25, fp4 13.5 / 2.25), the
# dtype label and the key prefix of recorded traffic.
PRECISIONS = {
    "bf16": {"elem_bytes": 2.0, "tensor_scale": 1.0, "dtype": "bf16", "key": ""},
    "mxfp8": {"elem_bytes": 1.0 + 1.0 / 32, "tensor_scale": 2.0, "dtype": "mxfp8-e4m3", "key": "mx_"},
    "nvfp4": {"elem_bytes": 0.5 + 1.0 / 16, "tensor_scale": 6.0, "dtype": "nvfp4-e2m1", "key": "nv_"},
}
NV_H_SCALE = 2.0 ** -8  # NVFP4 tensor scale of the SwiGLU output (|h| < 6 * 448 * 2^-8 = 10.5 here)


# ------------------------------------------------------------------------------ host logic

def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=500)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--config", default="large", choices=["tiny", "medium", "decode", "large", "skewed"],
                   help="the workload of the line (default: large, the largest single-GPU workload)")
    p.add_argument("--also", default="decode,medium",
                   help="comma-separated workloads measured after --config and reported as sub-records of "
                        "the same line, each under its own name (empty: none)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--precision", default="bf16", choices=sorted(PRECISIONS),
                   help="forward operands: bf16, MXFP8 E4M3 or NVFP4 E2M1 (block-scaled, prepared weights)")
    p.add_argument("--pass", dest="which", default="fwd", choices=["fwd", "bwd"],
                   help="fwd: the forward layer (the headline); bwd: its backward pass (one call per step)")
    p.add_argument("--pipeline", default="staged", choices=["staged", "mega"],
                   help="bf16 forward: separate GEMM kernels (staged) or both GEMMs in one grid (mega)")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--tokens", type=int, default=None,
                   help="replace the workload's T (smaller cases for profiling runs; no sub-records)")
    p.add_argument("--experts", type=int, default=None,
                   help="replace the workload's E (a weight-streaming case small enough for ncu; no sub-records)")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing on the host cores")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    p.add_argument("--sub-cpu-seconds", type=float, default=8.0,
                   help="target CPU time of the oracle sample of each sub-record")
    return p.parse_args(argv)


def dist_env():
    """(rank, world, local_rank) from the torchrun environment (1 process when absent)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def reduce_max(dist, value: float) -> float:
    """Max of a float over ranks (identity for one process)."""
    if dist is None:
        return value
    import torch

    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(seed: int, rank: int) -> int:
    """Tokens and routing of each replica differ; weights use the base seed on every rank."""
    return seed + 1009 * rank


def measured_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            peaks = json.load(fh)
        if peaks.get("hbm_gbs") and peaks.get("bf16_tflops"):
            return peaks, "measured"
    except (OSError, ValueError):
        pass
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_costs(T, D, F, E, K, touched, q=None):
    """Algorithmic flops and bytes per launch of each stage (tile padding not counted). q: bytes per
    element of the block-scaled operands (codes + scales), None for the bf16 forward."""
    R = T * K
    # dispatch: ids read twice (histogram, permute), perm and inv written, then the token-order
    # gather: each x row read once and written to its K routed rows
    if q is not None:
        return {
            "dispatch": {"flops": 0, "bytes": 2 * R * 4 + 2 * R * 4 + T * D * 2 + R * D * q},
            "gemm1_swiglu": {"flops": 4 * R * D * F, "bytes": touched * 2 * F * D * q + R * D * q + R * F * q},
            "gemm2_score": {"flops": 2 * R * D * F, "bytes": touched * D * F * q + R * F * q + R * D * 2 + R * 8},
            "combine": {"flops": 0, "bytes": R * D * 2 + T * D * 2 + R * 4},
        }
    return {
        "dispatch": {"flops": 0, "bytes": 2 * R * 4 + 2 * R * 4 + T * D * 2 + R * D * 2},
        "gemm1_swiglu": {"flops": 4 * R * D * F, "bytes": touched * 2 * F * D * 2 + R * D * 2 + R * F * 2},
        "gemm2_score": {"flops": 2 * R * D * F, "bytes": touched * D * F * 2 + R * F * 2 + R * D * 2 + R * 8},
        # both GEMMs in one grid: H stays inside the kernel, so only XP in and Y out count
        "fused_gemms": {"flops": 6 * R * D * F, "bytes": touched * 3 * F * D * 2 + R * D * 2 + R * D * 2 + R * 8},
        "combine": {"flops": 0, "bytes": R * D * 2 + T * D * 2 + R * 4},
    }


def path_costs(T, D, F, E, K, touched, wbytes=2.0):
    """The layer's algorithmic flops and bytes: touched experts' weights, x, out, ids, scores."""
    return 6 * T * K * D * F, touched * 3 * F * D * wbytes + 2 * T * D * 2 + T * K * 8


def overhead_bytes(T, D, F, K, q=2.0):
    """The implementation's intermediate round trips (written, then read back), which the
    algorithmic bytes leave out: the routed rows of x (XP, or XQ at q bytes per element), the SwiGLU
    output (H / HQ) and the bf16 score-weighted pair outputs (Y)."""
    R = T * K
    return {"xp": 2 * R * D * q, "h": 2 * R * F * q, "y": 2 * R * D * 2}


def roofline_entry(name, costs, seconds, peaks, sustained, traffic, tensor_scale=1.0):
    """tensor_scale multiplies the measured bf16 peak for another operand type (PRECISIONS)."""
    c = costs[name]
    ridge = tensor_scale * peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if c["flops"] > 0 and c["flops"] / max(c["bytes"], 1) >= ridge:
        peak = tensor_scale * (peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"])
        achieved = c["flops"] / seconds / 1e12
        kind = "sustained" if sustained else "burst"
        if tensor_scale != 1.0:
            kind += f" bf16 x {tensor_scale:g} (nominal dense ratio of the operand type to bf16)"
        return {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": name, "peak_kind": kind}
    achieved = c["bytes"] / seconds / 1e9
    peak = peaks["hbm_gbs"]
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": name, "peak_kind": "copy"}


def kernel_source_hash() -> str:
    """Hash of the grouped-GEMM sources; a recorded DRAM traffic is only valid for this hash."""
    h = hashlib.sha256()
    for rel in ("mixture_experts_routed_topk_gb300/csrc/grouped_gemm.cu",
                "mixture_experts_routed_topk_gb300/csrc/mxfp8.cu",
                "mixture_experts_routed_topk_gb300/csrc/nvfp4.cu",
                "mixture_experts_routed_topk_gb300/csrc/block_scaled.cuh",
                "mixture_experts_routed_topk_gb300/csrc/gemm_pipeline.cuh",
                "mixture_experts_routed_topk_gb300/csrc/ptx_sm103.cuh",
                "mixture_experts_routed_topk_gb300/csrc/routing.cu",
                "mixture_experts_routed_topk_gb300/csrc/combine.cu",
                "mixture_experts_routed_topk_gb300/csrc/backward.cu"):
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(config: str, kernel: str, touched: int | None = None):
    """DRAM bytes per launch recorded by an ncu capture (profiles/dram_traffic.md), or None when
    absent or taken on other kernel sources.

    A row's config is a workload name, or a name with its expert count cut for the capture
    ("decode (E=16)"): a weight-streaming kernel on a workload too large to capture under ncu is
    captured with fewer experts, and its traffic, which grows with the experts it touches, is scaled
    to `touched` experts by the ratio of touched experts (the row's last numeric column)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    src = kernel_source_hash()
    row = re.compile(r"^\|\s*(\w+)(?:\s*\(E=(\d+)\))?\s*\|\s*(\w+)\s*\|\s*([0-9a-f]{16})\s*\|\s*([0-9.eE+]+)\s*\|"
                     r"\s*[0-9.eE+]+\s*\|\s*[0-9.eE+]+\s*\|\s*(\d+)\s*\|", re.M)
    scaled = None
    for m in row.finditer(text):
        if m.group(1) != config or m.group(3) != kernel or m.group(4) != src:
            continue
        if m.group(2) is None:
            return float(m.group(5))
        if touched and scaled is None:
            scaled = float(m.group(5)) * touched / int(m.group(6))
    return round(scaled) if scaled is not None else None


def assemble_line(**kw) -> str:
    return json.dumps(kw, separators=(", ", ": "))


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", self.gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons, power = [], [], set(), []
        for ln in self.lines:
            f = [s.strip() for s in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        busy = [s for s, p in zip(sm, power) if p >= 0.5 * max(power)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


# ------------------------------------------------------------------------------ oracle timing

def oracle_sample(d, tokens: int):
    """Host copies of the first `tokens` tokens and the experts they touch (ids renumbered)."""
    import numpy as np
    import torch

    ids = d["topk_ids"][:tokens].cpu().numpy()
    E = d["w13"].shape[0]
    experts = np.unique(ids[(ids >= 0) & (ids < E)])
    remap = np.full(E, -1, np.int64)
    remap[experts] = np.arange(experts.size)
    ex = torch.from_numpy(experts).to(d["w13"].device)
    u16 = lambda t: t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    return {
        "x": u16(d["x"][:tokens]),
        "ids": remap[ids].astype(np.int32),
        "scores": d["topk_scores"][:tokens].cpu().numpy().astype(np.float32),
        "w13": u16(d["w13"].index_select(0, ex)),
        "w2": u16(d["w2"].index_select(0, ex)),
        "experts": int(experts.size),
    }


def oracle_tokens_for(seconds: float, wl, cores: int, gflops_per_core: float = 0.7) -> int:
    per_token = 6.0 * wl.K * wl.D * wl.F
    n = int(seconds * cores * gflops_per_core * 1e9 / per_token)
    return max(1, min(n, wl.T))


def bounded_tokens(ids_host, wl, n_tok: int, budget_bytes: int = 4 << 30) -> int:
    """Shrink the token sample until the weights of the experts it touches fit the host budget."""
    import numpy as np

    per_expert = 3 * wl.F * wl.D * 2
    while n_tok > 1:
        first = ids_host[:n_tok]
        touched = np.unique(first[(first >= 0) & (first < wl.E)]).size
        if touched * per_expert <= budget_bytes:
            break
        n_tok = max(1, n_tok // 2)
    return n_tok


def time_oracle(sample, nthreads: int) -> float:
    import oracle

    t0 = time.perf_counter()
    if "w13_nv" in sample:
        oracle.routed_experts_nvfp4(sample["x"], sample["ids"], sample["scores"], sample["w13_nv"],
                                    sample["w2_nv"], sample["gx"], sample["gh"], nthreads=nthreads)
    elif "w13_mx" in sample:
        oracle.routed_experts_mxfp8(sample["x"], sample["ids"], sample["scores"], sample["w13_mx"],
                                    sample["w2_mx"], nthreads=nthreads)
    else:
        oracle.routed_experts(sample["x"], sample["ids"], sample["scores"], sample["w13"], sample["w2"],
                              nthreads=nthreads)
    return time.perf_counter() - t0


def prepare_oracle_sample(sample, precision: str, gx: float = 0.0):
    """Quantized weights for the oracle's block-scaled forwards (prepared once, not timed). The
    NVFP4 weight scales come from the sample's experts."""
    import oracle

    if precision == "mxfp8":
        sample["w13_mx"] = oracle.mx_quantize_rows(sample["w13"])
        sample["w2_mx"] = oracle.mx_quantize_rows(sample["w2"])
    elif precision == "nvfp4":
        sample["w13_nv"] = oracle.nvfp4_prepare(sample["w13"])
        sample["w2_nv"] = oracle.nvfp4_prepare(sample["w2"])
        sample["gx"], sample["gh"] = gx, NV_H_SCALE


def cpu_baseline(d, wl, name: str, target_s: float, precision: str = "bf16", gx: float = 0.0) -> dict:
    """The oracle as it stands on the host cores: a bounded token sample, repeated to fill about
    target_s seconds; tokens/s = tokens processed / seconds. For a block-scaled precision, the
    oracle's forward of that format on weights it quantized beforehand."""
    cores = os.cpu_count() or 1
    ids_host = d["topk_ids"].cpu().numpy()
    rate = 0.7 if precision == "bf16" else 0.35
    n_tok = bounded_tokens(ids_host, wl, oracle_tokens_for(target_s, wl, cores, rate))
    sample = oracle_sample(d, n_tok)
    prepare_oracle_sample(sample, precision, gx)
    secs = [time_oracle(sample, cores)]
    reps = max(1, min(100, int(target_s / max(secs[0], 1e-6))))
    secs += [time_oracle(sample, cores) for _ in range(reps - 1)]
    total = sum(secs)
    return {"value": round(n_tok * len(secs) / total, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n_tok} tokens of the {name} workload ({sample['experts']} experts touched, full "
                      f"K={wl.K} per token) x {len(secs)} runs = {total:.1f} s on {cores} threads",
            "seconds": round(total, 2)}


# ------------------------------------------------------------------------------ our path

def workload_for(args, name):
    """The workload `name`, with the --tokens / --experts overrides applied to the primary one."""
    from mixture_experts_routed_topk_gb300 import workloads as W

    wl = W.WORKLOADS[name]
    if name == args.config:
        if args.tokens:
            wl = dataclasses.replace(wl, T=int(args.tokens))
        if args.experts:
            wl = dataclasses.replace(wl, E=int(args.experts))
    return wl


def workload_label(args, name, wl):
    base = __import__("mixture_experts_routed_topk_gb300.workloads", fromlist=["WORKLOADS"]).WORKLOADS[name]
    changed = [f"{k}={getattr(wl, k)}" for k in ("T", "E") if getattr(wl, k) != getattr(base, k)]
    return name if not changed else f"{name} ({', '.join(changed)})"


class WeightCache:
    """The expert weights of one (E, D, F) at a time, and their prepared block-scaled forms: the
    decode and large workloads share their shapes, so they share one 22.5 GB weight set."""

    def __init__(self, device, seed):
        self.device, self.seed, self.key, self.w, self.prepared = device, seed, None, None, {}

    def get(self, E, D, F):
        from mixture_experts_routed_topk_gb300 import workloads as W
        import torch

        if self.key != (E, D, F):
            self.w, self.prepared = None, {}
            torch.cuda.empty_cache()
            self.w = W.make_weights(E, D, F, self.seed, self.device)
            self.key = (E, D, F)
        return self.w

    def prepare(self, precision):
        """Block-scaled weights, prepared once per weight set (outside every timed region)."""
        from mixture_experts_routed_topk_gb300 import binding

        if precision not in self.prepared:
            w13, w2 = self.w
            if precision == "mxfp8":
                self.prepared[precision] = (binding.moe_mxfp8_prepare_weight(binding.MOE_WEIGHT_W13, w13),
                                            binding.moe_mxfp8_prepare_weight(binding.MOE_WEIGHT_W2, w2))
            else:
                self.prepared[precision] = (binding.moe_nvfp4_prepare_weight(binding.MOE_WEIGHT_W13, w13),
                                            binding.moe_nvfp4_prepare_weight(binding.MOE_WEIGHT_W2, w2))
        return self.prepared[precision]


def measure_forward(args, name, device, dist, rank, world, cache, cpu_seconds):
    """Times one workload's forward (the stage calls with events, then the whole call end to end on
    host buffers) and returns its fields for the JSON line (rank 0; None on the other ranks)."""
    import torch

    from mixture_experts_routed_topk_gb300 import binding
    from mixture_experts_routed_topk_gb300 import workloads as W

    wl = workload_for(args, name)
    T, D, F, E, K = wl.dims()
    rseed = replica_seed(args.seed, rank)
    x = W.make_x(T, D, rseed, device)
    ids = W.make_topk_ids(T, E, K, wl.routing, rseed, device)
    scores = W.make_scores(T, K, wl.scores, rseed, device)
    w13, w2 = cache.get(E, D, F)
    dims = (T, D, F, E, K)
    prec = PRECISIONS[args.precision]
    mx = args.precision == "mxfp8"
    nv = args.precision == "nvfp4"
    mega = args.pipeline == "mega"
    if mega and (mx or nv):
        raise SystemExit("--pipeline mega runs the bf16 forward")
    stages = MEGA_STAGES if mega else STAGES
    gx = 0.0
    if mx:  # prepared once, as the pages prepare block-scaled weights before execution
        w13_mx, w2_mx = cache.prepare("mxfp8")
        ws = binding.alloc_workspace(binding.moe_mxfp8_workspace_bytes(*dims), device)
    elif nv:  # weights prepared once; x's tensor scale calibrated from this batch, h's a constant
        w13_nv, w2_nv = cache.prepare("nvfp4")
        gx = float(torch.tensor(x.abs().max().float().item(), dtype=torch.float32) / 2688.0)
        ws = binding.alloc_workspace(binding.moe_nvfp4_workspace_bytes(*dims), device)
    elif mega:
        ws = binding.alloc_workspace(binding.moe_mega_workspace_bytes(*dims), device)
    else:
        ws = binding.alloc_workspace(binding.moe_workspace_bytes(*dims), device)
    out = torch.empty((T, D), dtype=torch.bfloat16, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step(ev=None):
        if mx or nv:
            for s in range(binding.MX_STAGES):
                if ev is not None:
                    ev[s].record(stream)
                if mx:
                    binding.moe_fwd_mxfp8_stages(x, ids, scores, w13_mx, w2_mx, out, ws, (F, E), s, s + 1, stream)
                else:
                    binding.moe_fwd_nvfp4_stages(x, ids, scores, w13_nv, w2_nv, out, ws, (F, E), gx, NV_H_SCALE, s,
                                                 s + 1, stream)
            if ev is not None:
                ev[binding.MX_STAGES].record(stream)
            return
        if mega:
            for s in range(binding.MEGA_STAGES):
                if ev is not None:
                    ev[s].record(stream)
                binding.moe_fwd_mega_stages(x, ids, scores, w13, w2, out, ws, s, s + 1, stream)
            if ev is not None:
                ev[binding.MEGA_STAGES].record(stream)
            return
        if ev is not None:
            ev[0].record(stream)
        binding.moe_fwd_dispatch(x, ids, dims, ws, stream)
        if ev is not None:
            ev[1].record(stream)
        binding.moe_fwd_gemm1(w13, dims, ws, stream)
        if ev is not None:
            ev[2].record(stream)
        binding.moe_fwd_gemm2(scores, w2, dims, ws, stream)
        if ev is not None:
            ev[3].record(stream)
        binding.moe_fwd_combine(ids, out, dims, ws, stream)
        if ev is not None:
            ev[4].record(stream)

    for _ in range(max(args.warmup, 0)):
        flush.zero_()
        step()
    torch.cuda.synchronize(device)
    status = binding.moe_get_status(ws, stream)
    if status != 0:
        raise RuntimeError(f"device status bits {status:#x} after warm-up ({name})")
    counts = (binding.moe_mxfp8_workspace_layout(*dims) if mx else
              binding.moe_nvfp4_workspace_layout(*dims) if nv else
              binding.moe_mega_workspace_layout(*dims) if mega else binding.moe_workspace_layout(*dims))
    cnt = ws[counts["counts"]:counts["counts"] + 4 * E].view(torch.int32)
    touched = int((cnt > 0).sum().item())

    # ------------------------------------------------------------------ device-timed region
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(args.steps)]
    props = torch.cuda.get_device_properties(device)
    gpu_id = "GPU-" + str(props.uuid) if hasattr(props, "uuid") else str(device.index)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    barrier(dist, device)
    torch.cuda.synchronize(device)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()  # outside the events: L2 holds no operand when a step starts
        step(events[i])
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - wall0
    barrier(dist, device)
    sampler.stop()
    stage_ms = {s: [events[i][j].elapsed_time(events[i][j + 1]) for i in range(args.steps)]
                for j, s in enumerate(stages)}
    step_ms = [events[i][0].elapsed_time(events[i][len(stages)]) for i in range(args.steps)]
    total_s = reduce_max(dist, sum(step_ms) / 1e3)

    # ------------------------------------------------------------------ end to end (host buffers)
    # Each step uploads its own x / ids / scores from pinned host memory and reads its output back,
    # all inside the timed region. Uploads and read-backs run on their own streams with two device
    # input/output sets, so step i+1's upload and step i-1's read-back overlap step i's compute, as a
    # serving loop would.
    x_h = [x.cpu().pin_memory() for _ in range(2)]
    ids_h = [ids.cpu().pin_memory() for _ in range(2)]
    scores_h = [scores.cpu().pin_memory() for _ in range(2)]
    out_h = [torch.empty((T, D), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x) for _ in range(2)]
    ids_d = [torch.empty_like(ids) for _ in range(2)]
    scores_d = [torch.empty_like(scores) for _ in range(2)]
    out_d = [torch.empty_like(out) for _ in range(2)]
    up_stream = torch.cuda.Stream(device)    # host -> device uploads
    down_stream = torch.cuda.Stream(device)  # device -> host read-backs
    uploaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    read_back = [torch.cuda.Event() for _ in range(2)]

    def upload(i):
        b = i % 2
        with torch.cuda.stream(up_stream):
            if i >= 2:
                up_stream.wait_event(computed[b])  # step i-2 has consumed this buffer set
            x_d[b].copy_(x_h[b], non_blocking=True)
            ids_d[b].copy_(ids_h[b], non_blocking=True)
            scores_d[b].copy_(scores_h[b], non_blocking=True)
            uploaded[b].record(up_stream)

    def e2e_run(n):
        upload(0)
        for i in range(n):
            b = i % 2
            stream.wait_event(uploaded[b])
            if i >= 2:
                stream.wait_event(read_back[b])  # out_d[b] of step i-2 has been read back
            if mx:
                binding.moe_routed_experts_fwd_mxfp8(x_d[b], ids_d[b], scores_d[b], w13_mx, w2_mx, out_d[b], ws,
                                                     (F, E), stream)
            elif nv:
                binding.moe_routed_experts_fwd_nvfp4(x_d[b], ids_d[b], scores_d[b], w13_nv, w2_nv, out_d[b], ws,
                                                     (F, E), gx, NV_H_SCALE, stream)
            elif mega:
                binding.moe_routed_experts_fwd_mega(x_d[b], ids_d[b], scores_d[b], w13, w2, out_d[b], ws, stream)
            else:
                binding.moe_routed_experts_fwd(x_d[b], ids_d[b], scores_d[b], w13, w2, out_d[b], ws, stream)
            computed[b].record(stream)
            if i + 1 < n:
                upload(i + 1)  # overlaps this step's compute
            with torch.cuda.stream(down_stream):
                down_stream.wait_event(computed[b])
                out_h[b].copy_(out_d[b], non_blocking=True)
                read_back[b].record(down_stream)

    e2e_run(max(args.warmup, 2))
    torch.cuda.synchronize(device)
    e2e_start = torch.cuda.Event(enable_timing=True)
    e2e_end = torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    torch.cuda.synchronize(device)
    e2e_start.record(stream)
    up_stream.wait_event(e2e_start)
    e2e_run(args.steps)
    stream.wait_stream(down_stream)
    e2e_end.record(stream)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    e2e_s = reduce_max(dist, e2e_start.elapsed_time(e2e_end) / 1e3)
    h2d = x.numel() * 2 + ids.numel() * 4 + scores.numel() * 4
    d2h = out.numel() * 2
    del x_d, out_d, ids_d, scores_d, flush

    if rank != 0:
        del ws, out
        return None

    peaks, peak_src = measured_peaks()
    costs = kernel_costs(T, D, F, E, K, touched, None if args.precision == "bf16" else prec["elem_bytes"])
    mean_stage = {s: statistics.mean(v) for s, v in stage_ms.items()}
    dominant = max(mean_stage, key=mean_stage.get)
    ms_per_step = total_s * 1e3 / args.steps
    sustained = ms_per_step * args.steps > 2000.0  # a seconds-long loop runs under the power cap
    tensor_scale = prec["tensor_scale"]
    label = workload_label(args, name, wl)
    roof = roofline_entry(dominant, costs, mean_stage[dominant] / 1e3, peaks, sustained,
                          recorded_traffic(name, prec["key"] + dominant, touched), tensor_scale)
    roof["peak_source"] = peak_src
    flops, alg_bytes = path_costs(T, D, F, E, K, touched, prec["elem_bytes"])
    step_s = ms_per_step / 1e3
    t_roof = max(flops / (tensor_scale * peaks["bf16_tflops"] * 1e12), alg_bytes / (peaks["hbm_gbs"] * 1e9))
    path_bound = "tensor" if flops / (tensor_scale * peaks["bf16_tflops"] * 1e12) >= alg_bytes / (
        peaks["hbm_gbs"] * 1e9) else "hbm"
    stage_roofs = {s: roofline_entry(s, costs, mean_stage[s] / 1e3, peaks, sustained,
                                     recorded_traffic(name, prec["key"] + s, touched), tensor_scale)
                   for s in stages}

    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline({"x": x, "topk_ids": ids, "topk_scores": scores, "w13": w13, "w2": w2}, wl,
                           label, cpu_seconds, args.precision, gx)
    del ws, out
    return {
        "value": round(world * T * args.steps / total_s, 1),
        "ms_per_step": round(ms_per_step, 4),
        "config": {"workload": label, "T": T, "D": D, "F": F, "E": E, "K": K,
                   "precision": args.precision, "pipeline": args.pipeline, "routing": wl.routing,
                   "experts_touched": touched, "global_batch": T * world, "parallelism": f"replicas{world}",
                   "l2": "flushed between steps (512 MB write)", "seed": args.seed},
        "tflops": round(world * flops / step_s / 1e12, 2),
        "path_roofline": {"bound": path_bound, "ms": round(t_roof * 1e3, 4), "frac": round(t_roof / step_s, 4),
                          "flops": flops, "alg_bytes": alg_bytes,
                          "hbm_gbs": round(alg_bytes / step_s / 1e9, 1),
                          "overhead_bytes": {k: int(v) for k, v in
                                             overhead_bytes(T, D, F, K, prec["elem_bytes"]).items()}},
        "roofline": roof,
        "stage_ms": {s: round(v, 4) for s, v in mean_stage.items()},
        "stage_roofline": {s: {k: r[k] for k in ("bound", "achieved", "unit", "frac", "traffic")}
                           for s, r in stage_roofs.items()},
        "e2e": {"value": round(world * T * args.steps / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": (MEGA_KERNELS_PER_STEP if mega else KERNELS_PER_STEP) * args.steps,
        "clocks": sampler.summary(),
        "wall_s": round(wall, 3),
        "cpu_baseline": cpu,
    }


def extra_workloads(args) -> list[str]:
    """The workloads measured after the primary one and reported as sub-records of its line."""
    if args.tokens or args.experts or not args.also:
        return []
    names = [n.strip() for n in args.also.split(",") if n.strip()]
    return [n for n in names if n != args.config]


def run_ours(args, rank, world, local_rank):
    import torch

    from mixture_experts_routed_topk_gb300 import binding, build

    build.build()
    binding.load()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist = dist_init(world, "nccl")
    cache = WeightCache(device, args.seed)
    prec = PRECISIONS[args.precision]

    main = measure_forward(args, args.config, device, dist, rank, world, cache, args.cpu_seconds)
    subs = {}
    for name in extra_workloads(args):
        subs[name] = measure_forward(args, name, device, dist, rank, world, cache, args.sub_cpu_seconds)
    if rank == 0:
        fields = dict(
            metric=METRIC,
            value=main["value"],
            unit="tokens/s",
            n_gpus=world,
            steps=args.steps,
            warmup=args.warmup,
            ms_per_step=main["ms_per_step"],
            higher_is_better=True,
            scaling="weak",
            vs_baseline=None,
            dtype=prec["dtype"],
            data="synthetic",
        )
        fields.update({k: v for k, v in main.items() if k not in ("value", "ms_per_step")})
        for name, rec in subs.items():
            fields[name] = rec
        print(assemble_line(**fields), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------------------------ backward pass

def bwd_stage_costs(T, D, F, E, K, touched):
    """Algorithmic flops and bytes of each backward stage (padding rows not counted): touched
    experts' weights, the routed rows each stage reads and writes, the weight gradients."""
    R = T * K
    ntf = -(-F // 256)  # dscores partial sums per pair (one per 256-column tile of the F axis)
    return {
        "dispatch": {"flops": 0, "bytes": 2 * R * 4 + 2 * R * 4 + 2 * T * D * 2 + 2 * R * D * 2},
        "recompute": {"flops": 4 * R * D * F, "bytes": touched * 2 * F * D * 2 + R * D * 2 + R * 3 * F * 2},
        "dgrad_down": {"flops": 2 * R * D * F,
                       "bytes": touched * D * F * 2 + R * D * 2 + R * 2 * F * 2 + R * 2 * F * 2 + R * ntf * 4},
        "dgrad_gate_up": {"flops": 4 * R * D * F, "bytes": touched * 2 * F * D * 2 + R * 2 * F * 2 + R * D * 2},
        "wgrad_down": {"flops": 2 * R * D * F, "bytes": R * D * 2 + R * F * 2 + E * D * F * 2},
        "wgrad_gate_up": {"flops": 4 * R * D * F, "bytes": R * 2 * F * 2 + R * D * 2 + E * 2 * F * D * 2},
        "reduce": {"flops": 0, "bytes": R * D * 2 + R * ntf * 4 + T * D * 2 + T * K * 4},
    }


def cpu_baseline_bwd(d, wl, name: str, target_s: float) -> dict:
    """The oracle's backward on the host cores: a bounded token sample, repeated to fill about
    target_s seconds (tokens/s = tokens processed / seconds)."""
    import oracle

    cores = os.cpu_count() or 1
    ids_host = d["topk_ids"].cpu().numpy()
    # the backward does about 16/6 of the forward's work per token (recompute, two dgrads, two wgrads)
    n_tok = bounded_tokens(ids_host, wl, max(1, oracle_tokens_for(target_s, wl, cores) * 6 // 16))
    sample = oracle_sample(d, n_tok)
    dout = d["dout"][:n_tok].float().cpu().numpy()

    def once():
        t0 = time.perf_counter()
        oracle.routed_experts_bwd(sample["x"], sample["ids"], sample["scores"], sample["w13"], sample["w2"], dout,
                                  nthreads=cores)
        return time.perf_counter() - t0

    secs = [once()]
    reps = max(1, min(100, int(target_s / max(secs[0], 1e-6))))
    secs += [once() for _ in range(reps - 1)]
    total = sum(secs)
    return {"value": round(n_tok * len(secs) / total, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"backward of the first {n_tok} tokens of the {name} workload ({sample['experts']} experts "
                      f"touched, full K={wl.K} per token) x {len(secs)} runs = {total:.1f} s on {cores} threads",
            "seconds": round(total, 2)}


def run_ours_bwd(args, rank, world, local_rank):
    """Times the backward as its seven stage calls (moe_bwd_stages), with events between them: dx,
    dscores, dw13, dw2 for one upstream gradient per step."""
    import torch

    from mixture_experts_routed_topk_gb300 import binding, build
    from mixture_experts_routed_topk_gb300 import workloads as W

    build.build()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist = dist_init(world, "nccl")
    wl = workload_for(args, args.config)
    T, D, F, E, K = wl.dims()
    rseed = replica_seed(args.seed, rank)
    x = W.make_x(T, D, rseed, device)
    ids = W.make_topk_ids(T, E, K, wl.routing, rseed, device)
    scores = W.make_scores(T, K, wl.scores, rseed, device)
    dout = W.make_x(T, D, rseed + 101, device)
    w13, w2 = W.make_weights(E, D, F, args.seed, device)
    ws = binding.alloc_workspace(binding.moe_bwd_workspace_bytes(T, D, F, E, K), device)
    dx = torch.empty_like(x)
    dscores = torch.empty((T, K), dtype=torch.float32, device=device)
    dw13, dw2 = torch.empty_like(w13), torch.empty_like(w2)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    stages = binding.BWD_STAGE_NAMES

    def step(ev=None):
        for s in range(binding.BWD_STAGES):
            if ev is not None:
                ev[s].record(stream)
            binding.moe_bwd_stages(x, ids, scores, w13, w2, dout, dx, dscores, dw13, dw2, ws, s, s + 1, stream)
        if ev is not None:
            ev[binding.BWD_STAGES].record(stream)

    for _ in range(max(args.warmup, 0)):
        flush.zero_()
        step()
    torch.cuda.synchronize(device)
    if binding.moe_get_status(ws, stream) != 0:
        raise RuntimeError("device status bits after warm-up")
    touched = int((torch.bincount(ids[(ids >= 0) & (ids < E)].long(), minlength=E) > 0).sum().item())
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(args.steps)]
    sampler = ClockSampler("GPU-" + str(torch.cuda.get_device_properties(device).uuid))
    sampler.start()
    barrier(dist, device)
    torch.cuda.synchronize(device)
    for i in range(args.steps):
        flush.zero_()
        step(events[i])
    torch.cuda.synchronize(device)
    barrier(dist, device)
    sampler.stop()
    stage_ms = {s: statistics.mean(events[i][j].elapsed_time(events[i][j + 1]) for i in range(args.steps))
                for j, s in enumerate(stages)}
    total_s = reduce_max(dist, sum(e[0].elapsed_time(e[len(stages)]) for e in events) / 1e3)

    # end to end: each step uploads x, ids, scores and dout from pinned host memory and reads dx and
    # dscores back, inside the timed region (the weight gradients stay on the device for the optimizer)
    x_h, ids_h, sc_h, go_h = (t.cpu().pin_memory() for t in (x, ids, scores, dout))
    dx_h = torch.empty((T, D), dtype=torch.bfloat16).pin_memory()
    ds_h = torch.empty((T, K), dtype=torch.float32).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    torch.cuda.synchronize(device)
    e0.record(stream)
    for _ in range(args.steps):
        x.copy_(x_h, non_blocking=True)
        ids.copy_(ids_h, non_blocking=True)
        scores.copy_(sc_h, non_blocking=True)
        dout.copy_(go_h, non_blocking=True)
        binding.moe_routed_experts_bwd(x, ids, scores, w13, w2, dout, dx, dscores, dw13, dw2, ws, stream)
        dx_h.copy_(dx, non_blocking=True)
        ds_h.copy_(dscores, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    e2e_s = reduce_max(dist, e0.elapsed_time(e1) / 1e3)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    peaks, peak_src = measured_peaks()
    R = T * K
    # recompute 4RDF + dgrad(down) 2RDF + dgrad(gate/up) 4RDF + wgrad(down) 2RDF + wgrad(gate/up) 4RDF
    flops = 16 * R * D * F
    step_s = total_s / args.steps
    achieved = world * flops / step_s / 1e12
    sustained = total_s > 2.0
    peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    costs = bwd_stage_costs(T, D, F, E, K, touched)
    label = workload_label(args, args.config, wl)
    stage_roofs = {s: roofline_entry(s, costs, stage_ms[s] / 1e3, peaks, sustained,
                                     recorded_traffic(args.config, "bwd_" + s, touched))
                   for s in stages}
    gemms = [s for s in stages if costs[s]["flops"] > 0]
    dominant = max(gemms, key=lambda s: stage_ms[s])
    furthest = min(gemms, key=lambda s: stage_roofs[s]["frac"])
    roof = dict(stage_roofs[dominant])
    roof["peak_source"] = peak_src
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline_bwd({"x": x, "topk_ids": ids, "topk_scores": scores, "w13": w13, "w2": w2,
                                "dout": dout}, wl, label, args.cpu_seconds)
    print(assemble_line(
        metric="routed-expert bwd tokens/s and TFLOP/s on 1 GB300; % of roofline",
        value=round(world * T * args.steps / total_s, 1), unit="tokens/s", n_gpus=world, steps=args.steps,
        warmup=args.warmup, ms_per_step=round(step_s * 1e3, 4), higher_is_better=True, scaling="weak",
        vs_baseline=None, dtype="bf16", data="synthetic",
        config={"workload": label, "T": T, "D": D, "F": F, "E": E, "K": K, "routing": wl.routing,
                "experts_touched": touched, "pass": "bwd", "l2": "flushed between steps (512 MB write)"},
        tflops=round(achieved, 2),
        path_roofline={"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                       "frac": round(achieved / peak, 4), "flops": flops,
                       "peak_kind": "sustained" if sustained else "burst"},
        roofline=roof,
        stage_ms={s: round(v, 4) for s, v in stage_ms.items()},
        stage_roofline={s: {k: r[k] for k in ("bound", "achieved", "unit", "frac", "traffic")}
                        for s, r in stage_roofs.items()},
        furthest_below_roof={"stage": furthest, "frac": stage_roofs[furthest]["frac"],
                             "achieved": stage_roofs[furthest]["achieved"], "unit": stage_roofs[furthest]["unit"]},
        e2e={"value": round(world * T * args.steps / e2e_s, 1), "unit": "tokens/s",
             "h2d_bytes_per_step": x.numel() * 2 + ids.numel() * 4 + scores.numel() * 4 + dout.numel() * 2,
             "d2h_bytes_per_step": dx.numel() * 2 + dscores.numel() * 4},
        gpu_launches=BWD_KERNELS_PER_STEP * args.steps, clocks=sampler.summary(), cpu_baseline=cpu,
    ), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------------------------ reference arm

def run_reference(args, rank, world, local_rank):
    """The CPU oracle as it stands, on the host cores, on bounded samples of the workload."""
    if rank != 0:
        return
    import torch

    import oracle
    from mixture_experts_routed_topk_gb300 import workloads as W

    oracle.build()
    wl = W.WORKLOADS[args.config]
    T, D, F, E, K = wl.dims()
    cores = os.cpu_count() or 1
    per_step_s = max(0.2, 60.0 / max(args.steps + args.warmup, 1))
    dev = torch.device("cuda", local_rank) if torch.cuda.is_available() else torch.device("cpu")
    x = W.make_x(T, D, args.seed, dev)
    ids = W.make_topk_ids(T, E, K, wl.routing, args.seed, dev)
    scores = W.make_scores(T, K, wl.scores, args.seed, dev)
    rate = 0.7 if args.precision == "bf16" else 0.35
    n_tok = bounded_tokens(ids.cpu().numpy(), wl, oracle_tokens_for(per_step_s, wl, cores, rate))
    first = ids[:n_tok].cpu()
    experts = sorted(set(first[(first >= 0) & (first < E)].tolist()))
    w13, w2 = W.make_weights(E, D, F, args.seed, dev, experts=experts)
    sample = oracle_sample({"x": x, "topk_ids": ids, "topk_scores": scores, "w13": w13, "w2": w2}, n_tok)
    del w13, w2
    gx = float(torch.tensor(x.abs().max().float().item(), dtype=torch.float32) / 2688.0)
    prepare_oracle_sample(sample, args.precision, gx)  # weights prepared once, outside the timed steps
    for _ in range(max(args.warmup, 0)):
        time_oracle(sample, cores)
    secs = [time_oracle(sample, cores) for _ in range(args.steps)]
    total = sum(secs)
    value = round(n_tok * args.steps / total, 3)
    desc = (f"each step: first {n_tok} tokens of the {args.config} workload ({sample['experts']} experts "
            f"touched), full K={K} per token, on {cores} threads")
    print(assemble_line(
        impl="reference", metric=METRIC, value=value, unit="tokens/s", n_gpus=world, steps=args.steps,
        warmup=args.warmup, ms_per_step=round(total * 1e3 / args.steps, 3), higher_is_better=True,
        scaling="weak", vs_baseline=None, dtype="f32", data="synthetic",
        config={"workload": args.config, "T": T, "D": D, "F": F, "E": E, "K": K, "routing": wl.routing,
                "precision": args.precision, "pipeline": args.pipeline, "sample_tokens": n_tok},
        cpu_baseline={"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
        e2e={"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    ), flush=True)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world, local_rank)
    elif args.which == "bwd":
        if args.precision != "bf16":
            raise SystemExit("the backward pass runs in bf16 only")
        run_ours_bwd(args, rank, world, local_rank)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
