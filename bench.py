#!/usr/bin/env python
"""Benchmark of the W4A16 fused-MoE layer on GB300.

One step = one pass of the whole hot path (routing alignment and the fp16
conversion of x in the prologue, GEMM1 with the fused activation, GEMM2,
combine) over one batch of seeded synthetic input,
replayed from a CUDA graph with inputs resident in HBM; L2 is flushed (a
write larger than L2) before every step and the step is bracketed by CUDA
events.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME --M M]

Under torchrun every rank runs an independent replica of the layer on its own
GPU (the path has no cross-GPU exchange); value = all ranks' tokens / the
slowest rank's time.  --impl reference times the CPU oracle on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from weight_only_bit_moe_gb300 import workloads as wk  # noqa: E402

# the largest single-GPU configuration: int4, K=4096, N=1536, E=128, top_k=8, Zipf(1.2) routing, M=4096
DEFAULT_WORKLOAD, DEFAULT_M = "int4-skew", 4096
DEFAULT_DECODE = "nvfp4-ep-norm:8"   # a decode-sized shape timed beside it


def launches_per_step(block_m: int, separate_align: bool, pairs_x_k: int) -> int:
    """Kernels one step launches: the alignment (its own launch when moe_align runs
    first, for decode-sized blocks and below 2^25 routed elements), the prologue,
    GEMM1, GEMM2, combine."""
    return 5 if (block_m <= 32 or separate_align or pairs_x_k < (1 << 25)) else 4
SWEEP = [("int4-bias", 123), ("int4-bias", 2304), ("mxfp4-alpha", 1), ("mxfp4-alpha", 32), ("mxfp4-alpha", 1024),
         ("nvfp4-ep-norm", 1), ("nvfp4-ep-norm", 8), ("nvfp4-ep-norm", 64), ("nvfp4-ep-norm", 512),
         ("int4-skew", 1), ("int4-skew", 16), ("int4-skew", 256), ("int4-skew", 4096), ("int4-uniform", 16),
         ("int4-uniform", 256), ("int4-uniform", 4096), ("int4-relu2", 123), ("int4-relu2", 2304)]
L2_FLUSH_BYTES = 512 << 20  # > 2x the 129 MB L2


# ---------------------------------------------------------------- algorithmic work

def touched_experts(wl, X) -> np.ndarray:
    local = X.topk_ids.reshape(-1) - wl.expert_base
    local = local[(local >= 0) & (local < wl.E)]
    return np.unique(local)


def local_pairs(wl, X) -> int:
    local = X.topk_ids.reshape(-1) - wl.expert_base
    return int(((local >= 0) & (local < wl.E)).sum())


def algorithmic(wl, W, X):
    """Bytes every step must move at least once and FLOPs over real pairs, per kernel."""
    M = X.x.shape[0]
    nt = len(touched_experts(wl, X))
    P = local_pairs(wl, X)

    def per_expert(a):
        return 0 if a is None else a.nbytes // a.shape[0]

    w13 = nt * (per_expert(W.w13) + per_expert(W.w13_s) + per_expert(W.b13) + (4 if W.w13_gs is not None else 0))
    w2 = nt * (per_expert(W.w2) + per_expert(W.w2_s) + per_expert(W.b2) + (4 if W.w2_gs is not None else 0))
    io = X.x.nbytes + M * wl.K * 2 + X.topk_ids.nbytes + X.topk_weights.nbytes
    if wl.post_norm:
        io += wl.K * 2
    f1 = 2.0 * P * wl.K * (2 if wl.gated else 1) * wl.N  # gate and up rows, or h rows only
    f2 = 2.0 * P * wl.N * wl.K
    return {"bytes": w13 + w2 + io, "bytes_gemm1": w13 + X.x.nbytes, "bytes_gemm2": w2,
            "flops": f1 + f2, "flops_gemm1": f1, "flops_gemm2": f2, "pairs": P, "touched": nt}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("common.cuh", "gemm.cuh", "gemm_small.cuh", "gemm_launch.cuh"):
        h.update(open(os.path.join(ROOT, "weight_only_bit_moe_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it still matches the kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
        e = d.get(f"{workload}:{kernel}")
        if e and e.get("src_sha") == kernel_source_hash():
            return e["dram_bytes_per_launch"]
    except Exception:
        return None
    return None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        self.file.flush()
        rows = []
        try:
            for line in open(self.file.name):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        finally:
            os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows if r[3].replace(".", "").isdigit()), default=None)}


# ---------------------------------------------------------------- replicas

def max_over_ranks(values, world: int, device="cpu"):
    """Each rank's per-step times -> the slowest rank's, on every rank (no-op for one rank)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def job_tokens_per_s(world: int, M: int, ms: float) -> float:
    """Whole-job throughput: every replica processes M tokens per step of `ms` (the slowest rank)."""
    return world * M / (ms * 1e-3)


# ---------------------------------------------------------------- our arm

def kernel_name(wl, B, dom):
    kfn = "moe_gemm_small_kernel" if B <= 32 else "moe_gemm_kernel"  # register-fed below 64-token blocks
    stage = ("gated" if wl.gated else "relu2") if dom == "gemm1" else "plain"
    return f"{kfn}<{wl.fmt},{stage},BN={B}>"


def roofline(wl, M, alg, kern, B):
    """Roofline of the dominant GEMM kernel: tensor-bound when the step's FLOPs at the
    tensor peak take longer than its bytes at the HBM peak, else HBM-bound."""
    hbm, tc_burst, tc_sus, src = peaks()
    t_hbm = alg["bytes"] / (hbm * 1e9)
    t_tc = alg["flops"] / (tc_burst * 1e12)
    tensor_bound = t_tc > t_hbm
    g1, g2 = kern["gemm1"], kern["gemm2"]
    dom = "gemm1" if g1 >= g2 else "gemm2"
    dom_ms = g1 if dom == "gemm1" else g2
    if tensor_bound:
        achieved = alg[f"flops_{dom}"] / (dom_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": tc_burst, "unit": "TFLOP/s",
                "frac": round(achieved / tc_burst, 4)}
    else:
        achieved = alg[f"bytes_{dom}"] / (dom_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4)}
    roof.update({"traffic": ncu_traffic(dom, f"{wl.name}:{M}"), "kernel": kernel_name(wl, B, dom),
                 "peak_source": src, "kernel_ms": round(dom_ms, 5)})
    step = {"bytes": alg["bytes"], "flops": alg["flops"], "t_roof_us": round(max(t_hbm, t_tc) * 1e6, 3),
            "bound": "tensor" if tensor_bound else "hbm"}
    return roof, step


def describe(wl, M):
    return (f"{wl.name} M={M}: {wl.fmt} W4A16, K={wl.K} N={wl.N} E={wl.E} top_k={wl.top_k} "
            f"group={wl.group}{' bias' if wl.bias_std else ''}, act={wl.act}"
            f"{', post-norm' if wl.post_norm else ''}, routed ids={wl.n_ids}, {wl.routing}")


class Case:
    """One workload shape on the device, ready to step through the public API."""

    def __init__(self, name, M, dev, block_m=0, separate_align=False):
        from weight_only_bit_moe_gb300.layer import MoELayer, batch_to_device
        import torch
        self.wl = wl = wk.WORKLOADS[name]
        self.M = M
        self.W = wk.make_weights(wl, wk.weight_seed(wl.name))
        self.X = wk.make_batch(wl, M, wk.batch_seed(wl.name, M))
        self.alg = algorithmic(wl, self.W, self.X)
        self.layer = MoELayer.from_numpy(self.W, device=dev)
        self.x, self.ids, self.tw, pnw = batch_to_device(self.X, dev)
        self.B = block_m or self.layer.choose_block_m(M, wl.top_k, wl.n_ids)
        self.separate = separate_align
        self.a = self.layer.alloc_align(M, wl.top_k, self.B) if separate_align else None
        self.out = torch.empty((M, wl.K), dtype=torch.bfloat16, device=dev)
        self.ws = self.layer.workspace(M, wl.top_k, self.B)
        self.kw = dict(expert_base=wl.expert_base, act=wl.act, alpha=wl.alpha, limit=wl.limit,
                       post_norm_w=pnw if wl.post_norm else None, norm_eps=wl.norm_eps, out=self.out,
                       workspace=self.ws, block_m=self.B)

    def step(self, x=None, ids=None, tw=None):
        """One pass of the layer: moe_align then the forward, or the forward aligning
        the routing itself."""
        x = self.x if x is None else x
        ids = self.ids if ids is None else ids
        tw = self.tw if tw is None else tw
        a = self.layer.align(ids, self.wl.expert_base, self.B, out=self.a) if self.separate else None
        self.layer.forward(x, ids, tw, a, **self.kw)


def time_case(case, args, stream, flush, world, clocks=None):
    """Graph-replayed steps with L2 flushed before each (CUDA events on the launching
    stream), then traced eager steps for per-kernel times."""
    import torch
    from weight_only_bit_moe_gb300 import binding
    with torch.cuda.stream(stream):
        for _ in range(3):  # eager warm-up: sets kernel attributes, caches device queries
            case.step()
        stream.synchronize()
        if case.layer.status() != 0:
            raise RuntimeError(f"device status not ok after warm-up ({case.wl.name} M={case.M})")
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            case.step()
        stream.synchronize()
        for _ in range(args.warmup):
            flush.fill_(1)
            graph.replay()
        stream.synchronize()

        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        if clocks is not None:
            clocks.__enter__()
        for i in range(args.steps):
            flush.fill_(1)
            starts[i].record(stream)
            graph.replay()
            ends[i].record(stream)
        torch.cuda.synchronize()
        if clocks is not None:
            clocks.__exit__(None, None, None)
        if world > 1:
            torch.distributed.barrier()
        step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

        # per-kernel times: traced eager steps, queued behind a spin so launches run ahead
        tev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(1)
            torch.cuda._sleep(2_000_000)
            t = tev[i]
            binding.moe_set_trace_events(t[1:5])
            t[0].record(stream)
            case.step()
            binding.moe_set_trace_events(None)
        stream.synchronize()
        if case.layer.status() != 0:
            raise RuntimeError(f"device status not ok after the timed steps ({case.wl.name} M={case.M})")
    kern = {k: statistics.mean(v) for k, v in zip(
        ("prologue", "gemm1", "gemm2", "combine"),
        zip(*[(t[0].elapsed_time(t[1]), t[1].elapsed_time(t[2]), t[2].elapsed_time(t[3]), t[3].elapsed_time(t[4]))
              for t in tev]))}
    del graph
    return step_ms, kern


def time_requant(name, args, stream, flush):
    """The FP8 requantisation kernel on one of its workloads: CUDA events around each
    launch (L2 flushed before each), algorithmic bytes = every valid row read and
    written once plus its scales."""
    import torch
    from weight_only_bit_moe_gb300 import binding
    wl = wk.REQUANT_WORKLOADS[name]
    X = wk.make_requant(wl, 77)
    E, max_m, K, G = wl.E, wl.max_m, wl.K, wl.K // wl.group
    dx = torch.from_numpy(X.x).cuda()
    ds = torch.from_numpy(X.scale).cuda()
    dm = torch.from_numpy(X.masked_m).cuda()
    dS = torch.tensor([X.tensor_scale], dtype=torch.float32, device="cuda")
    out = torch.empty_like(dx)
    rows = int(np.minimum(np.maximum(X.masked_m, 0), max_m).sum())
    hint = max(1, rows // E)
    call = lambda: binding.moe_requant_fp8(dx, ds, (G * max_m, max_m, 1), dm, E, max_m, K, wl.group, dS, out,
                                           hint, stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1)
            call()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a, b in ev:
            flush.fill_(1)
            a.record(stream)
            call()
            b.record(stream)
        stream.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    nbytes = rows * (2 * K + 4 * G) + 4 * E + 4
    hbm = peaks()[0]
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"{name}: E={E} max_m={max_m} K={K} group={wl.group}, {rows} valid rows ({wl.rows})",
            "us_per_launch": round(ms * 1e3, 3), "rows_per_s": round(rows / (ms * 1e-3), 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(gbs / hbm, 4), "bytes": nbytes, "kernel": "requant_kernel"}}


def run_ours(args, rank: int, world: int):
    import torch

    from weight_only_bit_moe_gb300 import binding, build

    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or not os.path.exists(binding.LIB_PATH):
        build.build()
    if world > 1:
        torch.distributed.barrier()
    binding.load()

    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    case = Case(args.workload, args.M, dev, args.block_m, args.align == "separate")
    wl, M, B = case.wl, case.M, case.B
    clk = ClockSampler(local_rank)
    step_ms, kern = time_case(case, args, stream, flush, world, clocks=clk)
    clocks = clk.summary()

    # ---- end to end through the public API with host buffers (pinned), copies inside
    hx = torch.from_numpy(np.ascontiguousarray(case.X.x).view(np.int16)).view(torch.bfloat16).pin_memory()
    hids = torch.from_numpy(case.X.topk_ids.astype(np.int32)).pin_memory()
    hw = torch.from_numpy(case.X.topk_weights.astype(np.float32)).pin_memory()
    hout = torch.empty((M, wl.K), dtype=torch.bfloat16).pin_memory()
    dx, dids, dw = torch.empty_like(case.x), torch.empty_like(case.ids), torch.empty_like(case.tw)
    e2e_ms = []
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            flush.fill_(1)
            stream.synchronize()
            t0 = time.perf_counter()
            dx.copy_(hx, non_blocking=True)
            dids.copy_(hids, non_blocking=True)
            dw.copy_(hw, non_blocking=True)
            case.step(dx, dids, dw)
            hout.copy_(case.out, non_blocking=True)
            stream.synchronize()
            if i >= args.warmup:
                e2e_ms.append((time.perf_counter() - t0) * 1e3)
    h2d = hx.numel() * 2 + hids.numel() * 4 + hw.numel() * 4
    d2h = hout.numel() * 2

    # ---- a decode-sized shape beside the headline (HBM-bound; same timing rules)
    decode = None
    if args.decode:
        dname, dM = args.decode.split(":")
        dcase = Case(dname, int(dM), dev, 0, args.align == "separate")
        d_step, d_kern = time_case(dcase, args, stream, flush, world)
        d_ms = max_over_ranks([statistics.mean(d_step)], world, dev)[0]
        d_roof, d_sr = roofline(dcase.wl, dcase.M, dcase.alg, d_kern, dcase.B)
        d_sr["frac_of_step"] = round(d_sr["t_roof_us"] * 1e-3 / d_ms, 4)
        decode = {"workload": describe(dcase.wl, dcase.M), "block_m": dcase.B,
                  "value": round(job_tokens_per_s(world, dcase.M, d_ms), 1), "unit": "tokens/s",
                  "ms_per_step": round(d_ms, 5), "roofline": d_roof, "step_roofline": d_sr,
                  "kernels_ms": {k: round(v, 5) for k, v in d_kern.items()}}
        del dcase
        torch.cuda.empty_cache()

    # ---- the W4AFP8 activation requantisation kernel beside it
    requant = None
    if args.requant:
        requant = [time_requant(n, args, stream, flush) for n in args.requant.split(",")]

    # ---- reduce over ranks
    ms, e2e = max_over_ranks([statistics.mean(step_ms), statistics.mean(e2e_ms)], world, dev)
    if rank != 0:
        return None

    roof, step_roof = roofline(wl, M, case.alg, kern, B)
    step_roof["frac_of_step"] = round(step_roof["t_roof_us"] * 1e-3 / ms, 4)

    # ---- CPU oracle on a bounded sample of the same batch
    cpu = cpu_baseline(wl, case.W, case.X, budget_s=args.cpu_budget) if args.cpu_budget > 0 else None

    value = job_tokens_per_s(world, M, ms)
    line = {
        "metric": "MoE layer tokens/s", "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp16",
        "dtype_detail": "4-bit weights dequantised exactly to fp16 tensor-core operands, activations fp16, "
                        "fp32 accumulation, scales, bias, activation and combine; bf16 in and out",
        "data": "synthetic",
        "config": {"workload": describe(wl, M), "M": M, "block_m": B, "parallelism": f"replicas x{world}",
                   "l2": "flushed before every step", "graph": "CUDA graph replay"},
        "roofline": roof,
        "step_roofline": step_roof,
        "kernels_ms": {k: round(v, 5) for k, v in kern.items()},
        "e2e": {"value": round(job_tokens_per_s(world, M, e2e), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e, 4)},
        "gpu_launches": launches_per_step(B, args.align == "separate", M * wl.top_k * wl.K) * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "decode": decode,
        "requant": requant,
    }
    return line


def cpu_baseline(wl, W, X, budget_s: float):
    import oracle
    oracle.build()
    M = X.x.shape[0]
    n = 1
    t_used = 0.0
    # grow the sample until it takes a few seconds, within the budget
    while True:
        toks = np.arange(min(n, M), dtype=np.int32)
        t0 = time.perf_counter()
        oracle.forward_workload(wl, W, X, tokens=toks)
        dt = time.perf_counter() - t0
        t_used += dt
        if dt > 3.0 or n >= M or t_used + 4 * dt > budget_s:
            break
        n *= 4
    return {"value": round(len(toks) / dt, 3), "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle", "sample": f"first {len(toks)} of {M} tokens, one pass, fp64 C oracle"}


# ---------------------------------------------------------------- reference arm (CPU oracle)

def run_reference(args, rank: int):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    wl = wk.WORKLOADS[args.workload]
    M = args.M
    W = wk.make_weights(wl, wk.weight_seed(wl.name))
    X = wk.make_batch(wl, M, wk.batch_seed(wl.name, M))
    per_step = min(M, args.ref_tokens)
    times = []
    for i in range(args.warmup + args.steps):
        toks = (np.arange(per_step) + i * per_step) % M
        t0 = time.perf_counter()
        oracle.forward_workload(wl, W, X, tokens=toks.astype(np.int32))
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = statistics.mean(times) * 1e3
    value = per_step / (ms * 1e-3)
    return {"metric": "MoE layer tokens/s", "value": round(value, 3), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": f"{wl.name} M={M}", "M": M, "sample_tokens_per_step": per_step},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": f"{per_step} of {M} tokens per step"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wk.WORKLOADS))
    ap.add_argument("--M", type=int, default=DEFAULT_M)
    ap.add_argument("--block-m", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--ref-tokens", type=int, default=32)
    ap.add_argument("--requant", default="requant-ll-1row,requant-ll-uniform,requant-ll-skew",
                    help="FP8 requantisation workloads timed beside the headline ('' to skip)")
    ap.add_argument("--align", choices=["separate", "internal"], default="internal",
                    help="moe_align before the forward, or the forward aligning the routing itself")
    ap.add_argument("--decode", default=DEFAULT_DECODE,
                    help="name:M of a decode shape timed beside the headline ('' to skip)")
    ap.add_argument("--sweep", action="store_true",
                    help="one line per workload shape of the parity suite (analysis; not the headline line)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.sweep:
        import torch
        sweep = SWEEP
        if os.environ.get("MOE_SWEEP_ONLY"):
            keep = set(os.environ["MOE_SWEEP_ONLY"].split(","))
            sweep = [(n, m) for n, m in SWEEP if f"{n}:{m}" in keep]
        args.decode = ""
        args.requant = ""
        for name, M in sweep:
            args.workload, args.M = name, M
            line = run_ours(args, 0, 1)
            print(json.dumps(line), flush=True)
            torch.cuda.empty_cache()
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        line = run_reference(args, rank)
    else:
        if world > 1:
            import torch
            torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        line = run_ours(args, rank, world)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
