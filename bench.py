#!/usr/bin/env python3
"""Benchmark of the warp-specialized pipeline library on one GB300.

Default step: one bf16 GEMM + bias + ReLU, M = N = K = 8192 (A, B ~ N(0,1)/sqrt(K)
cast to bf16, bias ~ N(0, 0.1), seed 3), persistent CTA pairs with 256x256 tiles and
a 3-stage ring of 128-K stages -- the workload the TFLOP/s half of the metric is quoted on.  The same run
also times the bandwidth half: the TMA staged copy of an fp32 [16384, 4096]
tensor (256 MiB, U[-1e3, 1e3], seed 1) with 128x64 tiles, reported under
"staged_copy" with its own roofline.

Prints ONE JSON line.  `--impl reference` times the CPU oracle instead (the
plain binary64 triple loop on the host cores, on a bounded sample of rows).
Under torchrun each rank runs its own replica of the workload (weak scaling);
timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TFLOP/s of ReLU(A·B+bias) and GB/s of TMA staged copy, as % of GB300 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_FILES = ["gbr_ptx.cuh", "gbr_common.cuh", "gbr_internal.h", "gemm_umma.cuh",
                "split_plan.cuh", "staged_copy.cu", "gemm_ffma.cu"]


# ----------------------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "mbarrier_gemm_pipelines_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source
    has not changed since it was captured (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel_key)
    if not rec:
        return None
    if rec.get("source_hash") != kernel_source_hash(rec.get("files", KERNEL_FILES)):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.out = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]),
                             "power": float(parts[3]) if parts[3] not in ("[N/A]", "") else None,
                             "hw": parts[5], "hw_thermal": parts[6], "sw_thermal": parts[7],
                             "sw_power": parts[8]})
            except ValueError:
                continue
        if not rows:
            return None
        loaded = [r for r in rows if r["power"] is None or r["power"] > 300] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(loaded)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def dist_max(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def emit(obj):
    print(json.dumps(obj), flush=True)


# ----------------------------------------------------------------------------- CPU baseline

def cpu_gemm_sample(A, B, bias, target_s=15.0):
    """Times the binary64 oracle on the first rows of the product, as many as fit
    in about target_s seconds (calibrated on one row per thread).  Returns (TFLOP/s, rows, s)."""
    import oracle
    A32, B32, b32 = A.float(), B.float(), bias.float()
    K, N = B32.shape
    nthr = oracle.max_threads()
    cal = max(4, nthr)
    for _ in range(2):                      # the first pass pages B in and starts the threads
        t0 = time.perf_counter()
        oracle.gemm_bias_relu(A32[:cal], B32, b32)
        dt = max(time.perf_counter() - t0, 1e-6)
    rows = int(max(cal, min(A32.shape[0], cal * target_s / dt)))
    t0 = time.perf_counter()
    oracle.gemm_bias_relu(A32[:rows], B32, b32)
    dt = time.perf_counter() - t0
    return 2.0 * rows * N * K / dt / 1e12, rows, dt


def cpu_copy_sample(src, target_s=5.0):
    import numpy as np
    import oracle
    x = src.numpy()
    y = np.empty_like(x)
    n = oracle.max_threads()
    reps, t_total = 0, 0.0
    while t_total < target_s and reps < 200:
        t0 = time.perf_counter()
        oracle.copy_into(x, y, nthreads=n)
        t_total += time.perf_counter() - t0
        reps += 1
    return 2.0 * x.nbytes * reps / t_total / 1e9, reps, t_total


# ----------------------------------------------------------------------------- workloads

def gemm_flops(M, N, K):
    return 2.0 * M * N * K


def time_launches(fn, steps, stream):
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3


def time_each(fn, steps, stream):
    """Each launch between its own pair of events (a separate pass, outside the
    timed region): the per-step distribution, in seconds."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize()
    evs[0].record(stream)
    for i in range(steps):
        fn()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    return [evs[i].elapsed_time(evs[i + 1]) / 1e3 for i in range(steps)]


def step_stats(times, work, scale):
    """Median and minimum of per-step times, with the throughput each gives."""
    med, lo = statistics.median(times), min(times)
    return {"steps": len(times), "median_ms": round(med * 1e3, 4), "min_ms": round(lo * 1e3, 4),
            "value_at_median": round(work / med / scale, 2), "value_at_min": round(work / lo / scale, 2)}


def measure_copy(gbr, peaks, stages=4, steps=40, warmup=5):
    import torch
    from mbarrier_gemm_pipelines_gb300 import inputs
    src = inputs.workload("copy").cuda()
    dst = torch.empty_like(src)
    stream = torch.cuda.current_stream()
    out = {}
    for S in (2, 4, 7):
        def run():
            gbr.staged_copy(src, dst, tile=(128, 64), stages=S)
        for _ in range(warmup):
            run()
        t = time_launches(run, steps, stream)
        gbr.check_device()
        gbs = 2.0 * src.numel() * 4 * steps / t / 1e9
        out[S] = gbs
    # The same S = 4 launches without programmatic dependent launch: each
    # kernel starts only once the previous one has finished.
    gbr.launch_overlap(False)
    try:
        t_plain = time_launches(lambda: gbr.staged_copy(src, dst, tile=(128, 64), stages=stages),
                                steps, stream)
    finally:
        gbr.launch_overlap(True)
    gbr.check_device()
    plain_gbs = 2.0 * src.numel() * 4 * steps / t_plain / 1e9
    per_step = step_stats(time_each(lambda: gbr.staged_copy(src, dst, tile=(128, 64), stages=stages),
                                    20, stream), 2.0 * src.numel() * 4, 1e9)
    gbr.check_device()
    t_ref = time_launches(lambda: dst.copy_(src), steps, stream)
    torch_copy_gbs = 2.0 * src.numel() * 4 * steps / t_ref / 1e9
    achieved = out[stages]
    # Kept short and printed last on the JSON line, so that a reader that keeps
    # only the line's tail still sees the GB/s half of the metric.
    return {
        "workload": "TMA staged copy fp32 16384x4096 (256 MiB), 128x64 tiles, S=%d" % stages,
        "value": round(achieved, 1), "unit": "GB/s",
        "frac": round(achieved / peaks["hbm_gbs"], 4), "peak": peaks["hbm_gbs"],
        "by_stages": {str(k): round(v, 1) for k, v in out.items()},
        "median_gbs": per_step["value_at_median"],
        "no_overlap_gbs": round(plain_gbs, 1), "torch_copy_gbs": round(torch_copy_gbs, 1),
        "traffic": recorded_traffic("staged_copy"), "bytes_per_launch": 2 * src.numel() * 4,
    }


def measure_config4_as_written(gbr, peaks, steps=20, warmup=3):
    """bf16 8192^3 with the ring the workload names: 4-6 stages of 64 K
    (128x256x64 per CTA; S = 5-6 only fit on the CTA pair), beside the
    default 3 x 128-K ring of the headline.  TFLOP/s and fraction of the
    measured bf16 peak."""
    import torch
    from mbarrier_gemm_pipelines_gb300 import inputs
    stream = torch.cuda.current_stream()
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    A, B, bias = inputs.workload("gemm_bf16")
    dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
    dC = torch.empty((8192, 8192), dtype=torch.bfloat16, device="cuda")
    f = gemm_flops(8192, 8192, 8192)
    out = {}
    for label, pair, S in (("pair_S4_64K", 2, 4), ("pair_S5_64K", 2, 5), ("pair_S6_64K", 2, 6),
                           ("one_cta_S4_64K", 1, 4)):
        gbr.gemm_tuning(pair, -1, -1, 1)
        fn = lambda: gbr.gemm_bias_relu(dA, dB, db, dC, dtype="bf16", stages=S)
        for _ in range(warmup):
            fn()
        t = time_launches(fn, steps, stream)
        gbr.check_device()
        v = f * steps / t / 1e12
        out[label] = {"value": round(v, 1), "frac": round(v / peak, 4)}
    gbr.gemm_tuning(-1, -1, -1, -1)
    return out


def compact(workloads):
    """{name: {value, frac}} of the secondary workloads, for the JSON line."""
    if not workloads:
        return workloads
    return {k: {"value": v["value"], "frac": v.get("roofline", {}).get("frac")}
            for k, v in workloads.items()}


def measure_workloads(gbr, peaks, sm_mhz=None, steps=20, warmup=3):
    """The other GEMM workloads, each against the roofline of its own unit."""
    import torch
    from mbarrier_gemm_pipelines_gb300 import inputs
    stream = torch.cuda.current_stream()
    bf16_peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    # The ALU peak at the maximum SM clock: conservative, and independent of the
    # clock the bf16 run happened to be capped at.
    clock_ghz = peaks.get("sm_max_mhz", 2070.0) / 1e3
    fp32_alu_peak = 152 * 128 * 2 * clock_ghz / 1e3          # TFLOP/s
    out = {}

    def timed(fn, flops):
        for _ in range(warmup):
            fn()
        t = time_launches(fn, steps, stream)
        gbr.check_device()
        return flops * steps / t / 1e12, t / steps * 1e3

    A, B, bias = inputs.workload("gemm_fp32")
    dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
    dC = torch.empty((4096, 4096), device="cuda")
    f = gemm_flops(4096, 4096, 4096)
    for dt, peak, bound, unit, stage_list in (
            ("ffma", fp32_alu_peak, "alu", "FP32 FMA lanes: 152 SM x 128 x 2 x f_SM", (3, 4)),
            ("tf32", bf16_peak * 0.5, "tensor",
             "measured bf16 x 0.5 (nominal TF32:bf16 dense ratio); B read in place, MN-major",
             (3, 4))):
        for S in stage_list:
            v, ms = timed(lambda: gbr.gemm_bias_relu(dA, dB, db, dC, dtype=dt, stages=S), f)
            out["gemm_fp32_4096_%s_S%d" % (dt, S)] = {
                "value": round(v, 2), "unit": "TFLOP/s", "ms_per_call": round(ms, 4),
                "roofline": {"bound": bound, "achieved": round(v, 2), "peak": round(peak, 1),
                             "unit": "TFLOP/s", "frac": round(v / peak, 4), "peak_note": unit}}
    # The pages' central comparison on GB300: the homogeneous load/sync/compute/
    # sync loop versus the warp-specialized ring at depths 1-4 (same tile, same
    # FFMA micro-kernel).
    v, ms = timed(lambda: gbr.gemm_bias_relu(dA, dB, db, dC, dtype="ffma_sync", stages=1), f)
    out["gemm_fp32_4096_ffma_homogeneous"] = {
        "value": round(v, 2), "unit": "TFLOP/s", "ms_per_call": round(ms, 4),
        "roofline": {"bound": "alu", "achieved": round(v, 2), "peak": round(fp32_alu_peak, 1),
                     "unit": "TFLOP/s", "frac": round(v / fp32_alu_peak, 4)}}
    for S in (1, 2):
        v, ms = timed(lambda: gbr.gemm_bias_relu(dA, dB, db, dC, dtype="ffma", stages=S), f)
        out["gemm_fp32_4096_ffma_S%d" % S] = {
            "value": round(v, 2), "unit": "TFLOP/s", "ms_per_call": round(ms, 4),
            "roofline": {"bound": "alu", "achieved": round(v, 2), "peak": round(fp32_alu_peak, 1),
                         "unit": "TFLOP/s", "frac": round(v / fp32_alu_peak, 4)}}
    # The 16-warp consumer layout (8x4 micro-tiles, 4 consumer warps per
    # scheduler) beside the default 8-warp one.
    gbr.ffma_tuning(16)
    v, ms = timed(lambda: gbr.gemm_bias_relu(dA, dB, db, dC, dtype="ffma", stages=4), f)
    gbr.ffma_tuning(-1)
    out["gemm_fp32_4096_ffma_16warps_S4"] = {
        "value": round(v, 2), "unit": "TFLOP/s", "ms_per_call": round(ms, 4),
        "roofline": {"bound": "alu", "achieved": round(v, 2), "peak": round(fp32_alu_peak, 1),
                     "unit": "TFLOP/s", "frac": round(v / fp32_alu_peak, 4)}}
    # The historical producer: the same ring and consumers, fed by a cp.async
    # warpgroup instead of one TMA lane.
    for S in (2, 4):
        v, ms = timed(lambda: gbr.gemm_bias_relu(dA, dB, db, dC, dtype="ffma_cpasync", stages=S), f)
        out["gemm_fp32_4096_ffma_cpasync_S%d" % S] = {
            "value": round(v, 2), "unit": "TFLOP/s", "ms_per_call": round(ms, 4),
            "roofline": {"bound": "alu", "achieved": round(v, 2), "peak": round(fp32_alu_peak, 1),
                         "unit": "TFLOP/s", "frac": round(v / fp32_alu_peak, 4)}}
    del dA, dB, db, dC
    A, B, bias = inputs.workload("gemm_small")
    dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
    dC = torch.empty((256, 256), device="cuda")
    v, ms = timed(lambda: gbr.gemm_bias_relu(dA, dB, db, dC, dtype="ffma", stages=2),
                  gemm_flops(256, 256, 256))
    out["gemm_fp32_256_ffma_S2"] = {"value": round(v, 3), "unit": "TFLOP/s",
                                    "us_per_call": round(ms * 1e3, 2),
                                    "note": "four 128x128 tiles on 4 of 152 SMs: bound by those SMs (the same replayed from a CUDA graph)"}
    counts, X, W, b = inputs.workload("grouped_bf16")
    dX, dW, db = X.cuda(), W.cuda(), b.cuda()
    dC = torch.empty((sum(counts), W.shape[2]), dtype=torch.bfloat16, device="cuda")
    f = 2.0 * sum(counts) * W.shape[1] * W.shape[2]
    v, ms = timed(lambda: gbr.gemm_bias_relu_grouped(dX, dW, db, counts, dC, stages=3), f)
    out["grouped_bf16_moe_S3"] = {
        "value": round(v, 2), "unit": "TFLOP/s", "ms_per_call": round(ms, 4), "counts": counts,
        "roofline": {"bound": "tensor", "achieved": round(v, 2), "peak": bf16_peak,
                     "unit": "TFLOP/s", "frac": round(v / bf16_peak, 4)}}
    # The same with every expert's last tile padded to 256 rows (thin tails off).
    gbr.gemm_thin_tail(False)
    v, ms = timed(lambda: gbr.gemm_bias_relu_grouped(dX, dW, db, counts, dC, stages=3), f)
    gbr.gemm_thin_tail(True)
    out["grouped_bf16_moe_S3_no_thin"] = {
        "value": round(v, 2), "unit": "TFLOP/s", "ms_per_call": round(ms, 4),
        "roofline": {"bound": "tensor", "achieved": round(v, 2), "peak": bf16_peak,
                     "unit": "TFLOP/s", "frac": round(v / bf16_peak, 4)}}
    del dX, dW, db, dC
    # Skewed expert sizes (halving from 2048 rows): tiles of the small experts
    # stream their whole weight matrix for few rows, so tiles differ in cost.
    # Static tile order versus tiles taken from an atomic counter.
    counts = [2048, 1024, 512, 256, 128, 64, 32, 32]
    _, X, W, b = inputs.grouped(tokens=sum(counts), experts=8, K=4096, N=14336, seed=4)
    dX, dW, db = X.cuda(), W.cuda(), b.cuda()
    dC = torch.empty((sum(counts), W.shape[2]), dtype=torch.bfloat16, device="cuda")
    f = 2.0 * sum(counts) * W.shape[1] * W.shape[2]
    for label, dyn in (("static", False), ("dynamic", True)):
        gbr.gemm_dynamic_schedule(dyn)
        v, ms = timed(lambda: gbr.gemm_bias_relu_grouped(dX, dW, db, counts, dC, stages=3), f)
        out["grouped_bf16_moe_skewed_%s_S3" % label] = {
            "value": round(v, 2), "unit": "TFLOP/s", "ms_per_call": round(ms, 4), "counts": counts,
            "roofline": {"bound": "tensor", "achieved": round(v, 2), "peak": bf16_peak,
                         "unit": "TFLOP/s", "frac": round(v / bf16_peak, 4)}}
    gbr.gemm_dynamic_schedule(False)
    return out


def run_ablation(args):
    """Ring depth on the tensor-core GEMM (bf16 8192^3): one CTA or a CTA pair per
    tile, one or two 128-byte K slices per stage, every depth that fits.  Prints one
    JSON line of TFLOP/s per variant."""
    import torch
    import mbarrier_gemm_pipelines_gb300 as gbr
    from mbarrier_gemm_pipelines_gb300 import inputs
    gbr.build()
    torch.cuda.set_device(0)
    A, B, bias = inputs.workload("gemm_bf16")
    dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
    dC = torch.empty((8192, 8192), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    f = gemm_flops(8192, 8192, 8192)
    res = {}
    for pair, ks, depths in ((1, 1, (1, 2, 3, 4)), (2, 1, (1, 2, 3, 4, 5, 6)), (2, 2, (1, 2, 3))):
        for S in depths:
            gbr.gemm_tuning(pair, -1, -1, ks)
            fn = lambda: gbr.gemm_bias_relu(dA, dB, db, dC, dtype="bf16", stages=S)
            for _ in range(3):
                fn()
            t = time_launches(fn, args.steps, stream)
            gbr.check_device()
            res["pair%d_kslices%d_S%d" % (pair, ks, S)] = round(f * args.steps / t / 1e12, 1)
    gbr.gemm_tuning(-1, -1, -1, -1)
    emit({"ablation": "tensor-core ring depth, bf16 8192^3", "unit": "TFLOP/s", "results": res})


def run_ours(args):
    import torch
    import mbarrier_gemm_pipelines_gb300 as gbr
    from mbarrier_gemm_pipelines_gb300 import inputs

    world, rank, local = dist_setup()
    gbr.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()

    M = N = K = 8192
    S = args.stages
    gbr.gemm_tuning(args.pair, -1)
    A, B, bias = inputs.workload("gemm_bf16")
    dA, dB, dbias = A.to(dev), B.to(dev), bias.to(dev)
    dC = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        gbr.gemm_bias_relu(dA, dB, dbias, dC, dtype="bf16", stages=S, stream=stream)

    for _ in range(args.warmup):
        step()
    gbr.check_device()

    sampler = ClockSampler(local)
    sampler.start()
    dist_barrier(world)
    launches0 = gbr.launch_count()
    t = time_launches(step, args.steps, stream)
    launches = gbr.launch_count() - launches0
    dist_barrier(world)
    clocks = sampler.stop()
    gbr.check_device()
    flops = gemm_flops(M, N, K)
    per_step = step_stats(time_each(step, 20, stream), flops, 1e12)
    gbr.check_device()
    value, t = aggregate(t, flops * args.steps, world)
    value /= 1e12
    per_launch = t / args.steps
    achieved = flops / per_launch / 1e12

    # End to end through the C ABI's host-buffer call: every step copies its
    # pinned host A, B and bias to the device, computes, and copies C back to
    # pinned host memory.  The library overlaps a call's copies with its
    # computation chunk by chunk; consecutive steps are issued on two streams,
    # like two independent requests, so that one step's copies overlap the
    # other's, each writing its own host C.
    hA, hB, hbias = A.pin_memory(), B.pin_memory(), bias.pin_memory()
    hCs = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    streams = [stream, torch.cuda.Stream(device=dev)]
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_run(steps):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(streams[0])
        streams[1].wait_event(start)
        for i in range(steps):
            gbr.gemm_bias_relu_host(hA, hB, hbias, hCs[i % 2], dtype="bf16", stages=S,
                                    stream=streams[i % 2], sync=False)
        streams[0].wait_stream(streams[1])
        end.record(streams[0])
        torch.cuda.synchronize()
        return start.elapsed_time(end) / 1e3

    e2e_run(2)
    t_e2e = dist_max(e2e_run(e2e_steps), world)
    gbr.check_device()
    hC = hCs[(e2e_steps - 1) % 2]
    h2d = hA.numel() * 2 + hB.numel() * 2 + hbias.numel() * 4
    d2h = hC.numel() * 2

    gbr.gemm_tuning(-1, -1)
    copy = measure_copy(gbr, peaks) if rank == 0 else None
    others = config4 = None
    if rank == 0 and not args.quick:
        others = measure_workloads(gbr, peaks, sm_mhz=(clocks or {}).get("sm_mhz"))
        config4 = measure_config4_as_written(gbr, peaks)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, rows, secs = cpu_gemm_sample(A, B, bias, target_s=args.cpu_seconds)
        import oracle
        cpu = {"value": round(v, 6), "unit": "TFLOP/s", "cores": oracle.max_threads(),
               "kind": "oracle",
               "sample": "first %d of %d rows of the 8192^3 product (binary64 i-k-j loop, "
                         "%.1f s)" % (rows, M, secs)}

    if rank != 0:
        return
    if args.details:
        with open(args.details, "w") as fh:
            json.dump({"other_workloads": others, "config4_as_written": config4,
                       "staged_copy": copy}, fh, indent=1)
    # Peak for the roofline: the burst cuBLAS figure for a short timed region,
    # the sustained (power-capped) one once the region is long enough for the
    # power cap to act (>= 100 ms) or the clock samples saw it acting.
    long_run = t >= 0.1 or "sw_power_cap" in (clocks or {}).get("reasons", [])
    peak_key = "bf16_tflops_sustained" if long_run and peaks.get("bf16_tflops_sustained") else "bf16_tflops"
    other_key = "bf16_tflops" if peak_key != "bf16_tflops" else "bf16_tflops_sustained"
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "bf16 GEMM+bias+ReLU M=N=K=8192, A,B~N(0,1)/sqrt(K)->bf16, "
                               "bias f32~N(0,0.1), seed 3; persistent CTA pairs (cta_group::2), "
                               "256x256 tile per pair, %d-stage TMA/mbarrier ring "
                               "(128 of K per stage when S<=3, else 64), tcgen05 MMA into TMEM" % S,
                   "M": M, "N": N, "K": K, "stages": S,
                   "l2": "inputs larger than L2 (A+B = 256 MiB > 129 MB); no flush",
                   "parallelism": "replica per GPU" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2),
                     "peak": peaks.get(peak_key, FALLBACK_PEAKS[peak_key]), "unit": "TFLOP/s",
                     "frac": round(achieved / peaks.get(peak_key, FALLBACK_PEAKS[peak_key]), 4),
                     "traffic": recorded_traffic("gemm_umma_bf16"),
                     "peak_source": "%s %s (%s cuBLAS bf16; timed region %.3f s)" % (
                         peak_src, peak_key,
                         "sustained" if peak_key.endswith("sustained") else "burst", t),
                     "frac_of_" + ("burst" if other_key == "bf16_tflops" else "sustained"):
                         (round(achieved / peaks[other_key], 4) if peaks.get(other_key) else None)},
        "e2e": {"value": round(flops * e2e_steps / t_e2e / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "steps": e2e_steps, "api": "gemm_bias_relu_host (C ABI, pinned host buffers)",
                "streams": 2},
        "gpu_launches": int(launches),
        "per_step": per_step,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "other_workloads": compact(others),
        "config4_as_written": config4,
        "staged_copy": copy,
    }
    emit(res)


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on the machine's host cores."""
    world, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return
    import oracle
    from mbarrier_gemm_pipelines_gb300 import inputs
    oracle.build()
    A, B, bias = inputs.workload("gemm_bf16")
    A, B, bias = A.float(), B.float(), bias.float()   # widened once, not per step
    # About 150 s of oracle work over the whole run, at least 0.25 s per step.
    per_step = max(0.25, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_gemm_sample(A, B, bias, target_s=per_step)
    vals, rows_used, secs = [], 0, 0.0
    for _ in range(args.steps):
        v, rows, s = cpu_gemm_sample(A, B, bias, target_s=per_step)
        vals.append(v)
        rows_used += rows
        secs += s
    value = statistics.median(vals)
    sample = ("per step: first ~%d of 8192 rows of the 8192^3 bf16 product, binary64 i-k-j loop"
              % (rows_used // max(1, args.steps)))
    res = {
        "metric": METRIC, "impl": "reference", "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / max(1, args.steps) * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "bf16 GEMM+bias+ReLU M=N=K=8192 (oracle on a row sample)",
                   "M": 8192, "N": 8192, "K": 8192},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s",
                         "cores": oracle.max_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    emit(res)


def aggregate(per_rank_seconds, units_per_rank, world):
    """Whole-job throughput under weak scaling: every rank processed
    units_per_rank in its own time; the job took the slowest rank's time."""
    t = dist_max(per_rank_seconds, world)
    return units_per_rank * world / t, t


def run_dist_selftest():
    """Exercises the multi-rank timing path without a GPU (gloo on CPU): each
    rank reports a synthetic elapsed time, rank 0 prints the aggregate."""
    world, rank, _ = dist_setup()
    dist_barrier(world)
    t_rank = 1.0 + 0.5 * rank                    # rank r "took" 1 + r/2 seconds
    value, t = aggregate(t_rank, 10.0, world)
    dist_barrier(world)
    if rank == 0:
        emit({"selftest": "dist", "n_ranks": world, "max_seconds": t, "value": value,
              "scaling": "weak"})
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_profile_case(case, launches=2, stages=4, pair=-1):
    """A short fixed invocation for Nsight Compute: `launches` launches of one
    kernel on its workload, nothing timed, nothing printed but a status line."""
    import torch
    import mbarrier_gemm_pipelines_gb300 as gbr
    from mbarrier_gemm_pipelines_gb300 import inputs
    gbr.build()
    torch.cuda.set_device(0)
    gbr.gemm_tuning(pair, -1)
    if case == "copy":
        src = inputs.workload("copy").cuda()
        dst = torch.empty_like(src)
        fn = lambda: gbr.staged_copy(src, dst, tile=(128, 64), stages=stages)
    elif case in ("gemm_bf16", "gemm_tf32", "gemm_ffma", "gemm_ffma_sync"):
        if case == "gemm_bf16":
            A, B, bias = inputs.workload("gemm_bf16")
        else:
            A, B, bias = inputs.workload("gemm_fp32")
        dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
        dt = case[len("gemm_"):]
        fn = lambda: gbr.gemm_bias_relu(dA, dB, db, dtype=dt, stages=stages)
    elif case == "grouped":
        counts, X, W, b = inputs.workload("grouped_bf16")
        dX, dW, db = X.cuda(), W.cuda(), b.cuda()
        fn = lambda: gbr.gemm_bias_relu_grouped(dX, dW, db, counts, stages=stages)
    else:
        raise SystemExit("unknown profile case %r" % case)
    for _ in range(launches):
        fn()
    gbr.check_device()
    print("profile case %s: %d launches ok" % (case, launches))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--stages", type=int, default=3)
    ap.add_argument("--pair", type=int, default=-1, choices=[-1, 1, 2],
                    help="tensor-core GEMM variant: -1 auto, 1 one CTA per tile, 2 CTA pair")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--details", metavar="PATH",
                    help="also write the secondary workloads' full records (JSON) to PATH")
    ap.add_argument("--quick", action="store_true",
                    help="skip the secondary workloads (fp32 4096^3, 256^3, grouped MoE)")
    ap.add_argument("--ablation", action="store_true",
                    help="ring-depth sweep of the tensor-core GEMM (one JSON line)")
    ap.add_argument("--dist-selftest", action="store_true",
                    help="check the multi-rank aggregation on CPU (gloo), no GPU work")
    ap.add_argument("--profile", metavar="CASE",
                    help="run two launches of one kernel for ncu: copy, gemm_bf16, gemm_tf32, "
                         "gemm_ffma, gemm_ffma_sync or grouped")
    args = ap.parse_args()
    if args.dist_selftest:
        run_dist_selftest()
        return
    if args.ablation:
        run_ablation(args)
        return
    if args.profile:
        run_profile_case(args.profile, stages=args.stages, pair=args.pair)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
