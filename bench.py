#!/usr/bin/env python3
"""Benchmark of the BF16 TN GEMM library on GB300.

One step = one call of the hot path (gemm_bf16_tn through the C ABI) on the
8192 x 28672 x 4096 MLP up-projection (A ~ N(0,1), B ~ N(0,1/4096), bf16
out), operands resident in HBM.  Operands (288 MiB) exceed L2 (126 MiB), so
no flush is needed between steps.  Alongside it, in the same run:

* ``secondary``: the 16 x 8192 x 8192 decode GEMM in GB/s (B rotated over
  four copies, 512 MiB, so it never sits in L2);
* ``fused_bias_gelu``: the same GEMM with bias + tanh-GELU in its epilogue;
* ``scheduler_clc`` / ``grouped``: the cluster-launch-control scheduler
  against the static one, and 64 small GEMMs as separate, batched and
  grouped calls;
* ``fp8``: the e4m3 variant on both shapes (per-tensor scales folded into
  alpha), against twice the measured bf16 peak and the copy bandwidth;
* ``stream_ceiling``: gemm_stream_read over each decode's weight matrix (the
  same TMA boxes and ring, nothing else done): the read ceiling each decode
  is compared with;
* ``mma_rate``: gemm_mma_rate, the cost of one tcgen05.mma at the skinny
  path's shapes (M = 128 per CTA or 256 per pair, N = 16..256);
* ``configs``: all five workloads, each timed and set against the roofline
  min(P_tc, BW * F/Q), with the oracle's parity on its outputs;
* ``e2e``: the same metric with host buffers — pinned host->device copies
  of A and B and the device->host copy of D inside every timed step;
* ``cpu_baseline``: the FP64 CPU oracle timed on a bounded row sample of
  the workload on the host's cores (its rows also double as a parity spot
  check of the GPU result);
* ``roofline``: achieved FLOP/s of the GEMM kernel (CUDA events on the
  launching stream) against the measured dense bf16 peak.

``--impl reference`` times the reference arm instead: the CPU oracle, on
bounded row samples of the same workload, one sample per step.

Multi-GPU (``torchrun --nproc-per-node N bench.py --gpus N``): every rank
runs the full workload on its own GPU (weak scaling, no data exchange);
elapsed time is the maximum over ranks and ``value`` sums all ranks' work.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import gemm_inputs as gi  # noqa: E402
from tensor_core_dense_tn_gb300 import roofline as rl  # noqa: E402

METRIC = "BF16 GEMM TFLOP/s at 8192×28672×4096 (% of tensor peak); GB/s at M=16"
MAIN = 3       # index of the 8192x28672x4096 workload
DECODE = 4     # index of the 16x8192x8192 workload
KERNEL_SOURCES = ("gemm_api.cu", "gemm_tiled.cu", "gemm_skinny.cu", "ptx.cuh", "kernels.h", "epilogue.cuh")
# the sources each profiled kernel is built from (its traffic stays valid while they are unchanged)
TILED_SOURCES = ("gemm_api.cu", "gemm_tiled.cu", "ptx.cuh", "kernels.h", "epilogue.cuh")
SKINNY_SOURCES = ("gemm_api.cu", "gemm_skinny.cu", "ptx.cuh", "kernels.h", "epilogue.cuh")
PATH_NAMES = {1: "1sm", 2: "2sm", 3: "skinny"}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------- distributed


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def finish(self):
        if self.pg:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.period), "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)  # let the sampler come up before the timed region

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float) -> dict:
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sms, maxes, reasons, n = [], [], set(), 0
        for ts, line in self.lines:
            if not (t0 <= ts <= t1 + 0.06):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            n += 1
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sms) if sms else None,
                "sm_max_mhz": max(maxes) if maxes else None,
                "reasons": sorted(reasons), "samples": n}


# ----------------------------------------------------------------------------- helpers


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, "tensor_core_dense_tn_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, if the sources of
    the profiled kernel (the entry's `sources`, else all kernel sources) are
    unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        d = json.load(open(p))
    except (OSError, ValueError):
        return None
    e = d.get(workload_name)
    if not e:
        return None
    try:
        h = kernel_source_hash(tuple(e.get("sources") or KERNEL_SOURCES))
    except OSError:
        return None
    if e.get("source_hash") != h:
        return None
    return e.get("dram_bytes_per_launch")


def dev_bf16(bits, torch, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


# ----------------------------------------------------------------------------- our arm


def time_steps(torch, stream, fn, steps):
    """CUDA-event time of `steps` back-to-back calls on `stream` (ms total)."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        fn(i)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def run_ours(args, dist):
    import torch
    import tensor_core_dense_tn_gb300 as g

    g.load()  # fail loudly without the CUDA library
    device = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(device)
    dist.init("nccl")
    stream = torch.cuda.current_stream(device)
    s_handle = stream.cuda_stream
    peaks = rl.load_peaks()
    warmup = max(args.warmup, 3)

    w = gi.WORKLOADS[args.workload]
    if args.shape:
        M, N, K = (int(x) for x in args.shape.split(","))
        w = gi.Workload(w.index, f"custom {M}x{N}x{K}", M, N, K, w.dist_a, w.dist_b, w.dist_c,
                        w.alpha, w.beta, w.out_dtype)
    fp8 = args.in_dtype != "bf16"
    fmt = gi.FP8_E5M2 if args.in_dtype == "e5m2" else gi.FP8_E4M3
    t_gen = time.time()
    A, B, C = gi.operands(w)
    if fp8:  # the fp8 variant of the same workload: codes plus per-tensor scales
        A8, B8, scale_a, scale_b = gi.fp8_operands(w, fmt)
        dA, dB = torch.from_numpy(A8).to(device), torch.from_numpy(B8).to(device)
        del A8, B8
    else:
        dA, dB = dev_bf16(A, torch, device), dev_bf16(B, torch, device)
    log(f"[bench] inputs for {w.name} generated in {time.time() - t_gen:.1f}s")
    out_t = torch.float32 if w.out_dtype == gi.OUT_F32 else torch.bfloat16
    dC = None
    if C is not None:
        dC = dev_bf16(C, torch, device) if w.out_dtype == gi.OUT_BF16 else torch.from_numpy(C).to(device)
    dD = torch.empty((w.M, w.N), dtype=out_t, device=device)
    sched = {"default": 0, "static": 1, "clc": 2}[args.scheduler]
    cfg = g.GemmConfig(path=args.path, scheduler=sched, l2_hints=args.l2_hints, raster_group=args.raster_group,
                       cluster_pref=args.cluster_pref, tiled_k_parts=args.tiled_k_parts)
    c_ptr = dC.data_ptr() if dC is not None else 0
    ldc = w.N if dC is not None else 0

    def step(_i):
        if fp8:
            rc = g.gemm_fp8_tn(w.M, w.N, w.K, dA.data_ptr(), w.K, dB.data_ptr(), w.K, fmt, scale_a, scale_b,
                               c_ptr, ldc, dD.data_ptr(), w.N, w.alpha, w.beta, w.out_dtype, s_handle)
        else:
            rc = g.gemm_bf16_tn_ex(w.M, w.N, w.K, dA.data_ptr(), w.K, dB.data_ptr(), w.K, c_ptr, ldc,
                                   dD.data_ptr(), w.N, w.alpha, w.beta, w.out_dtype, s_handle, cfg)
        if rc != 0:
            raise RuntimeError(f"gemm failed: {rc} {g.last_error()}")

    for i in range(warmup):
        step(i)
    st = g.gemm_get_status(s_handle)
    if st != 0:
        raise RuntimeError(f"device status {st}: {g.last_error()}")
    info = g.last_launch_info()

    vis = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    smi_index = int(vis[dist.local_rank]) if len(vis) > dist.local_rank and vis[dist.local_rank].isdigit() \
        else dist.local_rank
    sampler = ClockSampler(smi_index)
    sampler.start()
    dist.barrier()
    t0 = time.time()
    ms = time_steps(torch, stream, step, args.steps)
    t1 = time.time()
    dist.barrier()
    sampler.stop()
    st = g.gemm_get_status(s_handle)
    if st != 0:
        raise RuntimeError(f"device status {st}: {g.last_error()}")
    ms = dist.max(ms)
    clocks = sampler.summary(t0, t1)

    flops = rl.gemm_flops(w.M, w.N, w.K)
    qbytes = rl.gemm_bytes(w.M, w.N, w.K, 4 if w.out_dtype == gi.OUT_F32 else 2, w.beta != 0,
                           in_bytes=1 if fp8 else 2)
    per_step_s = ms / 1e3 / args.steps
    value = dist.world * flops / per_step_s / 1e12
    achieved = flops / per_step_s / 1e12          # per launch, per GPU
    traffic = profiled_traffic(w.name if not fp8 else f"{w.name} [{args.in_dtype}]")
    ratio = 2.0 if fp8 else 1.0                   # nominal fp8 : bf16 dense ratio (4.5 : 2.25 PFLOP/s)
    peak = ratio * peaks["bf16_tflops"]
    roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
            "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
            "traffic": traffic, "algorithmic_flops": flops, "algorithmic_bytes": qbytes,
            "peak_source": (f"{'2 x ' if fp8 else ''}{peaks['source']} burst bf16 (MEASURED_PEAKS.json)"
                            if peaks["source"] == "measured" else "fallback 1.9 PFLOP/s"),
            "frac_of_sustained": round(achieved / (ratio * peaks["bf16_tflops_sustained"]), 4),
            "kernel": info.get("kernel")}

    result = {
        "metric": METRIC if not fp8 else f"FP8 ({args.in_dtype}) GEMM TFLOP/s at {w.M}x{w.N}x{w.K}",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": warmup, "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": args.in_dtype, "data": "synthetic",
        "config": dict(w.describe(), path=PATH_NAMES.get(info.get("path"), info.get("path")),
                       grid=info.get("grid"), cluster=info.get("cluster"),
                       tile=[info.get("tile_m"), info.get("tile_n")], stages=info.get("stages"),
                       scheduler={1: "static", 2: "clc"}.get(info.get("scheduler"), None),
                       l2="operands (288 MiB) larger than L2; no flush" if args.workload == MAIN and not args.shape
                       else "see workload", parallelism=f"replicas x{dist.world}"),
        "roofline": roof,
        "gpu_launches": args.steps,
        "clocks": clocks,
    }

    if fp8:  # the other legs are the bf16 path's; the fp8 main step stands alone
        result["config"].update(A=f"{args.in_dtype} codes, scale {scale_a:g}",
                                B=f"{args.in_dtype} codes, scale {scale_b:g}")
        dist.finish()
        return result

    # ---------------------------------------------------------------- fused bias + GELU
    if not args.no_secondary:
        hb = gi.draw_bf16(w.N, 1, gi.Dist("normal", 1.0), w.seed(gi.TENSOR_C)).reshape(w.N)
        dbias = dev_bf16(hb, torch, device)
        dDf = torch.empty_like(dD)   # own output: dD keeps the plain GEMM for the CPU-sample check

        def fused(_i):
            rc = g.gemm_bf16_tn_bias_act(w.M, w.N, w.K, dA.data_ptr(), w.K, dB.data_ptr(), w.K, c_ptr, ldc,
                                         dDf.data_ptr(), w.N, w.alpha, w.beta, w.out_dtype,
                                         dbias.data_ptr(), 0, g.ACT_GELU_TANH, s_handle)
            if rc != 0:
                raise RuntimeError(f"fused gemm failed: {rc} {g.last_error()}")

        for i in range(3):
            fused(i)
        f_steps = max(10, min(args.steps, 50))
        f_ms = dist.max(time_steps(torch, stream, fused, f_steps))
        if g.gemm_get_status(s_handle) != 0:
            raise RuntimeError(g.last_error())
        result["fused_bias_gelu"] = {
            "value": round(dist.world * flops / (f_ms / 1e3 / f_steps) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(f_ms / f_steps, 4), "steps": f_steps,
            "op": "D = gelu_tanh(A B^T + bias) in the GEMM epilogue (gemm_bf16_tn_bias_act)"}
        del dDf

    # ---------------------------------------------------------------- e2e (host buffers)
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, g, torch, device, w, A, B, out_t, flops, dist)

    # ---------------------------------------------------------------- decode secondary
    if not args.no_secondary:
        result["secondary"] = run_decode(args, g, torch, device, peaks, dist)
        result["decode_b_static"] = run_decode(args, g, torch, device, peaks, dist, b_static=1)
        result["fp8"] = run_fp8(args, g, torch, device, peaks, dist)
        result["stream_ceiling"] = run_stream_ceiling(args, g, torch, device, peaks, dist, result)
        result["mma_rate"] = run_mma_rate(g, torch, device)
        result["configs"] = run_configs(args, g, torch, device, peaks, dist, result, w, A, B, dD)
        result["scheduler_clc"] = run_scheduler_study(args, g, torch, device, w, dA, dB, dD, flops, peaks, dist)
        result["grouped"] = run_grouped_leg(args, g, torch, device, dist)

    # ---------------------------------------------------------------- CPU oracle baseline
    if not args.no_cpu_baseline and dist.rank == 0:
        result["cpu_baseline"] = cpu_baseline(w, A, B, C, dD, out_t, torch, args.cpu_seconds)

    dist.finish()
    return result


def run_e2e(args, g, torch, device, w, A, B, out_t, flops, dist):
    """Every step copies A and B in from pinned host memory, runs the GEMM and
    copies D back out.  Steps are pipelined the way a serving loop would run
    them: step i's host->device copies and step i-1's device->host copy run
    on their own streams while the GEMM of the step in between computes, with
    two device buffers per operand.  Timed from the first copy in to the
    last copy out."""
    hA = torch.from_numpy(np.ascontiguousarray(A).view(np.int16)).pin_memory()
    hB = torch.from_numpy(np.ascontiguousarray(B).view(np.int16)).pin_memory()
    odt = torch.int16 if out_t == torch.bfloat16 else torch.float32
    hD = torch.empty((w.M, w.N), dtype=odt).pin_memory()
    dA = [torch.empty_like(hA, device=device) for _ in range(2)]
    dB = [torch.empty_like(hB, device=device) for _ in range(2)]
    dD = [torch.empty((w.M, w.N), dtype=odt, device=device) for _ in range(2)]
    s_in, s_gemm, s_out = (torch.cuda.Stream(device) for _ in range(3))
    ev = lambda: torch.cuda.Event()
    n = max(4, min(args.steps, 20))
    cfg = g.GemmConfig(path=args.path)

    def run(steps):
        copied = [ev() for _ in range(steps)]
        computed = [ev() for _ in range(steps)]
        drained = [ev() for _ in range(steps)]
        for i in range(steps):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(computed[i - 2])      # buffer b free to overwrite
                dA[b].copy_(hA, non_blocking=True)
                dB[b].copy_(hB, non_blocking=True)
                copied[i].record(s_in)
            s_gemm.wait_event(copied[i])
            if i >= 2:
                s_gemm.wait_event(drained[i - 2])         # D buffer b read out
            rc = g.gemm_bf16_tn_ex(w.M, w.N, w.K, dA[b].data_ptr(), w.K, dB[b].data_ptr(), w.K, 0, 0,
                                   dD[b].data_ptr(), w.N, w.alpha, w.beta, w.out_dtype, s_gemm.cuda_stream, cfg)
            if rc != 0:
                raise RuntimeError(f"e2e gemm failed: {rc} {g.last_error()}")
            computed[i].record(s_gemm)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[i])
                hD.copy_(dD[b], non_blocking=True)
                drained[i].record(s_out)

    run(2)
    torch.cuda.synchronize()
    # three timed rounds, the median reported (the host link is shared with
    # the machine's other GPUs, so single rounds vary)
    rounds = []
    for _ in range(3):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(s_in)
        run(n)
        end.record(s_out)
        torch.cuda.synchronize()
        rounds.append(dist.max(start.elapsed_time(end)))
    ms = statistics.median(rounds)
    st = g.gemm_get_status(s_gemm.cuda_stream)
    if st != 0:
        raise RuntimeError(f"device status {st}: {g.last_error()}")
    per = ms / 1e3 / n

    # The transfer bound: the same copies per step on the same streams, with
    # nothing computed (a reference measurement beside the e2e number).
    def copies_only(steps):
        for i in range(steps):
            b = i % 2
            with torch.cuda.stream(s_in):
                dA[b].copy_(hA, non_blocking=True)
                dB[b].copy_(hB, non_blocking=True)
            with torch.cuda.stream(s_out):
                hD.copy_(dD[b], non_blocking=True)

    copies_only(2)
    torch.cuda.synchronize()
    # three rounds, the fastest taken: the host link is shared with the
    # machine's other GPUs, and the bound is what the link allows at best
    copy_rounds = []
    for _ in range(3):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(s_in)
        s_out.wait_event(c0)
        copies_only(n)
        done = torch.cuda.Event()
        done.record(s_out)
        s_in.wait_event(done)
        c1.record(s_in)
        torch.cuda.synchronize()
        copy_rounds.append(dist.max(c0.elapsed_time(c1)) / n)
    copy_ms = min(copy_rounds)
    moved = hA.numel() * 2 + hB.numel() * 2 + hD.numel() * hD.element_size()
    return {"value": round(dist.world * flops / per / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": hA.numel() * 2 + hB.numel() * 2,
            "d2h_bytes_per_step": hD.numel() * hD.element_size(),
            "ms_per_step": round(ms / n, 3), "steps": n,
            "rounds_ms_per_step": [round(r / n, 3) for r in rounds],
            "copies_only_ms_per_step": round(copy_ms, 3),
            "copies_only_rounds_ms_per_step": [round(r, 3) for r in copy_rounds],
            "host_link_gbs": round(moved / (copy_ms / 1e3) / 1e9, 1),
            "of_transfer_bound": round(copy_ms / (ms / n), 4),
            "api": "gemm_bf16_tn_ex (C ABI); pinned host A, B in and D out every step, "
                   "copies on their own streams, two device buffers"}


def time_eager_and_graph(torch, stream, step, steps, dist):
    """(ms eager, ms graph) for `steps` launches on `stream`: first launched one
    by one from Python, then the same launches captured once in a CUDA graph
    and replayed (how a decode loop runs).  Each is the max over ranks."""
    ms_eager = dist.max(time_steps(torch, stream, step, steps))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(steps):
            step(i)
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        graph.replay()
        ms = dist.max(time_steps(torch, stream, lambda _i: graph.replay(), 1))
    return ms_eager, ms


def run_decode(args, g, torch, device, peaks, dist, b_static=0):
    """The 16 x 8192 x 8192 decode.  b_static = 1 times the same call with the
    caller's promise that nothing still running writes B (a decode loop's
    weights), which lets each call start loading its weights during the
    previous call's tail."""
    w = gi.WORKLOADS[DECODE]
    # own stream: graph capture needs a non-default stream
    stream = torch.cuda.Stream(device)
    s_handle = stream.cuda_stream
    A, B, _ = gi.operands(w)
    dA = dev_bf16(A, torch, device)
    copies = 4
    dBs = [dev_bf16(B, torch, device) for _ in range(copies)]
    dD = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device)
    cfg = g.GemmConfig(path=0, b_static=b_static)

    def step(i):
        rc = g.gemm_bf16_tn_ex(w.M, w.N, w.K, dA.data_ptr(), w.K, dBs[i % copies].data_ptr(), w.K, 0, 0,
                               dD.data_ptr(), w.N, w.alpha, w.beta, w.out_dtype, s_handle, cfg)
        if rc != 0:
            raise RuntimeError(f"decode gemm failed: {rc} {g.last_error()}")

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    torch.cuda.synchronize()
    info = g.last_launch_info()
    steps = max(args.steps, 50)
    # every step, eager or replayed, is one full GEMM on a rotated copy of B
    ms_eager, ms = time_eager_and_graph(torch, stream, step, steps, dist)
    st = g.gemm_get_status(s_handle)
    if st != 0:
        raise RuntimeError(f"device status {st}: {g.last_error()}")
    per = ms / 1e3 / steps
    qbytes = rl.gemm_bytes(w.M, w.N, w.K)
    gbs = qbytes / per / 1e9
    traffic = profiled_traffic(w.name)
    gbs_eager = qbytes / (ms_eager / 1e3 / steps) / 1e9
    return {"metric": "BF16 GEMM GB/s at 16x8192x8192", "value": round(dist.world * gbs, 1),
            "unit": "GB/s", "ms_per_step": round(ms / steps, 5), "steps": steps,
            "launch": "CUDA graph of the steps' launches" + (
                "; gemm_tn_config.b_static = 1 (B is not written by the preceding kernels)" if b_static else ""),
            "eager": {"value": round(dist.world * gbs_eager, 1), "ms_per_step": round(ms_eager / steps, 5)},
            "tflops": round(rl.gemm_flops(w.M, w.N, w.K) / per / 1e12, 2),
            "config": dict(w.describe(), path=PATH_NAMES.get(info.get("path")), grid=info.get("grid"),
                           stages=info.get("stages"), l2=f"B rotated over {copies} copies (512 MiB)"),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": traffic,
                         "algorithmic_bytes": qbytes, "kernel": info.get("kernel"),
                         "peak_source": "measured copy bandwidth (MEASURED_PEAKS.json)"
                         if peaks["source"] == "measured" else "fallback 6.8 TB/s"}}


def run_fp8(args, g, torch, device, peaks, dist):
    """The FP8 (e4m3) variant on the two headline shapes: the 8192x28672x4096
    up-projection (tensor bound) and the 16x8192x8192 decode (HBM bound), with
    per-tensor scales folded into alpha."""
    fmt = gi.FP8_E4M3
    stream = torch.cuda.Stream(device)
    s_handle = stream.cuda_stream
    out = {}
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    for name, idx in (("mlp_e4m3", MAIN), ("decode_e4m3", DECODE)):
        w = gi.WORKLOADS[idx]
        A, B, sa, sb = gi.fp8_operands(w, fmt)
        dA = torch.from_numpy(A).to(device)
        copies = 8 if idx == DECODE else 1
        dBs = [torch.from_numpy(B).to(device) for _ in range(copies)]
        dD = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device)

        def step(i, w=w, dA=dA, dBs=dBs, dD=dD, sa=sa, sb=sb):
            rc = g.gemm_fp8_tn(w.M, w.N, w.K, dA.data_ptr(), w.K, dBs[i % len(dBs)].data_ptr(), w.K, fmt, sa, sb,
                               0, 0, dD.data_ptr(), w.N, 1.0, 0.0, gi.OUT_BF16, s_handle)
            if rc != 0:
                raise RuntimeError(f"fp8 gemm failed: {rc} {g.last_error()}")

        cfg_bs = g.GemmConfig(b_static=1)

        def step_bs(i, w=w, dA=dA, dBs=dBs, dD=dD, sa=sa, sb=sb):
            rc = g.gemm_fp8_tn_ex(w.M, w.N, w.K, dA.data_ptr(), w.K, dBs[i % len(dBs)].data_ptr(), w.K, fmt, sa,
                                  sb, 0, 0, dD.data_ptr(), w.N, 1.0, 0.0, gi.OUT_BF16, s_handle, cfg_bs)
            if rc != 0:
                raise RuntimeError(f"fp8 gemm failed: {rc} {g.last_error()}")

        with torch.cuda.stream(stream):
            for i in range(max(args.warmup, 3)):
                step(i)
        torch.cuda.synchronize()
        info = g.last_launch_info()
        flops = rl.gemm_flops(w.M, w.N, w.K)
        qbytes = rl.gemm_bytes(w.M, w.N, w.K, in_bytes=1)
        if idx == DECODE:
            steps = max(args.steps, 50)
            ms_eager, ms = time_eager_and_graph(torch, stream, step, steps, dist)
            with torch.cuda.stream(stream):
                for i in range(3):
                    step_bs(i)
            ms_bs_eager, ms_bs = time_eager_and_graph(torch, stream, step_bs, steps, dist)
        else:
            steps = max(10, min(args.steps, 100))
            ms = dist.max(time_steps(torch, stream, step, steps))
            ms_eager = ms
        st = g.gemm_get_status(s_handle)
        if st != 0:
            raise RuntimeError(f"device status {st}: {g.last_error()}")
        per = ms / 1e3 / steps
        tf, gbs = flops / per / 1e12, qbytes / per / 1e9
        entry = {"op": f"D = (alpha*scale_a*scale_b) A B^T, A and B e4m3, bf16 out ({w.M}x{w.N}x{w.K})",
                 "ms_per_step": round(ms / steps, 5), "steps": steps,
                 "config": dict(w.describe(), A="e4m3 codes of N(0,1)", B="e4m3 codes of N(0,1)",
                                scale_a=sa, scale_b=sb, path=PATH_NAMES.get(info.get("path")),
                                grid=info.get("grid"), stages=info.get("stages"))}
        if idx == DECODE:
            entry.update({"value": round(dist.world * gbs, 1), "unit": "GB/s", "tflops": round(tf, 2),
                          "launch": "CUDA graph of the steps' launches",
                          "eager": {"value": round(dist.world * qbytes / (ms_eager / 1e3 / steps) / 1e9, 1),
                                    "ms_per_step": round(ms_eager / steps, 5)},
                          "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                                       "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                                       "traffic": profiled_traffic(f"{w.name} [e4m3]"),
                                       "algorithmic_bytes": qbytes, "kernel": info.get("kernel"),
                                       "peak_source": "measured copy bandwidth"}})
            entry["config"]["l2"] = f"B rotated over {copies} copies ({copies * w.N * w.K >> 20} MiB)"
            per_bs = ms_bs / 1e3 / steps
            gbs_bs = qbytes / per_bs / 1e9
            entry["b_static"] = {
                "value": round(dist.world * gbs_bs, 1), "unit": "GB/s", "ms_per_step": round(ms_bs / steps, 5),
                "eager_ms_per_step": round(ms_bs_eager / steps, 5),
                "frac": round(gbs_bs / peaks["hbm_gbs"], 4),
                "launch": "CUDA graph; gemm_tn_config.b_static = 1 (B is not written by the preceding kernels)"}
        else:
            entry.update({"value": round(dist.world * tf, 2), "unit": "TFLOP/s",
                          "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": fp8_peak,
                                       "unit": "TFLOP/s", "frac": round(tf / fp8_peak, 4),
                                       "traffic": profiled_traffic(f"{w.name} [e4m3]"),
                                       "algorithmic_flops": flops, "kernel": info.get("kernel"),
                                       "peak_source": "2 x measured burst bf16 (the nominal fp8:bf16 "
                                                      "dense ratio, 4.5:2.25 PFLOP/s)"}})
            entry["config"]["l2"] = "operands 144 MiB + D 448 MiB per step, larger than L2; no flush"
            # the same up-projection with bias + tanh-GELU fused into its epilogue
            hb = gi.draw_bf16(w.N, 1, gi.Dist("normal", 1.0), w.seed(gi.TENSOR_C)).reshape(w.N)
            dbias = dev_bf16(hb, torch, device)
            dDf = torch.empty_like(dD)

            def fused(_i, w=w, dA=dA, dBs=dBs, sa=sa, sb=sb):
                rc = g.gemm_fp8_tn_bias_act(w.M, w.N, w.K, dA.data_ptr(), w.K, dBs[0].data_ptr(), w.K, fmt, sa, sb,
                                            0, 0, dDf.data_ptr(), w.N, 1.0, 0.0, gi.OUT_BF16, dbias.data_ptr(), 0,
                                            g.ACT_GELU_TANH, s_handle)
                if rc != 0:
                    raise RuntimeError(f"fp8 fused gemm failed: {rc} {g.last_error()}")
            with torch.cuda.stream(stream):
                for i in range(3):
                    fused(i)
            f_ms = dist.max(time_steps(torch, stream, fused, steps))
            if g.gemm_get_status(s_handle) != 0:
                raise RuntimeError(g.last_error())
            entry["bias_gelu"] = {"value": round(dist.world * flops / (f_ms / 1e3 / steps) / 1e12, 2),
                                  "unit": "TFLOP/s", "ms_per_step": round(f_ms / steps, 5), "steps": steps,
                                  "op": "D = gelu_tanh(scale_a scale_b A B^T + bias) in the epilogue "
                                        "(gemm_fp8_tn_bias_act)"}
            del dDf
        out[name] = entry
        del dA, dBs, dD
    return out


def run_stream_ceiling(args, g, torch, device, peaks, dist, result):
    """The read ceiling of each decode's weight stream: gemm_stream_read pulls
    the decode's B matrix through the same TMA boxes (128 rows x 4 k-blocks)
    into the same 216 KiB ring on the same number of CTAs, and does nothing
    else.  B is rotated over the same number of copies as in the decode
    legs, and the launches are timed the same way (graph-replayed and eager)."""
    out = {"kernel": "gemm_stream_read (TMA boxes into a shared-memory ring, data discarded)"}
    legs = [("bf16_128MiB", result.get("secondary"), 8192, 8192 * 2, 4),
            ("e4m3_64MiB", (result.get("fp8") or {}).get("decode_e4m3"), 8192, 8192, 8)]
    stream = torch.cuda.Stream(device)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    for name, dec, rows, row_bytes, copies in legs:
        if not dec:
            continue
        grid = dec["config"].get("grid") or 128
        bufs = [torch.empty(rows * row_bytes, dtype=torch.uint8, device=device).fill_(0x3C) for _ in range(copies)]
        entry = {"bytes": rows * row_bytes, "box": "128 rows x 4 k-blocks of 128 B", "copies": copies}
        for label, gsize in (("decode_grid", grid), ("all_sms", sms)):
            def step(i, gsize=gsize):
                rc = g.gemm_stream_read(bufs[i % copies].data_ptr(), rows, row_bytes, 128, 4, gsize,
                                        stream.cuda_stream)
                if rc != 0:
                    raise RuntimeError(f"stream read failed: {rc} {g.last_error()}")
            with torch.cuda.stream(stream):
                for i in range(max(args.warmup, 3)):
                    step(i)
            torch.cuda.synchronize()
            steps = max(args.steps, 50)
            ms_eager, ms = time_eager_and_graph(torch, stream, step, steps, dist)
            us, us_e = ms * 1e3 / steps, ms_eager * 1e3 / steps
            gbs = rows * row_bytes / (us * 1e-6) / 1e9
            entry[label] = {"grid": gsize, "us": round(us, 3), "gbs": round(gbs, 1),
                            "frac_of_copy_peak": round(gbs / peaks["hbm_gbs"], 4),
                            "eager_us": round(us_e, 3)}
        if g.gemm_get_status(stream.cuda_stream) != 0:
            raise RuntimeError(g.last_error())
        dec_us = dec["ms_per_step"] * 1e3
        entry["decode_us"] = round(dec_us, 3)
        # the decode moves A and D as well; the ceiling streams B alone
        entry["decode_frac_of_stream_ceiling"] = round(entry["decode_grid"]["us"] / dec_us, 4)
        dec.setdefault("roofline", {})["frac_of_stream_ceiling"] = entry["decode_frac_of_stream_ceiling"]
        bs = result.get("decode_b_static") if name.startswith("bf16") else dec.get("b_static")
        if bs:
            bs_us = bs["ms_per_step"] * 1e3
            entry["decode_b_static_us"] = round(bs_us, 3)
            entry["decode_b_static_frac_of_stream_ceiling"] = round(entry["decode_grid"]["us"] / bs_us, 4)
        out[name] = entry
        del bufs
    return out


def run_mma_rate(g, torch, device):
    """gemm_mma_rate on every SM: nanoseconds per tcgen05.mma instruction at
    M = 128 rows per CTA (one CTA or a pair) against N, and the weight bytes
    each SM's tensor core consumes per nanosecond at that rate (each
    instruction reads 128 rows x 32 bytes of K per CTA)."""
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    out = torch.zeros(2, dtype=torch.int64, device=device)
    stream = torch.cuda.current_stream(device).cuda_stream
    reps = 4096
    res = {"reps": reps, "mma_per_rep": 4, "grid": sms}
    for fp8, kind in ((0, "bf16"), (1, "e4m3")):
        for cg in (1, 2):
            row = {}
            for n in (16, 32, 64, 128, 160, 192, 224, 256):
                for _ in range(2):
                    rc = g.gemm_mma_rate(n, cg, fp8, reps, sms - sms % cg, out.data_ptr(), stream)
                    if rc != 0:
                        raise RuntimeError(f"mma rate failed: {rc} {g.last_error()}")
                torch.cuda.synchronize()
                ns = float(out[0].item()) / (reps * 4)
                row[str(n)] = {"ns_per_mma": round(ns, 2), "weight_bytes_per_ns_per_sm": round(128 * 32 / ns, 1)}
            res[f"{kind}_cta_group{cg}"] = row
    if g.gemm_get_status(stream) != 0:
        raise RuntimeError(g.last_error())
    return res


def run_configs(args, g, torch, device, peaks, dist, result, w_main, A_main, B_main, dD_main):
    """All five workloads in one table: each timed in the launch configuration
    the automatic path picks, against the roofline min(P_tc, BW * F/Q) (the
    measured bf16 burst peak and copy bandwidth), with the oracle's parity on
    a sample of its outputs (every output for the two small-output shapes).
    Operand sets are rotated so that the bytes touched between two uses of
    one set exceed L2.  The up-projection and the decode reuse the main and
    secondary legs' timings."""
    import oracle
    l2 = torch.cuda.get_device_properties(device).L2_cache_size if hasattr(
        torch.cuda.get_device_properties(device), "L2_cache_size") else 126 << 20
    P, BW = peaks["bf16_tflops"], peaks["hbm_gbs"]
    out = {"roofline": "min(measured bf16 burst peak, measured copy GB/s x F/Q)", "l2_bytes": l2}
    stream = torch.cuda.Stream(device)
    sh = stream.cuda_stream
    for w in gi.WORKLOADS:
        out_bytes = 4 if w.out_dtype == gi.OUT_F32 else 2
        entry = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha, "beta": w.beta,
                 "out": "f32" if w.out_dtype == gi.OUT_F32 else "bf16"}
        if w.index == MAIN and args.workload == MAIN and not args.shape:
            A, B, C = A_main, B_main, None
            dD = dD_main
            us = result["ms_per_step"] * 1e3
            entry.update(us_per_call=round(us, 3), launch="eager (main leg)", steps=result["steps"])
        elif w.index == DECODE:
            A, B, C = gi.operands(w)
            sec = result["secondary"]
            us = sec["ms_per_step"] * 1e3
            entry.update(us_per_call=round(us, 3), launch="CUDA graph (secondary leg)", steps=sec["steps"],
                         eager_us_per_call=round(sec["eager"]["ms_per_step"] * 1e3, 3))
            dD = None
        else:
            A, B, C = gi.operands(w)
            set_bytes = rl.gemm_bytes(w.M, w.N, w.K, out_bytes, w.beta != 0)
            copies = max(2, -(-int(1.5 * l2) // set_bytes))
            dA = [dev_bf16(A, torch, device) for _ in range(copies)]
            dB = [dev_bf16(B, torch, device) for _ in range(copies)]
            dC = None
            if C is not None:
                dC = [dev_bf16(C, torch, device) if w.out_dtype == gi.OUT_BF16 else torch.from_numpy(C).to(device)
                      for _ in range(copies)]
            odt = torch.float32 if w.out_dtype == gi.OUT_F32 else torch.bfloat16
            dDs = [torch.empty((w.M, w.N), dtype=odt, device=device) for _ in range(copies)]

            def step(i, w=w, dA=dA, dB=dB, dC=dC, dDs=dDs, copies=copies):
                j = i % copies
                rc = g.gemm_bf16_tn(w.M, w.N, w.K, dA[j].data_ptr(), w.K, dB[j].data_ptr(), w.K,
                                    dC[j].data_ptr() if dC is not None else 0, w.N if dC is not None else 0,
                                    dDs[j].data_ptr(), w.N, w.alpha, w.beta, w.out_dtype, sh)
                if rc != 0:
                    raise RuntimeError(f"gemm failed: {rc} {g.last_error()}")

            with torch.cuda.stream(stream):
                for i in range(max(args.warmup, 3) + copies):
                    step(i)
            torch.cuda.synchronize()
            info = g.last_launch_info()
            steps = max(args.steps, 50) if w.index != 0 else max(args.steps, 400)
            ms_eager, ms = time_eager_and_graph(torch, stream, step, steps, dist)
            if g.gemm_get_status(sh) != 0:
                raise RuntimeError(g.last_error())
            us = ms * 1e3 / steps
            entry.update(us_per_call=round(us, 3), launch="CUDA graph of the steps' launches", steps=steps,
                         eager_us_per_call=round(ms_eager * 1e3 / steps, 3),
                         path=PATH_NAMES.get(info.get("path")), grid=info.get("grid"),
                         tile=[info.get("tile_m"), info.get("tile_n")],
                         l2=f"{copies} operand sets rotated ({copies * set_bytes >> 20} MiB)")
            dD = dDs[(steps - 1) % copies]
        roof = rl.roofline_entry(w.M, w.N, w.K, us * 1e-6, P, BW, out_bytes, w.beta != 0)
        entry["value"] = round(dist.world * roof["achieved_tflops"], 3)
        entry["unit"] = "TFLOP/s"
        entry["gbs"] = roof["achieved_gbs"]
        entry["roofline"] = roof
        if w.index == 0:
            entry["note"] = "launch-bound: 0.5 MiB of operands, a few microseconds per call"
        # parity: every output of the small-output shapes, sampled elsewhere
        if dD is None:  # decode: recompute on its own buffers
            dA1, dB1 = dev_bf16(A, torch, device), dev_bf16(B, torch, device)
            dD = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device)
            with torch.cuda.stream(stream):
                if g.gemm_bf16_tn(w.M, w.N, w.K, dA1.data_ptr(), w.K, dB1.data_ptr(), w.K, 0, 0, dD.data_ptr(), w.N,
                                  w.alpha, w.beta, w.out_dtype, sh) != 0:
                    raise RuntimeError(g.last_error())
            torch.cuda.synchronize()
        got = (dD.view(torch.int16).cpu().numpy().view(np.uint16) if w.out_dtype == gi.OUT_BF16
               else dD.cpu().numpy())
        cvals = None if C is None else (gi.bf16_bits_to_f32(C) if w.out_dtype == gi.OUT_BF16 else C)
        if w.M * w.N <= 1 << 18:
            ref, absdot = oracle.gemm_ref(A, B, C, w.alpha, w.beta)
            ok, worst, _ = oracle.check(got, ref, absdot, w.out_dtype, w.beta, cvals)
            exact = bool(np.array_equal(got, oracle.exact_f32(ref))) if w.index == 0 else None
            entry["parity"] = {"checked": "every output", "ok": bool(ok), "worst_err_over_bound": round(worst, 4)}
            if exact is not None:
                entry["parity"]["bit_exact"] = exact
        else:
            rng = np.random.default_rng(77 + w.index)
            rows = rng.integers(0, w.M, 3000)
            cols = rng.integers(0, w.N, 3000)
            rows = np.concatenate([rows, [0, w.M - 1, w.M - 1, 0]])
            cols = np.concatenate([cols, [0, w.N - 1, 0, w.N - 1]])
            ref, absdot = oracle.gemm_ref_sampled(A, B, rows, cols, C, w.alpha, w.beta)
            cs = None if cvals is None else cvals[rows, cols]
            ok, worst, _ = oracle.check(got[rows, cols], ref, absdot, w.out_dtype, w.beta, cs)
            entry["parity"] = {"checked": f"{rows.size} sampled outputs incl. corners", "ok": bool(ok),
                               "worst_err_over_bound": round(worst, 4)}
        out[str(w.index + 1)] = entry
        if "l2" in entry:
            del dA, dB, dC, dDs
        torch.cuda.empty_cache()
    return out


def run_scheduler_study(args, g, torch, device, w, dA, dB, dD, flops, peaks, dist):
    """The cluster-launch-control tile scheduler against the static persistent
    grid: (1) the main GEMM under CLC on an idle GPU; (2) an 8192x8192x4096
    GEMM started while another kernel (a 1-SM GEMM with one long tile per CTA)
    holds 64 of the SMs for ~0.45 ms, where a static grid cannot place all its
    CTAs and CLC lets the resident ones take the missing CTAs' tiles."""
    stream = torch.cuda.current_stream(device)
    s_handle = stream.cuda_stream

    def stepper(sched):
        cfg = g.GemmConfig(scheduler=sched)

        def step(_i):
            rc = g.gemm_bf16_tn_ex(w.M, w.N, w.K, dA.data_ptr(), w.K, dB.data_ptr(), w.K, 0, 0, dD.data_ptr(),
                                   w.N, w.alpha, w.beta, w.out_dtype, s_handle, cfg)
            if rc != 0:
                raise RuntimeError(f"gemm failed: {rc} {g.last_error()}")
        return step

    # interleaved rounds with equal step counts, so that clock and power
    # drift over the run falls on both schedulers alike
    steps = max(10, min(args.steps, 30))
    tf = {"static": [], "clc": []}
    for r in range(4):
        order = (("static", g.SCHED_STATIC), ("clc", g.SCHED_CLC))
        for name, sched in (order if r % 2 == 0 else order[::-1]):
            step = stepper(sched)
            for i in range(2):
                step(i)
            ms = dist.max(time_steps(torch, stream, step, steps))
            tf[name].append(flops / (ms / 1e3 / steps) / 1e12)
    if g.gemm_get_status(s_handle) != 0:
        raise RuntimeError(g.last_error())
    med = {k: statistics.median(v) for k, v in tf.items()}
    out = {"main_interleaved": {"unit": "TFLOP/s", "steps_per_round": steps, "rounds": 4,
                                "static": round(dist.world * med["static"], 2),
                                "clc": round(dist.world * med["clc"], 2),
                                "clc_over_static": round(med["clc"] / med["static"], 4)}}

    # shared GPU: background kernel on 64 SMs, then the GEMM on its own stream
    bg_ctas, kb = 64, 65536
    bgA = torch.zeros((128 * bg_ctas, kb), dtype=torch.bfloat16, device=device)
    bgB = torch.zeros((256, kb), dtype=torch.bfloat16, device=device)
    bgD = torch.empty((128 * bg_ctas, 256), dtype=torch.bfloat16, device=device)
    M = N = 8192
    K = 4096
    sA = dA[:M, :K] if dA.shape[0] >= M else None
    sB = dB[:N, :K] if dB.shape[0] >= N else None
    if sA is None or sB is None or w.K != K:
        return out
    s_bg, s_main = torch.cuda.Stream(device), torch.cuda.Stream(device)
    bg_cfg = g.GemmConfig(path=g.PATH_1SM, grid=bg_ctas, scheduler=g.SCHED_STATIC)
    dDs = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    times = {"static": [], "clc": []}
    for rep in range(4):
        for name, sched in (("static", g.SCHED_STATIC), ("clc", g.SCHED_CLC)):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            rc = g.gemm_bf16_tn_ex(128 * bg_ctas, 256, kb, bgA.data_ptr(), kb, bgB.data_ptr(), kb, 0, 0,
                                   bgD.data_ptr(), 256, 1.0, 0.0, gi.OUT_BF16, s_bg.cuda_stream, bg_cfg)
            if rc != 0:
                raise RuntimeError(g.last_error())
            with torch.cuda.stream(s_main):
                torch.cuda._sleep(40000)   # ~20 us: the background CTAs are resident by now
                e0.record(s_main)
                rc = g.gemm_bf16_tn_ex(M, N, K, sA.data_ptr(), w.K, sB.data_ptr(), w.K, 0, 0, dDs.data_ptr(), N,
                                       1.0, 0.0, gi.OUT_BF16, s_main.cuda_stream, g.GemmConfig(scheduler=sched))
                if rc != 0:
                    raise RuntimeError(g.last_error())
                e1.record(s_main)
            torch.cuda.synchronize()
            if rep > 0:  # the first round warms both paths up
                times[name].append(e0.elapsed_time(e1) * 1e3)
    if g.gemm_get_status(s_main.cuda_stream) != 0:
        raise RuntimeError(g.last_error())
    med = {k: statistics.median(v) for k, v in times.items()}
    out["shared_gpu"] = {"gemm": "8192x8192x4096 bf16", "other_kernel": f"1-SM GEMM on {bg_ctas} SMs, ~0.45 ms",
                         "static_us": round(med["static"], 1), "clc_us": round(med["clc"], 1),
                         "clc_speedup": round(med["static"] / med["clc"], 3), "repeats": len(times["clc"])}
    del bgA, bgB, bgD, dDs
    return out


def run_grouped_leg(args, g, torch, device, dist):
    """Many small GEMMs: 64 problems of the 256 x 256 x 256 shape as 64
    separate launches, as one strided batched call and as one grouped call.
    Each form is captured in a CUDA graph (10 calls) and replayed, so the
    numbers are GPU time, not host launch cost; the host time per call is
    given beside them."""
    P, M, N, K = 64, 256, 256, 256
    w0 = gi.WORKLOADS[0]
    A = dev_bf16(gi.draw_bf16(P * M, K, w0.dist_a, w0.seed(gi.TENSOR_A)), torch, device)
    B = dev_bf16(gi.draw_bf16(P * N, K, w0.dist_b, w0.seed(gi.TENSOR_B)), torch, device)
    D = torch.empty((P * M, N), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.Stream(device)
    sh = stream.cuda_stream
    probs = [g.GemmProblem(M=M, N=N, K=K, A=A.data_ptr() + 2 * p * M * K, lda=K, B=B.data_ptr() + 2 * p * N * K,
                           ldb=K, C=0, ldc=0, D=D.data_ptr() + 2 * p * M * N, ldd=N) for p in range(P)]

    def separate(_i):
        for q in probs:
            if g.gemm_bf16_tn(M, N, K, q.A, K, q.B, K, 0, 0, q.D, N, 1.0, 0.0, gi.OUT_BF16, sh) != 0:
                raise RuntimeError(g.last_error())

    def batched(_i):
        if g.gemm_bf16_tn_batched(P, M, N, K, A.data_ptr(), K, M * K, B.data_ptr(), K, N * K, 0, 0, 0,
                                  D.data_ptr(), N, M * N, 1.0, 0.0, gi.OUT_BF16, sh) != 0:
            raise RuntimeError(g.last_error())

    def grouped(_i):
        if g.gemm_bf16_tn_grouped(probs, 1.0, 0.0, gi.OUT_BF16, sh) != 0:
            raise RuntimeError(g.last_error())

    flops = 2.0 * P * M * N * K
    out = {"problems": f"{P} x {M}x{N}x{K} bf16 (int[-4,4] inputs)", "unit": "TFLOP/s"}
    calls = 10
    for name, fn, launches in (("separate", separate, P), ("batched", batched, 1), ("grouped", grouped, 2)):
        with torch.cuda.stream(stream):
            fn(0)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for i in range(calls):
                fn(i)
            torch.cuda.synchronize()
            host_us = (time.perf_counter() - t0) / calls * 1e6
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for i in range(calls):
                    fn(i)
            graph.replay()
            ms = dist.max(time_steps(torch, stream, lambda _i: graph.replay(), 5)) / 5
        per = ms / 1e3 / calls
        out[name] = {"value": round(dist.world * flops / per / 1e12, 2), "us_per_call": round(per * 1e6, 2),
                     "launches_per_call": launches, "host_us_per_call_eager": round(host_us, 1)}
    if g.gemm_get_status(sh) != 0:
        raise RuntimeError(g.last_error())
    del A, B, D
    return out


def cpu_baseline(w, A, B, C, dD, out_t, torch, seconds):
    """Time the CPU oracle on a row sample sized to ~`seconds`; compare those rows with the GPU."""
    import oracle
    threads = oracle.default_threads()
    per_row = 2.0 * w.N * w.K
    t = time.time()
    oracle.gemm_ref(A[:threads], B, None if C is None else C[:threads], w.alpha, w.beta)
    rate = threads * per_row / max(time.time() - t, 1e-3)
    rows = int(max(threads, min(w.M, seconds * rate / per_row)))
    r0 = (w.M - rows) // 2
    t = time.time()
    ref, absdot = oracle.gemm_ref(A[r0:r0 + rows], B, None if C is None else C[r0:r0 + rows], w.alpha, w.beta)
    dt = time.time() - t
    if out_t == torch.bfloat16:
        got = dD[r0:r0 + rows].view(torch.int16).cpu().numpy().view(np.uint16)
        od = gi.OUT_BF16
    else:
        got = dD[r0:r0 + rows].cpu().numpy()
        od = gi.OUT_F32
    cvals = None if C is None else (gi.bf16_bits_to_f32(C[r0:r0 + rows]) if od == gi.OUT_BF16 else C[r0:r0 + rows])
    ok, worst, _ = oracle.check(got, ref, absdot, od, w.beta, cvals)
    if not ok:
        log(f"[bench] WARNING: GPU rows disagree with the oracle on the CPU sample (worst {worst:.3g} x bound)")
    # one host thread on the two small workloads, in full: the 256^3 exact
    # GEMM and the 16 x 8192 x 8192 decode
    one_thread = {}
    for wi in (0, DECODE):
        ws = gi.WORKLOADS[wi]
        As, Bs, Cs = gi.operands(ws)
        t1 = time.time()
        oracle.gemm_ref(As, Bs, Cs, ws.alpha, ws.beta, nthreads=1)
        d1 = time.time() - t1
        one_thread[ws.name] = {"seconds": round(d1, 3), "value": round(ws.flops / d1 / 1e12, 6),
                               "unit": "TFLOP/s", "cores": 1, "sample": "every output"}
    return {"value": round(rows * per_row / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "sample": f"rows {r0}..{r0 + rows - 1} of {w.M} ({rows} x {w.N} outputs, "
                                        f"K={w.K}) in {dt:.1f}s",
            "parity_on_sample": {"ok": bool(ok), "worst_err_over_bound": round(worst, 4)},
            "one_thread": one_thread}



# ----------------------------------------------------------------------------- automatic-path check


def run_path_check(args):
    """The automatic path against every forced choice (1-SM and 2-SM tiles,
    each unsplit and in 2 and 4 k-parts, and the streaming kernel) over a
    grid of shapes: M 1..512 tokens, N 1024..28672, K 1024..8192, bf16,
    graph-replayed, B rotated over copies so that large weights stream from
    HBM.  Prints one JSON line: per shape the automatic choice's time and the
    fastest forced choice's, and the mean and worst ratio."""
    import torch
    import tensor_core_dense_tn_gb300 as g
    g.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    sh = stream.cuda_stream
    opts = [dict(path=0), dict(path=1, tiled_k_parts=1), dict(path=1, tiled_k_parts=2), dict(path=1, tiled_k_parts=4),
            dict(path=2, tiled_k_parts=1), dict(path=2, tiled_k_parts=2), dict(path=2, tiled_k_parts=4), dict(path=3)]
    names = ["auto", "1sm", "1sm_split2", "1sm_split4", "2sm", "2sm_split2", "2sm_split4", "skinny"]

    def timeit(M, N, K, Bs, A, D, opt):
        cfg = g.GemmConfig(**opt)

        def step(i):
            rc = g.gemm_bf16_tn_ex(M, N, K, A.data_ptr(), K, Bs[i % len(Bs)].data_ptr(), K, 0, 0, D.data_ptr(), N,
                                   1.0, 0.0, gi.OUT_BF16, sh, cfg)
            if rc != 0:
                raise ValueError(g.last_error())
        with torch.cuda.stream(stream):
            step(0)
            torch.cuda.synchronize()
            info = g.last_launch_info()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for i in range(30):
                    step(i)
            graph.replay()
            torch.cuda.synchronize()
            t = []
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                t.append(e0.elapsed_time(e1) / 30 * 1e3)
        if g.gemm_get_status(sh) != 0:
            raise RuntimeError(g.last_error())
        return sorted(t)[1], info

    rows, ratios = [], []
    Ms = [int(x) for x in args.path_check_m.split(",")]
    Ns = [int(x) for x in args.path_check_n.split(",")]
    Ks = [int(x) for x in args.path_check_k.split(",")]
    for K in Ks:
        for N in Ns:
            copies = max(2, min(4, int(600 * 2 ** 20 // (N * K * 2))))
            Bs = [torch.empty(N, K, device=dev, dtype=torch.bfloat16).normal_(0, 0.01) for _ in range(copies)]
            for M in Ms:
                A = torch.empty(M, K, device=dev, dtype=torch.bfloat16).normal_()
                D = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
                res = {}
                for name, opt in zip(names, opts):
                    try:
                        us, info = timeit(M, N, K, Bs, A, D, opt)
                        res[name] = (round(us, 2), info["path"], info["k_parts"])
                    except ValueError:
                        pass  # a forced path that cannot run the shape
                best_name = min((n for n in res if n != "auto"), key=lambda n: res[n][0])
                ratio = res["auto"][0] / res[best_name][0]
                ratios.append(ratio)
                rows.append({"shape": [M, N, K], "auto_us": res["auto"][0],
                             "auto_path": PATH_NAMES.get(res["auto"][1], res["auto"][1]),
                             "auto_k_parts": res["auto"][2], "best": best_name, "best_us": res[best_name][0],
                             "ratio": round(ratio, 4)})
                log(f"[path-check] {M}x{N}x{K}: auto {res['auto'][0]} us, best {best_name} {res[best_name][0]} us")
                del A, D
            del Bs
            torch.cuda.empty_cache()
    return {"path_check": {"shapes": len(rows), "mean_ratio": round(statistics.mean(ratios), 4),
                           "max_ratio": round(max(ratios), 4), "over_1.05": sum(r > 1.05 for r in ratios),
                           "launch": "CUDA graph of 30 calls, median of 3 replays, B rotated over copies",
                           "rows": rows}}


def run_box_rate(args):
    """gemm_stream_read over four copies of a 128 MiB matrix (8192 rows of
    16 KiB, as the decode's bf16 weights) on 128 CTAs, for each TMA box shape
    (rows x k-blocks of 128 bytes): microseconds per 128 MiB and GB/s per SM.
    The ring holds as many stages of the box as fit 216 KiB (at most 64)."""
    import torch
    import tensor_core_dense_tn_gb300 as g
    g.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    rows, row_bytes, copies, grid = 8192, 16384, 4, 128
    bufs = [torch.zeros(rows * row_bytes, dtype=torch.uint8, device=dev) for _ in range(copies)]
    out = []
    for box_rows, kgroup in ((32, 1), (64, 1), (128, 1), (64, 2), (128, 2), (128, 4), (256, 1), (64, 4)):
        def step(i, box_rows=box_rows, kgroup=kgroup):
            rc = g.gemm_stream_read(bufs[i % copies].data_ptr(), rows, row_bytes, box_rows, kgroup, grid,
                                    stream.cuda_stream)
            if rc != 0:
                raise RuntimeError(g.last_error())
        with torch.cuda.stream(stream):
            for i in range(6):
                step(i)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for i in range(40):
                    step(i)
            graph.replay()
            t = []
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                t.append(e0.elapsed_time(e1) * 1e3 / 40)
        us = statistics.median(t)
        box = box_rows * 128 * kgroup
        stages = min(64, 216 * 1024 // box)
        out.append({"box_rows": box_rows, "k_blocks": kgroup, "box_kib": box // 1024, "stages": stages,
                    "us": round(us, 2), "gbs": round(rows * row_bytes / us / 1e3, 1),
                    "gbs_per_sm": round(rows * row_bytes / us / 1e3 / grid, 1)})
    if g.gemm_get_status(stream.cuda_stream) != 0:
        raise RuntimeError(g.last_error())
    return {"box_rate": {"bytes": rows * row_bytes, "copies": copies, "grid": grid,
                         "launch": "CUDA graph of 40 calls, median of 3 replays", "rows": out}}


def run_stream_grid(args):
    """gemm_stream_read over four copies of a 128 MiB matrix with 8 to 152
    CTAs streaming, for 64 KiB boxes (128 rows x 4 k-blocks, the decode's)
    and 16 KiB boxes (128 rows x 1 k-block, the tiled kernels' B box):
    GB/s in all and per streaming SM.  Shows what one SM's TMA stream can
    take from HBM, which bounds GEMMs whose tiles occupy few SMs."""
    import torch
    import tensor_core_dense_tn_gb300 as g
    g.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rows, row_bytes, copies = 8192, 16384, 4
    bufs = [torch.zeros(rows * row_bytes, dtype=torch.uint8, device=dev) for _ in range(copies)]
    out = []
    for box_rows, kgroup in ((128, 4), (128, 1)):
        for grid in (8, 16, 32, 64, 96, 128, sms):
            def step(i, box_rows=box_rows, kgroup=kgroup, grid=grid):
                rc = g.gemm_stream_read(bufs[i % copies].data_ptr(), rows, row_bytes, box_rows, kgroup, grid,
                                        stream.cuda_stream)
                if rc != 0:
                    raise RuntimeError(g.last_error())
            n = 8 if grid < 32 else 20
            with torch.cuda.stream(stream):
                for i in range(4):
                    step(i)
                torch.cuda.synchronize()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=stream):
                    for i in range(n):
                        step(i)
                graph.replay()
                t = []
                for _ in range(3):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    graph.replay()
                    e1.record(stream)
                    torch.cuda.synchronize()
                    t.append(e0.elapsed_time(e1) * 1e3 / n)
            us = statistics.median(t)
            out.append({"box_rows": box_rows, "k_blocks": kgroup, "grid": grid, "us": round(us, 2),
                        "gbs": round(rows * row_bytes / us / 1e3, 1),
                        "gbs_per_sm": round(rows * row_bytes / us / 1e3 / grid, 1)})
    if g.gemm_get_status(stream.cuda_stream) != 0:
        raise RuntimeError(g.last_error())
    return {"stream_grid": {"bytes": rows * row_bytes, "copies": copies,
                            "launch": "CUDA graph of 8-20 calls, median of 3 replays", "rows": out}}


def run_sustained(args):
    """The up-projection (bf16, or --in-dtype e4m3) back to back for
    --sustained seconds: CUDA graphs of 20 calls replayed without a pause,
    each replay timed with events, the SM clock, power and throttle reasons
    sampled by nvidia-smi.  Reports the first replay, the settled rate (the
    median of the last half) and the clocks of each half: the power-capped
    regime a seconds-long GEMM settles into."""
    import torch
    import tensor_core_dense_tn_gb300 as g
    g.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fp8 = args.in_dtype != "bf16"
    w = gi.WORKLOADS[MAIN]
    M, N, K = w.M, w.N, w.K
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    if fp8:
        A = (torch.randn(M, K, device=dev, generator=gen) * 4).to(torch.float8_e4m3fn)
        B = (torch.randn(N, K, device=dev, generator=gen) * 4).to(torch.float8_e4m3fn)
    else:
        A = torch.randn(M, K, device=dev, generator=gen).bfloat16()
        B = (torch.randn(N, K, device=dev, generator=gen) / 64).bfloat16()
    D = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(dev)
    sh = stream.cuda_stream

    def call():
        if fp8:
            rc = g.gemm_fp8_tn(M, N, K, A.data_ptr(), K, B.data_ptr(), K, gi.FP8_E4M3, 0.25, 0.25, 0, 0,
                               D.data_ptr(), N, 1.0, 0.0, gi.OUT_BF16, sh)
        else:
            rc = g.gemm_bf16_tn(M, N, K, A.data_ptr(), K, B.data_ptr(), K, 0, 0, D.data_ptr(), N, 1.0, 0.0,
                                gi.OUT_BF16, sh)
        if rc != 0:
            raise RuntimeError(g.last_error())
    n = 20
    with torch.cuda.stream(stream):
        call()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(n):
                call()
        torch.cuda.synchronize()
        time.sleep(1.0)   # start from idle
        clocks = ClockSampler(torch.cuda.current_device(), period_ms=50)
        clocks.start()
        t_start = time.time()
        t_end = t_start + args.sustained
        evs = []
        while time.time() < t_end:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            evs.append((e0, e1))
            if len(evs) % 4 == 0:
                evs[-4][1].synchronize()
        torch.cuda.synchronize()
        t_stop = time.time()
        clocks.stop()
    if g.gemm_get_status(sh) != 0:
        raise RuntimeError(g.last_error())
    us = [e0.elapsed_time(e1) / n * 1e3 for e0, e1 in evs]
    half = len(us) // 2
    tf = lambda u: 2 * M * N * K / (u * 1e-6) / 1e12
    mid = t_start + (t_stop - t_start) / 2
    first, settled = us[0], statistics.median(us[half:])
    return {"sustained": {
        "workload": w.name, "dtype": "e4m3" if fp8 else "bf16", "seconds": round(t_stop - t_start, 2),
        "calls": len(us) * n, "launch": f"CUDA graph of {n} calls, replayed back to back",
        "first_replay_us_per_call": round(first, 1), "first_replay_tflops": round(tf(first), 1),
        "settled_us_per_call": round(settled, 1), "settled_tflops": round(tf(settled), 1),
        "clocks_first_half": clocks.summary(t_start, mid), "clocks_second_half": clocks.summary(mid, t_stop)}}


# ----------------------------------------------------------------------------- reference arm


def run_reference(args, dist):
    """The CPU oracle as the reference arm: one bounded row sample per step."""
    if dist.rank != 0:
        return None
    import oracle
    w = gi.WORKLOADS[args.workload]
    A, B, C = gi.operands(w)
    threads = oracle.default_threads()
    per_row = 2.0 * w.N * w.K
    t = time.time()
    oracle.gemm_ref(A[:threads], B, None if C is None else C[:threads], w.alpha, w.beta)
    rate = threads * per_row / max(time.time() - t, 1e-3)
    warmup = max(args.warmup, 3)
    budget = args.reference_seconds / (args.steps + warmup)
    rows = int(max(1, min(4 * threads, budget * rate / per_row)))
    for i in range(warmup):
        r0 = (i * rows) % (w.M - rows + 1)
        oracle.gemm_ref(A[r0:r0 + rows], B, None if C is None else C[r0:r0 + rows], w.alpha, w.beta)
    t = time.time()
    for i in range(args.steps):
        r0 = ((warmup + i) * rows) % (w.M - rows + 1)
        oracle.gemm_ref(A[r0:r0 + rows], B, None if C is None else C[r0:r0 + rows], w.alpha, w.beta)
    dt = time.time() - t
    value = args.steps * rows * per_row / dt / 1e12
    sample = f"{rows} rows x {w.N} outputs x K={w.K} per step"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": dist.world, "steps": args.steps, "warmup": warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": w.describe(),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=MAIN, help="index into gemm_inputs.WORKLOADS")
    ap.add_argument("--shape", default="", help="M,N,K override (profiling runs)")
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 1-SM, 2 2-SM, 3 skinny")
    ap.add_argument("--scheduler", choices=["default", "static", "clc"], default="default",
                    help="tile scheduler of the tiled paths (main step)")
    ap.add_argument("--l2-hints", type=int, default=0,
                    help="main step: L2 eviction hints of the tiled kernels (gemm_tn_config.l2_hints)")
    ap.add_argument("--raster-group", type=int, default=0,
                    help="main step: tiles along M per raster strip (0 = automatic)")
    ap.add_argument("--tiled-k-parts", type=int, default=0,
                    help="main step: k-parts per tile of the tiled paths (gemm_tn_config.tiled_k_parts)")
    ap.add_argument("--cluster-pref", type=int, default=0, choices=[0, 4, 8],
                    help="main step: preferred cluster size of the 2-SM path (gemm_tn_config.cluster_pref)")
    ap.add_argument("--in-dtype", choices=["bf16", "e4m3", "e5m2"], default="bf16",
                    help="input type of the main step (fp8 runs the main step alone)")
    ap.add_argument("--path-check", action="store_true",
                    help="time the automatic path against every forced choice over a grid of shapes and exit")
    ap.add_argument("--path-check-m", default="1,16,32,64,96,128,192,256,512")
    ap.add_argument("--path-check-n", default="1024,4096,8192,16384,28672")
    ap.add_argument("--path-check-k", default="1024,2048,4096,8192")
    ap.add_argument("--sustained", type=float, default=0.0,
                    help="only: the up-projection back to back for this many seconds, with clocks")
    ap.add_argument("--stream-grid", action="store_true",
                    help="only the HBM stream rate of gemm_stream_read against the number of streaming SMs")
    ap.add_argument("--box-rate", action="store_true",
                    help="time gemm_stream_read for each TMA box shape and exit")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--reference-seconds", type=float, default=120.0)
    args = ap.parse_args()
    dist = Dist()
    if args.path_check:
        print(json.dumps(run_path_check(args)), flush=True)
        return
    if args.box_rate:
        print(json.dumps(run_box_rate(args)), flush=True)
        return
    if args.stream_grid:
        print(json.dumps(run_stream_grid(args)), flush=True)
        return
    if args.sustained > 0:
        print(json.dumps(run_sustained(args)), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args, dist)
    else:
        res = run_ours(args, dist)
    if res is not None and dist.rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
