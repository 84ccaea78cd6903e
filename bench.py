#!/usr/bin/env python3
"""Benchmark of the W4A16 hot path on GB300.

One step = one pass of the whole path over one batch of synthetic inputs:
for every projection of the workload, RTN quantize/pack of its bf16 weight
(w4a16_quantize) followed by the W4A16 GEMM (w4a16_gemm).  Default workload:
the action-expert projections at M = 50 tokens, (N, K) = (2048, 1024),
(1024, 1024), (8192, 1024), (1024, 4096), seeds 1..4.

Timing: the steps are captured into CUDA graphs (the library's calls are
capture-safe), so no host launch overhead sits between kernels.  W untimed
warm-up steps replay first, then exactly K timed steps replay between CUDA
events on the launching stream, with a device synchronize (and, for N > 1,
a barrier) on both sides; the max over ranks is reported.  Every step reads
a different copy of all inputs and the copies together exceed 3x the L2
size, so each step streams its inputs from HBM.  Kernel durations for the
roofline come from a second replay of the same K steps with CUDA events
recorded around each launch on the same stream.  The e2e figure is the
eager public API (no graph) with pinned host inputs copied in and results
copied out every step.

`value` is whole-job algorithmic HBM bytes per second (GB/s): for each
quantize 2.515625 * N * K bytes (bf16 read, codes and scales written), for
each GEMM 0.515625 * N * K + 2 * M * K bytes (packed weight, scales and
activations read).  GEMM TFLOP/s and weight-stream GB/s are reported per
kernel alongside.

--impl reference times the CPU oracle (test infrastructure, never the
product path) on a bounded sample of the same workload.
Multi-GPU: the path is replicated (each rank runs the whole workload on its
own GPU); there is no collective on the data path.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
METRIC = "W4A16 GEMM TFLOPS & weight-stream GB/s vs roofline (M=1..8192), 1×GB300"


# ----------------------------------------------------------------- helpers
# bytes per weight of the codes and of the scales, per weight format: fp16
# scales per 128 values (INT4, INT8), one E8M0 byte per 32 (MXFP4), one E4M3
# byte per 16 (NVFP4)
FMT_BYTES = {"int4": (0.5, 2.0 / 128), "int8": (1.0, 2.0 / 128),
             "mxfp4": (0.5, 1.0 / 32), "nvfp4": (0.5, 1.0 / 16)}


def quant_bytes(N, K, fmt="int4"):
    """Algorithmic bytes of a quantize: bf16 weight in (NVFP4 reads it twice:
    the tensor absmax pass, then the packing pass), codes and scales out."""
    reads = 4.0 if fmt == "nvfp4" else 2.0
    return (reads + sum(FMT_BYTES[fmt])) * N * K


def weight_bytes(N, K, fmt="int4"):
    """Codes plus scales of an [N, K] weight."""
    return sum(FMT_BYTES[fmt]) * N * K


def gemm_bytes(M, N, K, fmt="int4"):
    return weight_bytes(N, K, fmt) + 2.0 * M * K


def gemm_flops(M, N, K):
    return 2.0 * M * N * K


def max_over_ranks(values, world, device=None):
    """Element-wise max of per-rank floats over all ranks (identity at N=1).
    Uses the process group already initialised: NCCL reduces on `device`,
    gloo on the CPU."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_rate(units_per_rank_step, steps, elapsed_ms, world):
    """Whole-job throughput: every rank processes `units_per_rank_step` per
    step (replicas), the job takes the slowest rank's `elapsed_ms`."""
    return world * units_per_rank_step * steps / (elapsed_ms * 1e-3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_only_int4_rtn_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:12]


def dram_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it
    was taken on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    cur = kernel_source_hash()
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#"):
                k, w, b, src = parts[:4]
                if k == kernel and w == workload and src == cur:
                    return float(b)
    return None


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(
                    ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=5)
                if out.returncode == 0 and out.stdout.strip():
                    self.samples.append([x.strip() for x in out.stdout.strip().split(",")])
            except Exception:
                pass
            self._stop.wait(0.2)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._t is not None:
            self._t.join(timeout=10)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in self.samples:
            for name, v in zip(names, s[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.samples)}


# ------------------------------------------------------------- GPU arm
def run_gpu(args, rank, world):
    import numpy as np
    import torch

    import weight_only_int4_rtn_gb300 as w4
    from weight_only_int4_rtn_gb300 import synthetic

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    cases = synthetic.WORKLOADS[args.workload]
    if args.grouped is None:
        # the projections are independent problems: one grouped launch of
        # each kind per step when they fit one launch (the grouped quantize
        # rounds to nearest)
        args.grouped = len(cases) <= w4.MAX_GROUP and args.sr_seed is None and args.weights == "int4"
    if args.grouped and len(cases) > w4.MAX_GROUP:
        raise SystemExit(f"--grouped takes at most {w4.MAX_GROUP} projections")
    if args.grouped and args.sr_seed is not None:
        raise SystemExit("--sr-seed quantizes per projection (no --grouped)")
    fmt = args.weights
    int8 = fmt == "int8"
    fp4 = fmt in ("mxfp4", "nvfp4")
    if fmt != "int4" and (args.grouped or args.sr_seed is not None or args.act != "bf16"):
        raise SystemExit(f"--weights {fmt}: bf16 activations, per projection, round to nearest")
    qname = {"int4": "rtn_quantize" if args.sr_seed is None else "sr_quantize",
             "int8": "rtn_quantize_int8", "mxfp4": "quantize_mxfp4", "nvfp4": "quantize_nvfp4"}[fmt]
    gname = {"int4": "w4a16_gemm_tc", "int8": "w8a16_gemm_tc", "mxfp4": "mxfp4_gemm_tc",
             "nvfp4": "nvfp4_gemm_tc"}[fmt]
    packed_bytes = w4.lib().w8a16_packed_bytes if int8 else w4.w4a16_packed_bytes

    def scales_like(c):
        if fp4:
            return torch.empty(c.K // (32 if fmt == "mxfp4" else 16), c.N, dtype=torch.uint8,
                               device=dev)
        return torch.empty(c.K // 128, c.N, dtype=torch.float16, device=dev)

    def quantize_one(s, st):
        if int8:
            w4.w8a16_quantize(s["W"], packed=s["packed"], scales=s["scales"], stream=st)
        elif fp4:
            w4.fp4a16_quantize(s["W"], fmt, packed=s["packed"], scales=s["scales"],
                               tensor_scale=s["ts"], stream=st)
        else:
            w4.w4a16_quantize(s["W"], packed=s["packed"], scales=s["scales"], stream=st,
                              seed=args.sr_seed)

    def gemm_one(A, packed, scales, Y, st, workspace, ts=None):
        if int8:
            w4.w8a16_gemm(A, packed, scales, Y=Y, workspace=workspace, stream=st)
        elif fp4:
            w4.fp4a16_gemm(A, packed, scales, fmt, tensor_scale=ts, Y=Y, workspace=workspace,
                           stream=st)
        else:
            w4.w4a16_gemm(A, packed, scales, Y=Y, workspace=workspace, stream=st)

    def variant_of(c):
        if int8:
            return w4.lib().w8a16_variant_name(w4.lib().w8a16_select_variant(c.M, c.N, c.K)).decode()
        if fp4:
            return w4.fp4a16_variant_name(w4.fp4a16_select_variant(c.M, c.N, c.K))
        return w4.w4a16_variant_name(w4.w4a16_select_variant(c.M, c.N, c.K))

    if args.tune and fmt != "int4":
        args.tune = False   # the INT8 and FP4 catalogues are chosen by the cost model
    shapes = [(c.M, c.N, c.K) for c in cases]
    if args.tune and args.tune_file and os.path.exists(args.tune_file):
        # replay choices an earlier run made by measurement (for profiling:
        # a profiler distorts the tuners' own timings)
        with open(args.tune_file) as f:
            saved = json.load(f)
        for (M, N, K), v in saved.get("table", []):
            w4.w4a16_table_set(M, N, K, v)
        if args.grouped and saved.get("group") is not None:
            w4.w4a16_set_grouped_variant(shapes, saved["group"])
    elif args.tune:
        # kernel choice by measurement, once per shape (or per set of shapes
        # of a grouped launch), outside the timed region; later calls use the
        # memoized choice
        saved = {"table": [], "group": None}
        if args.grouped:
            saved["group"] = w4.w4a16_tune_grouped(
                shapes, act=torch.float16 if args.act == "f16" else torch.bfloat16)
        else:
            for c in cases:
                saved["table"].append([[c.M, c.N, c.K], w4.w4a16_tune(c.M, c.N, c.K)])
        if args.tune_file:
            with open(args.tune_file, "w") as f:
                json.dump(saved, f)

    # one set of inputs per copy; the copies rotate step by step
    per_copy = sum(2 * c.N * c.K + c.N * c.K // 2 + 2 * c.N * c.K // 128 + 2 * c.M * c.K +
                   2 * c.M * c.N for c in cases)
    copies = max(1, min(64, -(-3 * L2_BYTES // per_copy)))
    host_sets = [synthetic.draw(c, act=args.act) for c in cases]
    act_dtype = torch.float16 if args.act == "f16" else torch.bfloat16
    sets = []
    for r in range(copies):
        s = []
        for c, (W, A, b) in zip(cases, host_sets):
            Wd = W.to(dev) if r == 0 else sets[0][len(s)]["W"].clone()
            Ad = A.to(dev) if r == 0 else sets[0][len(s)]["A"].clone()
            s.append(dict(W=Wd, A=Ad,
                          packed=torch.empty(packed_bytes(c.N, c.K), dtype=torch.uint8,
                                             device=dev),
                          scales=scales_like(c),
                          ts=torch.zeros(2, dtype=torch.float32, device=dev),
                          Y=torch.empty(c.M, c.N, dtype=act_dtype, device=dev)))
        sets.append(s)
    ws_bytes = max((w4.lib().w8a16_gemm_workspace_bytes(c.M, c.N, c.K) if int8 else
                    w4.lib().fp4a16_gemm_workspace_bytes(w4.FP4_FORMATS[fmt], c.M, c.N, c.K) if fp4
                    else w4.w4a16_gemm_workspace_bytes_max(c.M, c.N, c.K)) for c in cases)
    if args.grouped:
        probs, _, _ = w4._gemm_problems([s["A"] for s in sets[0]], [s["packed"] for s in sets[0]],
                                        [s["scales"] for s in sets[0]], None,
                                        [s["Y"] for s in sets[0]])
        ws_bytes = max(ws_bytes, w4.lib().w4a16_gemm_grouped_workspace_bytes(probs, len(cases), -1))
    ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    n_k = 2 if args.grouped else 2 * len(cases)

    def run_step(r, st, evs):
        """One step on stream `st`: per projection quantize then GEMM, or
        (--grouped) one grouped quantize then one grouped GEMM."""
        if args.grouped:
            sset = sets[r % copies]
            if evs is not None:
                evs[0][0].record(st)
            w4.w4a16_quantize_grouped([s["W"] for s in sset],
                                      outs=[(s["packed"], s["scales"]) for s in sset], stream=st)
            if evs is not None:
                evs[0][1].record(st)
                evs[1][0].record(st)
            w4.w4a16_gemm_grouped([s["A"] for s in sset], [s["packed"] for s in sset],
                                  [s["scales"] for s in sset], Ys=[s["Y"] for s in sset],
                                  workspace=ws, stream=st)
            if evs is not None:
                evs[1][1].record(st)
            return
        for j, c in enumerate(cases):
            s = sets[r % copies][j]
            if evs is not None:
                evs[2 * j][0].record(st)
            quantize_one(s, st)
            if evs is not None:
                evs[2 * j][1].record(st)
                evs[2 * j + 1][0].record(st)
            gemm_one(s["A"], s["packed"], s["scales"], s["Y"], st, ws, s["ts"])
            if evs is not None:
                evs[2 * j + 1][1].record(st)

    def step(r, evs=None):
        run_step(r, stream, evs)

    # eager warm-up (also sets kernel attributes outside any capture)
    for r in range(min(args.warmup, copies)):
        step(r)
    torch.cuda.synchronize(dev)
    if w4.w4a16_get_device_error() != w4.W4A16_OK:
        raise RuntimeError("device error during warm-up")

    # The timed steps run as one CUDA graph (no host launch overhead between
    # kernels): graph A holds warm-up + timed steps back to back; graph B is
    # the same steps with timing events around every kernel.
    def capture(n_steps, first, with_events):
        evs = None
        if with_events:
            evs = [[[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
                    for _ in range(n_k)] for _ in range(n_steps)]
        g = torch.cuda.CUDAGraph()
        cap_stream = torch.cuda.Stream(dev)
        cap_stream.wait_stream(torch.cuda.current_stream(dev))
        l0 = w4.w4a16_launch_count()
        with torch.cuda.stream(cap_stream):
            with torch.cuda.graph(g, stream=cap_stream):
                for r in range(n_steps):
                    step_on(first + r, cap_stream, None if evs is None else evs[r])
        torch.cuda.current_stream(dev).wait_stream(cap_stream)
        return g, evs, w4.w4a16_launch_count() - l0

    def step_on(r, st, evs):
        run_step(r, st, evs)

    g_warm, _, _ = capture(args.warmup, 0, False)
    g_timed, _, launches_per_replay = capture(args.steps, args.warmup, False)
    try:
        g_ev, kev, _ = capture(args.steps, args.warmup, True)
    except TypeError:
        g_ev, kev = None, None

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # --- timed region
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g_warm.replay()
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        # the NVTX range marks the timed steps for profilers (ncu --nvtx
        # --nvtx-include "bench_timed/" captures only these kernels)
        torch.cuda.nvtx.range_push("bench_timed")
        start.record(stream)
        g_timed.replay()
        end.record(stream)
        torch.cuda.synchronize(dev)
        torch.cuda.nvtx.range_pop()
    barrier()
    launches = launches_per_replay
    elapsed_ms = start.elapsed_time(end)

    # --- per-kernel durations: the same steps with events around each kernel
    if g_ev is not None:
        g_warm.replay()
        g_ev.replay()
        torch.cuda.synchronize(dev)
        kern_ms = [statistics.mean(kev[r][k][0].elapsed_time(kev[r][k][1]) for r in range(args.steps))
                   for k in range(n_k)]
    else:
        kern_ms = []
        for k in range(n_k):
            gk = torch.cuda.CUDAGraph()
            j, is_gemm = divmod(k, 2)
            with torch.cuda.graph(gk):
                for r in range(args.steps):
                    sset = sets[(args.warmup + r) % copies]
                    if args.grouped and is_gemm:
                        w4.w4a16_gemm_grouped([s["A"] for s in sset], [s["packed"] for s in sset],
                                              [s["scales"] for s in sset], Ys=[s["Y"] for s in sset],
                                              workspace=ws)
                    elif args.grouped:
                        w4.w4a16_quantize_grouped([s["W"] for s in sset],
                                                  outs=[(s["packed"], s["scales"]) for s in sset])
                    elif is_gemm:
                        s = sset[j]
                        gemm_one(s["A"], s["packed"], s["scales"], s["Y"], None, ws, s["ts"])
                    else:
                        quantize_one(sset[j], None)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            gk.replay()
            e0.record(stream)
            gk.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            kern_ms.append(e0.elapsed_time(e1) / args.steps)
    if w4.w4a16_get_device_error() != w4.W4A16_OK:
        raise RuntimeError("device error during timing")

    # --- e2e: pinned host inputs -> device, the path, result -> host
    pinned = [(W.pin_memory(), A.pin_memory()) for (W, A, b) in host_sets]
    yh = [torch.empty(c.M, c.N, dtype=act_dtype).pin_memory() for c in cases]
    h2d = sum(W.numel() * 2 + A.numel() * 2 for W, A in pinned)
    d2h = sum(c.M * c.N * 2 for c in cases)
    s0 = sets[0]

    def e2e_step():
        for j, c in enumerate(cases):
            s0[j]["W"].copy_(pinned[j][0], non_blocking=True)
            s0[j]["A"].copy_(pinned[j][1], non_blocking=True)
        run_step(0, stream, None)
        for j, c in enumerate(cases):
            yh[j].copy_(s0[j]["Y"], non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = e0.elapsed_time(e1)

    elapsed_ms, e2e_ms = max_over_ranks([elapsed_ms, e2e_ms], world, dev)

    bytes_step = sum(quant_bytes(c.N, c.K, fmt) + gemm_bytes(c.M, c.N, c.K, fmt) for c in cases)
    flops_step = sum(gemm_flops(c.M, c.N, c.K) for c in cases)
    ms_step = elapsed_ms / args.steps
    value = job_rate(bytes_step, args.steps, elapsed_ms, world) / 1e9
    e2e_value = job_rate(bytes_step, args.steps, e2e_ms, world) / 1e9

    peaks = load_peaks()
    kernels = []
    if args.grouped:
        tq, tg = kern_ms[0], kern_ms[1]
        qb = sum(quant_bytes(c.N, c.K, fmt) for c in cases)
        gb = sum(gemm_bytes(c.M, c.N, c.K, fmt) for c in cases)
        kernels.append(dict(kernel="rtn_quantize", grouped=len(cases), us=round(tq * 1e3, 3),
                            gbs=round(qb / (tq * 1e-3) / 1e9, 1)))
        kernels.append(dict(kernel="w4a16_gemm_tc", grouped=len(cases), us=round(tg * 1e3, 3),
                            tflops=round(flops_step / (tg * 1e-3) / 1e12, 2),
                            gbs=round(gb / (tg * 1e-3) / 1e9, 1)))
    for j, c in enumerate([] if args.grouped else cases):
        tq, tg = kern_ms[2 * j], kern_ms[2 * j + 1]
        kernels.append(dict(kernel=qname, shape=[c.N, c.K], us=round(tq * 1e3, 3),
                            gbs=round(quant_bytes(c.N, c.K, fmt) / (tq * 1e-3) / 1e9, 1)))
        kernels.append(dict(kernel=gname, shape=[c.M, c.N, c.K], us=round(tg * 1e3, 3),
                            variant=variant_of(c),
                            tflops=round(gemm_flops(c.M, c.N, c.K) / (tg * 1e-3) / 1e12, 2),
                            weight_gbs=round(weight_bytes(c.N, c.K, fmt) / (tg * 1e-3) / 1e9, 1),
                            gbs=round(gemm_bytes(c.M, c.N, c.K, fmt) / (tg * 1e-3) / 1e9, 1)))
    # dominant kernel: the kind with the larger share of kernel time
    t_q = sum(kern_ms[0::2])
    t_g = sum(kern_ms[1::2])
    launches_kind = 1 if args.grouped else len(cases)
    if t_q >= t_g:
        dom, dom_bytes = qname, sum(quant_bytes(c.N, c.K, fmt) for c in cases)
        dom_ms, launches_dom = t_q, launches_kind
        bound, achieved, peak, unit = "hbm", None, peaks["hbm_gbs"], "GB/s"
        achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    else:
        dom_ms, launches_dom = t_g, launches_kind
        big = max(cases, key=lambda c: gemm_flops(c.M, c.N, c.K) / max(gemm_bytes(c.M, c.N, c.K, fmt), 1))
        ai = gemm_flops(big.M, big.N, big.K) / gemm_bytes(big.M, big.N, big.K, fmt)
        tensor_bound = ai > peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
        dom = gname
        if tensor_bound:
            bound, peak, unit = "tensor", peaks["bf16_tflops"], "TFLOP/s"
            achieved = sum(gemm_flops(c.M, c.N, c.K) for c in cases) / (dom_ms * 1e-3) / 1e12
        else:
            bound, peak, unit = "hbm", peaks["hbm_gbs"], "GB/s"
            achieved = sum(gemm_bytes(c.M, c.N, c.K, fmt) for c in cases) / (dom_ms * 1e-3) / 1e9
    traffic = dram_traffic(dom, args.workload + ("_grouped" if args.grouped else "") +
                           ("_sr" if args.sr_seed is not None else ""))

    # --- each GEMM shape alone: a CUDA graph of back-to-back launches on
    # weight copies rotating through more than 3x L2 (launch overhead
    # amortised, no quantize in between), against the roofline of the shape
    b2b = []
    for c in {(c.M, c.N, c.K): c for c in cases}.values():
        s0 = sets[0][cases.index(c)]
        nb = packed_bytes(c.N, c.K) + s0["scales"].numel() * s0["scales"].element_size()
        ncp = max(1, min(16, -(-3 * L2_BYTES // nb)))
        cps = [(s0["packed"], s0["scales"])] + [(s0["packed"].clone(), s0["scales"].clone())
                                                for _ in range(ncp - 1)]
        reps = max(8, 2 * ncp)
        gb = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream(dev)
        cs.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cs):
            with torch.cuda.graph(gb, stream=cs):
                for r in range(reps):
                    gemm_one(s0["A"], cps[r % ncp][0], cps[r % ncp][1], s0["Y"], cs, ws, s0["ts"])
        torch.cuda.current_stream(dev).wait_stream(cs)
        gb.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gb.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) / reps * 1e3
        t_hbm = gemm_bytes(c.M, c.N, c.K, fmt) / (peaks["hbm_gbs"] * 1e9) * 1e6
        t_tc = gemm_flops(c.M, c.N, c.K) / (peaks["bf16_tflops"] * 1e12) * 1e6
        b2b.append(dict(shape=[c.M, c.N, c.K], variant=variant_of(c), us=round(us, 3),
                        weight_gbs=round(weight_bytes(c.N, c.K, fmt) / (us * 1e-6) / 1e9, 1),
                        tflops=round(gemm_flops(c.M, c.N, c.K) / (us * 1e-6) / 1e12, 2),
                        bound="hbm" if t_hbm >= t_tc else "tensor",
                        roofline_frac=round(max(t_hbm, t_tc) / us, 4), weight_copies=ncp))
        if args.swiglu and "gate_up" in c.name and not (int8 or fp4) and args.act == "bf16":
            # the same weight copies through the SwiGLU epilogue (rows read as
            # interleaved up/gate pairs; Y is [M, N/2]), each eligible tcgen05
            # variant timed the same way, the fastest reported (the epilogue's
            # own choice by measurement, passed as w4a16_gemm_swiglu's variant)
            Yh = torch.empty(c.M, c.N // 2, dtype=torch.bfloat16, device=dev)
            best = None
            for vid in range(w4.w4a16_variant_count()):
                vname = w4.w4a16_variant_name(vid)
                if vname.startswith("simt_") or not w4.w4a16_variant_eligible(vid, c.M, c.N, c.K):
                    continue
                wsh = torch.zeros(max(w4.w4a16_variant_workspace_bytes(vid, c.M, c.N, c.K), 256),
                                  dtype=torch.uint8, device=dev)
                gh = torch.cuda.CUDAGraph()
                with torch.cuda.stream(cs):
                    for r in range(2):   # outside the capture: kernel attributes
                        w4.w4a16_gemm_swiglu(s0["A"], cps[r % ncp][0], cps[r % ncp][1], Y=Yh,
                                             workspace=wsh, stream=cs, variant=vid)
                    with torch.cuda.graph(gh, stream=cs):
                        for r in range(reps):
                            w4.w4a16_gemm_swiglu(s0["A"], cps[r % ncp][0], cps[r % ncp][1], Y=Yh,
                                                 workspace=wsh, stream=cs, variant=vid)
                torch.cuda.current_stream(dev).wait_stream(cs)
                gh.replay()
                e0.record(stream)
                gh.replay()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                us = e0.elapsed_time(e1) / reps * 1e3
                if best is None or us < best[0]:
                    best = (us, vname)
                del gh, wsh
            us, vname = best
            b2b.append(dict(shape=[c.M, c.N, c.K], epilogue="swiglu", variant=vname,
                            us=round(us, 3),
                            weight_gbs=round(weight_bytes(c.N, c.K, fmt) / (us * 1e-6) / 1e9, 1),
                            tflops=round(gemm_flops(c.M, c.N, c.K) / (us * 1e-6) / 1e12, 2),
                            bound="hbm" if t_hbm >= t_tc else "tensor",
                            roofline_frac=round(max(t_hbm, t_tc) / us, 4), weight_copies=ncp))
            del Yh
        del cps, gb
    if w4.w4a16_get_device_error() != w4.W4A16_OK:
        raise RuntimeError("device error during the back-to-back GEMM timing")
    roofline = dict(bound=bound, achieved=round(achieved, 2), peak=peak, unit=unit,
                    frac=round(achieved / peak, 4),
                    traffic=None if traffic is None else traffic,
                    kernel=dom, launches_per_step=launches_dom, peak_source=peaks["source"])

    out = dict(metric=METRIC, value=round(value, 2), unit="GB/s", n_gpus=world, steps=args.steps,
               warmup=args.warmup, ms_per_step=round(ms_step, 5), higher_is_better=True,
               scaling="weak", vs_baseline=None, dtype=args.act, data="synthetic",
               config=dict(workload=args.workload, activations=args.act, weights=args.weights,
                           shapes=[[c.M, c.N, c.K] for c in cases],
                           step=("one grouped rtn_quantize launch over all projections + one grouped "
                                 "w4a16_gemm launch" if args.grouped else
                                 "INT8 rtn_quantize + w8a16_gemm per projection" if int8 else
                                 f"{fmt.upper()} quantize + fp4a16_gemm per projection" if fp4 else
                                 "rtn_quantize + w4a16_gemm per projection" if args.sr_seed is None
                                 else "stochastic-rounding quantize (seed %d) + w4a16_gemm per "
                                 "projection" % args.sr_seed),
                           l2="inputs rotate over %d copies (%.0f MB > 3x L2)" % (copies, copies * per_copy / 2**20),
                           selection=("per-shape table tuned by measurement before timing" if args.tune
                                      else "cost-model rule"),
                           parallelism=f"replicas x{world}"),
               gemm=dict(tflops=round(job_rate(flops_step, args.steps, elapsed_ms, world) / 1e12, 3)),
               kernels=kernels, roofline=roofline, clocks=clk.summary(),
               gemm_back_to_back=b2b,
               gpu_launches=int(launches),
               e2e=dict(value=round(e2e_value, 2), unit="GB/s", h2d_bytes_per_step=int(h2d),
                        d2h_bytes_per_step=int(d2h)))
    return out


# ------------------------------------------------------------- CPU oracle
def time_oracle(workload: str, budget_s: float, sr_seed=None, weights="int4"):
    """The oracle as it stands, on the host cores, over whole passes of the
    workload (quantize + GEMM per projection; the stochastic-rounding quantize
    when `sr_seed` is given) until `budget_s` is used."""
    import numpy as np

    import oracle
    from weight_only_int4_rtn_gb300 import synthetic

    cases = synthetic.WORKLOADS[workload]
    inputs = []
    for c in cases:
        W, A, b = synthetic.draw(c)
        inputs.append((synthetic.bits(W), synthetic.bits(A)))
    # bounded sample: for very large workloads only the first rows of A
    sample_rows = [min(c.M, 64) for c in cases]
    done_bytes = 0.0
    passes = 0
    t0 = time.perf_counter()
    while True:
        for c, (wb, ab), mr in zip(cases, inputs, sample_rows):
            if weights == "int8":
                p, s = oracle.quantize8(wb)
                oracle.gemm8(ab[:mr], p, s)
            elif weights == "mxfp4":
                p, s = oracle.quantize_mxfp4_f32(oracle.bf16_bits_to_f32(wb))
                oracle.gemm_fp4(ab[:mr], oracle.dequantize_mxfp4(p, s))
            elif weights == "nvfp4":
                p, s, g = oracle.quantize_nvfp4_f32(oracle.bf16_bits_to_f32(wb))
                oracle.gemm_fp4(ab[:mr], oracle.dequantize_nvfp4(p, s, g))
            else:
                p, s = oracle.quantize(wb) if sr_seed is None else oracle.quantize_sr(wb, sr_seed)
                oracle.gemm(ab[:mr], p, s)
            done_bytes += quant_bytes(c.N, c.K, weights) + gemm_bytes(mr, c.N, c.K, weights)
        passes += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = (f"{passes} pass(es) of {workload}: oracle "
              + ({"int8": "INT8 ", "mxfp4": "MXFP4 ", "nvfp4": "NVFP4 "}.get(weights, "")
                 if weights != "int4" else "" if sr_seed is None else "stochastic-rounding ")
              + "quantize + FP32 GEMM per projection"
              + ("" if all(mr == c.M for mr, c in zip(sample_rows, cases)) else
                 ", GEMM on the first 64 rows of A"))
    return dict(value=round(done_bytes / dt / 1e9, 4), unit="GB/s", cores=cores, kind="oracle",
                sample=sample, seconds=round(dt, 2))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="expert_m50",
                    choices=["tiny", "expert_m50", "prefix_m816", "sweep", "large"])
    ap.add_argument("--act", default="bf16", choices=["bf16", "f16"],
                    help="activation type of the GEMMs (A, bias, Y)")
    ap.add_argument("--grouped", dest="grouped", action="store_true", default=None,
                    help="one grouped quantize and one grouped GEMM launch per step (the "
                         "projections are independent problems; the default when the "
                         "workload has at most 8 projections)")
    ap.add_argument("--per-projection", dest="grouped", action="store_false",
                    help="one quantize and one GEMM launch per projection")
    ap.add_argument("--weights", default="int4", choices=["int4", "int8", "mxfp4", "nvfp4"],
                    help="weight scheme: INT4 (W4A16), INT8 (W8A16), MXFP4 or NVFP4 weights")
    ap.add_argument("--sr-seed", type=int, default=None,
                    help="quantize with seeded stochastic rounding (w4a16_quantize_sr) instead "
                         "of round to nearest")
    ap.add_argument("--swiglu", action="store_true",
                    help="also time each gate/up projection's GEMM with the SwiGLU epilogue "
                         "(w4a16_gemm_swiglu) back to back, with the variant that measures "
                         "fastest (INT4 weights, bf16 activations)")
    ap.add_argument("--tune-file", default=None,
                    help="write the tuned choices to this JSON file, or replay them from it "
                         "when it exists (no timing under a profiler)")
    ap.add_argument("--no-tune", dest="tune", action="store_false", default=True,
                    help="select kernels by the cost-model rule instead of tuning each "
                         "shape by measurement first")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        t_budget = max(5.0, min(60.0, args.cpu_budget * (args.steps + args.warmup) / 10))
        cb = time_oracle(args.workload, t_budget, args.sr_seed, args.weights)
        line = dict(metric=METRIC, value=cb["value"], unit="GB/s", n_gpus=world, steps=args.steps,
                    warmup=args.warmup, ms_per_step=None, higher_is_better=True, scaling="weak",
                    vs_baseline=None, dtype="f32", data="synthetic", impl="reference",
                    config=dict(workload=args.workload), cpu_baseline=cb,
                    e2e=dict(value=cb["value"], unit="GB/s", h2d_bytes_per_step=0,
                             d2h_bytes_per_step=0))
        print(json.dumps(line), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")

    from __graft_entry__ import build
    build()
    out = run_gpu(args, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = time_oracle(args.workload, args.cpu_budget, args.sr_seed, args.weights)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
