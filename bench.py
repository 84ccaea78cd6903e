#!/usr/bin/env python3
"""Benchmark of the W4A16 GEMM on GB300.

Metric: W4A16 GEMM TFLOP/s and weight-stream GB/s against the roofline over
M = 1 .. 8192.  One step = one pass of the GEMM over one batch of synthetic
inputs: the W4A16 GEMM of every projection of the workload, on INT4 weights
that were RTN-quantized at load and stay resident in HBM (one grouped launch
when the workload has 2 .. 8 projections).  The quantize/pack is load-time
work: it is timed apart and reported under `kernels`, outside the step.

Default workload: `large` (M = N = K = 8192), the compute-bound end of the
metric's M range; `value` is its GEMM TFLOP/s.  The same line carries
`sweep`: the bandwidth-bound end (M in {1, 4, 16, 64} x (N, K) in {(16384,
2048), (2048, 16384), (8192, 8192)}), every shape's GEMM alone, back to back,
with its weight GB/s and roofline fraction.

Timing: the steps are captured into CUDA graphs (the library's calls are
capture-safe), so no host launch overhead sits between kernels.  W untimed
warm-up steps replay first, then exactly K timed steps replay between CUDA
events on the launching stream, with a device synchronize (and, for N > 1, a
barrier) on both sides; the max over ranks is reported.  Every step reads a
different copy of the weights and activations, and the copies together
exceed 3x the L2 size, so each step streams its inputs from HBM.  SM clocks
and throttle reasons are sampled during the timed region (NVML, read only).
The e2e figure is the same steps through the public API with the
activations copied in from pinned host memory and the outputs copied back,
every step, pipelined over copy-in, compute and copy-out streams.

--impl reference times the CPU oracle (test infrastructure, never the
product path) on a bounded sample of the same workload, in the same unit.
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


def code_only(text: str) -> str:
    """C/C++/CUDA source text without its comments, whitespace runs collapsed
    to one space: what the compiler sees (string and character literals are
    kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash():
    """A digest of the kernel sources' code (comments and layout left out), the
    key under which measured DRAM traffic is recorded."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_only_int4_rtn_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                h.update(f.encode() + b"\0" + code_only(fh.read()).encode() + b"\0")
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
    """SM clocks and throttle reasons of one GPU, sampled every 2 ms while
    the context is open: NVML through ctypes (read-only queries; the device
    found by its PCI bus id), else nvidia-smi every 200 ms."""

    NVML_CLOCK_SM = 1
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.device = device
        self.samples = []          # (host time, sm_mhz, max_mhz, {reason names})
        self.window = None         # host-time window of the timed region
        self.source = None
        self._stop = threading.Event()
        self._t = None
        self._nvml = None
        self._handle = None

    def _open_nvml(self):
        import ctypes
        import torch
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return False
            p = torch.cuda.get_device_properties(self.device)
            bus = "%08X:%02X:%02X.0" % (getattr(p, "pci_domain_id", 0), p.pci_bus_id,
                                        p.pci_device_id)
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                return False
            self._nvml, self._handle = nv, h
            return True
        except Exception:
            return False

    def _sample_nvml(self):
        import ctypes
        nv, h = self._nvml, self._handle
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if nv.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(clk)) != 0:
            return
        nv.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx))
        fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        fn(h, ctypes.byref(rs))
        names = {n for bit, n in self.REASONS.items() if rs.value & bit}
        self.samples.append((time.perf_counter(), float(clk.value), float(mx.value), names))

    def _sample_smi(self):
        out = subprocess.run(
            ["nvidia-smi", "-i", str(self.device.index), f"--query-gpu={self.FIELDS}",
             "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=5)
        if out.returncode == 0 and out.stdout.strip():
            s = [x.strip() for x in out.stdout.strip().split(",")]
            if s[0].replace(".", "").isdigit() and s[1].replace(".", "").isdigit():
                names = {n for n, v in zip(["hw_slowdown", "hw_thermal_slowdown",
                                            "sw_thermal_slowdown", "sw_power_cap"], s[4:8])
                         if v.strip().lower() == "active"}
                self.samples.append((time.perf_counter(), float(s[0]), float(s[1]), names))

    def _run(self):
        use_nvml = self._open_nvml()
        self.source = "nvml" if use_nvml else "nvidia-smi"
        while not self._stop.is_set():
            try:
                self._sample_nvml() if use_nvml else self._sample_smi()
            except Exception:
                pass
            self._stop.wait(0.002 if use_nvml else 0.2)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        time.sleep(0.05)   # sampling runs before the timed region starts
        return self

    def mark(self, t0, t1):
        """The timed region's host-time window; summary() keeps the samples
        inside it (and the one just before it, so a very short region still
        has one)."""
        self.window = (t0, t1)

    def __exit__(self, *exc):
        self._stop.set()
        if self._t is not None:
            self._t.join(timeout=10)

    def summary(self):
        samples = self.samples
        if self.window is not None:
            t0, t1 = self.window
            before = [s for s in samples if s[0] < t0][-1:]
            samples = before + [s for s in samples if t0 <= s[0] <= t1]
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        reasons = set()
        for s in samples:
            reasons |= s[3]
        return {"sm_mhz": statistics.median(s[1] for s in samples),
                "sm_max_mhz": max(s[2] for s in samples),
                "reasons": sorted(reasons), "samples": len(samples), "source": self.source}


# ------------------------------------------------------------- GPU arm
class Formats:
    """The calls of one weight scheme (INT4, INT8, MXFP4, NVFP4) through the
    binding: quantize (load time), GEMM (the step), variant names."""

    def __init__(self, w4, fmt, act, sr_seed, dev):
        import torch
        self.w4, self.fmt, self.act, self.sr_seed, self.dev = w4, fmt, act, sr_seed, dev
        self.int8 = fmt == "int8"
        self.fp4 = fmt in ("mxfp4", "nvfp4")
        self.act_dtype = torch.float16 if act == "f16" else torch.bfloat16
        self.qname = {"int4": "rtn_quantize" if sr_seed is None else "sr_quantize",
                      "int8": "rtn_quantize_int8", "mxfp4": "quantize_mxfp4",
                      "nvfp4": "quantize_nvfp4"}[fmt]
        self.gname = {"int4": "w4a16_gemm_tc", "int8": "w8a16_gemm_tc", "mxfp4": "mxfp4_gemm_tc",
                      "nvfp4": "nvfp4_gemm_tc"}[fmt]

    def packed_bytes(self, N, K):
        L = self.w4.lib()
        return L.w8a16_packed_bytes(N, K) if self.int8 else self.w4.w4a16_packed_bytes(N, K)

    def new_weight(self, N, K):
        """Empty (packed, scales, tensor scale) buffers of an [N, K] weight."""
        import torch
        packed = torch.empty(self.packed_bytes(N, K), dtype=torch.uint8, device=self.dev)
        if self.fp4:
            scales = torch.empty(K // (32 if self.fmt == "mxfp4" else 16), N, dtype=torch.uint8,
                                 device=self.dev)
        else:
            scales = torch.empty(K // 128, N, dtype=torch.float16, device=self.dev)
        ts = torch.zeros(2, dtype=torch.float32, device=self.dev)
        return dict(packed=packed, scales=scales, ts=ts)

    def quantize(self, W, wt, st=None):
        w4 = self.w4
        if self.int8:
            w4.w8a16_quantize(W, packed=wt["packed"], scales=wt["scales"], stream=st)
        elif self.fp4:
            w4.fp4a16_quantize(W, self.fmt, packed=wt["packed"], scales=wt["scales"],
                               tensor_scale=wt["ts"], stream=st)
        else:
            w4.w4a16_quantize(W, packed=wt["packed"], scales=wt["scales"], stream=st,
                              seed=self.sr_seed)

    def gemm(self, A, wt, Y, ws, st=None):
        w4 = self.w4
        if self.int8:
            w4.w8a16_gemm(A, wt["packed"], wt["scales"], Y=Y, workspace=ws, stream=st)
        elif self.fp4:
            w4.fp4a16_gemm(A, wt["packed"], wt["scales"], self.fmt, tensor_scale=wt["ts"], Y=Y,
                           workspace=ws, stream=st)
        else:
            w4.w4a16_gemm(A, wt["packed"], wt["scales"], Y=Y, workspace=ws, stream=st)

    def workspace_bytes(self, M, N, K):
        L = self.w4.lib()
        if self.int8:
            return L.w8a16_gemm_workspace_bytes(M, N, K)
        if self.fp4:
            return L.fp4a16_gemm_workspace_bytes(self.w4.FP4_FORMATS[self.fmt], M, N, K)
        return self.w4.w4a16_gemm_workspace_bytes_max(M, N, K)

    def tune(self, M, N, K, swiglu=False):
        """Choose this catalogue's variant for the shape by measurement (the
        library's tuners; memoized in its table)."""
        w4 = self.w4
        if swiglu:
            return w4.w4a16_tune_swiglu(M, N, K)
        if self.int8:
            return w4.w8a16_tune(M, N, K)
        if self.fp4:
            return w4.fp4a16_tune(M, N, K, self.fmt)
        return w4.w4a16_tune(M, N, K)

    def variant(self, M, N, K):
        w4 = self.w4
        if self.int8:
            L = w4.lib()
            return L.w8a16_variant_name(L.w8a16_select_variant(M, N, K)).decode()
        if self.fp4:
            return w4.fp4a16_variant_name(w4.fp4a16_select_variant(M, N, K))
        return w4.w4a16_variant_name(w4.w4a16_select_variant(M, N, K))


def graph_of(dev, fn, n):
    """A CUDA graph of n calls fn(i, stream), captured on a side stream."""
    import torch
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream(dev)
    cs.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            for i in range(n):
                fn(i, cs)
    torch.cuda.current_stream(dev).wait_stream(cs)
    return g


def time_graph_us(dev, g, reps, trials=20):
    """Device time per call of a replayed graph of `reps` calls: the median
    over `trials` replays, each between CUDA events on the current stream,
    after one untimed replay."""
    import torch
    stream = torch.cuda.current_stream(dev)
    g.replay()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(trials)]
    for e0, e1 in evs:
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) / reps * 1e3


def back_to_back(fx, c, peaks, wcache, tune, dev, swiglu=False):
    """One GEMM shape alone: a CUDA graph of back-to-back launches on weight
    copies that rotate through more than 3x L2 (every launch reads from HBM), no
    other kernel in between, against the roofline of the shape.  swiglu: the
    same weights through w4a16_gemm_swiglu (rows read as interleaved up/gate
    pairs, Y of [M, N/2]), its variant chosen by its own tuner."""
    import torch

    from weight_only_int4_rtn_gb300 import synthetic
    w4 = fx.w4
    if tune:
        fx.tune(c.M, c.N, c.K, swiglu)
    key = (c.N, c.K, c.seed, c.wdist)
    if key not in wcache:
        wcache.clear()
        W = synthetic.draw_weight_only(c.seed, c.N, c.K, c.wdist).to(dev)
        wt = fx.new_weight(c.N, c.K)
        fx.quantize(W, wt)
        torch.cuda.synchronize(dev)   # weights complete before any GEMM may read them early
        del W
        wcache[key] = wt
    wt = wcache[key]
    _, A, _ = synthetic.draw(c, act=fx.act)
    A = A.to(dev)
    Y = torch.empty(c.M, c.N // 2 if swiglu else c.N, dtype=fx.act_dtype, device=dev)
    nb = sum(t.numel() * t.element_size() for t in (wt["packed"], wt["scales"]))
    ncp = max(1, min(16, -(-3 * L2_BYTES // nb)))
    cps = [wt] + [{k: v.clone() for k, v in wt.items()} for _ in range(ncp - 1)]
    ws = torch.zeros(max(fx.workspace_bytes(c.M, c.N, c.K), 256), dtype=torch.uint8, device=dev)
    reps = max(8, 2 * ncp)

    def one(i, st=None):
        if swiglu:
            w4.w4a16_gemm_swiglu(A, cps[i % ncp]["packed"], cps[i % ncp]["scales"], Y=Y,
                                 workspace=ws, stream=st)
        else:
            fx.gemm(A, cps[i % ncp], Y, ws, st)

    for i in range(2):   # kernel attributes are set outside the capture
        one(i)
    g = graph_of(dev, one, reps)
    us = time_graph_us(dev, g, reps)
    t_hbm = gemm_bytes(c.M, c.N, c.K, fx.fmt) / (peaks["hbm_gbs"] * 1e9) * 1e6
    t_tc = gemm_flops(c.M, c.N, c.K) / (peaks["bf16_tflops"] * 1e12) * 1e6
    del g, cps, ws
    out = dict(shape=[c.M, c.N, c.K],
               variant=(w4.w4a16_variant_name(w4.lib().w4a16_select_variant(c.M, c.N, c.K))
                        if not swiglu else None) or fx.variant(c.M, c.N, c.K),
               us=round(us, 3),
               weight_gbs=round(weight_bytes(c.N, c.K, fx.fmt) / (us * 1e-6) / 1e9, 1),
               tflops=round(gemm_flops(c.M, c.N, c.K) / (us * 1e-6) / 1e12, 2),
               bound="hbm" if t_hbm >= t_tc else "tensor",
               roofline_frac=round(max(t_hbm, t_tc) / us, 4), weight_copies=ncp)
    if swiglu:
        out["epilogue"] = "swiglu"
        out["variant"] = "tuned (w4a16_tune_swiglu)"
    elif fx.fmt != "int4":
        out["variant"] = fx.variant(c.M, c.N, c.K)
    return out


def grouped_back_to_back(w4, cases, epilogues, peaks, tune, dev):
    """The projections of one block as one grouped launch (optionally with
    the SwiGLU epilogue on some problems), back to back on weight copies
    rotating through more than 3x L2, plan tuned by measurement."""
    import torch

    from weight_only_int4_rtn_gb300 import synthetic
    shapes = [(c.M, c.N, c.K, e) for c, e in zip(cases, epilogues)]
    vname = None
    if tune:
        vname = w4.w4a16_variant_name(w4.w4a16_tune_grouped(shapes))
    drawn = [synthetic.draw(c) for c in cases]
    q = w4.w4a16_quantize_grouped([W.to(dev) for W, _, _ in drawn])
    torch.cuda.synchronize(dev)   # weights complete before any GEMM may read them early
    nb = sum(p.numel() + s.numel() * 2 for p, s in q)
    ncp = max(1, min(16, -(-3 * L2_BYTES // nb)))
    cps = [q] + [[(p.clone(), s.clone()) for p, s in q] for _ in range(ncp - 1)]
    As = [A.to(dev) for _, A, _ in drawn]
    Ys = [torch.empty(c.M, c.N // 2 if e else c.N, dtype=torch.bfloat16, device=dev)
          for c, e in zip(cases, epilogues)]
    probs, _, _ = w4._gemm_problems(As, [p for p, _ in q], [s for _, s in q], None, Ys, epilogues)
    ws = torch.zeros(max(w4.lib().w4a16_gemm_grouped_workspace_bytes(probs, len(cases), -1), 256),
                     dtype=torch.uint8, device=dev)
    reps = max(8, 2 * ncp)

    def one(i, st=None):
        cp = cps[i % ncp]
        w4.w4a16_gemm_grouped(As, [p for p, _ in cp], [s for _, s in cp], Ys=Ys, workspace=ws,
                              stream=st, epilogues=epilogues)

    for i in range(2):
        one(i)
    g = graph_of(dev, one, reps)
    us = time_graph_us(dev, g, reps)
    del g, cps, ws
    byts = sum(gemm_bytes(c.M, c.N, c.K) for c in cases)
    flops = sum(gemm_flops(c.M, c.N, c.K) for c in cases)
    t_hbm = byts / (peaks["hbm_gbs"] * 1e9) * 1e6
    t_tc = flops / (peaks["bf16_tflops"] * 1e12) * 1e6
    return dict(shapes=[[c.M, c.N, c.K] for c in cases], epilogues=["swiglu" if e else "none"
                                                                    for e in epilogues],
                variant=vname, us=round(us, 3), gbs=round(byts / (us * 1e-6) / 1e9, 1),
                tflops=round(flops / (us * 1e-6) / 1e12, 2),
                bound="hbm" if t_hbm >= t_tc else "tensor",
                roofline_frac=round(max(t_hbm, t_tc) / us, 4), weight_copies=ncp)


def workload_cases(args):
    """The workload's projections, or (--shape M,N,K) one projection of that
    shape (N(0, 0.02) weights, seed 0), e.g. a smaller case of a kernel for a
    profiler."""
    from weight_only_int4_rtn_gb300 import synthetic
    if args.shape:
        M, N, K = (int(x) for x in args.shape.split(","))
        return [synthetic.Case(f"shape_m{M}_n{N}_k{K}", M, N, K, 0)]
    return synthetic.WORKLOADS[args.workload]


def run_gpu(args, rank, world):
    import torch

    import weight_only_int4_rtn_gb300 as w4
    from weight_only_int4_rtn_gb300 import synthetic

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    cases = workload_cases(args)
    fmt = args.weights
    fx = Formats(w4, fmt, args.act, args.sr_seed, dev)
    if fmt != "int4" and (args.grouped or args.act != "bf16"):
        raise SystemExit(f"--weights {fmt}: bf16 activations, one launch per projection")
    if args.grouped is None:
        # the projections are independent problems: one grouped GEMM launch
        # per step when they fit one launch (INT4 weights)
        args.grouped = len(cases) > 1 and len(cases) <= w4.MAX_GROUP and fmt == "int4"
    if args.grouped and len(cases) > w4.MAX_GROUP:
        raise SystemExit(f"--grouped takes at most {w4.MAX_GROUP} projections")
    peaks = load_peaks()

    # --- kernel choice by measurement, once per shape (or per set of shapes
    # of a grouped launch), outside the timed region
    # the block's gate/up projection with the SwiGLU epilogue (--swiglu)
    epilogues = [1 if (args.swiglu and "gate_up" in c.name) else 0 for c in cases]
    if any(epilogues) and (not args.grouped or fmt != "int4" or args.act != "bf16"):
        raise SystemExit("--swiglu: INT4 weights, bf16 activations, grouped step")
    shapes = [(c.M, c.N, c.K, e) for c, e in zip(cases, epilogues)]
    if args.variant is not None:
        # one catalogue variant for every projection of the step, set in the
        # library's table (no tuning): to time or profile that kernel
        vid = w4.variant_id(args.variant)
        if fmt != "int4" or args.grouped or any(epilogues):
            raise SystemExit("--variant: INT4 weights, one launch per projection, no epilogue")
        for c in cases:
            if not w4.w4a16_variant_eligible(vid, c.M, c.N, c.K):
                raise SystemExit(f"--variant {args.variant} is not eligible for {c.M}x{c.N}x{c.K}")
            w4.w4a16_table_set(c.M, c.N, c.K, vid)
        args.tune = False
    if args.tune:
        if args.grouped:
            w4.w4a16_tune_grouped(shapes, act=fx.act_dtype)
        else:
            for c in cases:
                fx.tune(c.M, c.N, c.K)

    # --- resident inputs: the weights are quantized at load (once per copy);
    # the copies rotate step by step so that every step reads its weights and
    # activations from HBM (more than 3x L2 in total)
    host = [synthetic.draw(c, act=args.act) for c in cases]
    in_bytes = sum(gemm_bytes(c.M, c.N, c.K, fmt) for c in cases)
    copies = max(2, min(64, -(-3 * L2_BYTES // int(in_bytes))))
    W_dev = [W.to(dev) for (W, _, _) in host]
    sets = []
    for r in range(copies):
        s = []
        for j, c in enumerate(cases):
            wt = fx.new_weight(c.N, c.K)
            fx.quantize(W_dev[j], wt)
            s.append(dict(wt=wt, A=host[j][1].to(dev),
                          Y=torch.empty(c.M, c.N // 2 if epilogues[j] else c.N,
                                        dtype=fx.act_dtype, device=dev)))
        sets.append(s)
    torch.cuda.synchronize(dev)
    # inference: no kernel writes the weights between steps (they are
    # quantized above, at load), so each GEMM may request its first codes
    # and scales before the previous kernel on the stream has finished
    w4.w4a16_set_weights_static(args.static_weights)
    ws_bytes = max(fx.workspace_bytes(c.M, c.N, c.K) for c in cases)
    if args.grouped:
        probs, _, _ = w4._gemm_problems([s["A"] for s in sets[0]],
                                        [s["wt"]["packed"] for s in sets[0]],
                                        [s["wt"]["scales"] for s in sets[0]], None,
                                        [s["Y"] for s in sets[0]], epilogues)
        ws_bytes = max(ws_bytes, w4.lib().w4a16_gemm_grouped_workspace_bytes(probs, len(cases), -1))
    ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(r, st, evs=None):
        """One step: the GEMM of every projection on copy r % copies (one
        grouped launch, or one launch per projection)."""
        sset = sets[r % copies]
        if args.grouped:
            if evs is not None:
                evs[0][0].record(st)
            w4.w4a16_gemm_grouped([s["A"] for s in sset], [s["wt"]["packed"] for s in sset],
                                  [s["wt"]["scales"] for s in sset], Ys=[s["Y"] for s in sset],
                                  workspace=ws, stream=st, epilogues=epilogues)
            if evs is not None:
                evs[0][1].record(st)
            return
        for j, s in enumerate(sset):
            if evs is not None:
                evs[j][0].record(st)
            fx.gemm(s["A"], s["wt"], s["Y"], ws, st)
            if evs is not None:
                evs[j][1].record(st)

    n_launch = 1 if args.grouped else len(cases)
    # eager warm-up (also sets kernel attributes outside any capture)
    for r in range(min(args.warmup, copies)):
        step(r, stream)
    torch.cuda.synchronize(dev)
    if w4.w4a16_get_device_error() != w4.W4A16_OK:
        raise RuntimeError("device error during warm-up")

    # graph A: warm-up steps; graph B: the timed steps back to back; graph C:
    # the same steps with events around every launch (per-launch durations)
    g_warm = graph_of(dev, lambda i, st: step(i, st), args.warmup)
    l0 = w4.w4a16_launch_count()
    g_timed = graph_of(dev, lambda i, st: step(args.warmup + i, st), args.steps)
    launches = w4.w4a16_launch_count() - l0
    kev = [[[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
            for _ in range(n_launch)] for _ in range(args.steps)]
    try:
        g_ev = graph_of(dev, lambda i, st: step(args.warmup + i, st, kev[i]), args.steps)
    except (TypeError, RuntimeError):
        g_ev = None

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # --- timed region
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g_warm.replay()
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev) as clk:
        # the NVTX range marks the timed steps for profilers
        torch.cuda.nvtx.range_push("bench_timed")
        t0 = time.perf_counter()
        start.record(stream)
        g_timed.replay()
        end.record(stream)
        torch.cuda.synchronize(dev)
        clk.mark(t0, time.perf_counter())
        torch.cuda.nvtx.range_pop()
    barrier()
    elapsed_ms = start.elapsed_time(end)

    # --- per-launch durations (one launch per step: the timed region itself)
    if n_launch == 1:
        launch_ms = [elapsed_ms / args.steps]
    elif g_ev is not None:
        g_warm.replay()
        g_ev.replay()
        torch.cuda.synchronize(dev)
        launch_ms = [statistics.mean(kev[r][j][0].elapsed_time(kev[r][j][1])
                                     for r in range(args.steps)) for j in range(n_launch)]
    else:
        launch_ms = [elapsed_ms / args.steps / n_launch] * n_launch
    if w4.w4a16_get_device_error() != w4.W4A16_OK:
        raise RuntimeError("device error during timing")

    # --- the load-time quantize, timed apart: a graph of back-to-back
    # launches (grouped over the projections when the step is grouped) on
    # the resident bf16 weights
    qreps = max(4, min(args.steps, 20))
    if args.grouped:
        qouts = [(s["wt"]["packed"], s["wt"]["scales"]) for s in sets[0]]
        w4.w4a16_quantize_grouped(W_dev, outs=qouts)
        gq = graph_of(dev, lambda i, st: w4.w4a16_quantize_grouped(W_dev, outs=qouts, stream=st),
                      qreps)
        q_us = [time_graph_us(dev, gq, qreps)]
    else:
        q_us = []
        for j, c in enumerate(cases):
            gq = graph_of(dev, lambda i, st: fx.quantize(W_dev[j], sets[0][j]["wt"], st), qreps)
            q_us.append(time_graph_us(dev, gq, qreps))
    del gq

    # --- e2e: the public API on host buffers, every step: the step's
    # activations copied in from pinned host memory, its GEMMs on the
    # resident weights, its outputs copied back to pinned host memory.  The
    # steps are pipelined over three streams (copy in, compute, copy out)
    # with two device buffers for A and Y: step i's copies overlap the GEMMs
    # of steps i - 1 and i + 1, and a buffer is reused only after the copy
    # that last read it has finished.  The timed region runs from the first
    # copy in to the last copy out.
    a_host = [A.pin_memory() for (_, A, _) in host]
    y_host = [torch.empty(c.M, c.N // 2 if e else c.N, dtype=fx.act_dtype).pin_memory()
              for c, e in zip(cases, epilogues)]
    h2d = sum(a.numel() * a.element_size() for a in a_host)
    d2h = sum(y.numel() * y.element_size() for y in y_host)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = [[dict(A=torch.empty_like(s["A"]), Y=torch.empty_like(s["Y"])) for s in sets[0]] for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_gemm = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = i % 2
        wset = sets[i % copies]
        s_in.wait_event(ev_gemm[b])              # A[b]'s last GEMM is done
        with torch.cuda.stream(s_in):
            for j in range(len(cases)):
                bufs[b][j]["A"].copy_(a_host[j], non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])              # Y[b]'s last copy out is done
        if args.grouped:
            w4.w4a16_gemm_grouped([x["A"] for x in bufs[b]], [s["wt"]["packed"] for s in wset],
                                  [s["wt"]["scales"] for s in wset], Ys=[x["Y"] for x in bufs[b]],
                                  workspace=ws, stream=stream, epilogues=epilogues)
        else:
            for j, s in enumerate(wset):
                fx.gemm(bufs[b][j]["A"], s["wt"], bufs[b][j]["Y"], ws, stream)
        ev_gemm[b].record(stream)
        s_out.wait_event(ev_gemm[b])
        with torch.cuda.stream(s_out):
            for j in range(len(cases)):
                y_host[j].copy_(bufs[b][j]["Y"], non_blocking=True)
        ev_out[b].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)

    # the host link alone, outside the timed region: one step's copies in,
    # then its copies out, each direction by itself (median of 3)
    def copies_ms(fn, st):
        ts = []
        for _ in range(3):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(st)
            with torch.cuda.stream(st):
                fn()
            c1.record(st)
            torch.cuda.synchronize(dev)
            ts.append(c0.elapsed_time(c1))
        return statistics.median(ts)

    t_in = copies_ms(lambda: [bufs[0][j]["A"].copy_(a_host[j], non_blocking=True) for j in range(len(cases))],
                     s_in)
    t_out = copies_ms(lambda: [y_host[j].copy_(bufs[0][j]["Y"], non_blocking=True) for j in range(len(cases))],
                      s_out)

    def both_ms():
        # a step's copies in and out at once, on their two streams
        ts = []
        cur = torch.cuda.current_stream(dev)
        for _ in range(3):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(cur)
            for st, fn in ((s_in, lambda: [bufs[0][j]["A"].copy_(a_host[j], non_blocking=True)
                                           for j in range(len(cases))]),
                           (s_out, lambda: [y_host[j].copy_(bufs[1][j]["Y"], non_blocking=True)
                                            for j in range(len(cases))])):
                st.wait_event(c0)
                with torch.cuda.stream(st):
                    fn()
                done = torch.cuda.Event()
                done.record(st)
                cur.wait_event(done)
            c1.record(cur)
            torch.cuda.synchronize(dev)
            ts.append(c0.elapsed_time(c1))
        return statistics.median(ts)

    t_both = both_ms()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(s_in)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    if w4.w4a16_get_device_error() != w4.W4A16_OK:
        raise RuntimeError("device error during the end-to-end steps")

    elapsed_ms, e2e_ms = max_over_ranks([elapsed_ms, e2e_ms], world, dev)
    flops_step = sum(gemm_flops(c.M, c.N, c.K) for c in cases)
    bytes_step = sum(gemm_bytes(c.M, c.N, c.K, fmt) for c in cases)
    wbytes_step = sum(weight_bytes(c.N, c.K, fmt) for c in cases)
    value = job_rate(flops_step, args.steps, elapsed_ms, world) / 1e12
    e2e_value = job_rate(flops_step, args.steps, e2e_ms, world) / 1e12

    # --- kernels: the step's GEMM launches, then the load-time quantize
    kernels = []
    if args.grouped:
        kernels.append(dict(kernel=fx.gname, grouped=len(cases), us=round(launch_ms[0] * 1e3, 3),
                            tflops=round(flops_step / (launch_ms[0] * 1e-3) / 1e12, 2),
                            weight_gbs=round(wbytes_step / (launch_ms[0] * 1e-3) / 1e9, 1),
                            gbs=round(bytes_step / (launch_ms[0] * 1e-3) / 1e9, 1)))
        qb = sum(quant_bytes(c.N, c.K, fmt) for c in cases)
        kernels.append(dict(kernel=fx.qname, grouped=len(cases), us=round(q_us[0], 3),
                            gbs=round(qb / (q_us[0] * 1e-6) / 1e9, 1),
                            when="load time, outside the step"))
    else:
        for j, c in enumerate(cases):
            t = launch_ms[j]
            kernels.append(dict(kernel=fx.gname, shape=[c.M, c.N, c.K], us=round(t * 1e3, 3),
                                variant=fx.variant(c.M, c.N, c.K),
                                tflops=round(gemm_flops(c.M, c.N, c.K) / (t * 1e-3) / 1e12, 2),
                                weight_gbs=round(weight_bytes(c.N, c.K, fmt) / (t * 1e-3) / 1e9, 1),
                                gbs=round(gemm_bytes(c.M, c.N, c.K, fmt) / (t * 1e-3) / 1e9, 1)))
        for j, c in enumerate(cases):
            kernels.append(dict(kernel=fx.qname, shape=[c.N, c.K], us=round(q_us[j], 3),
                                gbs=round(quant_bytes(c.N, c.K, fmt) / (q_us[j] * 1e-6) / 1e9, 1),
                                when="load time, outside the step"))

    # --- roofline of the step's kernel family (the GEMM): algorithmic work
    # per launch over the launches' measured durations
    dom_ms = sum(launch_ms)
    t_hbm = bytes_step / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops_step / (peaks["bf16_tflops"] * 1e12)
    if t_tc >= t_hbm:
        bound, peak, unit = "tensor", peaks["bf16_tflops"], "TFLOP/s"
        achieved = flops_step / (dom_ms * 1e-3) / 1e12
    else:
        bound, peak, unit = "hbm", peaks["hbm_gbs"], "GB/s"
        achieved = bytes_step / (dom_ms * 1e-3) / 1e9
    # the recorded traffic is keyed by workload (or --shape) and, when one
    # was forced, the variant: another workload's figure never applies
    tkey = ("shape_" + args.shape.replace(",", "x") if args.shape else args.workload) + \
        ("_grouped" if args.grouped else "") + ("" if fmt == "int4" else "_" + fmt) + \
        ("_f16" if args.act == "f16" else "") + ("_" + args.variant if args.variant else "")
    traffic = dram_traffic(fx.gname, tkey)
    roofline = dict(bound=bound, achieved=round(achieved, 2), peak=peak, unit=unit,
                    frac=round(achieved / peak, 4),
                    traffic=None if traffic is None else traffic / n_launch,
                    traffic_source=(None if traffic is None else
                                    "profiles/dram_traffic.txt: ncu dram__bytes_read.sum + "
                                    "dram__bytes_write.sum per launch, taken on kernel sources "
                                    "hash %s (the current ones)" % kernel_source_hash()),
                    kernel=fx.gname, launches_per_step=n_launch, peak_source=peaks["source"],
                    algorithmic=("%.0f flops per step" % flops_step if bound == "tensor" else
                                 "%.0f bytes per step (codes + scales + activations)" % bytes_step))

    # --- each distinct GEMM shape of the workload alone, back to back; and
    # (default run) the metric's bandwidth-bound end: the M in {1, 4, 16, 64}
    # sweep, every shape back to back with its roofline fraction
    del g_timed, g_warm, g_ev
    wcache = {}
    b2b = [back_to_back(fx, c, peaks, wcache, args.tune, dev) for c in
           {(c.M, c.N, c.K): c for c in cases}.values()] if len(cases) > 1 else []
    if args.swiglu:
        b2b += [back_to_back(fx, c, peaks, wcache, args.tune, dev, swiglu=True)
                for c, e in zip(cases, epilogues) if e]
    sweep = block = None
    if (args.workload == "large" and not args.shape and not args.no_sweep and fmt == "int4"
            and args.act == "bf16"):
        del sets, W_dev
        torch.cuda.empty_cache()
        sweep = [back_to_back(fx, c, peaks, wcache, args.tune, dev) for c in synthetic.SWEEP]
        # the action-expert block (M = 50) as one grouped launch, plain and
        # with the SwiGLU epilogue on its gate/up projection
        ex = synthetic.EXPERT_M50
        block = [grouped_back_to_back(w4, ex, [0] * len(ex), peaks, args.tune, dev),
                 grouped_back_to_back(w4, ex, [1 if "gate_up" in c.name else 0 for c in ex],
                                      peaks, args.tune, dev)]
        # the same projections at decode sizes (M = 1 and 4): one grouped
        # launch, whose plan may take the row-block kernel
        import dataclasses
        for m in (1, 4):
            dec = [dataclasses.replace(c, M=m, name=c.name.replace("m50", f"m{m}")) for c in ex]
            block.append(grouped_back_to_back(w4, dec, [0] * len(dec), peaks, args.tune, dev))
    if w4.w4a16_get_device_error() != w4.W4A16_OK:
        raise RuntimeError("device error during the back-to-back GEMM timing")

    out = dict(metric=METRIC, value=round(value, 3), unit="TFLOP/s", n_gpus=world, steps=args.steps,
               warmup=args.warmup, ms_per_step=round(elapsed_ms / args.steps, 5),
               higher_is_better=True, scaling="weak", vs_baseline=None, dtype=args.act,
               data="synthetic",
               config=dict(workload=args.workload if not args.shape else "shape " + args.shape,
                           activations=args.act, weights=fmt,
                           shapes=[[c.M, c.N, c.K] for c in cases],
                           step=("one grouped W4A16 GEMM launch over all projections"
                                 if args.grouped else "one GEMM launch per projection") +
                                (" (gate/up with the SwiGLU epilogue)" if any(epilogues) else "") +
                                " on weights quantized at load (the quantize is timed apart, "
                                "under kernels)",
                           l2="inputs rotate over %d copies (%.0f MB of weights and activations "
                              "> 3x L2)" % (copies, copies * in_bytes / 2**20),
                           selection=(f"forced: {args.variant}" if args.variant is not None
                                      else "tuned by measurement before timing" if args.tune
                                      else "cost-model rule"),
                           weights_static=bool(args.static_weights),
                           parallelism=f"replicas x{world}"),
               gemm=dict(tflops=round(value, 3),
                         weight_gbs=round(job_rate(wbytes_step, args.steps, elapsed_ms, world) / 1e9, 1),
                         gbs=round(job_rate(bytes_step, args.steps, elapsed_ms, world) / 1e9, 1)),
               kernels=kernels, roofline=roofline, clocks=clk.summary(),
               gpu_launches=int(launches),
               e2e=dict(value=round(e2e_value, 3), unit="TFLOP/s", h2d_bytes_per_step=int(h2d),
                        d2h_bytes_per_step=int(d2h),
                        pipeline="copy in, GEMM and copy out on three streams, two device "
                                 "buffers for A and Y: step i's copies overlap the GEMMs of "
                                 "its neighbours",
                        link=dict(h2d_gbs=round(h2d / (t_in * 1e-3) / 1e9, 1),
                                  d2h_gbs=round(d2h / (t_out * 1e-3) / 1e9, 1),
                                  h2d_ms=round(t_in, 4), d2h_ms=round(t_out, 4),
                                  both_ms=round(t_both, 4),
                                  note="one step's copies outside the timed region: each "
                                       "direction alone, then both at once (both_ms: the "
                                       "shortest step the link allows)")))
    if b2b:
        out["gemm_back_to_back"] = b2b
    if block is not None:
        out["expert_block_grouped"] = block
    if sweep is not None:
        out["sweep"] = sweep
        out["sweep_roofline_frac"] = dict(
            min=min(e["roofline_frac"] for e in sweep), max=max(e["roofline_frac"] for e in sweep),
            bound="hbm", peak=peaks["hbm_gbs"], unit="GB/s",
            note="each sweep shape alone, back to back, weight copies > 3x L2; roofline = max of "
                 "(codes + scales + activations) / HBM peak and flops / bf16 peak")
    return out


# ------------------------------------------------------------- CPU oracle
def time_oracle(workload, budget_s: float, weights="int4", rows=1024):
    """The oracle as it stands, on the host cores: each projection's weight
    quantized once by the oracle (load time, untimed), then the oracle's GEMM
    (dequantize + FP32 matmul) on the first `rows` rows of the activations,
    projection after projection, until `budget_s` is used.  Returns the rate
    in the metric's unit (TFLOP/s of the GEMM flops done)."""
    import numpy as np  # noqa: F401

    import oracle
    from weight_only_int4_rtn_gb300 import synthetic

    cases = synthetic.WORKLOADS[workload] if isinstance(workload, str) else workload
    name = workload if isinstance(workload, str) else cases[0].name
    prepared = []
    for c in cases:
        W, A, _ = synthetic.draw(c)
        wb, ab = synthetic.bits(W), synthetic.bits(A)
        mr = min(c.M, rows)
        if weights == "int8":
            p, s = oracle.quantize8(wb)
            fn = (lambda a, p=p, s=s: oracle.gemm8(a, p, s))
        elif weights == "mxfp4":
            p, s = oracle.quantize_mxfp4_f32(oracle.bf16_bits_to_f32(wb))
            fn = (lambda a, p=p, s=s: oracle.gemm_fp4(a, oracle.dequantize_mxfp4(p, s)))
        elif weights == "nvfp4":
            p, s, g = oracle.quantize_nvfp4_f32(oracle.bf16_bits_to_f32(wb))
            fn = (lambda a, p=p, s=s, g=g: oracle.gemm_fp4(a, oracle.dequantize_nvfp4(p, s, g)))
        else:
            p, s = oracle.quantize(wb)
            fn = (lambda a, p=p, s=s: oracle.gemm(a, p, s))
        prepared.append((c, ab[:mr], mr, fn))
    flops = 0.0
    passes = 0
    t0 = time.perf_counter()
    while True:
        for c, a, mr, fn in prepared:
            fn(a)
            flops += gemm_flops(mr, c.N, c.K)
        passes += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sampled = any(mr < c.M for c, _, mr, _ in prepared)
    sample = (f"{passes} pass(es) of {name}: the oracle's "
              + ({"int8": "INT8 ", "mxfp4": "MXFP4 ", "nvfp4": "NVFP4 "}.get(weights, ""))
              + "GEMM (dequantize + FP32 matmul) per projection"
              + (f" on the first {rows} rows of A" if sampled else "")
              + "; weights quantized once by the oracle beforehand (load time, untimed)")
    return dict(value=round(flops / dt / 1e12, 6), unit="TFLOP/s", cores=cores, kind="oracle",
                sample=sample, seconds=round(dt, 2), passes=passes)


# the shapes on which the selection rule is checked against measurement: the
# metric's M range on the sweep's and the workloads' weight shapes
REGRET_NK = [(16384, 2048), (2048, 16384), (8192, 8192), (4096, 4096), (2048, 8192),
             (28672, 4096), (1024, 4096), (4096, 14336)]
REGRET_SHAPES = ([(m, n, k) for m in (1, 2, 4, 8, 16, 32, 64) for n, k in REGRET_NK] +
                 [(m, n, k) for m in (50, 128, 256, 816)
                  for n, k in ((8192, 8192), (2048, 2048), (32768, 2048), (1024, 4096))])


def rule_regret(dev, trials=10):
    """Every eligible INT4 (bf16) variant timed back to back on each shape of
    REGRET_SHAPES (weights static, copies rotating past 3x L2): the variant
    the library's cost-model rule selects on this device against the fastest
    measured one.  The measured, memoized choice ("Kernel dispatch and
    Humming quantization in PhyAI", section "Keep selection work out of
    repeated inference") is the tuners'; this checks the rule that shapes
    without a table entry take."""
    import torch
    import weight_only_int4_rtn_gb300 as w4
    from weight_only_int4_rtn_gb300 import synthetic
    w4.w4a16_set_weights_static(True)
    rows = []
    for (M, N, K) in REGRET_SHAPES:
        case = synthetic.Case("regret", M, N, K, 3)
        W = synthetic.draw_weight_only(case.seed, N, K, case.wdist).to(dev)
        packed, scales = w4.w4a16_quantize(W)
        torch.cuda.synchronize(dev)
        del W
        _, A, _ = synthetic.draw(case)
        A = A.to(dev)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        nb = packed.numel() + scales.numel() * 2
        ncp = max(1, min(16, -(-3 * L2_BYTES // nb)))
        cps = [(packed, scales)] + [(packed.clone(), scales.clone()) for _ in range(ncp - 1)]
        reps = max(8, 2 * ncp)
        times = {}
        for v in range(w4.w4a16_variant_count()):
            if not w4.w4a16_variant_eligible(v, M, N, K):
                continue
            ws = torch.zeros(max(w4.w4a16_variant_workspace_bytes(v, M, N, K), 256),
                             dtype=torch.uint8, device=dev)

            def one(i, st=None, v=v, ws=ws):
                w4.w4a16_gemm(A, cps[i % ncp][0], cps[i % ncp][1], Y=Y, workspace=ws, variant=v,
                              stream=st)
            for i in range(2):
                one(i)
            g = graph_of(dev, one, reps)
            times[w4.w4a16_variant_name(v)] = time_graph_us(dev, g, reps, trials)
            del g
        if w4.w4a16_get_device_error() != w4.W4A16_OK:
            raise RuntimeError("device error while timing the variants")
        pick = w4.w4a16_variant_name(w4.w4a16_select_variant(M, N, K))
        best = min(times, key=times.get)
        rows.append(dict(shape=[M, N, K], rule=pick, rule_us=round(times[pick], 3), best=best,
                         best_us=round(times[best], 3),
                         regret=round(times[pick] / times[best] - 1.0, 4)))
        del cps, packed, scales
    regrets = [r["regret"] for r in rows]
    return dict(metric="selection rule regret (rule's variant / fastest variant - 1)",
                unit="fraction", shapes=len(rows), mean=round(sum(regrets) / len(regrets), 4),
                worst=max(regrets), above_5pct=sum(1 for x in regrets if x > 0.05),
                kernel_sources=kernel_source_hash(), rows=rows)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large",
                    choices=["tiny", "expert_m50", "prefix_m816", "sweep", "large"])
    ap.add_argument("--act", default="bf16", choices=["bf16", "f16"],
                    help="activation type of the GEMMs (A, bias, Y)")
    ap.add_argument("--grouped", dest="grouped", action="store_true", default=None,
                    help="one grouped GEMM launch per step (the projections are independent "
                         "problems; the default when the workload has 2 to 8 projections)")
    ap.add_argument("--per-projection", dest="grouped", action="store_false",
                    help="one GEMM launch per projection")
    ap.add_argument("--weights", default="int4", choices=["int4", "int8", "mxfp4", "nvfp4"],
                    help="weight scheme: INT4 (W4A16), INT8 (W8A16), MXFP4 or NVFP4 weights")
    ap.add_argument("--sr-seed", type=int, default=None,
                    help="quantize at load with seeded stochastic rounding (w4a16_quantize_sr) "
                         "instead of round to nearest")
    ap.add_argument("--shape", default=None,
                    help="M,N,K: one projection of this shape instead of the workload's")
    ap.add_argument("--variant", default=None,
                    help="INT4: run every projection of the step with this catalogue variant "
                         "(set in the library's table; no tuning)")
    ap.add_argument("--swiglu", action="store_true",
                    help="the gate/up projection takes the SwiGLU epilogue: inside the grouped "
                         "step, and back to back through w4a16_gemm_swiglu (INT4, bf16)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="leave out the M in {1, 4, 16, 64} sweep of the default line")
    ap.add_argument("--no-tune", dest="tune", action="store_false", default=True,
                    help="select kernels by the cost-model rule instead of tuning each "
                         "shape by measurement first")
    ap.add_argument("--dynamic-weights", dest="static_weights", action="store_false", default=True,
                    help="do not declare the weights static (w4a16_set_weights_static): every GEMM "
                         "then waits for the previous kernel before its first weight copy")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rule-regret", action="store_true",
                    help="instead of the step: time every eligible INT4 variant on a grid of "
                         "72 shapes and report the selection rule's regret (one JSON line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        # each step a bounded sample of the workload: about 1.2 s of oracle work
        t_budget = max(5.0, min(90.0, 1.2 * (args.steps + args.warmup)))
        cb = time_oracle(workload_cases(args), t_budget, args.weights)
        # a step of this arm is one sampled pass of the oracle (see the sample)
        line = dict(metric=METRIC, value=cb["value"], unit="TFLOP/s", n_gpus=world,
                    steps=args.steps, warmup=args.warmup,
                    ms_per_step=round(cb["seconds"] * 1e3 / max(cb["passes"], 1), 3),
                    higher_is_better=True,
                    scaling="weak", vs_baseline=None, dtype="f32", data="synthetic",
                    impl="reference",
                    config=dict(workload=args.workload if not args.shape else "shape " + args.shape,
                                weights=args.weights),
                    cpu_baseline=cb,
                    e2e=dict(value=cb["value"], unit="TFLOP/s", h2d_bytes_per_step=0,
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
    if args.rule_regret:
        import torch
        if rank == 0:
            print(json.dumps(rule_regret(torch.device("cuda", 0))), flush=True)
        return 0
    out = run_gpu(args, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = time_oracle(workload_cases(args), args.cpu_budget, args.weights)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
