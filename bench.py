#!/usr/bin/env python3
"""Benchmark of the MX block-scaled GEMM hot path on one GB300 (or N, as
independent replicas: weak scaling).

One step = the whole path on one batch of synthetic input resident in HBM:
  mx_quantize(A fp32 8192 x 8192 -> E4M3 + UE8M0)
  mx_quantize(B fp32 8192 x 8192, row-major K x N -> E4M3 + UE8M0, K-major)
  mx_gemm(A_mx, B_mx -> C bf16 8192 x 8192)
value = 2*M*N*K / step time, in TFLOP/s.  The fp32 sources (268 MB each) are
larger than L2 (129 MB), so no step finds its inputs in L2.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
                  [--workload mxfp8_8192|mxfp4_8192|bf16_4096|...]

--impl reference times the CPU oracle (float64, OpenMP) on a bounded sample
of the same workload (rows of C computed from the fp32 sources) on the host
cores.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# nominal dense tensor rate of each kind relative to bf16 (2.25 / 4.5 / 13.5
# PFLOP/s for bf16 / fp8 / fp4); an E2M1 operand beside an 8-bit one runs at
# the FP8 rate
NOMINAL_RATIO = {"bf16": 1.0, "f16": 1.0, "mxfp8": 2.0, "mxfp4": 6.0,
                 "mxfp8_e5m2": 2.0, "w4a8": 2.0,
                 # weight-only: B dequantized to bf16, the bf16 tensor rate
                 "w8a16": 1.0, "w4a16": 1.0, "w2a16": 1.0}
# the per-clock rate of each kind's tcgen05.mma relative to bf16, measured on
# GB300 with back-to-back MMAs in the forms the kernels issue (cta_group::2,
# M = 256, N = 256, and the 1-CTA forms): fp8 2x, every FP4 form 4x (not the
# nominal 6x); profiles/mx_gemm_mxfp4_8192.md
INSTRUCTION_RATIO = dict(NOMINAL_RATIO, mxfp4=4.0)
DTYPE_NAME = {"mxfp8": "e4m3", "mxfp4": "e2m1", "mxfp8_e5m2": "e5m2",
              "w4a8": "e4m3 x e2m1"}
# dense flop per clock per SM of each kind's MMA, measured on this machine's
# GB300 (profiles/mx_gemm_mxfp4_8192.md): the clock-normalised peak is
# SM count x this x the SM clock the work ran at
PER_CLOCK = {k: 8192.0 * v for k, v in INSTRUCTION_RATIO.items()}
# NVIDIA's nominal dense figures for one GB300, TFLOP/s (context)
NOMINAL_TFLOPS = {"bf16": 2250.0, "f16": 2250.0, "mxfp8": 4500.0,
                  "mxfp8_e5m2": 4500.0, "w4a8": 4500.0, "mxfp4": 13500.0,
                  "w8a16": 2250.0, "w4a16": 2250.0, "w2a16": 2250.0}
NOMINAL_HBM_GBS = 7900.0


PROFILES = os.path.join(ROOT, "profiles")
GEMM_SOURCES = [os.path.join(ROOT, "block_scaled_quantized_mx_gb300", "csrc", f)
                for f in ("gemm.cu", "gemm_kernel.cuh", "gemm_mxf8.cu", "gemm_common.cuh",
                          "mx_rule.cuh", "ptx.cuh", "common.cuh")]


def gemm_source_hash() -> str:
    h = hashlib.sha256()
    for p in GEMM_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the GEMM kernel on this workload, from the
    traffic record of a committed ncu summary under profiles/, or None when
    there is none or the kernel's sources changed since it was taken."""
    want = gemm_source_hash()
    try:
        names = sorted(os.listdir(PROFILES))
    except OSError:
        return None
    for name in names:
        with open(os.path.join(PROFILES, name)) as f:
            for line in f:
                line = line.strip()
                if not line.startswith("traffic-record:"):
                    continue
                kv = dict(t.split("=", 1) for t in line.split()[1:])
                if kv.get("workload") == workload and kv.get("sources") == want:
                    return int(kv["bytes_per_launch"])
    return None


def ws_format(fa, fb):
    """The format mx_gemm_workspace_bytes takes for an operand pair."""
    return fa if fa == fb else 1


def peaks():
    try:
        with open(MEASURED_PEAKS) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "measured")
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ------------------------------------------------------------------ clocks

# NVML clock-event reason bits (nvmlClocksEventReason*)
_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class NvmlClock:
    """Query-only NVML readings of one GPU through ctypes (libnvidia-ml): the
    SM clock, its maximum, the clock-event reasons and the power draw.
    Nothing is set.  Raises OSError / RuntimeError when NVML is missing."""

    def __init__(self, index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index),
                                                  ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle for GPU %d" % index)
        reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = reasons or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        v = ctypes.c_uint()
        self.max_mhz = (float(v.value) if self.lib.nvmlDeviceGetMaxClockInfo(
            self.h, 1, ctypes.byref(v)) == 0 else None)

    def read(self):
        ct = self.ct
        clk, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        ok = self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk)) == 0   # SM
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw))
        self.reasons_fn(self.h, ct.byref(rs))
        return (float(clk.value) if ok else None, pw.value / 1000.0, int(rs.value))


class ClockSampler:
    """SM clock, power and clock-event reasons sampled every 2 ms from a
    thread while the timed work runs (NVML; nvidia-smi at its 100 ms
    floor when NVML cannot be loaded)."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_s: float = 0.002):
        self.index = index
        self.period = period_s
        self.rows = []
        self.thread = None
        self.proc = None
        self.path = None
        try:
            self.nvml = NvmlClock(index)
        except Exception:
            self.nvml = None

    def start(self):
        import threading
        self.rows = []
        if self.nvml is not None:
            self.stop_flag = threading.Event()

            def loop():
                while not self.stop_flag.is_set():
                    try:
                        self.rows.append(self.nvml.read())
                    except Exception:
                        pass
                    time.sleep(self.period)
            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            time.sleep(0.01)
            return
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.thread is not None:
            time.sleep(0.01)
            self.stop_flag.set()
            self.thread.join(timeout=2)
            self.thread = None
            rows = [r for r in self.rows if r[0] is not None]
            if not rows:
                return None
            sm = [r[0] for r in rows]
            bits = 0
            for r in rows:
                bits |= r[2]
            return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm),
                    "sm_max_mhz": self.nvml.max_mhz or max(sm),
                    "power_w_max": max(r[1] for r in rows),
                    "samples": len(rows), "source": "NVML, 2 ms",
                    "reasons": sorted(n for b, n in _REASONS.items() if bits & b)}
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for ln in open(self.path):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        sm = [r[0] for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2])
                          if v.lower().startswith("active")})
        loaded = [s for s in sm if s >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded),
                "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "source": "nvidia-smi, 100 ms",
                "reasons": reasons}


# ------------------------------------------------------------------ our arm

def flops_of(c):
    return 2.0 * c.M * c.N * c.K


def metric_name(c):
    """The metric both arms print for a workload (identical strings, so that
    the two lines can be divided)."""
    return "%s GEMM TFLOP/s" % c.kind


def step_description(c):
    """What one step of the workload computes (both arms do this work)."""
    if workloads.is_mx(c):
        return ("mx_quantize(A fp32) + mx_quantize(B fp32, K-strided) + "
                "mx_gemm(A_mx, B_mx) -> %s C; TFLOP/s = 2 M N K / step time"
                % c.out)
    return "gemm_f16(A, B) -> %s C; TFLOP/s = 2 M N K / step time" % c.out


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """Largest elapsed time over all ranks (every rank gets the result).
    Ranks are independent replicas of the step, so the job's time is the
    slowest rank's; with one rank this is the identity."""
    if world <= 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank: float, world: int, ms: float) -> float:
    """Whole-job TFLOP/s: the work of all ranks over the slowest rank's time."""
    return flops_per_rank * world / (ms * 1e-3) / 1e12


L2_BYTES = 129 * 2 ** 20


class L2Flusher:
    """Writes a buffer larger than L2 so that the next kernel starts cold."""

    def __init__(self, dev):
        self.buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32,
                               device=dev)

    def __call__(self):
        self.buf.fill_(1.0)


def event_time(f, iters=20, flusher=None):
    """Mean CUDA-event time (ms) of f() on the current stream, after 3
    untimed calls; L2 flushed (untimed) before every call when a flusher is
    given."""
    for _ in range(3):
        f()
    stream = torch.cuda.current_stream()
    tot = 0.0
    for _ in range(iters):
        if flusher is not None:
            flusher()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        f()
        e1.record(stream)
        e1.synchronize()
        tot += e0.elapsed_time(e1)
    return tot / iters


def time_gemm_only(mx, c, dev, iters=20, flusher=None, splitk=False):
    """CUDA-event time of the GEMM kernel alone on pre-quantized operands
    (mean over iters; L2 flushed before every launch when a flusher is
    given).  Returns (ms, TFLOP/s)."""
    A, B = workloads.sources(c)
    dA, dB = A.to(dev), B.to(dev)
    out_dt = torch.bfloat16 if c.out == "bf16" else torch.float32
    C = torch.empty((c.M, c.N), dtype=out_dt, device=dev)
    if workloads.is_dequant(c):
        qb = mx.mx_quantize(B.to(dev), workloads.formats(c)[1], k_strided=True)
        # the K-split whenever the tiles leave SMs idle (decode shapes)
        nb = mx.gemm_dequant_workspace_bytes(c.M, c.N, c.K)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None
        f = lambda: mx.gemm_dequant(dA, qb, out_dtype=out_dt, out=C,  # noqa
                                    workspace=ws)
    elif workloads.is_mx(c):
        fa, fb = workloads.formats(c)
        qa = mx.mx_quantize(dA, fa)
        qb = mx.mx_quantize(dB, fb, k_strided=True)
        del dA, dB
        nb = (mx.mx_gemm_workspace_bytes(ws_format(fa, fb), c.M, c.N, c.K)
              if splitk else 0)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None
        f = lambda: mx.mx_gemm(qa, qb, out_dtype=out_dt, out=C, workspace=ws)  # noqa
    else:
        nb = mx.gemm_f16_workspace_bytes(c.M, c.N, c.K) if splitk else 0
        ws = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None
        f = lambda: mx.gemm_f16(dA, dB, out=C, workspace=ws)  # noqa
    ms = event_time(f, iters, flusher)
    assert mx.mx_last_error() == 0
    return ms, flops_of(c) / (ms * 1e-3) / 1e12


def time_gemm_graph(mx, c, dev, min_bytes=3 * L2_BYTES, replays=5):
    """Mean time per GEMM of a CUDA graph of back-to-back launches over R
    distinct operand sets whose bytes together exceed L2 (so every launch
    finds its operands outside L2), replayed between CUDA events on the
    current stream: a stream of independent GEMMs, each launch's host cost
    removed by the graph.  The K-split workspace is used where the library
    asks for one.  Returns (ms per GEMM, R)."""
    A, B = workloads.sources(c)
    dA0, dB0 = A.to(dev), B.to(dev)
    out_dt = torch.bfloat16 if c.out == "bf16" else torch.float32
    if workloads.is_dequant(c):
        fb = workloads.formats(c)[1]
        q0 = mx.mx_quantize(dB0, fb, k_strided=True)
        set_bytes = dA0.numel() * 2 + q0.data.numel() + q0.scales.numel()
        nb = mx.gemm_dequant_workspace_bytes(c.M, c.N, c.K)
    elif workloads.is_mx(c):
        fa, fb = workloads.formats(c)
        qa0 = mx.mx_quantize(dA0, fa)
        qb0 = mx.mx_quantize(dB0, fb, k_strided=True)
        set_bytes = (qa0.data.numel() + qa0.scales.numel() + qb0.data.numel() +
                     qb0.scales.numel())
        nb = mx.mx_gemm_workspace_bytes(ws_format(fa, fb), c.M, c.N, c.K)
    else:
        set_bytes = (dA0.numel() + dB0.numel()) * 2
        nb = mx.gemm_f16_workspace_bytes(c.M, c.N, c.K)
    set_bytes += c.M * c.N * (2 if out_dt == torch.bfloat16 else 4)
    R = max(2, min(64, -(-min_bytes // set_bytes)))
    ws = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None
    calls = []
    for i in range(R):
        C = torch.empty((c.M, c.N), dtype=out_dt, device=dev)
        if workloads.is_dequant(c):
            a = dA0.clone()
            qb = mx.MXTensor(q0.data.clone(), q0.scales.clone(), q0.fmt, q0.outer, q0.K)
            calls.append(lambda s, a=a, qb=qb, C=C: mx.gemm_dequant(
                a, qb, out_dtype=out_dt, out=C, workspace=ws, stream=s))
        elif workloads.is_mx(c):
            qa = mx.MXTensor(qa0.data.clone(), qa0.scales.clone(), qa0.fmt, qa0.outer, qa0.K)
            qb = mx.MXTensor(qb0.data.clone(), qb0.scales.clone(), qb0.fmt, qb0.outer, qb0.K)
            calls.append(lambda s, qa=qa, qb=qb, C=C: mx.mx_gemm(
                qa, qb, out_dtype=out_dt, out=C, workspace=ws, stream=s))
        else:
            a, b = dA0.clone(), dB0.clone()
            calls.append(lambda s, a=a, b=b, C=C: mx.gemm_f16(
                a, b, out=C, workspace=ws, stream=s))
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for f in calls:
            f(s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for f in calls:
            f(s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(replays):
        g.replay()
    e1.record()
    e1.synchronize()
    assert mx.mx_last_error() == 0
    ms = e0.elapsed_time(e1) / (replays * R)
    del g, calls
    return ms, R


def back_to_back_time(f, n=20):
    """Mean CUDA-event time (ms) of n calls of f launched back to back
    between one pair of events (after 3 untimed calls), so that host launch
    latency is hidden behind the GPU's work; for kernels whose inputs exceed
    L2."""
    for _ in range(3):
        f()
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n):
        f()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / n


def time_quantize_formats(mx, dA, dB, fmts, rows, K):
    """mx_quantize throughput of every element format on the step's fp32
    sources (each larger than L2), calls back to back: GB/s of algorithmic
    bytes for the A (K-contiguous) and B (K-strided, transposing) layouts."""
    out = {}
    for fmt, name in fmts:
        qa = mx.empty_mx(fmt, rows, K, dA.device)
        qb = mx.empty_mx(fmt, rows, K, dA.device)
        ta = back_to_back_time(lambda: mx.mx_quantize(dA, fmt, out=qa))
        tb = back_to_back_time(lambda: mx.mx_quantize(dB, fmt, k_strided=True, out=qb))
        gb = quant_bytes(fmt, rows, K)
        out[name] = {"a_ms": ta, "b_ms": tb, "a_gbs": gb / ta / 1e6,
                     "b_gbs": gb / tb / 1e6}
    assert mx.mx_last_error() == 0
    return out


def time_fused(mx, c, dev, flusher):
    """The fused epilogue against the decomposed path on one MX workload
    (the RIGEL summary's fused GEMM + bias + GELU, Main findings section 4):
      gemm             mx_gemm, bf16 C (no epilogue work)
      fused            mx_gemm_fused, bias + GELU, bf16 C
      decomposed       mx_gemm fp32 C, then bias + GELU as a separate
                       elementwise pass (torch), bf16 result
      fused_quantize   mx_gemm_fused_quantize, bias + GELU, C as E4M3 MX
      two_step_quantize  mx_gemm_fused fp32 C, then mx_quantize
    Every launch starts with L2 flushed.  Returns milliseconds and the gains
    of the fused forms."""
    fa, fb = workloads.formats(c)
    A, B = workloads.sources(c)
    qa = mx.mx_quantize(A.to(dev), fa)
    qb = mx.mx_quantize(B.to(dev), fb, k_strided=True)
    bias = (torch.randn(c.N, generator=torch.Generator().manual_seed(9)) *
            0.5).to(dev)
    Cb = torch.empty((c.M, c.N), dtype=torch.bfloat16, device=dev)
    Cf = torch.empty((c.M, c.N), dtype=torch.float32, device=dev)
    q = mx.empty_mx(mx.E4M3, c.M, c.N, dev)
    gelu = torch.nn.functional.gelu

    def decomposed():
        mx.mx_gemm(qa, qb, out_dtype=torch.float32, out=Cf)
        Cb.copy_(gelu(Cf + bias))

    def two_step():
        mx.mx_gemm_fused(qa, qb, bias, mx.ACT_GELU, out_dtype=torch.float32,
                         out=Cf)
        mx.mx_quantize(Cf, mx.E4M3, out=q)

    t = {
        "gemm": event_time(lambda: mx.mx_gemm(qa, qb, out=Cb), flusher=flusher),
        "fused": event_time(lambda: mx.mx_gemm_fused(qa, qb, bias, mx.ACT_GELU,
                                                     out=Cb), flusher=flusher),
        "decomposed": event_time(decomposed, flusher=flusher),
        "fused_quantize": event_time(
            lambda: mx.mx_gemm_fused_quantize(qa, qb, mx.E4M3, bias,
                                              mx.ACT_GELU, out=q),
            flusher=flusher),
        "two_step_quantize": event_time(two_step, flusher=flusher),
    }
    assert mx.mx_last_error() == 0
    out = {k + "_ms": v for k, v in t.items()}
    out["fused_gain_vs_decomposed"] = t["decomposed"] / t["fused"] - 1.0
    out["fused_cost_vs_gemm"] = t["fused"] / t["gemm"] - 1.0
    out["fused_quantize_gain_vs_two_step"] = \
        t["two_step_quantize"] / t["fused_quantize"] - 1.0
    out["fused_tflops"] = flops_of(c) / (t["fused"] * 1e-3) / 1e12
    return out


def time_attention(mx, c, dev, flusher):
    """flash_attention on one attention workload (L2 flushed before each
    launch): ms, TFLOP/s (4 BH Lq Lk d flop: the two matmuls), the fraction of
    the bf16 peak, and torch's scaled_dot_product_attention on the same
    tensors as library context."""
    Q, K, V = (t.to(dev) for t in workloads.attn_sources(c))
    O = torch.empty(Q.shape, dtype=torch.bfloat16, device=dev)
    ms_whole = event_time(lambda: mx.flash_attention(Q, K, V, out_dtype=torch.bfloat16,
                                                     out=O), flusher=flusher)
    # the key-split entry point, when the (head, 256-query) units leave a
    # partial last wave of SMs
    nbytes = mx.flash_attention_workspace_bytes(c.BH, c.Lq, c.Lk, c.d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None
    ms = event_time(lambda: mx.flash_attention(Q, K, V, out_dtype=torch.bfloat16,
                                               out=O, workspace=ws), flusher=flusher)
    assert mx.mx_last_error() == 0
    flops = 4.0 * c.BH * c.Lq * c.Lk * c.d
    sdpa = torch.nn.functional.scaled_dot_product_attention
    lib_ms = event_time(lambda: sdpa(Q.unsqueeze(0), K.unsqueeze(0), V.unsqueeze(0)),
                        flusher=flusher)
    return {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12,
            "split_kv": nbytes > 0, "unsplit_ms": ms_whole,
            "library_reference_ms": lib_ms,
            "library_reference": "torch scaled_dot_product_attention (context only)"}


def cublaslt_mx_reference(c, qa, qb, out_dt, C, mx):
    """Context only: cuBLASLt's MXFP8 GEMM (torch._scaled_mm with UE8M0
    block scales) on the step's own quantized planes -- the scale plane is
    the tensor-core layout both read -- timed the same way as the step's
    GEMM (mean CUDA-event time, L2 flushed before every launch), and
    whether its C equals ours bit for bit."""
    try:
        af = qa.data.view(torch.float8_e4m3fn).view(c.M, c.K)
        bf = qb.data.view(torch.float8_e4m3fn).view(c.N, c.K)
        sa = qa.scales.view(torch.float8_e8m0fnu)
        sb = qb.scales.view(torch.float8_e8m0fnu)
        f = lambda: torch._scaled_mm(af, bf.t(), scale_a=sa, scale_b=sb,  # noqa
                                     out_dtype=out_dt)
        Ct = f()
        same = bool(torch.equal(Ct, C))
        ms = event_time(f, flusher=L2Flusher(C.device))
    except Exception as e:                     # no block-scaled path in torch
        return {"unavailable": "%s: %s" % (type(e).__name__, str(e)[:120])}
    return {"library": "cuBLASLt MXFP8 via torch._scaled_mm (context only)",
            "ms": ms, "tflops": flops_of(c) / (ms * 1e-3) / 1e12,
            "bit_identical_c": same}


def dequant_bytes(c):
    """Algorithmic bytes of one gemm_dequant: bf16 A read, B's codes and
    scales read, C written."""
    bits = {4: 8, 5: 4, 6: 2}[workloads.formats(c)[1]]
    out_b = 2 if c.out == "bf16" else 4
    return 2.0 * c.M * c.K + c.N * c.K * bits / 8 + c.N * c.K / 32 + out_b * c.M * c.N


def quant_bytes(fmt, rows, K):
    """Algorithmic bytes of one mx_quantize: fp32 in, codes + scales out."""
    code = rows * K / 2 if fmt == 2 else rows * K           # E2M1: 4 bits
    return 4.0 * rows * K + code + rows * K / 32


def run_ours(args, rank, world, local_rank):
    import block_scaled_quantized_mx_gb300 as mx
    mx.build()
    mx.lib()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    c = workloads.case(args.workload)
    if workloads.is_dequant(c):
        raise SystemExit("%s is timed in gemm_only_other_workloads; the step "
                         "workload is an MX or 16-bit case" % c.name)
    hbm, bf16, bf16_sus, peak_src = peaks()
    stream = torch.cuda.current_stream()

    A, B = workloads.sources(c)
    is_mx = workloads.is_mx(c)
    fa, fb = workloads.formats(c) if is_mx else (None, None)
    out_dt = torch.bfloat16 if c.out == "bf16" else torch.float32
    dA, dB = A.to(dev), B.to(dev)
    C = torch.empty((c.M, c.N), dtype=out_dt, device=dev)
    if is_mx:
        qa = mx.empty_mx(fa, c.M, c.K, dev)
        qb = mx.empty_mx(fb, c.N, c.K, dev)
        ws_bytes = mx.mx_gemm_workspace_bytes(ws_format(fa, fb), c.M, c.N, c.K)
    else:
        ws_bytes = mx.gemm_f16_workspace_bytes(c.M, c.N, c.K)
    # scratch for the K-split of the last wave of tiles (allocated here,
    # once); off by default: measured on GB300 it does not beat the unsplit
    # kernel on the default workload
    ws = (torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
          if ws_bytes and args.splitk else None)

    # per-kernel events so every launch's duration is known
    def step(ev=None):
        if is_mx:
            if ev is not None:
                ev[0].record(stream)
            mx.mx_quantize(dA, fa, out=qa)
            if ev is not None:
                ev[1].record(stream)
            mx.mx_quantize(dB, fb, k_strided=True, out=qb)
            if ev is not None:
                ev[2].record(stream)
            mx.mx_gemm(qa, qb, out_dtype=out_dt, out=C, workspace=ws)
            if ev is not None:
                ev[3].record(stream)
        else:
            if ev is not None:
                ev[0].record(stream)
            mx.gemm_f16(dA, dB, out=C, workspace=ws)
            if ev is not None:
                ev[1].record(stream)

    # our kernels per step: 2 quantizes (MX) + the GEMM (the K-split, when
    # active, sums its partials inside the same GEMM launch)
    launches_per_step = 3 if is_mx else 1
    # operands smaller than L2: flush it between timed steps, and take the
    # step time from the kernels' own events (the flush is not timed)
    src_bytes = A.numel() * A.element_size() + B.numel() * B.element_size()
    flusher = L2Flusher(dev) if src_bytes < 2 * L2_BYTES else None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert mx.mx_last_error() == 0

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    nev = 4 if is_mx else 2
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)]
           for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device()
                          if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else local_rank)
    clocks.start()
    barrier()
    t0.record(stream)
    for i in range(args.steps):
        if flusher is not None:
            flusher()
        step(evs[i])
    t1.record(stream)
    barrier()
    clk = clocks.stop()
    assert mx.mx_last_error() == 0
    ms = t0.elapsed_time(t1)
    per_kernel = [[e[j].elapsed_time(e[j + 1]) for e in evs]
                  for j in range(nev - 1)]
    if flusher is not None:
        ms = sum(e[0].elapsed_time(e[nev - 1]) for e in evs)
    ms = max_over_ranks(ms, world, dev)
    ms_step = ms / args.steps
    tflops = job_throughput(flops_of(c), world, ms_step)

    gemm_ms = statistics.mean(per_kernel[-1])
    gemm_tf = flops_of(c) / (gemm_ms * 1e-3) / 1e12
    peak = bf16 * NOMINAL_RATIO[c.kind]
    extra = {"gemm_ms": gemm_ms, "gemm_tflops": gemm_tf,
             "gemm_frac_of_peak": gemm_tf / peak}
    if is_mx:
        qa_ms = statistics.mean(per_kernel[0])
        qb_ms = statistics.mean(per_kernel[1])
        extra["quantize_a_ms"] = qa_ms
        extra["quantize_b_ms"] = qb_ms
        extra["quantize_a_gbs"] = quant_bytes(fa, c.M, c.K) / qa_ms / 1e6
        extra["quantize_b_gbs"] = quant_bytes(fb, c.N, c.K) / qb_ms / 1e6
        extra["quantize_a_frac_hbm"] = extra["quantize_a_gbs"] / hbm
        extra["quantize_b_frac_hbm"] = extra["quantize_b_gbs"] / hbm
        if rank == 0 and fa == fb == 1:
            extra["library_reference"] = cublaslt_mx_reference(c, qa, qb, out_dt, C, mx)

    window = None

    nsm = torch.cuda.get_device_properties(dev).multi_processor_count

    def clock_peak(kind, mhz):
        return nsm * PER_CLOCK[kind] * mhz * 1e6 / 1e12 if mhz else None

    clk_mhz = (clk or {}).get("sm_mhz")
    if is_mx and rank == 0 and not args.no_quant_formats:
        others_q = [(1, "e4m3"), (2, "e2m1"), (3, "e5m2")]
        extra["quantize_formats"] = time_quantize_formats(mx, dA, dB, others_q, c.M, c.K)
        for v in extra["quantize_formats"].values():
            v["a_frac_hbm"] = v["a_gbs"] / hbm
            v["b_frac_hbm"] = v["b_gbs"] / hbm

    # ---- end to end through the C ABI with host buffers
    # Every step copies its fp32 inputs from pinned host memory and its
    # result back, inside the timed region.  Steps are pipelined on three
    # streams (copy in, compute, copy out) with double-buffered device
    # buffers, so step i+1's inputs stream in while step i computes and
    # copies out: the host link, not the GPU, sets the pace.
    e2e = None
    if not args.no_e2e:
        hA = A.pin_memory()
        hB = B.pin_memory()
        hC = [torch.empty((c.M, c.N), dtype=out_dt).pin_memory() for _ in range(2)]
        dAs = [dA, torch.empty_like(dA)]
        dBs = [dB, torch.empty_like(dB)]
        Cs = [C, torch.empty_like(C)]
        s_in, s_cmp, s_out = (torch.cuda.Stream(dev), torch.cuda.Stream(dev),
                              torch.cuda.Stream(dev))
        ev = {k: [torch.cuda.Event(), torch.cuda.Event()]
              for k in ("in", "used", "done", "out")}
        for k in ("used", "out"):
            for e_ in ev[k]:
                e_.record(stream)            # buffers start free

        def e2e_step(i):
            b = i % 2
            s_in.wait_event(ev["used"][b])       # step i-2 has read dA/dB[b]
            with torch.cuda.stream(s_in):
                dAs[b].copy_(hA, non_blocking=True)
                dBs[b].copy_(hB, non_blocking=True)
                ev["in"][b].record(s_in)
            s_cmp.wait_event(ev["in"][b])
            s_cmp.wait_event(ev["out"][b])       # step i-2's C[b] is copied out
            if is_mx:
                mx.mx_quantize(dAs[b], fa, out=qa, stream=s_cmp)
                mx.mx_quantize(dBs[b], fb, k_strided=True, out=qb, stream=s_cmp)
                ev["used"][b].record(s_cmp)
                mx.mx_gemm(qa, qb, out_dtype=out_dt, out=Cs[b], workspace=ws,
                           stream=s_cmp)
            else:
                mx.gemm_f16(dAs[b], dBs[b], out=Cs[b], workspace=ws,
                            stream=s_cmp)
                ev["used"][b].record(s_cmp)
            ev["done"][b].record(s_cmp)
            s_out.wait_event(ev["done"][b])
            with torch.cuda.stream(s_out):
                hC[b].copy_(Cs[b], non_blocking=True)
                ev["out"][b].record(s_out)

        for i in range(max(2, args.warmup // 2)):
            e2e_step(i)
        barrier()
        n_e2e = max(2, args.e2e_steps)
        t_start = time.perf_counter()
        for i in range(n_e2e):
            e2e_step(i)
        torch.cuda.synchronize()
        ems = (time.perf_counter() - t_start) * 1e3 / n_e2e
        barrier()
        assert mx.mx_last_error() == 0
        ems = max_over_ranks(ems, world, dev)
        e2e = {"value": job_throughput(flops_of(c), world, ems),
               "unit": "TFLOP/s", "ms_per_step": ems,
               "h2d_bytes_per_step": int(hA.numel() * hA.element_size() +
                                         hB.numel() * hB.element_size()),
               "d2h_bytes_per_step": int(hC[0].numel() * hC[0].element_size()),
               "timing": "host wall clock around n steps, synchronized",
               "pipelining": "3 streams (copy in / compute / copy out), "
                             "double-buffered device inputs and outputs"}

    others = {}
    if not args.no_others and rank == 0:
        fl = L2Flusher(dev)
        for name in args.others.split(","):
            if not name or name == c.name:
                continue
            oc = workloads.case(name)
            ms_o, tf_o = time_gemm_only(mx, oc, dev, flusher=fl,
                                        splitk=not args.no_splitk_others)
            others[name] = {"gemm_ms": ms_o, "tflops": tf_o,
                            "frac_of_peak": tf_o / (bf16 * NOMINAL_RATIO[oc.kind]),
                            "frac_of_nominal": tf_o / NOMINAL_TFLOPS[oc.kind]}
            if not args.no_graph_others:
                gms, nsets = time_gemm_graph(mx, oc, dev)
                gtf = flops_of(oc) / (gms * 1e-3) / 1e12
                others[name].update({
                    "graph_ms": gms, "graph_tflops": gtf,
                    "graph_frac_of_peak": gtf / (bf16 * NOMINAL_RATIO[oc.kind]),
                    "graph_operand_sets": nsets})
            if INSTRUCTION_RATIO[oc.kind] != NOMINAL_RATIO[oc.kind]:
                others[name]["frac_of_instruction_rate"] = \
                    tf_o / (bf16 * INSTRUCTION_RATIO[oc.kind])
            if workloads.is_dequant(oc):
                gbs = dequant_bytes(oc) / ms_o / 1e6
                others[name].update({"gbs": gbs, "frac_of_hbm": gbs / hbm})
        # the four projections of one transformer layer (QKV, out, up, down):
        # their summed flops over their summed times
        projs = [n for n in ("proj_qkv", "proj_out", "proj_up", "proj_down") if n in others]
        if len(projs) == 4:
            flop = sum(flops_of(workloads.case(n)) for n in projs)
            ms = sum(others[n]["gemm_ms"] for n in projs)
            agg = {"gemms": projs, "gemm_ms": ms, "tflops": flop / (ms * 1e-3) / 1e12}
            agg["frac_of_peak"] = agg["tflops"] / (bf16 * NOMINAL_RATIO["mxfp8"])
            if all("graph_ms" in others[n] for n in projs):
                gms = sum(others[n]["graph_ms"] for n in projs)
                agg.update({"graph_ms": gms, "graph_tflops": flop / (gms * 1e-3) / 1e12})
                agg["graph_frac_of_peak"] = agg["graph_tflops"] / (bf16 * NOMINAL_RATIO["mxfp8"])
            others["proj_layer_aggregate"] = agg
        del fl
    attention = {}
    if not args.no_attention and rank == 0:
        fl = L2Flusher(dev)
        for name in args.attention.split(","):
            if name:
                a = time_attention(mx, workloads.attn_case(name), dev, fl)
                a["frac_of_peak"] = a["tflops"] / bf16
                attention[name] = a
        del fl
    fused = {}
    if not args.no_fused and rank == 0:
        fl = L2Flusher(dev)
        for name in args.fused.split(","):
            if name:
                fused[name] = time_fused(mx, workloads.case(name), dev, fl)
        del fl

    # ---- the SM clock under this load: the same step back to back for
    # about a second with the 2 ms sampler running (the timed region itself
    # lasts only steps x ms_per_step, a few samples)
    if not args.no_clock_window:
        n_win = int(min(5000, max(20, args.clock_window_s * 1e3 / ms_step)))
        cs = ClockSampler(clocks.index)
        w0 = torch.cuda.Event(enable_timing=True)
        w1 = torch.cuda.Event(enable_timing=True)
        cs.start()
        w0.record(stream)
        for _ in range(n_win):
            if flusher is not None:
                flusher()
            step()
        w1.record(stream)
        w1.synchronize()
        cw = cs.stop()
        assert mx.mx_last_error() == 0
        w_ms = w0.elapsed_time(w1) / n_win
        window = {"steps": n_win, "ms_per_step": w_ms, "clocks": cw,
                  "note": "ms_per_step includes the L2 flush" if flusher is not None
                  else "back-to-back steps"}

    roofline = {"bound": "tensor", "kernel": "mx_gemm" if is_mx else "gemm_f16",
                "achieved": gemm_tf, "peak": peak, "unit": "TFLOP/s",
                "frac": gemm_tf / peak,
                "traffic": profiled_traffic(c.name) if is_mx else None,
                "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum "
                                  "per launch, ncu capture summarised in "
                                  "profiles/ (null once the kernel changed)",
                "peak_source": "%s bf16 burst x nominal %s/bf16 ratio %g" %
                (peak_src, c.kind, NOMINAL_RATIO[c.kind]),
                "frac_of_nominal": gemm_tf / NOMINAL_TFLOPS[c.kind],
                "nominal_peak": NOMINAL_TFLOPS[c.kind]}
    if clk_mhz:
        cp = clock_peak(c.kind, clk_mhz)
        roofline["clock_normalised"] = {
            "sm_mhz": clk_mhz, "peak": cp, "frac": gemm_tf / cp,
            "peak_source": "%d SMs x %d flop/clk/SM (measured %s MMA rate) x "
                           "median SM clock sampled in the timed region"
                           % (nsm, PER_CLOCK[c.kind], c.kind)}
    if window and window.get("clocks") and window["clocks"].get("sm_mhz"):
        wm = window["clocks"]["sm_mhz"]
        window["step_tflops"] = flops_of(c) / (window["ms_per_step"] * 1e-3) / 1e12
        window["clock_normalised_peak"] = clock_peak(c.kind, wm)
    line = {
        "metric": metric_name(c),
        "step": step_description(c),
        "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE_NAME.get(c.kind, c.kind),
        "data": "synthetic (seeded)",
        "config": {"workload": c.name, "M": c.M, "N": c.N, "K": c.K,
                   "out": c.out, "dist": c.dist_a,
                   "l2": ("inputs larger than L2 (sources %d MB + %d MB)" %
                          (src_bytes // 2 ** 21, src_bytes // 2 ** 21))
                         if flusher is None else
                         "L2 flushed between steps (258 MB write, not timed)",
                   "parallelism": "replicas%d" % world},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roofline,
        "breakdown": extra,
        "gemm_only_other_workloads": others,
        "fused_epilogue": fused,
        "attention": attention,
        "e2e": e2e,
        "clocks": clk,
        "clock_window": window,
    }
    return line


# ------------------------------------------------------------------ provenance

def source_hash() -> str:
    """sha256 (first 16 hex digits) of every CUDA source and header the
    library is built from: identifies the code where no git metadata is."""
    import glob
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "block_scaled_quantized_mx_gb300", "csrc", "*"))
                   + glob.glob(os.path.join(ROOT, "include", "*.h")))
    for f in files:
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode() + fh.read())
    return h.hexdigest()[:16]


def provenance_rows(line):
    """One record per measured operation of a bench line: the code
    (source hash, and the git commit where there is one), the workload's
    shapes and seeds, times, throughput, fractions of peak, SM clock and the
    environment."""
    try:
        commit = subprocess.run(["git", "-C", ROOT, "rev-parse", "HEAD"],
                                capture_output=True, text=True,
                                timeout=5).stdout.strip() or None
    except Exception:
        commit = None
    env = {"sources": source_hash(), "commit": commit,
           "utc": time.strftime("%Y-%m-%dT%H:%M:%SZ", time.gmtime()),
           "torch": torch.__version__, "cuda": torch.version.cuda,
           "device": torch.cuda.get_device_name(0) if torch.cuda.is_available() else None,
           "nproc": os.cpu_count(),
           "sm_mhz": (line.get("clocks") or {}).get("sm_mhz"),
           "clock_reasons": (line.get("clocks") or {}).get("reasons")}

    def case_fields(name):
        try:
            c = workloads.case(name)
            return {"M": c.M, "N": c.N, "K": c.K, "seed_a": c.seed_a,
                    "seed_b": c.seed_b, "kind": c.kind, "out": c.out}
        except KeyError:
            c = workloads.attn_case(name)
            return {"BH": c.BH, "Lq": c.Lq, "Lk": c.Lk, "d": c.d,
                    "seed": c.seed, "kind": "attention", "out": "bf16"}

    cfg = line["config"]
    rows = [dict(env, op="step", workload=cfg["workload"],
                 **case_fields(cfg["workload"]), ms=line["ms_per_step"],
                 tflops=line["value"],
                 frac_of_peak=(line.get("roofline") or {}).get("frac"),
                 breakdown=line.get("breakdown"))]
    for name, r in (line.get("gemm_only_other_workloads") or {}).items():
        if name == "proj_layer_aggregate":
            rows.append(dict(env, op="gemm_aggregate", workload=name, gemms=r["gemms"],
                             ms=r["gemm_ms"], tflops=r["tflops"],
                             frac_of_peak=r["frac_of_peak"]))
            continue
        rows.append(dict(env, op="gemm", workload=name, **case_fields(name),
                         ms=r["gemm_ms"], tflops=r["tflops"],
                         frac_of_peak=r["frac_of_peak"],
                         frac_of_instruction_rate=r.get("frac_of_instruction_rate"),
                         gbs=r.get("gbs")))
    for name, r in (line.get("fused_epilogue") or {}).items():
        rows.append(dict(env, op="fused_epilogue", workload=name,
                         **case_fields(name), ms=r["fused_ms"],
                         tflops=r.get("fused_tflops"), plain_ms=r["gemm_ms"],
                         decomposed_ms=r["decomposed_ms"],
                         fused_quantize_ms=r["fused_quantize_ms"]))
    for name, r in (line.get("attention") or {}).items():
        rows.append(dict(env, op="attention", workload=name,
                         **case_fields(name), ms=r["ms"], tflops=r["tflops"],
                         frac_of_peak=r.get("frac_of_peak"),
                         unsplit_ms=r.get("unsplit_ms")))
    if line.get("e2e"):
        rows.append(dict(env, op="e2e", workload=cfg["workload"],
                         **case_fields(cfg["workload"]),
                         ms=line["e2e"]["ms_per_step"],
                         tflops=line["e2e"]["value"]))
    return rows


# ------------------------------------------------------------------ oracle

def oracle_sample(c, budget_s: float):
    """Rows of C from the fp32 sources with the CPU oracle, until the time
    budget is spent: quantize the whole B once, then quantize and multiply
    A rows in chunks.  Returns (flops done, seconds, rows, threads)."""
    import oracle
    A, B = workloads.sources(c)
    t0 = time.perf_counter()
    if c.kind in ("f16", "bf16"):
        bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)  # noqa
        Ab, Bb = bits(A), bits(B)
        code = oracle.F16 if c.kind == "f16" else oracle.BF16
        rows = 0
        chunk = 8
        while rows < c.M:
            r = list(range(rows, min(c.M, rows + chunk)))
            oracle.gemm_f16(Ab, Bb, code, rows=r)
            rows += len(r)
            if time.perf_counter() - t0 > budget_s:
                break
    else:
        fa, fb = workloads.formats(c)
        cb, sb = oracle.quantize(B.numpy(), fb, k_axis=0)
        An = A.numpy()
        rows = 0
        chunk = 16
        while rows < c.M:
            ca, sa = oracle.quantize(An[rows:rows + chunk], fa, k_axis=1)
            oracle.gemm_mx(ca, sa, cb, sb, fa, fmt_b=fb)
            rows += ca.shape[0]
            if time.perf_counter() - t0 > budget_s:
                break
    dt = time.perf_counter() - t0
    return 2.0 * rows * c.N * c.K, dt, rows, oracle.num_threads()


def oracle_extras(c, budget_s: float):
    """Two more figures of the CPU oracle, each on a bounded sample: its
    quantizer in GB/s of algorithmic bytes on all host cores (rows of the
    workload's A source), and its MX GEMM in GFLOP/s on one core at
    1024 x 1024 x 1024 (rows of C from seeded random codes)."""
    import oracle
    if not workloads.is_mx(c):
        return None
    fa, fb = workloads.formats(c)
    per_elem = 4.0 + (0.5 if fa == oracle.E2M1 else 1.0) + 1.0 / 32
    A, _ = workloads.sources(c)
    An = A.numpy()
    rows, t0 = 0, time.perf_counter()
    while rows < c.M and time.perf_counter() - t0 < budget_s / 2:
        oracle.quantize(An[rows:rows + 256], fa, k_axis=1)
        rows += min(256, c.M - rows)
    q_dt = time.perf_counter() - t0
    q_rows = rows
    n = 1024
    ca, sa = workloads.random_codes((n, n), fa, seed=n + 1)
    cb, sb = workloads.random_codes((n, n), fb, seed=n + 2)
    oracle.set_num_threads(1)
    try:
        rows, t0 = 0, time.perf_counter()
        while rows < n and time.perf_counter() - t0 < budget_s / 2:
            oracle.gemm_mx(ca[rows:rows + 8], sa[rows:rows + 8], cb, sb, fa,
                           fmt_b=fb)
            rows += 8
        g_dt = time.perf_counter() - t0
    finally:
        oracle.set_num_threads(0)
    return {
        "quantize_gbs": q_rows * c.K * per_elem / q_dt / 1e9,
        "quantize_cores": oracle.num_threads(),
        "quantize_sample": "%d rows of the %d x %d A source, %.1f s"
                           % (q_rows, c.M, c.K, q_dt),
        "gemm_1core_gflops": 2.0 * rows * n * n / g_dt / 1e9,
        "gemm_1core_sample": "%d rows of C of a %d^3 product, %.1f s"
                             % (rows, n, g_dt),
    }


def run_reference(args):
    c = workloads.case(args.workload)
    budget = max(1.0, args.ref_budget / max(1, args.steps))
    vals = []
    secs = []
    last = None
    for _ in range(args.warmup if args.warmup < 1 else 1):
        oracle_sample(c, min(budget, 2.0))
    for _ in range(args.steps):
        fl, dt, rows, thr = oracle_sample(c, budget)
        vals.append(fl / dt / 1e12)
        secs.append(dt)
        last = (rows, thr, dt)
    v = statistics.median(vals)
    rows, thr, dt = last
    sample = ("rows of C computed from the fp32 sources: quantize all of B, "
              "then %d rows of A quantized and multiplied (%.1f s per step)"
              % (rows, dt)) if workloads.is_mx(c) else \
        ("%d rows of C (%.1f s per step)" % (rows, dt))
    return {
        "impl": "reference",
        "metric": metric_name(c), "step": step_description(c),
        "value": v, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        # each step is a bounded sample of the workload (its rows of C)
        "ms_per_step": statistics.mean(secs) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": c.name, "M": c.M, "N": c.N, "K": c.K,
                   "out": c.out},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": thr,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mxfp8_8192")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline key")
    ap.add_argument("--ref-budget", type=float, default=60.0,
                    help="total seconds of oracle work for --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--others", default="mxfp8_4096,mxfp4_8192,mxfp4_4096,"
                    "mxfp8_e5m2_8192,w4a8_8192,w4a16_8192,w2a16_8192,"
                    "w4a16_decode,w4a16_decode_m1,"
                    "bf16_4096,f16_4096,bf16_2048,bf16_1024,proj_qkv,proj_out,"
                    "proj_up,proj_down,mx256",
                    help="workloads whose GEMM alone is also timed (L2 "
                         "flushed before each launch)")
    ap.add_argument("--no-others", action="store_true")
    ap.add_argument("--fused", default="proj_up,mxfp8_4096",
                    help="MX workloads on which the fused bias + GELU epilogue "
                         "is timed against the decomposed path")
    ap.add_argument("--no-fused", action="store_true")
    ap.add_argument("--attention", default="attn_sam_d64,attn_sam_d128,attn_long_d128",
                    help="attention workloads timed with flash_attention")
    ap.add_argument("--no-attention", action="store_true")
    ap.add_argument("--jsonl", default=None,
                    help="append one provenance record per measured operation "
                         "(code hash, shapes, seeds, times, clocks, environment)")
    ap.add_argument("--splitk", action="store_true",
                    help="use the K-split GEMM entry points (with a workspace) "
                         "in the step")
    ap.add_argument("--no-splitk-others", action="store_true",
                    help="time the other workloads without the K-split "
                         "workspace the library asks for")
    ap.add_argument("--no-graph-others", action="store_true",
                    help="skip the CUDA-graph timing of the other workloads")
    ap.add_argument("--no-clock-window", action="store_true")
    ap.add_argument("--clock-window-s", type=float, default=1.0,
                    help="seconds of back-to-back steps sampled for the SM clock")
    ap.add_argument("--no-quant-formats", action="store_true",
                    help="skip the E2M1 / E5M2 quantizer timings")
    return ap.parse_args(argv)


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        # the CPU oracle runs once, on rank 0; other ranks exit without work
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(
            "nccl", device_id=torch.device("cuda", local_rank))
    line = run_ours(args, rank, world, local_rank)
    if rank == 0 and not args.no_cpu_baseline:
        c = workloads.case(args.workload)
        fl, dt, rows, thr = oracle_sample(c, args.cpu_budget)
        line["cpu_baseline"] = {
            "value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": thr,
            "kind": "oracle",
            "sample": "%d rows of C from the fp32 sources (all of B "
                      "quantized), %.1f s" % (rows, dt)}
        try:
            extra = oracle_extras(c, 4.0)
        except Exception as e:   # a context figure: report, never lose the line
            extra = {"error": "%s: %s" % (type(e).__name__, e)}
        if extra is not None:
            line.setdefault("breakdown", {})["oracle_cpu"] = extra
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
        if args.jsonl:
            with open(args.jsonl, "a") as f:
                for row in provenance_rows(line):
                    f.write(json.dumps(row) + "\n")


if __name__ == "__main__":
    main()
