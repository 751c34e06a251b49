#!/usr/bin/env python3
"""Benchmark of the ternary (PQ2) x INT8 small-batch projection on GB300.

Workload (one GPU): attn_qkv, K=5120 inputs, N=10240 outputs, M = 1, 2, 3, 4
tokens; ternary 2-bit codes iid uniform over {0,1,2} with fp16 group-128
scales uniform in [0.005, 0.05]; bf16 activations N(0,1) with a seeded 1% of
the channels scaled by 20; INT8 per-128-group activation quantisation, fp32
accumulation, bf16 output.

A step is one complete projection call (quantise + GEMV) for each of M = 1..4,
every call on a different weight matrix; the distinct matrices (more than 4x
the L2 size in total) rotate, so weights always stream from HBM.  Steps are
replayed from CUDA graphs and timed with CUDA events on the launching stream.

  value       microseconds per complete call (device time) for the whole job:
              the slowest rank's step time over all ranks' calls (N replicas)
  e2e         the same through host buffers, all inside the timed region:
              per step one copy of the step's x (M = 1..4, one pinned host
              buffer) to the device, the calls, one copy of the step's y
              back to pinned host memory
  roofline    pq2_mmv alone: packed weight bytes K*N*34/128 per launch over
              its CUDA-event time per launch, against the measured HBM peak
  cpu_baseline the CPU oracle on the host cores, on a bounded sample
  per_m       attn_qkv per M: pq2_mmv in independent calls and in a
              dependent chain, and the complete call, with HBM fractions
  sweep       the GEMV on every configured shape (4096x14336 at M = 1; the
              layer shapes 5120x10240, 5120x6144, 5120x17408, 17408x5120 at
              M = 1..8, with the batch-invariance check): microseconds, GB/s
              and fraction, independent, dependent and complete calls
  prefill     pq2_mm, pq2_mm_f8 and pq2_linear on ffn_up K=5120 N=17408 at
              M = 16 .. 4096: microseconds, TOPS and the fraction of the
              measured dense tensor peak of the kernel's own operand type
  prep        the fused preparation (pq2_norm_hadamard_quantize) at K=5120,
              M = 1..4, 16, 64, 256 and 4096, with the stand-alone quantisation beside it
  gated       the gated gate/up projection (pq2_mmv_gated, silu(gate) * up
              in the GEMV's epilogue) on ffn gate/up (K=5120, 2 x 17408
              rows) at M = 1..4: microseconds, HBM GB/s and fraction, the
              plain GEMV on the same rows and the complete gated call

`--impl reference` times the CPU oracle on the same workload instead (the
reference arm of this comparison).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("µs/call and HBM GB/s (frac of peak) for ternary×INT8 matmul at "
          "M=1–8; prefill TOPS")
K_DIM, N_DIM, MS = 5120, 10240, (1, 2, 3, 4)
PREFILL_K, PREFILL_N, PREFILL_MS = 5120, 17408, (16, 128, 512, 2048, 4096)
PREFILL_GROUPED_MS = (128, 512, 4096)  # the grouped calls the pages time, and the largest
GATED_K, GATED_I = 5120, 17408
# The GEMV sweep: the layer shapes at every M in 1..8 (with the batch
# invariance check) and the 4096 x 14336 shape at M = 1, as (K, N, Ms, name).
SWEEP = ((4096, 14336, (1,), "4096x14336"),
         (5120, 10240, tuple(range(1, 9)), "attn_qkv"),
         (5120, 6144, tuple(range(1, 9)), "5120x6144"),
         (5120, 17408, tuple(range(1, 9)), "ffn_up"),
         (17408, 5120, tuple(range(1, 9)), "ffn_down"))
MMV_PROFILE = os.path.join(ROOT, "profiles", "pq2_mmv_attn_qkv_full.md")
MMV_SOURCES = ("ternary_weight_int8_gb300/csrc/pq2_mmv.cu",
               "ternary_weight_int8_gb300/csrc/pq2_device.cuh")
WORKLOAD = ("attn_qkv K=5120 N=10240, M=1,2,3,4 per step (quantise + GEMV each); ternary "
            "codes U{0,1,2}, fp16 group-128 scales U[0.005,0.05]; bf16 x N(0,1) with 1% "
            "channels x20; fp32 accumulate, bf16 out")


def max_over_ranks(value: float, device=None) -> float:
    """The largest value over the ranks of the process group (an all-reduce
    MAX), or the value itself without one: the job's time is its slowest
    rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_call(ms: float, calls_per_rank: int, world: int) -> float:
    """Whole-job microseconds per call: `world` replicas each made
    `calls_per_rank` calls in `ms` (the slowest rank's time)."""
    return ms * 1e3 / (calls_per_rank * world)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def recorded_traffic():
    """DRAM bytes (read + write) per pq2_mmv launch on attn_qkv from the
    committed ncu summary, or None when the kernel's sources have changed
    since that capture (the summary records their hash) or no record exists."""
    import hashlib
    try:
        with open(MMV_PROFILE) as f:
            line = next(ln for ln in f if ln.startswith("traffic-record:"))
        fields = dict(kv.split("=", 1) for kv in line.split()[1:])
        h = hashlib.sha256()
        for rel in MMV_SOURCES:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] != fields["sources_sha256_16"]:
            return None
        return int(fields["dram_bytes_per_launch"])
    except (OSError, StopIteration, KeyError, ValueError):
        return None


def measured_tensor_peak():
    """Dense 16-bit tensor peak in TFLOP/s (fp16 and bf16 run at one rate)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- reference
def oracle_linear_threads(O, x_bits, codes, scales, threads):
    """The oracle's complete call (widen, quantise, group dots, scale) with
    the output rows split into `threads` contiguous slices, one host thread
    each.  Every slice runs the unchanged oracle on its rows (quantising x
    itself), so the result equals the single-threaded call bit for bit; the
    oracle is a C library and its calls release the interpreter lock, so the
    slices run on separate cores."""
    import numpy as np
    from concurrent.futures import ThreadPoolExecutor
    N = codes.shape[0]
    if threads <= 1:
        return O.linear(x_bits, "bf16", codes, scales)
    cuts = [N * i // threads for i in range(threads + 1)]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda i: O.linear(x_bits, "bf16", codes[cuts[i]:cuts[i + 1]],
                                               scales[cuts[i]:cuts[i + 1]]),
                            range(threads)))
    return np.concatenate(parts, axis=1)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def run_reference(args):
    """The CPU oracle on the same workload: each step is one complete call
    for M = 1..4 on the full attn_qkv shape, the output rows split over every
    host core (oracle_linear_threads)."""
    from oracle import oracle as O
    from ternary_weight_int8_gb300 import synth

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cores = host_cores()
    raw = synth.raw_weights(N_DIM, K_DIM, seed=1234)
    codes, scales = O.prepare(raw.numpy(), K_DIM)
    xs = {M: synth.bits_u16(synth.activations(M, K_DIM, seed=77 + M, outlier_frac=0.01))
          for M in MS}
    O.load()

    def step():
        for M in MS:
            oracle_linear_threads(O, xs[M], codes, scales, cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    us = dt / (args.steps * len(MS)) * 1e6
    sample = (f"{args.steps} steps of complete M=1..4 calls on the full {K_DIM}x{N_DIM} shape, "
              f"output rows split over {cores} host threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 3), "unit": "us/call",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "i8", "data": "synthetic",
        "config": {"workload": WORKLOAD,
                   "runs": f"CPU oracle (plain C, IEEE fp32/fp64), {cores} host threads"},
        "cpu_baseline": {"value": round(us, 3), "unit": "us/call", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(us, 3), "unit": "us/call", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------- ours
def host_mapped(t) -> bool:
    """True when the pinned host tensor `t` is addressable by the device at
    its own address (unified addressing): then kernels can read and write it
    directly, over NVLink-C2C on a Grace-Blackwell node.  Asked of the CUDA
    runtime (cudaPointerGetAttributes), never by touching it from the GPU."""
    import ctypes

    class Attr(ctypes.Structure):
        _fields_ = [("type", ctypes.c_int), ("device", ctypes.c_int),
                    ("devicePointer", ctypes.c_void_p), ("hostPointer", ctypes.c_void_p),
                    ("reserved", ctypes.c_long * 16)]
    for name in ("libcudart.so", "libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            rt = None
    if rt is None:
        return False
    a = Attr()
    rc = rt.cudaPointerGetAttributes(ctypes.byref(a), ctypes.c_void_p(t.data_ptr()))
    return rc == 0 and a.type == 1 and a.devicePointer == t.data_ptr()


def cpu_baseline_sample(budget_s=8.0):
    """The oracle as it stands on the host cores: complete calls for M = 1..4
    on the full attn_qkv shape, repeated for about budget_s seconds on every
    core (output rows split over one thread per core), then for about
    budget_s / 2 seconds on one core."""
    from oracle import oracle as O
    from ternary_weight_int8_gb300 import synth
    raw = synth.raw_weights(N_DIM, K_DIM, seed=4321)
    codes, scales = O.prepare(raw.numpy(), K_DIM)
    xs = {M: synth.bits_u16(synth.activations(M, K_DIM, seed=5 + M, outlier_frac=0.01))
          for M in MS}
    O.load()
    cores = host_cores()

    def run(threads, budget):
        calls, t0 = 0, time.perf_counter()
        while True:
            for M in MS:
                oracle_linear_threads(O, xs[M], codes, scales, threads)
                calls += 1
            if time.perf_counter() - t0 > budget:
                break
        return calls, time.perf_counter() - t0

    calls, dt = run(cores, budget_s)
    calls1, dt1 = run(1, budget_s / 2)
    return {"value": round(dt / calls * 1e6, 3), "unit": "us/call", "cores": cores,
            "kind": "oracle",
            "sample": f"{calls} complete attn_qkv calls (M=1..4 cycled) in {dt:.1f} s, output "
                      f"rows split over {cores} host threads",
            "single_core_value": round(dt1 / calls1 * 1e6, 3),
            "single_core_sample": f"{calls1} calls in {dt1:.1f} s on one thread"}


def prefill_leg(args, dev, stream, timed, capture):
    """Prefill: ffn_up (K=5120, N=17408) at M = 16 .. 4096 through pq2_mm
    (kernel only, on pre-quantised fp16 activations) and pq2_linear
    (quantise + GEMM); 8 rotated weight matrices (190 MB, above the L2
    size).  TOPS = 2*M*N*K / time; the fraction is of the measured dense
    16-bit tensor peak, the rate of the tensor-core kind the kernel uses."""
    import torch
    from ternary_weight_int8_gb300 import pq2, synth
    lib = pq2.lib()
    K, N, nm = PREFILL_K, PREFILL_N, 8
    mats = []
    for i in range(nm):
        raw = synth.raw_weights(N, K, seed=5000 + i, device=dev)
        mats.append(pq2.pq2_prepare(raw, K))
        del raw
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sp = stream.cuda_stream
    peak, kind = measured_tensor_peak()
    out = {"workload": f"ffn_up K={K} N={N}, bf16 x N(0,1), bf16 out, {nm} rotated matrices",
           "peak_tflops": peak, "peak_source": kind, "by_m": {}}
    for M in PREFILL_MS:
        x = synth.activations(M, K, seed=900 + M, device=dev)
        q, sx, qs = pq2.pq2_quantize_act(x, pq2.PQ2_Q_F16)
        q8, _, _ = pq2.pq2_quantize_act(x, pq2.PQ2_Q_F8)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(pq2.linear_workspace_bytes(M, K), dtype=torch.uint8, device=dev)

        def mm_f8_calls():
            for c, sc in mats:
                st = lib.pq2_mm_f8(q8.data_ptr(), sx.data_ptr(), qs.data_ptr(), c.data_ptr(),
                                   sc.data_ptr(), y.data_ptr(), pq2.PQ2_BF16, M, N, K,
                                   status.data_ptr(), sp)
                if st:
                    raise RuntimeError(f"pq2_mm_f8 failed ({st})")

        def mm_calls():
            for c, sc in mats:
                st = lib.pq2_mm(q.data_ptr(), sx.data_ptr(), qs.data_ptr(), c.data_ptr(),
                                sc.data_ptr(), y.data_ptr(), pq2.PQ2_BF16, M, N, K,
                                status.data_ptr(), sp)
                if st:
                    raise RuntimeError(f"pq2_mm failed ({st})")

        def linear_calls():
            for c, sc in mats:
                st = lib.pq2_linear(x.data_ptr(), pq2.PQ2_BF16, K, M, N, K, c.data_ptr(),
                                    sc.data_ptr(), y.data_ptr(), pq2.PQ2_BF16, ws.data_ptr(),
                                    ws.numel(), status.data_ptr(), sp)
                if st:
                    raise RuntimeError(f"pq2_linear failed ({st})")

        reps = max(3, min(50, 20000 // M))
        k_ms = timed([capture(mm_calls)], reps, 3) / (reps * nm)
        k8_ms = timed([capture(mm_f8_calls)], reps, 3) / (reps * nm)
        c_ms = timed([capture(linear_calls)], reps, 3) / (reps * nm)
        tops = 2.0 * M * N * K / (k_ms * 1e-3) / 1e12
        out["by_m"][str(M)] = {"mm_us": round(k_ms * 1e3, 2), "mm_tflops": round(tops, 1),
                               "frac": round(tops / peak, 3),
                               "mm_f8_us": round(k8_ms * 1e3, 2),
                               # pq2_mm_f8 runs 2 e4m3 MMAs per K step (the two
                               # planes of q): 4MNK executed operations at the
                               # e4m3 rate, twice the 16-bit one
                               "f8_pipe_frac": round(4.0 * M * N * K / (k8_ms * 1e-3) / 1e12
                                                     / (2 * peak), 3),
                               "f8_e4m3_frac": round(2.0 * M * N * K / (k8_ms * 1e-3) / 1e12
                                                     / (2 * peak), 3),
                               "complete_us": round(c_ms * 1e3, 2),
                               "complete_tflops": round(2.0 * M * N * K / (c_ms * 1e-3) / 1e12, 1)}
        del x, q, q8, sx, qs, y, ws
    # Activation groups of 128 / 64 / 32 (the pages time the complete call at
    # M = 128 and 512): the 8-bit grouped GEMM alone and pq2_linear_grouped.
    out["grouped"] = {}
    for M in PREFILL_GROUPED_MS:
        x = synth.activations(M, K, seed=950 + M, device=dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        by_a = {}
        for A in (128, 64, 32):
            q8, sx, qs = pq2.pq2_quantize_act_grouped(x, A, pq2.PQ2_Q_F8)
            ws = torch.empty(pq2.linear_grouped_workspace_bytes(M, K, A), dtype=torch.uint8,
                             device=dev)

            def mm_calls():
                for c, sc in mats:
                    st = lib.pq2_mm_f8_grouped(q8.data_ptr(), sx.data_ptr(), qs.data_ptr(),
                                               c.data_ptr(), sc.data_ptr(), y.data_ptr(),
                                               pq2.PQ2_BF16, M, N, K, A, status.data_ptr(), sp)
                    if st:
                        raise RuntimeError(f"pq2_mm_f8_grouped failed ({st})")

            def linear_calls():
                for c, sc in mats:
                    st = lib.pq2_linear_grouped(x.data_ptr(), pq2.PQ2_BF16, K, M, N, K,
                                                c.data_ptr(), sc.data_ptr(), A, y.data_ptr(),
                                                pq2.PQ2_BF16, ws.data_ptr(), ws.numel(),
                                                status.data_ptr(), sp)
                    if st:
                        raise RuntimeError(f"pq2_linear_grouped failed ({st})")

            reps = max(3, min(50, 20000 // M))
            k_ms = timed([capture(mm_calls)], reps, 3) / (reps * nm)
            c_ms = timed([capture(linear_calls)], reps, 3) / (reps * nm)
            by_a[str(A)] = {"mm_f8_us": round(k_ms * 1e3, 2),
                            "mm_f8_tops": round(2.0 * M * N * K / (k_ms * 1e-3) / 1e12, 1),
                            "complete_us": round(c_ms * 1e3, 2)}
            del q8, sx, qs, ws
        for A in ("64", "32"):
            by_a[A]["complete_cost_vs_128"] = round(
                by_a[A]["complete_us"] / by_a["128"]["complete_us"] - 1.0, 3)
        out["grouped"][str(M)] = by_a
        del x, y
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    del mats
    torch.cuda.empty_cache()
    return out


def gated_leg(args, dev, stream, timed, capture):
    """The gated gate/up projection (silu(gate) * up in the GEMV's epilogue)
    on the ffn gate/up shape: K=5120, N = 2 x 17408 weight rows,
    max(16, ceil(4 L2 / B)) rotated matrices (above 4x the L2 size), M = 1..4.
    Per call: pq2_mmv_gated
    alone (back-to-back independent calls on pre-quantised activations),
    the complete pq2_linear_gated call, and pq2_mmv on the same N rows
    without the gated epilogue; GB/s of packed weight bytes K*N*34/128."""
    import torch
    from ternary_weight_int8_gb300 import pq2, synth
    lib = pq2.lib()
    K, N = GATED_K, 2 * GATED_I
    nm = rotation_count(torch.cuda.get_device_properties(dev).L2_cache_size, N * K * 34 // 128)
    mats = []
    for i in range(nm):
        raw = synth.raw_weights(N, K, seed=7000 + i, device=dev)
        mats.append(pq2.pq2_prepare(raw, K))
        del raw
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sp = stream.cuda_stream
    hbm, hbm_kind = measured_peaks()
    nbytes = N * K * 34 // 128
    out = {"workload": f"ffn gate/up K={K} N=2x{GATED_I} (gate rows, then up rows), "
                       f"bf16 x N(0,1) with 1% outliers, bf16 out, {nm} rotated matrices",
           "bytes_per_call": nbytes, "peak_gbs": hbm, "peak_source": hbm_kind, "by_m": {}}
    for M in MS:
        x = synth.activations(M, K, seed=300 + M, device=dev, outlier_frac=0.01)
        q, sx, qs = pq2.pq2_quantize_act(x, pq2.PQ2_Q_PLANES)
        o = torch.empty((M, N // 2), dtype=torch.bfloat16, device=dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(pq2.linear_workspace_bytes(M, K), dtype=torch.uint8, device=dev)

        def gated_calls():
            for c, sc in mats:
                st = lib.pq2_mmv_gated(q.data_ptr(), sx.data_ptr(), qs.data_ptr(), c.data_ptr(),
                                       sc.data_ptr(), o.data_ptr(), pq2.PQ2_BF16, M, N, K,
                                       pq2.PQ2_MMV_INDEPENDENT, status.data_ptr(), sp)
                if st:
                    raise RuntimeError(f"pq2_mmv_gated failed ({st})")

        def plain_calls():
            for c, sc in mats:
                st = lib.pq2_mmv_ex(q.data_ptr(), sx.data_ptr(), qs.data_ptr(), c.data_ptr(),
                                    sc.data_ptr(), y.data_ptr(), pq2.PQ2_BF16, M, N, K,
                                    lib.pq2_mmv_decoder(M), pq2.PQ2_MMV_INDEPENDENT,
                                    status.data_ptr(), sp)
                if st:
                    raise RuntimeError(f"pq2_mmv failed ({st})")

        def complete_calls():
            for c, sc in mats:
                st = lib.pq2_linear_gated(x.data_ptr(), pq2.PQ2_BF16, K, M, N, K, c.data_ptr(),
                                          sc.data_ptr(), o.data_ptr(), pq2.PQ2_BF16,
                                          ws.data_ptr(), ws.numel(), status.data_ptr(), sp)
                if st:
                    raise RuntimeError(f"pq2_linear_gated failed ({st})")

        reps = 50
        g_ms = timed([capture(gated_calls)], reps, 3) / (reps * nm)
        p_ms = timed([capture(plain_calls)], reps, 3) / (reps * nm)
        c_ms = timed([capture(complete_calls)], reps, 3) / (reps * nm)
        gbs = nbytes / (g_ms * 1e-3) / 1e9
        out["by_m"][str(M)] = {"gated_us": round(g_ms * 1e3, 3), "gated_gbs": round(gbs, 1),
                               "gated_frac": round(gbs / hbm, 3),
                               "mmv_same_rows_us": round(p_ms * 1e3, 3),
                               "complete_us": round(c_ms * 1e3, 3)}
        del x, q, sx, qs, o, y, ws
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    del mats
    torch.cuda.empty_cache()
    return out


def grouped_leg(args, dev, stream, timed, capture, mats, wbytes):
    """Activation groups of 64 and 32 on the step's attn_qkv shape and its
    rotated weight matrices (inputs larger than L2): pq2_mmv_grouped alone
    (back-to-back independent calls on pre-quantised activations) and
    pq2_quantize_act_grouped, M = 1..4, 5 and 8 (M > 4: two passes over the
    weights); GB/s of packed weight bytes."""
    import torch
    from ternary_weight_int8_gb300 import pq2, synth
    lib = pq2.lib()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sp = stream.cuda_stream
    hbm, hbm_kind = measured_peaks()
    out = {"workload": f"attn_qkv K={K_DIM} N={N_DIM}, bf16 x N(0,1) with 1% outliers, "
                       f"bf16 out, {len(mats)} rotated matrices",
           "bytes_per_call": wbytes, "peak_gbs": hbm, "peak_source": hbm_kind, "by_a": {}}
    for A in (64, 32):
        by_m = {}
        for M in tuple(MS) + (5, 8):  # M > 4: two passes over the weights
            x = synth.activations(M, K_DIM, seed=500 + M + A, device=dev, outlier_frac=0.01)
            q, sx, qs = pq2.pq2_quantize_act_grouped(x, A, pq2.PQ2_Q_PLANES)
            y = torch.empty((M, N_DIM), dtype=torch.bfloat16, device=dev)

            def mmv_calls():
                for c, sc in mats:
                    st = lib.pq2_mmv_grouped(q.data_ptr(), sx.data_ptr(), qs.data_ptr(),
                                             c.data_ptr(), sc.data_ptr(), y.data_ptr(),
                                             pq2.PQ2_BF16, M, N_DIM, K_DIM, A,
                                             pq2.PQ2_MMV_INDEPENDENT, status.data_ptr(), sp)
                    if st:
                        raise RuntimeError(f"pq2_mmv_grouped failed ({st})")

            def quant_calls():
                for _ in mats:
                    st = lib.pq2_quantize_act_grouped(x.data_ptr(), pq2.PQ2_BF16, K_DIM, M,
                                                      K_DIM, A, q.data_ptr(), pq2.PQ2_Q_PLANES,
                                                      sx.data_ptr(), qs.data_ptr(), sp)
                    if st:
                        raise RuntimeError(f"pq2_quantize_act_grouped failed ({st})")

            reps = 30
            k_ms = timed([capture(mmv_calls)], reps, 3) / (reps * len(mats))
            q_ms = timed([capture(quant_calls)], reps, 3) / (reps * len(mats))
            gbs = wbytes / (k_ms * 1e-3) / 1e9
            by_m[str(M)] = {"mmv_us": round(k_ms * 1e3, 3), "mmv_gbs": round(gbs, 1),
                            "mmv_frac": round(gbs / hbm, 3), "quant_us": round(q_ms * 1e3, 3)}
            del x, q, sx, qs, y
        out["by_a"][str(A)] = by_m
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    return out


def ptq_leg(args, dev, stream, timed, capture):
    """PTQ1_0 weights (28 bytes per 128 weights) on the attn_qkv shape, 48
    rotated matrices (550 MB, above L2), activation groups of 32 (the pages'
    PTQ1_0 path) and 128, M = 1..4: pq2_ptq_mmv alone (back-to-back
    independent calls) and the complete call pq2_ptq_linear (grouped
    quantisation, then the GEMV streaming its weights while the quantisation
    runs)."""
    import torch
    from ternary_weight_int8_gb300 import pq2, synth
    lib = pq2.lib()
    K, N, nm = K_DIM, N_DIM, 48
    mats = []
    for i in range(nm):
        raw = synth.ptq_raw_weights(N, K, seed=9000 + i, device=dev)
        mats.append(pq2.pq2_ptq_prepare(raw, K))
        del raw
    sp = stream.cuda_stream
    hbm, hbm_kind = measured_peaks()
    nbytes = N * K * 28 // 128
    out = {"workload": f"attn_qkv K={K} N={N} PTQ1_0 (bytes uniform, fp16 d in [0.005, 0.05]), "
                       f"bf16 x N(0,1) with 1% outliers, bf16 out, {nm} rotated matrices",
           "bytes_per_call": nbytes, "peak_gbs": hbm, "peak_source": hbm_kind, "by_a": {}}
    for A in (32, 128):
        by_m = {}
        for M in MS:
            x = synth.activations(M, K, seed=700 + M + A, device=dev, outlier_frac=0.01)
            q, sx, qs = pq2.pq2_quantize_act_grouped(x, A, pq2.PQ2_Q_ROWS)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

            wsb = torch.empty(lib.pq2_ptq_linear_workspace_bytes(M, K, A), dtype=torch.uint8,
                              device=dev)

            def mmv_calls():
                for wq, ws in mats:
                    st = lib.pq2_ptq_mmv(q.data_ptr(), sx.data_ptr(), qs.data_ptr(), wq.data_ptr(),
                                         ws.data_ptr(), y.data_ptr(), pq2.PQ2_BF16, M, N, K, A,
                                         pq2.PQ2_MMV_INDEPENDENT, sp)
                    if st:
                        raise RuntimeError(f"pq2_ptq_mmv failed ({st})")

            def complete_calls():
                for wq, ws in mats:
                    st = lib.pq2_ptq_linear(x.data_ptr(), pq2.PQ2_BF16, K, M, N, K, wq.data_ptr(),
                                            ws.data_ptr(), A, y.data_ptr(), pq2.PQ2_BF16,
                                            wsb.data_ptr(), wsb.numel(), sp)
                    if st:
                        raise RuntimeError(f"pq2_ptq_linear failed ({st})")

            reps = 30
            k_ms = timed([capture(mmv_calls)], reps, 3) / (reps * nm)
            c_ms = timed([capture(complete_calls)], reps, 3) / (reps * nm)
            gbs = nbytes / (k_ms * 1e-3) / 1e9
            by_m[str(M)] = {"mmv_us": round(k_ms * 1e3, 3), "mmv_gbs": round(gbs, 1),
                            "mmv_frac": round(gbs / hbm, 3), "complete_us": round(c_ms * 1e3, 3)}
            del x, q, sx, qs, y, wsb
        out["by_a"][str(A)] = by_m
    del mats
    torch.cuda.empty_cache()
    return out


def prep_leg(args, dev, stream, timed, capture):
    """The fused preparation (pq2_norm_hadamard_quantize: RMSNorm with a
    residual, signs, 1024-point Walsh-Hadamard, group-128 INT8 in the plane
    layout) at K=5120 for M = 1..4, 16, 64, 256 and 4096, against the stand-alone
    quantisation of the same rows; HBM bytes per call: x and residual in
    (2 x 2MK), w and signs (3K), q out (MK), s_x and sum(q) (8MK/128)."""
    import torch
    from ternary_weight_int8_gb300 import pq2, synth
    lib = pq2.lib()
    K = K_DIM
    hbm, hbm_kind = measured_peaks()
    g = torch.Generator().manual_seed(17)
    w = (torch.randn(K, generator=g) * 0.1).to(torch.bfloat16).to(dev)
    sign = (torch.randint(0, 2, (K,), generator=g) * 2 - 1).to(torch.int8).to(dev)
    sp = stream.cuda_stream
    out = {"workload": f"K={K}, bf16 x and residual, eps 1e-6, q in plane order",
           "peak_gbs": hbm, "peak_source": hbm_kind, "by_m": {}}
    for M in tuple(MS) + (16, 64, 256, 4096):
        n_in = 8 if M < 64 else 1  # rotate inputs of small calls
        xs = [synth.activations(M, K, seed=40 + i, device=dev).to(torch.bfloat16)
              for i in range(n_in)]
        rs = [synth.activations(M, K, seed=80 + i, device=dev).to(torch.bfloat16)
              for i in range(n_in)]
        q = torch.empty((M, K), dtype=torch.int8, device=dev)
        sx = torch.empty((M, K // 128), dtype=torch.float32, device=dev)
        qs = torch.empty((M, K // 128), dtype=torch.int32, device=dev)
        calls = 8

        def fused():
            for i in range(calls):
                st = lib.pq2_norm_hadamard_quantize(
                    xs[i % n_in].data_ptr(), rs[i % n_in].data_ptr(), None, w.data_ptr(),
                    sign.data_ptr(), 1e-6, M, K, None, q.data_ptr(), pq2.PQ2_Q_PLANES,
                    sx.data_ptr(), qs.data_ptr(), sp)
                if st:
                    raise RuntimeError(f"pq2_norm_hadamard_quantize failed ({st})")

        def quant_only():
            for i in range(calls):
                st = lib.pq2_quantize_act(xs[i % n_in].data_ptr(), pq2.PQ2_BF16, K, M, K,
                                          q.data_ptr(), pq2.PQ2_Q_PLANES, sx.data_ptr(),
                                          qs.data_ptr(), sp)
                if st:
                    raise RuntimeError(f"pq2_quantize_act failed ({st})")

        reps = 20 if M >= 64 else 100
        f_ms = timed([capture(fused)], reps, 3) / (reps * calls)
        q_ms = timed([capture(quant_only)], reps, 3) / (reps * calls)
        nbytes = 4 * M * K + 3 * K + M * K + 8 * M * K // 128
        out["by_m"][str(M)] = {"fused_us": round(f_ms * 1e3, 3),
                               "gbs": round(nbytes / (f_ms * 1e-3) / 1e9, 1),
                               "frac": round(nbytes / (f_ms * 1e-3) / 1e9 / hbm, 3),
                               "quantize_only_us": round(q_ms * 1e3, 3)}
        del xs, rs, q, sx, qs
    torch.cuda.empty_cache()
    return out


def rotation_count(l2_bytes: int, matrix_bytes: int) -> int:
    """Distinct weight matrices to rotate so that a call never finds its
    weights in L2: max(16, ceil(4 L2 / B))."""
    return max(16, math.ceil(4 * l2_bytes / matrix_bytes))


def compact(by_m: dict, key: str, frac_key: str | None = None) -> str:
    """'M:us/frac' pairs in one short string (the summary keys)."""
    out = []
    for M, d in by_m.items():
        s = f"{M}:{d[key]:.2f}"
        if frac_key:
            s += f"/{d[frac_key]:.2f}"
        out.append(s)
    return " ".join(out)


def sweep_leg(args, dev, stream, timed, capture):
    """The GEMV on every configured shape (SWEEP), each rotating
    rotation_count() distinct weight matrices, per M:
      mmv_us   pq2_mmv alone, back-to-back PQ2_MMV_INDEPENDENT calls (each
               call may read its inputs and compute while the previous call
               finishes)
      dep_us   pq2_mmv in a dependent chain: PQ2_MMV_OVERLAP_WEIGHTS calls,
               each waiting for the previous call to complete before it
               reads its activations (the position of a GEMV in a decode
               step; the weights still stream early)
      complete_us  pq2_linear (quantise + GEMV), chained
    with GB/s of packed weight bytes K*N*34/128 and the fraction of the
    measured HBM peak.  Batch invariance: for each shape, y (fp32) of the
    first M rows of an 8-row activation matrix, for every M, is compared bit
    for bit with rows 0..M-1 of the M = 8 call."""
    import torch
    from ternary_weight_int8_gb300 import pq2, synth
    lib = pq2.lib()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sp = stream.cuda_stream
    hbm, hbm_kind = measured_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = {"peak_gbs": hbm, "peak_source": hbm_kind, "shapes": {}}
    for K, N, Ms, name in SWEEP:
        wbytes = N * K * 34 // 128
        n_mats = rotation_count(l2, wbytes)
        mats = []
        for i in range(n_mats):
            raw = synth.raw_weights(N, K, seed=20000 + 100 * K + i, device=dev)
            mats.append(pq2.pq2_prepare(raw, K))
            del raw
        x8 = synth.activations(max(Ms), K, seed=31 + K + N, device=dev)
        shape = {"K": K, "N": N, "bytes_per_call": wbytes, "matrices": n_mats, "by_m": {}}
        ref = None
        invariant = True
        for M in sorted(Ms, reverse=True):
            x = x8[:M]
            q, sx, qs = pq2.pq2_quantize_act(x, pq2.PQ2_Q_PLANES)
            qt, sxt, corr = pq2.pq2_quantize_act(x, pq2.PQ2_Q_MMV16)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = torch.empty(pq2.linear_workspace_bytes(M, K), dtype=torch.uint8, device=dev)
            # batch invariance on the first matrix, fp32 output
            c0, s0 = mats[0]
            y32 = pq2.pq2_mmv(q, sx, qs, c0, s0, out_dtype=torch.float32)
            torch.cuda.synchronize()
            if ref is None:
                ref = y32
            elif not torch.equal(y32.view(torch.int32), ref[:M].view(torch.int32)):
                invariant = False

            def calls(flag):
                def run():
                    for c, sc in mats:
                        st = lib.pq2_mmv_ex(q.data_ptr(), sx.data_ptr(), qs.data_ptr(),
                                            c.data_ptr(), sc.data_ptr(), y.data_ptr(),
                                            pq2.PQ2_BF16, M, N, K, lib.pq2_mmv_decoder(M), flag,
                                            status.data_ptr(), sp)
                        if st:
                            raise RuntimeError(f"pq2_mmv_ex failed ({st})")
                return run

            def tc_calls(flag):
                def run():
                    for c, sc in mats:
                        st = lib.pq2_mmv_tc(qt.data_ptr(), sxt.data_ptr(), corr.data_ptr(),
                                            c.data_ptr(), sc.data_ptr(), y.data_ptr(),
                                            pq2.PQ2_BF16, M, N, K, flag, status.data_ptr(), sp)
                        if st:
                            raise RuntimeError(f"pq2_mmv_tc failed ({st})")
                return run

            def complete_calls():
                for c, sc in mats:
                    st = lib.pq2_linear(x.data_ptr(), pq2.PQ2_BF16, K, M, N, K, c.data_ptr(),
                                        sc.data_ptr(), y.data_ptr(), pq2.PQ2_BF16, ws.data_ptr(),
                                        ws.numel(), status.data_ptr(), sp)
                    if st:
                        raise RuntimeError(f"pq2_linear failed ({st})")

            reps = 10
            k_ms = timed([capture(calls(pq2.PQ2_MMV_INDEPENDENT))], reps, 3) / (reps * n_mats)
            d_ms = timed([capture(calls(pq2.PQ2_MMV_OVERLAP_WEIGHTS))], reps, 3) / (reps * n_mats)
            c_ms = timed([capture(complete_calls)], reps, 3) / (reps * n_mats)
            t_ms = timed([capture(tc_calls(pq2.PQ2_MMV_INDEPENDENT))], reps, 3) / (reps * n_mats)
            td_ms = timed([capture(tc_calls(pq2.PQ2_MMV_OVERLAP_WEIGHTS))], reps, 3) / (
                reps * n_mats)
            # the tensor-core GEMV's y must equal the dp4a GEMV's (same bits)
            yt = pq2.pq2_mmv_tc(qt, sxt, corr, c0, s0, out_dtype=torch.float32)
            torch.cuda.synchronize()
            if not torch.equal(yt.view(torch.int32), y32.view(torch.int32)):
                raise RuntimeError(f"pq2_mmv_tc differs from pq2_mmv ({name}, M={M})")
            frac = lambda ms: round(wbytes / (ms * 1e-3) / 1e9 / hbm, 3)  # noqa: E731
            shape["by_m"][str(M)] = {"mmv_us": round(k_ms * 1e3, 3),
                                     "mmv_gbs": round(wbytes / (k_ms * 1e-3) / 1e9, 1),
                                     "mmv_frac": frac(k_ms),
                                     "dep_us": round(d_ms * 1e3, 3), "dep_frac": frac(d_ms),
                                     "tc_us": round(t_ms * 1e3, 3), "tc_frac": frac(t_ms),
                                     "tc_dep_us": round(td_ms * 1e3, 3),
                                     "tc_dep_frac": frac(td_ms),
                                     "complete_us": round(c_ms * 1e3, 3)}
            del q, sx, qs, y, ws, y32, qt, sxt, corr, yt
        shape["by_m"] = dict(sorted(shape["by_m"].items(), key=lambda kv: int(kv[0])))
        if len(Ms) > 1:
            shape["batch_invariant"] = invariant
        out["shapes"][name] = shape
        del mats, x8, ref
        torch.cuda.empty_cache()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist
    from ternary_weight_int8_gb300 import pq2, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = pq2.lib()

    # -------------------------------------------------- inputs (resident)
    wbytes = N_DIM * K_DIM * 34 // 128
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_mats = max(16, math.ceil(4 * l2 / wbytes))
    n_mats = (n_mats + len(MS) - 1) // len(MS) * len(MS)
    mats = []
    for i in range(n_mats):
        raw = synth.raw_weights(N_DIM, K_DIM, seed=1000 * rank + i, device=dev)
        mats.append(pq2.pq2_prepare(raw, K_DIM))
        del raw
    xs = {M: synth.activations(M, K_DIM, seed=77 + M, device=dev, outlier_frac=0.01)
          for M in MS}
    qbuf = {M: pq2.pq2_quantize_act(xs[M], pq2.PQ2_Q_PLANES) for M in MS}
    # The step's outputs (M = 1..4) live in one contiguous buffer, [sum M][N].
    y_all = torch.empty((sum(MS), N_DIM), dtype=torch.bfloat16, device=dev)
    row0 = {M: sum(MS[:i]) for i, M in enumerate(MS)}
    ys = {M: y_all[row0[M]:row0[M] + M] for M in MS}
    # End-to-end leg: the step's inputs in one pinned host buffer [sum M][K]
    # (one host->device copy per step) and its outputs read back with one
    # device->host copy per step.
    hx_all = torch.cat([xs[M].cpu() for M in MS]).pin_memory()
    hy_all = torch.empty((sum(MS), N_DIM), dtype=torch.bfloat16).pin_memory()
    dx_all = torch.empty((sum(MS), K_DIM), dtype=torch.bfloat16, device=dev)
    dx = {M: dx_all[row0[M]:row0[M] + M] for M in MS}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream

    wss = {M: torch.empty(pq2.linear_workspace_bytes(M, K_DIM), dtype=torch.uint8, device=dev)
           for M in MS}

    def complete(M, mat, x, s, y=None):
        """One complete call through the public entry point: quantise + GEMV."""
        c, sc = mats[mat]
        y = ys[M] if y is None else y
        st = lib.pq2_linear(x.data_ptr(), pq2.PQ2_BF16, K_DIM, M, N_DIM, K_DIM, c.data_ptr(),
                            sc.data_ptr(), y.data_ptr(), pq2.PQ2_BF16, wss[M].data_ptr(),
                            wss[M].numel(), status.data_ptr(), s)
        if st:
            raise RuntimeError(f"pq2_linear failed ({st})")

    def mmv_only(M, mat, s):
        """The GEMV alone on pre-quantised activations: back-to-back
        independent projections (nothing in flight writes their inputs), so
        each call may stream its inputs while the previous call finishes."""
        q, sx, qs = qbuf[M]
        c, sc = mats[mat]
        st = lib.pq2_mmv_ex(q.data_ptr(), sx.data_ptr(), qs.data_ptr(), c.data_ptr(),
                            sc.data_ptr(), ys[M].data_ptr(), pq2.PQ2_BF16, M, N_DIM, K_DIM,
                            lib.pq2_mmv_decoder(M), pq2.PQ2_MMV_INDEPENDENT,
                            status.data_ptr(), s)
        if st:
            raise RuntimeError(f"pq2_mmv failed ({st})")

    n_graphs = n_mats // len(MS)
    # A graph holds `chunk` consecutive steps (a divisor of the step count,
    # at most one full rotation over the matrices), as a decode step captured
    # in one graph would; programmatic dependent launch overlaps neighbouring
    # kernels inside a graph but not across graph launches.
    chunk = max(d for d in range(1, n_graphs + 1) if args.steps % d == 0)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()  # warm the launch path (sets kernel attributes) outside capture
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=stream):
                fn()
        return g

    def step_calls(j):
        """Step j: the 4 complete calls (M = 1..4) on matrices 4j'..4j'+3."""
        j %= n_graphs
        for i, M in enumerate(MS):
            complete(M, 4 * j + i, xs[M], sp)

    def e2e_staged_step(j):
        j %= n_graphs
        dx_all.copy_(hx_all, non_blocking=True)
        for i, M in enumerate(MS):
            complete(M, 4 * j + i, dx[M], sp)
        hy_all.copy_(y_all, non_blocking=True)

    # Mapped end to end: the calls read x from the pinned host buffer and
    # write y into the pinned host buffer themselves (unified addressing over
    # NVLink-C2C), so the step has no staging copies between its kernels.
    mapped = host_mapped(hx_all) and host_mapped(hy_all)
    hx = {M: hx_all[row0[M]:row0[M] + M] for M in MS}
    hy = {M: hy_all[row0[M]:row0[M] + M] for M in MS}

    def e2e_mapped_step(j):
        j %= n_graphs
        for i, M in enumerate(MS):
            complete(M, 4 * j + i, hx[M], sp, y=hy[M])

    e2e_step = e2e_mapped_step if mapped else e2e_staged_step

    n_chunks = n_graphs // math.gcd(n_graphs, chunk)
    step_graphs = [capture(lambda j=j: [step_calls(j * chunk + t) for t in range(chunk)])
                   for j in range(n_chunks)]
    e2e_graphs = [capture(lambda j=j: [e2e_step(j * chunk + t) for t in range(chunk)])
                  for j in range(n_chunks)]
    staged_graphs = ([capture(lambda j=j: [e2e_staged_step(j * chunk + t) for t in range(chunk)])
                      for j in range(n_chunks)] if mapped else e2e_graphs)

    def timed(graphs, replays, warmup):
        with torch.cuda.stream(stream):
            for i in range(warmup):
                graphs[i % len(graphs)].replay()
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(replays):
                graphs[i % len(graphs)].replay()
            e1.record(stream)
            torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1), dev)

    warm_replays = -(-args.warmup // chunk)
    # soak (untimed) while the clock sampler runs, then the timed region; the
    # sampler stays open over every leg below, so its summary covers them all
    clocks = ClockSampler(local).__enter__()
    t_end = time.time() + 1.5
    while time.time() < t_end:
        timed(step_graphs, 20, 0)
    total_ms = timed(step_graphs, args.steps // chunk, warm_replays)
    e2e_ms = timed(e2e_graphs, args.steps // chunk, warm_replays)
    staged_ms = timed(staged_graphs, args.steps // chunk, warm_replays)
    ms_step = total_ms / args.steps
    us_call = job_us_per_call(ms_step, len(MS), world)
    e2e_us = job_us_per_call(e2e_ms / args.steps, len(MS), world)
    staged_us = job_us_per_call(staged_ms / args.steps, len(MS), world)
    if mapped:
        # the mapped outputs equal the device path's, bit for bit
        with torch.cuda.stream(stream):
            e2e_mapped_step(0)
            step_calls(0)
        torch.cuda.synchronize()
        if not torch.equal(hy_all.view(torch.int16), y_all.cpu().view(torch.int16)):
            raise RuntimeError("mapped end-to-end outputs differ from the device path")

    # ------------------------------------------- per-M and kernel-only legs
    per_m = {}
    peak, peak_kind = measured_peaks()

    def mmv_dep(M, mat, s):
        """The GEMV in a dependent chain: each call waits for the kernel
        before it to complete before reading its activations."""
        q, sx, qs = qbuf[M]
        c, sc = mats[mat]
        st = lib.pq2_mmv_ex(q.data_ptr(), sx.data_ptr(), qs.data_ptr(), c.data_ptr(),
                            sc.data_ptr(), ys[M].data_ptr(), pq2.PQ2_BF16, M, N_DIM, K_DIM,
                            lib.pq2_mmv_decoder(M), pq2.PQ2_MMV_OVERLAP_WEIGHTS,
                            status.data_ptr(), s)
        if st:
            raise RuntimeError(f"pq2_mmv failed ({st})")

    for M in MS:
        # one graph = one call on each of the n_mats matrices in turn
        g_c = [capture(lambda: [complete(M, i, xs[M], sp) for i in range(n_mats)])]
        g_k = [capture(lambda: [mmv_only(M, i, sp) for i in range(n_mats)])]
        g_d = [capture(lambda: [mmv_dep(M, i, sp) for i in range(n_mats)])]
        reps = max(20, args.steps // 10)
        c_ms = timed(g_c, reps, 3) / (reps * n_mats)
        k_ms = timed(g_k, reps, 3) / (reps * n_mats)
        d_ms = timed(g_d, reps, 3) / (reps * n_mats)
        per_m[str(M)] = {
            "complete_us": round(c_ms * 1e3, 3),
            "complete_frac": round(wbytes / (c_ms * 1e-3) / 1e9 / peak, 3),
            "mmv_us": round(k_ms * 1e3, 3),
            "mmv_gbs": round(wbytes / (k_ms * 1e-3) / 1e9, 1),
            "mmv_frac": round(wbytes / (k_ms * 1e-3) / 1e9 / peak, 3),
            "dep_us": round(d_ms * 1e3, 3),
            "dep_frac": round(wbytes / (d_ms * 1e-3) / 1e9 / peak, 3),
        }
    sweep = sweep_leg(args, dev, stream, timed, capture) if not args.no_sweep else None
    prefill = prefill_leg(args, dev, stream, timed, capture) if not args.no_prefill else None
    gated = gated_leg(args, dev, stream, timed, capture) if not args.no_gated else None
    prep = prep_leg(args, dev, stream, timed, capture) if not args.no_prep else None
    grouped = (grouped_leg(args, dev, stream, timed, capture, mats, wbytes)
               if not args.no_grouped else None)
    ptq = ptq_leg(args, dev, stream, timed, capture) if not args.no_ptq else None
    clocks.__exit__(None, None, None)
    # dominant kernel: pq2_mmv over the step's M mix, kernel-only
    mean_k_us = statistics.mean(per_m[str(M)]["mmv_us"] for M in MS)
    mean_d_us = statistics.mean(per_m[str(M)]["dep_us"] for M in MS)
    achieved = wbytes / (mean_k_us * 1e-6) / 1e9
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 3),
                "traffic": recorded_traffic(),
                "kernel": "pq2_mmv", "peak_source": peak_kind,
                "bytes_per_launch": wbytes,
                "timing": "independent calls (PQ2_MMV_INDEPENDENT), mean over M=1..4",
                "dep_frac": round(wbytes / (mean_d_us * 1e-6) / 1e9 / peak, 3),
                "dep_timing": "dependent chain (each call waits for the previous one before "
                              "reading its activations), mean over M=1..4",
                "attn_qkv_indep_us_frac": compact(per_m, "mmv_us", "mmv_frac"),
                "attn_qkv_dep_us_frac": compact(per_m, "dep_us", "dep_frac"),
                "attn_qkv_complete_us": compact(per_m, "complete_us")}
    if sweep:
        for name, sh in sweep["shapes"].items():
            roofline[f"{name}_indep_us_frac"] = compact(sh["by_m"], "mmv_us", "mmv_frac")
            roofline[f"{name}_dep_us_frac"] = compact(sh["by_m"], "dep_us", "dep_frac")
            roofline[f"{name}_tc_indep_us_frac"] = compact(sh["by_m"], "tc_us", "tc_frac")
            roofline[f"{name}_complete_us"] = compact(sh["by_m"], "complete_us")
            if "batch_invariant" in sh:
                roofline[f"{name}_batch_invariant"] = sh["batch_invariant"]
    if prefill:
        for M, d in prefill["by_m"].items():
            for k in ("mm_us", "frac", "mm_f8_us", "f8_pipe_frac", "f8_e4m3_frac",
                      "complete_us"):
                prefill[f"m{M}_{k}"] = d[k]
        # activation groups of 64 / 32: "A:f8 GEMM us/complete us/cost" per M
        for M, by_a in prefill.get("grouped", {}).items():
            prefill[f"grouped_m{M}"] = " ".join(
                f"{A}:{v['mm_f8_us']}/{v['complete_us']}"
                + (f"/{v['complete_cost_vs_128']:+.3f}" if "complete_cost_vs_128" in v else "")
                for A, v in by_a.items())

    result = {
        "metric": METRIC, "value": round(us_call, 3), "unit": "us/call", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "i8",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {n_mats} distinct weight matrices "
                         f"({n_mats * wbytes / 1e6:.0f} MB) rotated",
                   "timing": f"CUDA graphs of {chunk} steps ({chunk * len(MS)} calls) "
                             "replayed, CUDA events on the launching stream"},
        "e2e": {"value": round(e2e_us, 3), "unit": "us/call",
                "h2d_bytes_per_step": sum(M * K_DIM * 2 for M in MS),
                "d2h_bytes_per_step": sum(M * N_DIM * 2 for M in MS),
                "transfer": ("x read and y written by the calls in mapped pinned host memory "
                             "(unified addressing, NVLink-C2C)" if mapped else
                             "one pinned host-to-device copy of x and one device-to-host copy "
                             "of y per step"),
                "staged_value": round(staged_us, 3),
                "staged_transfer": "one pinned host-to-device copy of x and one "
                                   "device-to-host copy of y per step"},
        "gpu_launches": 2 * len(MS) * args.steps,
        "roofline": roofline,
        "per_m": per_m,
        "sweep": sweep,
        "prefill": prefill,
        "gated": gated,
        "prep": prep,
        "grouped": grouped,
        "ptq": ptq,
        "clocks": clocks.summary(),
    }
    if rank == 0 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline_sample()
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_profile_case(args):
    """A short fixed sequence for an ncu capture: the attn_qkv GEMV
    (pq2_mmv, or pq2_mmv_tc for "mmvtc", INDEPENDENT calls over 8 rotated
    matrices), the fused preparation ("prep", K=5120 with a residual), or the
    ffn_up prefill
    GEMM (pq2_mm, pq2_mm_f8 for "mm8", pq2_mm_f8_grouped with
    --profile-act-group for "mm8g"), at --profile-m columns; 3 warm-up calls
    then 3 calls."""
    import torch
    from ternary_weight_int8_gb300 import pq2, synth
    dev = torch.device("cuda", 0)
    M = args.profile_m
    if args.profile_case == "ptq":
        K, N, nm, A = K_DIM, N_DIM, 8, args.profile_act_group
        mats = [pq2.pq2_ptq_prepare(synth.ptq_raw_weights(N, K, seed=9000 + i, device=dev), K)
                for i in range(nm)]
        x = synth.activations(M, K, seed=11, device=dev, outlier_frac=0.01)
        q, sx, qs = pq2.pq2_quantize_act_grouped(x, A, pq2.PQ2_Q_ROWS)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        for i in range(6):
            wq, ws = mats[i % nm]
            pq2.pq2_ptq_mmv(q, sx, qs, wq, ws, A, y=y, flags=pq2.PQ2_MMV_INDEPENDENT)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": "ptq", "M": M, "N": N, "K": K, "act_group": A,
                          "launches": 6, "ok": True}))
        return 0
    if args.profile_case == "prep":
        K = K_DIM
        g = torch.Generator().manual_seed(17)
        w = (torch.randn(K, generator=g) * 0.1).to(torch.bfloat16).to(dev)
        sign = (torch.randint(0, 2, (K,), generator=g) * 2 - 1).to(torch.int8).to(dev)
        xs = [synth.activations(M, K, seed=40 + i, device=dev).to(torch.bfloat16) for i in range(6)]
        rs = [synth.activations(M, K, seed=80 + i, device=dev).to(torch.bfloat16) for i in range(6)]
        for i in range(6):
            pq2.pq2_norm_hadamard_quantize(xs[i], w, sign, 1e-6, residual=rs[i])
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": "prep", "M": M, "K": K, "launches": 6, "ok": True}))
        return 0
    if args.profile_case in ("mmv", "mmvtc"):
        K, N, nm = K_DIM, N_DIM, 8
        layout = pq2.PQ2_Q_PLANES if args.profile_case == "mmv" else pq2.PQ2_Q_MMV16
    else:
        K, N, nm = PREFILL_K, PREFILL_N, 2
        layout = pq2.PQ2_Q_F8 if args.profile_case in ("mm8", "mm8g") else pq2.PQ2_Q_F16
    mats = [pq2.pq2_prepare(synth.raw_weights(N, K, seed=7000 + i, device=dev), K)
            for i in range(nm)]
    x = synth.activations(M, K, seed=11, device=dev, outlier_frac=0.01)
    A = args.profile_act_group if args.profile_case == "mm8g" else 128
    q, sx, qs = pq2.pq2_quantize_act_grouped(x, A, layout)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    for i in range(6):
        c, sc = mats[i % nm]
        if args.profile_case == "mmv":
            pq2.pq2_mmv(q, sx, qs, c, sc, y=y, flags=pq2.PQ2_MMV_INDEPENDENT)
        elif args.profile_case == "mmvtc":
            pq2.pq2_mmv_tc(q, sx, qs, c, sc, y=y, flags=pq2.PQ2_MMV_INDEPENDENT)
        elif args.profile_case == "mm8":
            pq2.pq2_mm_f8(q, sx, qs, c, sc, y=y)
        elif args.profile_case == "mm8g":
            pq2.pq2_mm_f8_grouped(q, sx, qs, c, sc, A, y=y)
        else:
            pq2.pq2_mm(q, sx, qs, c, sc, y=y)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": args.profile_case, "M": M, "N": N, "K": K,
                      "act_group": A, "launches": 6, "ok": True}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill (pq2_mm) leg")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the GEMV sweep over the configured shapes and M = 1..8")
    ap.add_argument("--no-gated", action="store_true",
                    help="skip the gated gate/up (pq2_mmv_gated) leg")
    ap.add_argument("--no-prep", action="store_true",
                    help="skip the fused preparation (pq2_norm_hadamard_quantize) leg")
    ap.add_argument("--no-grouped", action="store_true",
                    help="skip the activation-group 64/32 (pq2_mmv_grouped) leg")
    ap.add_argument("--no-ptq", action="store_true",
                    help="skip the PTQ1_0 weight-format (pq2_ptq_mmv) leg")
    ap.add_argument("--profile-case", choices=["mmv", "mmvtc", "mm", "mm8", "mm8g", "ptq",
                                               "prep"],
                    default=None,
                    help="run a short fixed call sequence for an ncu capture and exit")
    ap.add_argument("--profile-m", type=int, default=1, help="columns for --profile-case")
    ap.add_argument("--profile-act-group", type=int, default=32,
                    help="activation group for --profile-case ptq and mm8g")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.profile_case:
        return run_profile_case(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
