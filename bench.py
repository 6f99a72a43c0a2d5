#!/usr/bin/env python3
"""Benchmark of the GB300 dense projection Y = X·Wᵀ (+ bias).

One step = one call of the whole hot path (proj_run: weight stream, multiply-
accumulate, split-K reduction, bias and bf16 epilogue) over one batch of
synthetic inputs.  The default workload is the decode projection
X [16,8192] · W [8192,8192]ᵀ + bias → bf16 Y, the M=16, K=8192 shape the
metric is quoted on.

Measurement (methodology of "How I made Muse's GPU projections 1.32× faster in
the Open Kernel Challenge", section "How I checked whether an idea was actually
faster": CUDA-graph replay, cold L2, fresh weights):
  * inputs are resident in HBM; W rotates over enough copies that the copies
    together exceed twice the L2, so every step streams W from HBM; each copy is
    packed once into the handle's tile-contiguous layout before timing (the
    preparation step of section "Preparation is not secretly computing the
    answer"; ``--no-packed`` runs on W as stored);
  * the K timed steps are replayed from CUDA graphs, timed with CUDA events on
    the launching stream, bracketed by a barrier and device synchronisation,
    max over ranks;
  * e2e repeats the K steps through proj_run_host (X copied host→device and Y
    device→host every step, pinned buffers; W stays resident);
  * ``repeats``: the spread (median, p10, p90 of per-call µs) over 7 shorter
    timed regions of the same kind; ``cold_call``: single calls, each after
    writing twice the L2, timed alone;
  * ``library_baseline``: the same projection through cuBLAS (torch.addmm /
    torch.mm), informational only;
  * the fp64 oracle is timed on the host cores as the CPU baseline, and the
    output of the timed steps is checked against it on the sampled columns;
  * nvidia-smi clocks are sampled while the GPU is under load.

Multi-GPU: independent replicas (one per rank, no collective on the data path);
``value`` is the aggregate over ranks ("scaling": "weak").

``--impl reference`` times the fp64 CPU oracle as the reference arm instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "projection µs & weight HBM GB/s (M=16,K=8192) / TFLOP/s at M≥512 vs roofline"
DEFAULT_WORKLOAD = "decode_bias"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300 datasheet figures (nominal, not measured): HBM3e bandwidth and dense
# bf16 tensor throughput.  Reported beside the measured-peak fractions.
DATASHEET = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}
PROFILE_DIR = os.path.join(ROOT, "profiles")
CSRC_DIR = os.path.join(ROOT, "dense_linear_projection_gb300", "csrc")


# ---------------------------------------------------------------- pure helpers
def roofline_time_s(bytes_moved: float, flops: float, bw_bytes_per_s: float,
                    flops_per_s: float) -> float:
    """Lower bound on time: the slower of moving the bytes and doing the FLOPs
    (section "A rough way to ask how much room was left": t ≥ max(F/P, B/Q))."""
    return max(bytes_moved / bw_bytes_per_s, flops / flops_per_s)


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


# Files that decide what the kernel reads and writes: its device code, the
# shared work decomposition and the planner (host launch code does not).
TRAFFIC_SOURCES = ("proj_kernel.cuh", "proj_internal.h", "planner.cpp")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES:
        with open(os.path.join(CSRC_DIR, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def profile_traffic(workload: str):
    """Per-launch DRAM bytes from the committed ncu summary of this workload,
    or None if there is none or the kernel sources changed since it was taken."""
    path = os.path.join(PROFILE_DIR, f"proj_tc_kernel_{workload}.md")
    try:
        text = open(path, encoding="utf-8").read()
    except OSError:
        return None, None
    fields = {}
    for line in text.splitlines():
        line = line.strip().strip("`")
        if ":" in line and line.split(":", 1)[0] in ("traffic_bytes_per_launch",
                                                    "kernel_source_sha256"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("kernel_source_sha256") != kernel_source_hash():
        return None, os.path.relpath(path, ROOT)
    try:
        return int(fields["traffic_bytes_per_launch"]), os.path.relpath(path, ROOT)
    except (KeyError, ValueError):
        return None, os.path.relpath(path, ROOT)


def hold_stream(stream, seconds: float = 50e-6) -> None:
    """Queue a short spin kernel on ``stream``: while it runs, the host queues
    the start event and the timed graph behind it, so the timed region holds
    the device time of the steps alone, not the host's launch latency (the
    blocking-kernel technique of GPU benchmark harnesses)."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(seconds * 2.0e9))


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_over_ranks(value: float, op: str, device=None) -> float:
    """max/sum of a host scalar over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, seconds_per_rank: float, device=None) -> dict:
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    t_max = reduce_over_ranks(seconds_per_rank, "max", device)
    units = reduce_over_ranks(units_per_rank, "sum", device)
    return {"seconds": t_max, "units": units, "per_second": units / t_max if t_max > 0 else 0.0}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling (200 ms) of SM clocks and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.out_path = None

    def start(self):
        import tempfile
        fd, self.out_path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.out_path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.out_path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.out_path)
        return summarize_clocks(rows)


def summarize_clocks(rows) -> dict:
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    sm, mx, reasons, power = [], [], set(), []
    for r in rows:
        try:
            sm.append(float(r[1]))
            mx.append(float(r[2]))
            power.append(float(r[3]))
        except ValueError:
            continue
        for i, nm in enumerate(names):
            if r[5 + i].lower().startswith("active"):
                reasons.add(nm)
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(mx) if mx else None,
            "power_w_max": max(power) if power else None,
            "samples": len(sm), "reasons": sorted(reasons)}


def visible_gpu_id(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# ---------------------------------------------------------------- CPU oracle
def _oracle_project(w, X, W, bias):
    """The oracle's product for workload ``w``: bf16 weights, or the exact
    fp32-weight product for router weights."""
    import oracle
    if w.w_dtype == "f32":
        return oracle.project_f32w(X, W, w.w_layout, bias)
    return oracle.project(X, W, w.w_layout, bias)


def cpu_oracle_timing(w, inp, target_s: float, y_gpu=None, act: str = "none", residual=None) -> dict:
    """Time the fp64 oracle on the host cores on a bounded sample of the
    workload: all M token rows against the first n_cols output columns (or the
    whole workload, repeated, if that is quick).  Returns weight GB/s.  With
    ``y_gpu`` (the output the timed steps left, as float64), the sampled
    columns of it are also checked against the oracle's result."""
    import numpy as np
    import oracle
    threads = oracle.max_threads()
    X, W, b = inp["X"], inp["W"], inp["bias"]

    def cols_slice(nc):
        if w.w_layout == 0:
            return np.ascontiguousarray(W[:nc]), None if b is None else b[:nc]
        return np.ascontiguousarray(W[:, :nc]), None if b is None else b[:nc]

    probe = min(w.N, 64)
    Wp, bp = cols_slice(probe)
    t0 = time.perf_counter()
    _oracle_project(w, X[: min(w.M, 256)], Wp, bp)
    dt = max(time.perf_counter() - t0, 1e-6)
    per_col = dt / probe * (w.M / min(w.M, 256))
    n_cols = int(max(1, min(w.N, target_s / per_col)))
    reps = 1
    if n_cols == w.N:
        reps = max(1, min(10, int(target_s / max(per_col * w.N, 1e-6))))
    Ws, bs = cols_slice(n_cols)
    t0 = time.perf_counter()
    for _ in range(reps):
        r = _oracle_project(w, X, Ws, bs)
    elapsed = time.perf_counter() - t0
    wbytes = 2.0 * n_cols * w.K * reps
    sample = (f"all {w.M} token rows x {n_cols} of {w.N} output columns"
              + (f", {reps} repetitions" if reps > 1 else "") + f", {elapsed:.2f} s")
    out = {"value": wbytes / elapsed / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": sample, "seconds": elapsed}
    if y_gpu is not None:
        # The fused epilogue, if any, on the oracle's columns (fp64).
        if act == "gelu":
            r = oracle.gelu(r)
        if residual is not None:
            r = r + residual[:, :n_cols]
        # The tolerance of the parity tests: |u - r| <= 1e-3 + 5e-3·|r|.
        u = y_gpu[:, :n_cols]
        bad = int(np.count_nonzero(~(np.abs(u - r) <= 1e-3 + 5e-3 * np.abs(r))))
        out["timed_output_check"] = {"cells": int(u.size), "out_of_tolerance": bad}
    return out


def swiglu_output_check(w, inp, y_gpu, residual, features: int = 64) -> dict:
    """The first ``features`` outputs of every token row against the oracle's
    SwiGLU (their gate rows f and up rows F + f)."""
    import numpy as np
    import oracle
    F = w.N // 2
    nf = min(features, F)
    W = inp["W"]
    if w.w_layout == 0:
        Wsub = np.ascontiguousarray(np.vstack([W[:nf], W[F:F + nf]]))
    else:
        Wsub = np.ascontiguousarray(np.hstack([W[:, :nf], W[:, F:F + nf]]))
    r = oracle.project_swiglu(inp["X"], Wsub, w.w_layout,
                              None if residual is None else residual[:, :nf])
    u = y_gpu[:, :nf]
    bad = int(np.count_nonzero(~(np.abs(u - r) <= 1e-3 + 5e-3 * np.abs(r))))
    return {"cells": int(u.size), "out_of_tolerance": bad}


# ---------------------------------------------------------------- every config
def oracle_report(w, inp, y64: np.ndarray, rows) -> dict:
    """Accuracy of the GPU output against the fp64 oracle on the given token
    rows (all columns): the elementwise rule of the parity tests, relative L2
    over those rows, and the row rule of section "The actual error rule,
    including what L2 means" (each row's error norm over max(row norm, a tenth
    of the mean row norm)).  Also returns the all-thread oracle time of the
    sample."""
    import oracle
    Xs = np.ascontiguousarray(inp["X"][rows])
    t0 = time.perf_counter()
    r = oracle.project(Xs, inp["W"], w.w_layout, inp["bias"])
    t_all = time.perf_counter() - t0
    u = y64[rows]
    bad = int(np.count_nonzero(~(np.abs(u - r) <= 1e-3 + 5e-3 * np.abs(r))))
    diff = np.linalg.norm(u - r, axis=1)
    rn = np.linalg.norm(r, axis=1)
    denom = np.maximum(rn, 0.1 * rn.mean())
    return {"rows_checked": int(len(rows)), "cells": int(u.size), "out_of_tolerance": bad,
            "max_abs_err": float(np.abs(u - r).max()),
            "rel_l2": float(np.linalg.norm(u - r) / np.linalg.norm(r)),
            "row_rule_max": float((diff / denom).max())}, t_all


def oracle_single_thread_ms(w, inp, target_s: float = 0.4) -> tuple:
    """Single-thread oracle time of one whole call, extrapolated from a block
    of output columns (all token rows, or the first 64 of many)."""
    import oracle
    X, W, b = inp["X"], inp["W"], inp["bias"]
    m = min(w.M, 64)
    Xs = np.ascontiguousarray(X[:m])

    def cols(nc):
        Wc = np.ascontiguousarray(W[:nc] if w.w_layout == 0 else W[:, :nc])
        return Wc, (None if b is None else b[:nc])

    prev = oracle.max_threads()
    oracle.set_threads(1)
    try:
        Wc, bc = cols(min(w.N, 8))
        t0 = time.perf_counter()
        oracle.project(Xs, Wc, w.w_layout, bc)
        per_col = max(time.perf_counter() - t0, 1e-6) / Wc.shape[0 if w.w_layout == 0 else 1]
        nc = int(max(8, min(w.N, target_s / per_col)))
        Wc, bc = cols(nc)
        t0 = time.perf_counter()
        oracle.project(Xs, Wc, w.w_layout, bc)
        dt = time.perf_counter() - t0
    finally:
        oracle.set_threads(prev)
    full = dt * (w.N / nc) * (w.M / m)
    return full * 1e3, f"{m} of {w.M} token rows x {nc} of {w.N} columns, scaled to the whole call"


def measure_workloads(args, device, peaks: dict) -> dict:
    """Every configuration the metric names, each timed like the headline:
    packed weights rotating through copies larger than twice the L2, the
    --steps steps replayed from one CUDA graph (warmed once), device time of
    the steps alone.  Per config: µs per call, weight GB/s, TFLOP/s, the
    roofline fraction (measured and datasheet peaks), the oracle's time on
    the host cores (all threads and one thread) and its accuracy report."""
    import torch
    import dense_linear_projection_gb300 as dlp
    import oracle
    import synth

    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    stream = torch.cuda.Stream(device)
    out = {}
    cores = oracle.max_threads()

    def dev_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)

    def one(key, w, inp):
        X = dev_bf16(inp["X"])
        W0 = dev_bf16(inp["W"])
        bias = dev_bf16(inp["bias"]) if w.has_bias else None
        n_copies = max(2, math.ceil(2 * l2 / w.weight_bytes) + 1)
        proj = dlp.Projection(w.M, w.N, w.K, w.w_layout,
                              dlp.PROJ_F32 if w.y_dtype == "f32" else dlp.PROJ_BF16, w.has_bias,
                              overlap={"none": dlp.PROJ_OVERLAP_NONE, "prologue": dlp.PROJ_OVERLAP_PROLOGUE,
                                       "weights": dlp.PROJ_OVERLAP_WEIGHTS}[args.overlap])
        Wp = [proj.pack(W0)] + [proj.pack(W0.clone()) for _ in range(n_copies - 1)]
        del W0
        Y = torch.empty((w.M, w.N), dtype=torch.float32 if w.y_dtype == "f32" else torch.bfloat16,
                        device=device)
        torch.cuda.synchronize()  # inputs and packing (current stream) before the runs on `stream`
        steps = max(args.steps, 2 * n_copies)
        with torch.cuda.stream(stream):
            proj(X, Wp[0], bias, out=Y, stream=stream, packed=True)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(steps):
                proj(X, Wp[i % n_copies], bias, out=Y, stream=stream, packed=True)
        with torch.cuda.stream(stream):
            g.replay()  # warm-up: the same graph (its first launch also uploads it)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_stream(stream)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        st = proj.status(stream)
        if st != dlp.PROJ_OK:
            raise RuntimeError(f"{key}: device status {dlp.proj_status_string(st)}")
        t = e0.elapsed_time(e1) / 1e3 / steps
        y64 = Y.float().cpu().numpy().astype(np.float64)
        plan = proj.plan
        proj.close()
        del Wp, g
        torch.cuda.empty_cache()
        bytes_alg, flops = w.algorithmic_bytes, w.flops
        hbm_t = bytes_alg / (peaks["hbm_gbs"] * 1e9)
        ten_t = flops / (peaks["bf16_tflops"] * 1e12)
        if hbm_t >= ten_t:
            achieved = bytes_alg / t / 1e9
            roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / peaks["hbm_gbs"],
                    "datasheet": {"peak": DATASHEET["hbm_gbs"], "frac": achieved / DATASHEET["hbm_gbs"]}}
        else:
            achieved = flops / t / 1e12
            roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": achieved / peaks["bf16_tflops"],
                    "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                    "datasheet": {"peak": DATASHEET["bf16_tflops"],
                                  "frac": achieved / DATASHEET["bf16_tflops"]}}
        roof["peak_source"] = "of measured" if peaks["source"] == "measured" else "of fallback"
        roof["bytes_per_launch"] = bytes_alg
        roof["flops_per_launch"] = flops
        # Accuracy against the oracle: every token row up to 256, else 128
        # rows spread over the output (first, last and evenly spaced).
        rows = (np.arange(w.M) if w.M <= 256
                else np.unique(np.linspace(0, w.M - 1, 128).astype(np.int64)))
        acc, t_all = oracle_report(w, inp, y64, rows)
        ms_1t, sample_1t = oracle_single_thread_ms(w, inp)
        out[key] = {
            "M": w.M, "N": w.N, "K": w.K, "w_layout": "NK" if w.w_layout == 0 else "KN",
            "bias": w.has_bias, "y_dtype": w.y_dtype, "seed": w.seed, "steps": steps,
            "us_per_call": t * 1e6, "weight_gbs": w.weight_bytes / t / 1e9,
            "tflops": flops / t / 1e12, "roofline": roof,
            "plan": {k: plan[k] for k in ("block_t", "block_n", "grid", "stages", "cluster_split",
                                          "cta_pair", "tiles_dp", "tiles_sk")},
            "oracle": {"cores": cores,
                       "ms_all_threads": t_all * 1e3 * (w.M / len(rows)),
                       "all_threads_sample": (f"all {w.M} token rows" if len(rows) == w.M else
                                              f"{len(rows)} of {w.M} token rows, scaled to the whole call"),
                       "ms_single_thread": ms_1t, "single_thread_sample": sample_1t},
            "accuracy_vs_oracle": acc,
        }

    for name in args.workload_list:
        if name == "ffn_up_sweep":
            base = synth.workload(name, max(synth.FFN_SWEEP_M))
            full = synth.make_inputs(base)  # X rows of smaller M are a prefix (same seed)
            for M in synth.FFN_SWEEP_M:
                w = base.with_m(M)
                one(f"ffn_up_sweep_m{M}", w, dict(full, X=np.ascontiguousarray(full["X"][:M])))
            del full
        else:
            w = synth.workload(name)
            one(name, w, synth.make_inputs(w))
    return out


# ---------------------------------------------------------------- GPU arm
def run_gpu_arm(args) -> dict:
    import numpy as np
    import torch
    import torch.distributed as dist

    import dense_linear_projection_gb300 as dlp
    import synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    w = synth.workload(args.workload, args.m)
    inp = synth.make_inputs(w)

    def dev_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)

    X = dev_bf16(inp["X"])
    fp32_w = w.w_dtype == "f32"  # router weights: packed runs only (high/low split)
    W0 = torch.from_numpy(np.ascontiguousarray(inp["W"])).to(device) if fp32_w else dev_bf16(inp["W"])
    bias = dev_bf16(inp["bias"]) if w.has_bias else None
    if fp32_w and not args.packed:
        raise SystemExit("fp32 router weights run only packed (the split is the packing)")
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    n_copies = max(2, math.ceil(2 * l2 / w.weight_bytes) + 1)
    Ws = [W0] + [W0.clone() for _ in range(n_copies - 1)]
    y_dt = torch.float32 if w.y_dtype == "f32" else torch.bfloat16
    swiglu = args.activation == "swiglu"
    if swiglu and (not args.packed or w.has_bias or fp32_w or w.N % 2):
        raise SystemExit("swiglu runs packed, without bias, on bf16 weights with an even N")
    n_out = w.N // 2 if swiglu else w.N
    Y = torch.empty((w.M, n_out), dtype=y_dt, device=device)
    # Each step's kernel may start its set-up while the previous step
    # finishes (programmatic dependent launch).  Mode "weights" (the default)
    # also streams its first weight stages early, which the library does for
    # plans that occupy every SM; everything else waits for the previous
    # step to complete.  W is never written by the preceding kernel here.
    overlap = {"none": dlp.PROJ_OVERLAP_NONE, "prologue": dlp.PROJ_OVERLAP_PROLOGUE,
               "weights": dlp.PROJ_OVERLAP_WEIGHTS}[args.overlap]
    proj = dlp.Projection(w.M, w.N, w.K, w.w_layout,
                          dlp.PROJ_F32 if w.y_dtype == "f32" else dlp.PROJ_BF16, w.has_bias,
                          overlap=overlap, w_dtype=dlp.PROJ_F32 if fp32_w else dlp.PROJ_BF16)
    stream = torch.cuda.Stream(device)
    # Fused epilogue (optional): activation and a residual input R.  The
    # activation is set before packing (SwiGLU interleaves gate and up rows).
    proj.set_activation({"none": dlp.PROJ_ACT_NONE, "gelu": dlp.PROJ_ACT_GELU,
                         "swiglu": dlp.PROJ_ACT_SWIGLU}[args.activation])
    R = (torch.randn((w.M, n_out), device=device, generator=torch.Generator(device).manual_seed(w.seed))
         .to(y_dt) if args.residual else None)
    # Weights packed once per copy into the handle's tile-contiguous layout:
    # the preparation step, outside every timed region.
    Wrun = [proj.pack(Wc) for Wc in Ws] if args.packed else Ws
    torch.cuda.synchronize()

    def step(Wc, strm):
        proj(X, Wc, bias, out=Y, stream=strm, packed=args.packed, residual=R)

    # Graphs of back-to-back steps, each step on the next W copy.
    def capture(nsteps, offset):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(nsteps):
                step(Wrun[(offset + i) % n_copies], stream)
        return g

    with torch.cuda.stream(stream):
        step(Wrun[0], stream)  # first call encodes the tensor maps
    torch.cuda.synchronize()
    chunk = n_copies * max(1, 64 // n_copies)
    g_chunk = capture(chunk, 0)
    rem = args.steps % chunk
    g_rem = capture(rem, 0) if rem else None

    def run_steps(k):
        """Replay exactly k steps (k = the timed step count, or whole chunks)."""
        for _ in range(k // chunk):
            g_chunk.replay()
        if k % chunk:
            assert g_rem is not None and k % chunk == rem
            g_rem.replay()

    sampler = ClockSampler(visible_gpu_id(local)).start()
    with torch.cuda.stream(stream):
        # Warm-up replays the very graphs the timed region replays (a graph's
        # first launch also uploads it), at least `warmup` steps in all.
        for _ in range(max(1, math.ceil(args.warmup / args.steps))):
            run_steps(args.steps)
        # Untimed soak so the clock sampler sees the GPU under load even when
        # the timed region itself is only milliseconds long.
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < args.soak:
            run_steps(chunk)
            torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(stream)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        run_steps(args.steps)
        ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    seconds = ev0.elapsed_time(ev1) / 1e3
    status = proj.status(stream)
    if status != dlp.PROJ_OK:
        raise RuntimeError(f"device status after timing: {dlp.proj_status_string(status)}")

    agg = aggregate_throughput(w.weight_bytes * args.steps, seconds, device)
    t_step = agg["seconds"] / args.steps

    # ---- Spread: R shorter timed regions of the same kind (per-call µs).
    repeats = None
    if args.repeats > 0:
        r_steps = chunk * max(1, (args.steps // 10) // chunk)
        per_call = []
        with torch.cuda.stream(stream):
            for _ in range(args.repeats):
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                hold_stream(stream)
                a.record(stream)
                for _ in range(r_steps // chunk):
                    g_chunk.replay()
                b_.record(stream)
                b_.synchronize()
                per_call.append(a.elapsed_time(b_) * 1e3 / r_steps)
        qs = statistics.quantiles(per_call, n=10)
        repeats = {"n": args.repeats, "steps_each": r_steps, "median_us": statistics.median(per_call),
                   "p10_us": qs[0], "p90_us": qs[-1]}

    # ---- One call after an L2 flush (a write of twice the L2), not overlapped.
    cold = None
    if args.cold_calls > 0:
        flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=device)
        times = []
        with torch.cuda.stream(stream):
            for i in range(args.cold_calls):
                flush.fill_(float(i))
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                hold_stream(stream)
                a.record(stream)
                step(Wrun[i % n_copies], stream)
                b_.record(stream)
                b_.synchronize()
                times.append(a.elapsed_time(b_) * 1e3)
        del flush
        cold = {"calls": args.cold_calls, "median_us": statistics.median(times),
                "what": "one proj_run after writing 2x L2, events around the call alone (device time)"}

    # ---- Informational: the same projection through cuBLAS (torch), never the target.
    library = None
    if args.library:
        # bf16 weights: bf16 GEMM, bf16 output; fp32 router weights: fp32 GEMM
        # of X cast to fp32 (torch keeps TF32 off for matmul by default).
        Xl = X.float() if fp32_w else X
        bl = None if bias is None else (bias.float() if fp32_w else bias)
        Yl = torch.empty((w.M, w.N), dtype=torch.float32 if fp32_w else torch.bfloat16, device=device)

        def lib_call(Wc):
            Wm = Wc.t() if w.w_layout == 0 else Wc
            if bl is not None:
                torch.addmm(bl, Xl, Wm, out=Yl)
            else:
                torch.mm(Xl, Wm, out=Yl)

        with torch.cuda.stream(stream):
            lib_call(W0)
        torch.cuda.synchronize()
        gl = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gl, stream=stream):
            for i in range(chunk):
                lib_call(Ws[i % n_copies])
        l_steps = chunk * max(1, (args.steps // 4) // chunk)
        with torch.cuda.stream(stream):
            for _ in range(max(1, math.ceil(args.warmup / chunk))):
                gl.replay()
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            hold_stream(stream)
            a.record(stream)
            for _ in range(l_steps // chunk):
                gl.replay()
            b_.record(stream)
        torch.cuda.synchronize()
        t_lib = a.elapsed_time(b_) / 1e3 / l_steps
        library = {"impl": ("torch.mm (cuBLAS fp32 GEMM, X cast to fp32), fp32 output" if fp32_w
                            else "torch.addmm / torch.mm (cuBLAS), bf16 output"), "steps": l_steps,
                   "us_per_call": t_lib * 1e6, "value": w.weight_bytes / t_lib / 1e9, "unit": "GB/s",
                   "note": "informational; same inputs, W rotation and CUDA-graph replay"}
        del Yl, gl
    peaks = load_peaks()
    fused = args.activation != "none" or args.residual
    traffic, profile_path = (None, None) if fused else profile_traffic(
        args.workload if args.m is None else f"{args.workload}_m{args.m}")
    # A residual is one more output-sized array read; SwiGLU writes N/2 columns.
    ysz = 4 if w.y_dtype == "f32" else 2
    alg_bytes = (w.algorithmic_bytes - (w.M * (w.N - n_out) * ysz)
                 + (w.M * n_out * ysz if args.residual else 0))
    hbm_bound = roofline_time_s(alg_bytes, w.flops, peaks["hbm_gbs"] * 1e9,
                                peaks["bf16_tflops"] * 1e12)
    if alg_bytes / (peaks["hbm_gbs"] * 1e9) >= w.flops / (peaks["bf16_tflops"] * 1e12):
        roof = {"bound": "hbm", "achieved": alg_bytes / t_step / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        peak_tf = peaks["bf16_tflops_sustained"] if agg["seconds"] > 1.0 else peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": w.flops / t_step / 1e12, "peak": peak_tf,
                "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    ds = DATASHEET["hbm_gbs"] if roof["bound"] == "hbm" else DATASHEET["bf16_tflops"]
    roof["datasheet"] = {"peak": ds, "frac": roof["achieved"] / ds}
    roof["traffic"] = traffic
    roof["peak_source"] = ("of measured" if peaks["source"] == "measured" else "of fallback")
    roof["bytes_per_launch"] = alg_bytes
    roof["flops_per_launch"] = w.flops
    roof["bound_us"] = hbm_bound * 1e6
    if profile_path:
        roof["profile"] = profile_path

    # ---- e2e: the user-facing call with host activations, every step.
    e2e = None
    if not args.no_e2e and not fused:  # the host-buffer call has no fused epilogue
        Xh = torch.from_numpy(np.ascontiguousarray(inp["X"]).view(np.int16)).view(
            torch.bfloat16).pin_memory()
        Yh = torch.empty((w.M, w.N), dtype=y_dt).pin_memory()
        sptr = stream.cuda_stream
        run_host = dlp.proj_run_host_packed if args.packed else dlp.proj_run_host
        for i in range(max(3, args.warmup)):
            run_host(proj.handle, Xh, Wrun[i % n_copies], bias, Yh, sptr)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            run_host(proj.handle, Xh, Wrun[i % n_copies], bias, Yh, sptr)
        e1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e_agg = aggregate_throughput(w.weight_bytes * args.steps, e0.elapsed_time(e1) / 1e3,
                                     device)
        ybytes = w.M * w.N * (4 if w.y_dtype == "f32" else 2)
        e2e = {"value": e_agg["per_second"] / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": 2 * w.M * w.K, "d2h_bytes_per_step": ybytes,
               "us_per_step": e_agg["seconds"] / args.steps * 1e6,
               "path": ("proj_run_host_packed" if args.packed else "proj_run_host")
                       + " per step (X H2D by a copy kernel; Y written to pinned host by the epilogue; W resident)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # Y still holds the timed steps' output (every W copy is the same W).
        step(Wrun[0], stream)  # the output of one plain call, to be safe
        torch.cuda.synchronize()
        y64 = Y.float().cpu().numpy().astype(np.float64)
        cpu = cpu_oracle_timing(w, inp, args.cpu_seconds, y_gpu=None if swiglu else y64,
                                act=args.activation,
                                residual=None if R is None else R.double().cpu().numpy())
        if swiglu:
            cpu["timed_output_check"] = swiglu_output_check(w, inp, y64, None if R is None else
                                                            R.double().cpu().numpy())
        cpu.pop("seconds", None)

    # ---- The allocation-free entry point against proj_run on the same weights
    # as stored (it takes no packed weights): eager calls, so the host-side
    # cost of each call shows (host µs per call) beside the device time.
    noalloc = None
    if rank == 0 and world == 1 and not args.no_noalloc and not fp32_w and not fused:
        y_code = dlp.PROJ_F32 if w.y_dtype == "f32" else dlp.PROJ_BF16
        calls = 64

        def eager(fn):
            for i in range(8):
                fn(i)
            torch.cuda.synchronize()
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            h0 = time.perf_counter()
            for i in range(calls):
                fn(i)
            host = time.perf_counter() - h0
            b_.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b_) * 1e3 / calls, host * 1e6 / calls

        run_us, run_host = eager(lambda i: dlp.proj_run(proj.handle, X, Ws[i % n_copies], bias, Y, stream))
        na_us, na_host = eager(lambda i: dlp.proj_run_noalloc(w.M, w.N, w.K, w.w_layout, y_code, X,
                                                              Ws[i % n_copies], bias, Y, stream))
        st_na = dlp.proj_noalloc_device_status(stream)
        if st_na != dlp.PROJ_OK:
            raise RuntimeError(f"allocation-free path status: {dlp.proj_status_string(st_na)}")
        noalloc = {"calls": calls, "proj_run_us_per_call": run_us, "proj_run_host_us_per_call": run_host,
                   "noalloc_us_per_call": na_us, "noalloc_host_us_per_call": na_host,
                   "what": "eager back-to-back calls on the weights as stored (no graph), events around "
                           "the loop; host µs = enqueue time per call"}

    plan = proj.plan
    proj.close()
    workloads = None
    if rank == 0 and world == 1 and args.workload_list:
        torch.cuda.empty_cache()
        workloads = measure_workloads(args, device, peaks)
    line = {
        "metric": METRIC,
        "value": agg["per_second"] / 1e9,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_step * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 (fp32 weights as high/low bf16 parts)" if fp32_w else "bf16",
        "data": "synthetic (seeded SplitMix64/Box-Muller normals, bf16)",
        "config": {
            "workload": w.name, "M": w.M, "N": w.N, "K": w.K,
            "w_layout": "NK" if w.w_layout == 0 else "KN", "bias": w.has_bias,
            "y_dtype": w.y_dtype, "seed": w.seed,
            "l2": f"rotating {n_copies} W copies ({n_copies * w.weight_bytes / 2**20:.0f} MiB > "
                  f"2x L2 of {l2 / 2**20:.0f} MiB); inputs resident in HBM",
            "timing": "CUDA-graph replay of the K steps, CUDA events on the launching stream",
            "overlap": f"programmatic dependent launch, mode '{args.overlap}'",
            "weights": ("pre-packed tile-contiguous by proj_pack_weights, once per copy before "
                        "timing (the preparation step)" if args.packed else "as stored"),
            "epilogue": ("act(X·Wᵀ + b) + R" if args.residual else "act(X·Wᵀ + b)")
                        + f", act = {args.activation}",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "us_per_call": t_step * 1e6,
        "tflops": w.flops / t_step / 1e12,
        "repeats": repeats,
        "cold_call": cold,
        "library_baseline": library,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "plan": {k: plan[k] for k in ("kernel", "block_t", "stages", "grid", "tiles_dp",
                                      "tiles_sk", "units_sk")},
        "noalloc": noalloc,
        "workloads": workloads,
    }
    if world > 1:
        dist.destroy_process_group()
    return line if rank == 0 else None


# ---------------------------------------------------------------- reference arm
def run_reference_arm(args) -> dict:
    """The fp64 CPU oracle as the reference implementation, on this arm's
    workload: every step is a bounded sample (all token rows against a block of
    output columns) sized so warm-up + timed steps take about a minute."""
    import numpy as np
    import oracle
    import synth

    rank, world, _ = dist_env()
    if rank != 0:
        return None
    w = synth.workload(args.workload, args.m)
    inp = synth.make_inputs(w)
    X, W, b = inp["X"], inp["W"], inp["bias"]
    threads = oracle.max_threads()
    probe = min(w.N, 32)
    Wp = W[:probe] if w.w_layout == 0 else np.ascontiguousarray(W[:, :probe])
    t0 = time.perf_counter()
    _oracle_project(w, X, Wp, None if b is None else b[:probe])
    per_col = max(time.perf_counter() - t0, 1e-6) / probe
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    n_cols = int(max(1, min(w.N, budget / per_col)))
    Ws = W[:n_cols] if w.w_layout == 0 else np.ascontiguousarray(W[:, :n_cols])
    bs = None if b is None else b[:n_cols]
    for _ in range(args.warmup):
        _oracle_project(w, X, Ws, bs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_project(w, X, Ws, bs)
    elapsed = time.perf_counter() - t0
    value = 2.0 * n_cols * w.K * args.steps / elapsed / 1e9
    sample = f"each step: all {w.M} token rows x {n_cols} of {w.N} output columns"
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded SplitMix64/Box-Muller normals, bf16)",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
                   "w_layout": "NK" if w.w_layout == 0 else "KN", "bias": w.has_bias,
                   "y_dtype": w.y_dtype, "seed": w.seed},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="decode_f32out | decode_bias | ffn_up_sweep | qkv_kn_bias | prefill"
                         " | router_f32w")
    ap.add_argument("--m", type=int, default=None, help="token rows (overrides the workload's M)")
    ap.add_argument("--soak", type=float, default=1.0,
                    help="seconds of untimed load before timing (clock sampling)")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--overlap", choices=["none", "prologue", "weights"], default="weights",
                    help="overlap of consecutive steps (programmatic dependent launch)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--repeats", type=int, default=7,
                    help="shorter timed regions for the median/p10/p90 spread (0: none)")
    ap.add_argument("--cold-calls", type=int, default=10,
                    help="single calls timed after an L2 flush (0: none)")
    ap.add_argument("--no-noalloc", action="store_true",
                    help="skip the allocation-free entry point's per-call timing")
    ap.add_argument("--no-library", dest="library", action="store_false",
                    help="skip the informational cuBLAS timing")
    ap.add_argument("--no-packed", dest="packed", action="store_false",
                    help="run on the weights as stored instead of pre-packed ones")
    ap.add_argument("--activation", choices=["none", "gelu", "swiglu"], default="none",
                    help="fused activation on projection + bias (proj_set_activation); swiglu "
                         "reads W as [gate rows; up rows] and writes N/2 columns")
    ap.add_argument("--residual", action="store_true",
                    help="fused residual add: Y = act(X·Wᵀ + b) + R, R an [M,N] input")
    ap.add_argument("--workloads", default="decode_f32out,decode_bias,ffn_up_sweep,qkv_kn_bias,prefill",
                    help="comma-separated configs also timed into the line's 'workloads' object "
                         "(single GPU only; empty: none)")
    args = ap.parse_args(argv)
    args.workload_list = [x for x in args.workloads.split(",") if x]
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 1:
        ap.error("--steps must be positive")
    return args


def main(argv=None):
    args = parse_args(argv)
    line = run_reference_arm(args) if args.impl == "reference" else run_gpu_arm(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
