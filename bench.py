#!/usr/bin/env python3
"""Benchmark of the hot path: the 8192x8192x16384 column-major FP16 GEMM and
the 34816x5120 BF16 decode GEMV (n = 1, 4, 8), on one GB300 per process.

One step = one pass of the whole path on one batch of synthetic input:
    gemm_f16_colmajor(A, B, C, 8192, 8192, 16384)
    gemv_bf16(W_i, x_n, y_n, 34816, 5120, n)   4 times back to back, for n in (1, 4, 8)
(three copies W_i of the weights rotate, so no GEMV launch finds W in L2; the
GEMM's operands, 537 MB, are larger than L2 too).  W = warm-up steps are run
first, then exactly K steps are timed with CUDA events on the launching
stream, bracketed by a barrier and a device synchronize.

Reported (one JSON line, rank 0):
  value      GEMM TFLOP/s: 2*M*N*K / mean GEMM kernel time (events around
             each GEMM launch), times the number of ranks (replicas).
  roofline_gemv  (last on the line) the GEMV's HBM GB/s per n against the
             measured copy bandwidth: algorithmic bytes / average launch time
             over each chain of 4 launches (events at the chain's ends, as in a
             decode loop); single_launch_us is one launch after the GEMM with
             events on both sides (which stops the overlap of the launch with
             the kernel before it); cuda_core_best is the fastest CUDA-core
             GEMV kernel for that n, timed the same way.
  e2e        the same metrics through the C-ABI calls on host buffers
             (gemm_f16_colmajor_host, gemv_bf16_host; pinned memory): the
             copies of the step's inputs in and of the result out happen
             inside the call, overlapped with the compute in blocks.
  roofline   for the dominant kernel (the GEMM) against the measured bf16
             peak (FP16 and BF16 dense rates are equal on this part).
  other_configs  device time of the remaining workloads (256^3 and 4095x4097x4100
             FP16 GEMMs, the 4096-token BF16 prefill projection, gemm_f16 in
             other storage forms with a fused bias, and the FP8 GEMM), measured
             after the step.
  decode_attention  split-KV decode attention at 8K/16K/32K tokens (KV-cache GB/s),
             back-to-back calls (and, separately, each call between events).
  cpu_baseline  the oracle timed on a bounded sample on the host cores: the
             headline GEMM, and every other workload in `configs`.

``--impl reference`` times the oracle (the plain CPU triple loop) on the same
workload instead, on the host cores, each step a bounded sample of columns.
Multi-GPU: one process per GPU under torchrun runs an independent replica.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GEMM_M, GEMM_N, GEMM_K = 8192, 8192, 16384
GEMV_M, GEMV_K, GEMV_NS = 34816, 5120, (1, 4, 8)
# A decode step runs GEMVs back to back: each n is timed over a chain of this
# many launches (events at the chain's ends only), rotating three weight copies
# so that no launch finds its W in L2.
GEMV_CHAIN = 4
S_PREFILL = 4096
METRIC = "FP16 GEMM TFLOP/s @8192x8192x16384; BF16 GEMV HBM GB/s (fraction of peak)"
WORKLOAD = "gemm_f16_colmajor 8192x8192x16384 + gemv_bf16 34816x5120 n=1,4,8"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def gemm_flops() -> int:
    return 2 * GEMM_M * GEMM_N * GEMM_K


def gemv_bytes(n: int) -> int:
    """Algorithmic bytes of one decode GEMV: W once, x once, y once (BF16)."""
    return 2 * (GEMV_M * GEMV_K + n * GEMV_K + n * GEMV_M)


def tile_stage_bytes(block_m: int, block_n: int, block_k: int, elem_bytes: int = 2) -> int:
    """Bytes of one pipeline stage of a tiled GEMM: (BLOCK_M + BLOCK_N) * BLOCK_K * element size
    ("Hygon 优化", section 软件流水线)."""
    return (block_m + block_n) * block_k * elem_bytes


def roofline(peak: float, bandwidth: float, intensity: float) -> float:
    """Attainable rate min(P_peak, B * I) of the roofline model (DCU decode-GEMV
    article, section 3); units follow the arguments (e.g. TFLOP/s, TB/s, FLOP/B)."""
    return min(peak, bandwidth * intensity)


# ---------------------------------------------------------------------------
# environment: ranks, peaks, clocks, ncu traffic
# ---------------------------------------------------------------------------

def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist

    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, dist, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity for one rank)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units: float, seconds: float, dist, device=None) -> float:
    """Units processed by all ranks divided by the slowest rank's time."""
    if dist is None:
        return units / seconds
    import torch

    t = torch.tensor([units, seconds], dtype=torch.float64, device=device)
    u = t[:1].clone()
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    m = t[1:].clone()
    dist.all_reduce(m, op=dist.ReduceOp.MAX)
    return float(u.item()) / float(m.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# The code each measured launch is built from: (file, text that starts the
# file's host-only part or None), or (file, (first, end)) for the part of a
# file from the text `first` up to the text `end`.  Host-side launch code does
# not change the kernel, so it is left out of the digest -- except the GEMM's
# planning and launch set-up in api.cu (pack, tile width and height, schedule,
# tile order, k order), whose choices change the kernel's DRAM traffic.
KERNEL_SOURCES = {
    "gemm": (("gemm_tcgen05.cuh", "inline CUtensorMapDataType tmap_type("), ("ptx.cuh", None),
             ("bsk_internal.h", "using TmapEncodeFn"),
             ("api.cu", ("// Which operands must be packed before the TMA can read them",
                         "// Elements a stored matrix"))),
    "gemv": (("gemv.cu", "int launch_vec(const GemvLaunch& g"), ("bsk_internal.h", "using TmapEncodeFn")),
}


def source_digest(kernel: str, cdir: str | None = None) -> str:
    """Hash of one kernel's device code (comments and whitespace left out); a
    committed traffic figure is only reported while that code is unchanged
    since it was measured.  `cdir`: the source directory (default: the
    package's csrc/)."""
    h = hashlib.sha256()
    cdir = cdir or os.path.join(ROOT, "bf16_gemm_skinny_gb300", "csrc")
    for name, host_start in KERNEL_SOURCES[kernel]:
        with open(os.path.join(cdir, name), "rb") as f:
            text = f.read()
        if isinstance(host_start, tuple):
            first, end = (text.find(m.encode()) for m in host_start)
            if first < 0 or end < first:
                raise RuntimeError(f"{name}: markers {host_start!r} not found in order")
            text = text[first:end]
        elif host_start is not None:
            cut = text.find(host_start.encode())
            if cut < 0:
                raise RuntimeError(f"{name}: host-code marker {host_start!r} not found")
            text = text[:cut]
        # comments and layout do not change the kernel
        code = re.sub(rb"/\*.*?\*/", b"", text, flags=re.S)
        code = re.sub(rb"//[^\n]*", b"", code)
        code = b" ".join(code.split())
        h.update(name.encode() + b"\0" + code)
    return h.hexdigest()[:16]


def committed_traffic(kernel_key: str):
    """DRAM bytes per launch from profiles/traffic.txt (lines: key digest bytes)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    digest = source_digest(kernel_key.split("_")[0])
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel_key:
                    return float(parts[2]) if parts[1] == digest else None
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.count(",") >= 8]
        self.file.close()
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample
# ---------------------------------------------------------------------------

def oracle_gemm_sample(A, B, seconds: float, max_cols: int = 4096):
    """Runs the oracle on growing batches of output columns of the GEMM until
    about `seconds` of CPU work; returns (flops, elapsed, cols, threads)."""
    import oracle

    threads = oracle.max_threads()
    done, elapsed, batch, col = 0, 0.0, max(1, threads), 0
    while elapsed < seconds and done < max_cols:
        cols = [(col + i * 977) % GEMM_N for i in range(batch)]
        t0 = time.perf_counter()
        oracle.gemm_f16_colmajor(A, B, GEMM_M, GEMM_N, GEMM_K, cols=cols, threads=threads)
        elapsed += time.perf_counter() - t0
        done += batch
        col += 1
    return 2 * GEMM_M * GEMM_K * done, elapsed, done, threads


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, else the implementer/part codes)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read().splitlines()
    except OSError:
        return "unknown"
    for key in ("model name", "Model name", "CPU part"):
        for line in info:
            if line.split(":")[0].strip() == key:
                value = line.split(":", 1)[1].strip()
                if key == "CPU part":
                    impl = next((ln.split(":", 1)[1].strip() for ln in info
                                 if ln.split(":")[0].strip() == "CPU implementer"), "?")
                    return f"implementer {impl}, part {value}"
                return value
    return "unknown"


def single_thread_rates():
    """The oracle on one thread: the whole 256^3 GEMM, and 64 output features of
    the n = 1 GEMV at 34816x5120 (about a second each)."""
    import oracle
    from bf16_gemm_skinny_gb300 import inputs

    A, B = inputs.gemm_operands(256, 256, 256, "uniform")
    t0 = time.perf_counter()
    oracle.gemm_f16_colmajor(A, B, 256, 256, 256, threads=1)
    t_gemm = time.perf_counter() - t0
    W, x = inputs.linear_operands(GEMV_M, GEMV_K, 1, "normal0.02", "normal1")
    js = list(range(0, GEMV_M, GEMV_M // 64))[:64]
    t0 = time.perf_counter()
    oracle.linear_bf16(W, x, GEMV_M, GEMV_K, 1, js=js, threads=1)
    t_gemv = time.perf_counter() - t0
    return {"gemm_256_ms": round(t_gemm * 1e3, 2),
            "gemm_256_gflops": round(2 * 256 ** 3 / t_gemm / 1e9, 3),
            "gemv_n1_gbs": round(len(js) * GEMV_K * 2 / t_gemv / 1e9, 3),
            "gemv_n1_sample": f"{len(js)} output features of 34816 (K = 5120)"}


def timed_batches(run_batch, seconds: float, first: int, cap: int):
    """Calls run_batch(i0, count) on batches of growing size until about `seconds`
    of work; returns (units done, elapsed seconds)."""
    done, elapsed, batch = 0, 0.0, max(1, first)
    while elapsed < seconds and done < cap:
        count = min(batch, cap - done)
        t0 = time.perf_counter()
        run_batch(done, count)
        elapsed += time.perf_counter() - t0
        done += count
        batch *= 2
    return done, elapsed


def oracle_configs(seconds_each: float, threads: int):
    """The oracle on `threads` host threads for every workload, each on a bounded
    sample of its outputs (whole output columns of a GEMM, whole output features
    of a linear layer): rate, sample and seconds per workload.  The thread count
    is passed to every call: the oracle's OpenMP setting persists between calls."""
    import oracle
    from bf16_gemm_skinny_gb300 import inputs

    out = {}
    for name, (M, N, K, dist) in (("gemm_256x256x256", (256, 256, 256, "uniform")),
                                   ("gemm_4095x4097x4100", (4095, 4097, 4100, "normal0.5"))):
        A, B = inputs.gemm_operands(M, N, K, dist)
        if M == 256:
            reps, el = timed_batches(lambda i0, c: [oracle.gemm_f16_colmajor(A, B, M, N, K, threads=threads)
                                                    for _ in range(c)], seconds_each, 1, 1 << 16)
            out[name] = {"tflops": 2.0 * M * N * K * reps / el / 1e12, "sample": f"the whole GEMM, {reps} times",
                         "s": round(el, 2)}
        else:
            cols, el = timed_batches(lambda i0, c: oracle.gemm_f16_colmajor(
                A, B, M, N, K, cols=[(i0 + i) * 131 % N for i in range(c)], threads=threads), seconds_each, threads, N)
            out[name] = {"tflops": 2.0 * M * K * cols / el / 1e12,
                         "sample": f"{cols} of {N} output columns", "s": round(el, 2)}
    W, _ = inputs.linear_operands(GEMV_M, GEMV_K, 1, "normal0.02", "normal1")
    for n in GEMV_NS:
        _, x = inputs.linear_operands(1, GEMV_K, n, "normal0.02", "normal1")
        rows, el = timed_batches(lambda i0, c: oracle.linear_bf16(
            W, x, GEMV_M, GEMV_K, n, js=[(i0 + i) * 977 % GEMV_M for i in range(c)], threads=threads), seconds_each,
            4 * threads, GEMV_M)
        out[f"gemv_34816x5120_n{n}"] = {"gbs": rows * GEMV_K * 2 / el / 1e9, "sample": f"{rows} of {GEMV_M} output "
                                        "features (GB/s of weights read)", "s": round(el, 2)}
    _, X = inputs.linear_operands(1, GEMV_K, S_PREFILL, "normal0.02", "normal1")
    feats, el = timed_batches(lambda i0, c: oracle.linear_bf16(
        W, X, GEMV_M, GEMV_K, S_PREFILL, js=[(i0 + i) * 977 % GEMV_M for i in range(c)], threads=threads),
        seconds_each, threads, GEMV_M)
    out["prefill_4096x34816x5120"] = {"tflops": 2.0 * S_PREFILL * GEMV_K * feats / el / 1e12,
                                      "sample": f"{feats} of {GEMV_M} output features", "s": round(el, 2)}
    for v in out.values():
        v["threads"] = threads
        for key in ("tflops", "gbs"):
            if key in v:
                v[key] = round(v[key], 5)
    return out


def cpu_baseline(A, B, seconds: float, seconds_each: float = 2.5):
    flops, elapsed, cols, threads = oracle_gemm_sample(A, B, seconds)
    configs = oracle_configs(seconds_each, threads)
    return {"value": flops / elapsed / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{cols} output columns of the 8192x8192x16384 GEMM (each 8192x16384 FMAs, FP64), "
                      f"{elapsed:.1f} s",
            "cpu": cpu_model(), "configs": configs, "single_thread": single_thread_rates()}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def time_launches(fn, iters: int, warmup: int = 3) -> float:
    """Mean device time (ms) of `fn`'s launches on the current stream, CUDA events."""
    import torch

    for _ in range(warmup):
        fn()
    stream = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(iters + 1)]
    torch.cuda.synchronize()
    evs[0].record(stream)
    for i in range(iters):
        fn()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    return statistics.fmean(evs[i].elapsed_time(evs[i + 1]) for i in range(iters))


def time_device(fn, iters: int, warmup: int = 3, blocker_cycles: int = 4_000_000) -> float:
    """Median device time (ms) of one call of `fn`: CUDA events recorded around
    each call in the stream, behind a spin kernel of about 2 ms queued first, so
    that the host has enqueued every call before the GPU reaches it.  The calls
    then run back to back, each bracketed by its events (which also stop the
    programmatic-launch overlap of consecutive calls), and the host's per-call
    overhead does not show."""
    import torch

    for _ in range(warmup):
        fn()
    stream = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(iters + 1)]
    torch.cuda.synchronize()
    torch.cuda._sleep(blocker_cycles)
    evs[0].record(stream)
    for i in range(iters):
        fn()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    return statistics.median(evs[i].elapsed_time(evs[i + 1]) for i in range(iters))


def time_chain_ahead(fn, iters: int, warmup: int = 3, blocker_cycles: int = 4_000_000) -> float:
    """Mean device time (ms) per call of `iters` back-to-back calls of `fn`, with
    events at the chain's ends only, behind a spin kernel of about 2 ms so that
    the host has enqueued every call before the GPU reaches the first."""
    import torch

    for _ in range(warmup):
        fn()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    torch.cuda._sleep(blocker_cycles)
    e0.record(stream)
    for _ in range(iters):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def time_chain(fn, iters: int, warmup: int = 3) -> float:
    """Mean device time (ms) per call of `iters` back-to-back calls of `fn` on the
    current stream, CUDA events at the chain's ends only (an event between two
    launches would stop the programmatic-dependent overlap of consecutive calls)."""
    import torch

    for _ in range(warmup):
        fn()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(iters):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def other_configs(W_prefill, dev, peaks):
    """Device time of the other workloads (256^3, the ragged 4095x4097x4100 GEMM
    and the 4096-token prefill projection, other storage forms, FP8), each on
    its own seeded inputs, with the host ahead of the GPU.  For the two FP16
    GEMMs of the workload list, `us` is the mean per call over 20 calls back to
    back (events at the chain's ends); `us_between_events` is the median over
    calls each bracketed by events (an event between two kernels costs about
    4 us on its own on GB300: a trivial kernel measures 4.3 us that way and
    2.2 us back to back), and `us_host_paced` the same with the calls issued as
    Python reaches them.  The larger workloads report the median between
    events."""
    import numpy as np
    import torch

    from bf16_gemm_skinny_gb300 import _native as bsk
    from bf16_gemm_skinny_gb300 import inputs

    to_dev = lambda bits: torch.from_numpy(bits.view(np.int16)).to(dev)  # noqa: E731
    peak_t = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    out = {}
    for name, (M, N, K, dist) in (("gemm_256x256x256", (256, 256, 256, "uniform")),
                                   ("gemm_4095x4097x4100", (4095, 4097, 4100, "normal0.5"))):
        A, B = inputs.gemm_operands(M, N, K, dist)
        Ad, Bd = to_dev(A), to_dev(B)
        C = torch.empty(M * N, dtype=torch.int16, device=dev)
        call = lambda: bsk.gemm_f16_colmajor_enqueue(Ad, Bd, C, M, N, K)  # noqa: E731
        ms = time_chain_ahead(call, 20)
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        out[name] = {"us": round(ms * 1e3, 2), "tflops": round(tf, 1), "frac_of_peak": round(tf / peak_t, 4),
                     "us_between_events": round(time_device(call, 20) * 1e3, 2),
                     "us_host_paced": round(time_launches(call, 20) * 1e3, 2),
                     "note": "includes the pack of unaligned operands" if M % 8 else ""}
        del Ad, Bd, C
    # The same GEMM in other storage forms with a fused bias (gemm_f16): column-major
    # NT, and a row-major FP16 linear layer Y = X W^T + b over the prefill shape.
    for name, (order, ta, tb, M, N, K) in (
            ("gemm_f16_nt_bias_8192x8192x8192", (0, 0, 1, 8192, 8192, 8192)),
            ("linear_f16_rowmajor_bias_4096x34816x5120", (1, 0, 1, S_PREFILL, GEMV_M, GEMV_K))):
        A, B = inputs.gemm_operands(M, N, K, "uniform")
        Ad, Bd = to_dev(A), to_dev(B)
        bias = to_dev(inputs.to_f16_bits(inputs.draw("uniform", N, 41)))
        C = torch.empty(M * N, dtype=torch.int16, device=dev)
        lda = (K if ta else M) if order == 0 else (M if ta else K)
        ldb = (N if tb else K) if order == 0 else (K if tb else N)
        ldc = M if order == 0 else N
        ms = time_device(lambda: bsk.gemm_f16_enqueue(order, ta, tb, Ad, lda, Bd, ldb, C, ldc, M, N, K, bias,
                                                      bsk.BIAS_COLUMN), 20)
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        out[name] = {"us": round(ms * 1e3, 2), "tflops": round(tf, 1), "frac_of_peak": round(tf / peak_t, 4),
                     "layout": {"order": "row" if order else "column", "transa": ta, "transb": tb,
                                "bias": "per column"}}
        del Ad, Bd, C, bias
    # FP8 (E4M3) GEMMs with FP32 accumulation and BF16 output: the square
    # shape, and FP8 weights over the prefill projection (A = W, B = X).
    fp8_peak = 2.0 * peak_t   # FP8 dense rate = 2x the measured BF16 rate (nominal ratio)
    for name, (M, N, K) in (("gemm_fp8_e4m3_8192x8192x8192", (8192, 8192, 8192)),
                            ("linear_fp8_e4m3_34816x4096x5120", (GEMV_M, S_PREFILL, GEMV_K))):
        A, B = inputs.fp8_operands(M, N, K, "normal1", "e4m3")
        Ad = torch.from_numpy(A).to(dev)
        Bd = torch.from_numpy(B).to(dev)
        C = torch.empty(M * N, dtype=torch.int16, device=dev)
        ms = time_device(lambda: bsk.gemm_fp8_enqueue(bsk.FP8_E4M3, Ad, K, Bd, K, C, M, bsk.OUT_BF16, M, N, K,
                                                      1.0), 20)
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        out[name] = {"us": round(ms * 1e3, 2), "tflops": round(tf, 1), "frac_of_fp8_peak": round(tf / fp8_peak, 4),
                     "fp8_peak": round(fp8_peak, 1), "out": "bf16"}
        del Ad, Bd, C
    S = S_PREFILL
    _, X = inputs.linear_operands(1, GEMV_K, S, "normal0.02", "normal1")
    Xd = to_dev(X)
    Y = torch.empty(S * GEMV_M, dtype=torch.int16, device=dev)
    ms = time_device(lambda: bsk.gemv_bf16_enqueue(W_prefill, Xd, Y, GEMV_M, GEMV_K, S), 10)
    tf = 2.0 * S * GEMV_M * GEMV_K / (ms * 1e-3) / 1e12
    out["prefill_4096x34816x5120"] = {"us": round(ms * 1e3, 2), "tflops": round(tf, 1),
                                      "frac_of_peak": round(tf / peak_t, 4)}
    bsk.stream_check()
    return out


def attention_configs(dev, hbm_peak):
    """Split-KV decode attention at the page's head shape (16 query heads over 4 KV
    heads, head_dim 256, 784-token pages) for 8K / 16K / 32K tokens, with the
    automatic segment count and with the page's 16 / 32 rule.  `us` is the mean
    device time per call over 20 back-to-back calls (each on a cache copy not in
    L2), enqueued behind a spin kernel so the host is ahead of the GPU;
    `per_call_events_us` brackets every call with events (host ahead too);
    `us_host_paced` is the back-to-back mean with the calls issued as Python
    reaches them (no spin kernel first), where the host's per-call cost shows
    if it exceeds the GPU's."""
    import numpy as np
    import torch

    from bf16_gemm_skinny_gb300 import _native as bsk
    from bf16_gemm_skinny_gb300 import inputs

    nqh, nkv, hd, bs = 16, 4, 256, 784
    out = {}
    for L in (8192, 16384, 32768):
        nb = -(-L // bs)
        n = nb * bs * nkv * hd
        k = torch.from_numpy(inputs.to_bf16_bits(inputs.draw("normal1", n, 31)).view(np.int16)).to(dev)
        v = torch.from_numpy(inputs.to_bf16_bits(inputs.draw("normal1", n, 32)).view(np.int16)).to(dev)
        q = torch.from_numpy(inputs.to_bf16_bits(inputs.draw("normal1", nqh * hd, 33)).view(np.int16)).to(dev)
        bt = torch.from_numpy(np.random.default_rng(34).permutation(nb).astype(np.int32)).to(dev)
        sl = torch.tensor([L], dtype=torch.int32, device=dev)
        o = torch.empty(nqh * hd, dtype=torch.int16, device=dev)
        kv_bytes = L * nkv * hd * 2 * 2
        # Enough copies of the cache that successive calls never find it in L2
        # (together at least twice the 129 MB L2).
        copies = max(2, -(-260_000_000 // kv_bytes))
        kvs = [(k, v)] + [(k.clone(), v.clone()) for _ in range(copies - 1)]
        row = {}
        for name, segs in (("auto", 0), ("page_rule", 32 if L >= 12288 else 16)):
            it = [0]

            def call():
                kc, vc = kvs[it[0] % copies]
                it[0] += 1
                bsk.decode_attention_bf16_enqueue(q, kc, vc, bt, sl, o, 1, nqh, nkv, hd, bs, nb, nb, L, 1.0 / 16.0,
                                                  segs)

            ms = time_chain_ahead(call, 20)
            gbs = kv_bytes / (ms * 1e-3) / 1e9
            row[name] = {"segments": segs, "us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                         "frac_of_hbm": round(gbs / hbm_peak, 4),
                         "per_call_events_us": round(time_device(call, 20) * 1e3, 2),
                         "us_host_paced": round(time_chain(call, 20) * 1e3, 2)}
        row["kv_copies"] = copies
        out[f"L{L}"] = row
        del k, v, kvs
    bsk.stream_check()
    return out


def run_ours(args):
    import numpy as np
    import torch

    from bf16_gemm_skinny_gb300 import _native as bsk
    from bf16_gemm_skinny_gb300 import build as bsk_build
    from bf16_gemm_skinny_gb300 import inputs

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    bsk_build.build()
    bsk.load()

    # ---- inputs: seeded, synthetic, shaped like the workload ----
    A_h, B_h = inputs.gemm_operands(GEMM_M, GEMM_N, GEMM_K, "uniform")
    W_h, _ = inputs.linear_operands(GEMV_M, GEMV_K, 1, "normal0.02", "normal1")
    xs_h = {n: inputs.linear_operands(1, GEMV_K, n, "normal0.02", "normal1")[1] for n in GEMV_NS}

    def pinned(a):
        t = torch.from_numpy(a.view(np.int16)).pin_memory()
        return t

    A_p, B_p, W_p = pinned(A_h), pinned(B_h), pinned(W_h)
    x_p = {n: pinned(xs_h[n]) for n in GEMV_NS}
    A = A_p.to(dev)
    B = B_p.to(dev)
    C = torch.empty(GEMM_M * GEMM_N, dtype=torch.int16, device=dev)
    Ws = [W_p.to(dev) for _ in range(3)]          # weight copies, rotated: consecutive launches differ
    xs = {n: x_p[n].to(dev) for n in GEMV_NS}
    ys = {n: torch.empty(n * GEMV_M, dtype=torch.int16, device=dev) for n in GEMV_NS}
    C_p = torch.empty(GEMM_M * GEMM_N, dtype=torch.int16).pin_memory()
    y_p = {n: torch.empty(n * GEMV_M, dtype=torch.int16).pin_memory() for n in GEMV_NS}
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev["g0"].record(stream)
        bsk.gemm_f16_colmajor_enqueue(A, B, C, GEMM_M, GEMM_N, GEMM_K, stream)
        if ev is not None:
            ev["g1"].record(stream)
        j = 0
        for n in GEMV_NS:
            if ev is not None:
                ev[f"v0_{n}"].record(stream)
            for _ in range(GEMV_CHAIN):
                bsk.gemv_bf16_enqueue(Ws[j % len(Ws)], xs[n], ys[n], GEMV_M, GEMV_K, n, stream)
                j += 1
            if ev is not None:
                ev[f"v1_{n}"].record(stream)

    for _ in range(args.warmup):
        step()
    bsk.stream_check(stream)
    torch.cuda.synchronize()
    barrier(dist, dev)

    keys = ["g0", "g1"] + [f"v{j}_{n}" for n in GEMV_NS for j in (0, 1)]
    evs = [{k: torch.cuda.Event(enable_timing=True) for k in keys} for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    bsk.stream_check(stream)
    barrier(dist, dev)

    total_ms = t_start.elapsed_time(t_end)
    gemm_ms = [e["g0"].elapsed_time(e["g1"]) for e in evs]
    gemv_ms = {n: [e[f"v0_{n}"].elapsed_time(e[f"v1_{n}"]) / GEMV_CHAIN for e in evs] for n in GEMV_NS}
    gemm_ms_mean = statistics.fmean(gemm_ms)

    def pct(values):
        v = sorted(values)
        q = lambda f: v[min(len(v) - 1, int(round(f * (len(v) - 1))))]  # noqa: E731
        return {"mean": round(statistics.fmean(v) * 1e3, 2), "p10": round(q(0.1) * 1e3, 2),
                "p50": round(q(0.5) * 1e3, 2), "p90": round(q(0.9) * 1e3, 2)}

    timing_us = {"gemm": pct(gemm_ms), **{f"gemv_n{n}": pct(v) for n, v in gemv_ms.items()}}
    total_ms_max = max_over_ranks(total_ms, dist, dev)
    gemv_ms_mean = {n: max_over_ranks(statistics.fmean(v), dist, dev) for n, v in gemv_ms.items()}

    # ---- end to end through the blocking C-ABI calls, host buffers ----
    e2e_steps = max(2, min(5, args.steps))
    barrier(dist, dev)
    torch.cuda.synchronize()
    e2e_gemm, e2e_gemv = [], {n: [] for n in GEMV_NS}
    for it in range(e2e_steps + 1):            # the first pass warms the copy paths, untimed
        t0 = time.perf_counter()
        bsk.gemm_f16_colmajor_host(A_p, B_p, C_p, GEMM_M, GEMM_N, GEMM_K, stream)
        if it:
            e2e_gemm.append(time.perf_counter() - t0)
        for n in GEMV_NS:
            t0 = time.perf_counter()
            bsk.gemv_bf16_host(W_p, x_p[n], y_p[n], GEMV_M, GEMV_K, n, stream)
            if it:
                e2e_gemv[n].append(time.perf_counter() - t0)
    e2e_gemm_s = max_over_ranks(statistics.median(e2e_gemm), dist, dev)
    # the blocking call alone (device buffers, host sync inside), wall clock
    blocking = []
    for it in range(e2e_steps + 1):
        t0 = time.perf_counter()
        bsk.gemm_f16_colmajor(A, B, C, GEMM_M, GEMM_N, GEMM_K, stream)
        if it:
            blocking.append(time.perf_counter() - t0)
    blocking_ms = max_over_ranks(statistics.median(blocking), dist, dev) * 1e3
    e2e_gemv_s = {n: max_over_ranks(statistics.median(v), dist, dev) for n, v in e2e_gemv.items()}
    # one GEMV launch right after a GEMM, bracketed on its own (events on both
    # sides stop the next launch from overlapping this one's tail), for each n
    single = {n: [] for n in GEMV_NS}
    single_steps = max(3, min(20, args.steps))
    sev = []
    for it in range(single_steps + 1):
        row = {}
        for i, n in enumerate(GEMV_NS):
            bsk.gemm_f16_colmajor_enqueue(A, B, C, GEMM_M, GEMM_N, GEMM_K, stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            bsk.gemv_bf16_enqueue(Ws[(it + i) % len(Ws)], xs[n], ys[n], GEMV_M, GEMV_K, n, stream)
            e1.record(stream)
            row[n] = (e0, e1)
        if it:
            sev.append(row)
    torch.cuda.synchronize()
    bsk.stream_check(stream)
    for row in sev:
        for n, (e0, e1) in row.items():
            single[n].append(e0.elapsed_time(e1))
    single_ms = {n: max_over_ranks(statistics.median(v), dist, dev) for n, v in single.items()}
    # The best CUDA-core GEMV kernel for each n, timed like the default (chains of
    # GEMV_CHAIN launches, median of five chains); the default runs n >= 4 on the
    # tensor-core skinny GEMM.
    cuda_core = {}
    for n in GEMV_NS:
        best = None
        for kern in (1, 2, 3, 4):
            if kern == 4 and n < 5:
                continue
            bsk.set_option("gemv_kernel", kern)
            it = [0]

            def call_cc(n=n, it=it):
                bsk.gemv_bf16_enqueue(Ws[it[0] % len(Ws)], xs[n], ys[n], GEMV_M, GEMV_K, n, stream)
                it[0] += 1

            ms = statistics.median(time_chain(call_cc, GEMV_CHAIN, warmup=1) for _ in range(5))
            if best is None or ms < best[1]:
                best = (kern, ms)
        bsk.set_option("gemv_kernel", 0)
        cuda_core[n] = (best[0], max_over_ranks(best[1], dist, dev))
    bsk.stream_check(stream)

    peaks, peak_src = load_peaks()
    value = whole_job_rate(gemm_flops(), gemm_ms_mean * 1e-3, dist, dev) / 1e12
    per_launch_tflops = gemm_flops() / (gemm_ms_mean * 1e-3) / 1e12
    gemm_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    kernel_names = {1: "register streaming", 2: "cp.async pipeline, x FP32", 3: "cp.async pipeline, x BF16",
                    4: "token-paired accumulators"}
    gemv = {}
    for n in GEMV_NS:
        gbs = gemv_bytes(n) / (gemv_ms_mean[n] * 1e-3) / 1e9
        kc, ms_cc = cuda_core[n]
        gemv[f"n{n}"] = {
            "achieved": round(world * gbs, 1), "frac": round(gbs / hbm_peak, 4),
            "us": round(gemv_ms_mean[n] * 1e3, 2),
            "single_launch_us": round(single_ms[n] * 1e3, 2),
            "single_launch_frac": round(gemv_bytes(n) / (single_ms[n] * 1e-3) / 1e9 / hbm_peak, 4),
            "kernel": ("gemv_bf16_kernel (CUDA cores, register streaming)" if n <= 3 else
                       "gemm_tcgen05_kernel<BN 32, K-major A, BF16> (tensor cores, 128 x 32 tiles)"),
            "cuda_core_best": {"kernel": kernel_names[kc], "us": round(ms_cc * 1e3, 2),
                               "frac": round(gemv_bytes(n) / (ms_cc * 1e-3) / 1e9 / hbm_peak, 4)},
            "e2e_gbs": round(world * gemv_bytes(n) / e2e_gemv_s[n] / 1e9, 1)}
    gemv_n1_gbs = gemv_bytes(1) / (gemv_ms_mean[1] * 1e-3) / 1e9

    h2d = (A.numel() + B.numel() + sum(W.numel() for W in Ws) + sum(x.numel() for x in xs.values())) * 2
    d2h = (C.numel() + sum(y.numel() for y in ys.values())) * 2
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms_max / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16/bf16 in, f32 accumulate",
        "data": "synthetic (seeded PCG64: GEMM A,B uniform[-1,1] FP16; W N(0,0.02), x N(0,1) BF16)",
        "config": {"workload": WORKLOAD, "gemm": [GEMM_M, GEMM_N, GEMM_K], "gemv": [GEMV_M, GEMV_K, list(GEMV_NS)],
                   "parallelism": f"replicas x{world}", "gemm_tile": [512, 256, 64],
                   "gemm_stage_bytes_per_sm": tile_stage_bytes(256, 128, 64),
                   "l2": "inputs larger than L2 (GEMM operands 537 MB; consecutive GEMV launches read different "
                         "356 MB weight copies, three in rotation)",
                   "gemv_timing": f"per-launch average over a chain of {GEMV_CHAIN} back-to-back launches per n "
                                  "(events at the chain's ends); single_launch_us: one launch after the GEMM with "
                                  "events on both sides"},
        "timing_us": timing_us,
        "blocking_call_ms": {"gemm_f16_colmajor": round(blocking_ms, 4)},
        "e2e": {"value": round(world * gemm_flops() / e2e_gemm_s / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "gemv_gbs": {f"n{n}": gemv[f"n{n}"].pop("e2e_gbs") for n in GEMV_NS},
                "note": "host-buffer C-ABI calls gemm_f16_colmajor_host / gemv_bf16_host on pinned memory: "
                        "H2D of A,B (GEMM) and W,x (GEMV), D2H of C / y inside the call, overlapped with the "
                        "compute in blocks"},
        "roofline": {"bound": "tensor", "achieved": round(per_launch_tflops, 2), "peak": gemm_peak,
                     "unit": "TFLOP/s", "frac": round(per_launch_tflops / gemm_peak, 4),
                     "frac_of_sustained": round(per_launch_tflops / float(
                         peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])), 4),
                     "traffic": committed_traffic("gemm_f16_8192x8192x16384"),
                     "peak_source": f"{peak_src} bf16_tflops (FP16 dense rate = BF16 on this part)",
                     "kernel": "gemm_tcgen05_pair_kernel<MN-major A, FP16, 2 row blocks> (CTA pairs, 512x256 tiles)"},
        "gpu_launches": args.steps * (1 + GEMV_CHAIN * len(GEMV_NS)),
        "clocks": clocks,
    }
    if not args.no_other_configs:
        line["other_configs"] = other_configs(Ws[0], dev, peaks)
        line["decode_attention"] = attention_configs(dev, hbm_peak)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(A_h, B_h, args.cpu_seconds)
    # Last on the line: the decode GEMV per n against the HBM roofline (the
    # top-level achieved / frac / traffic are n = 1's, the register-streaming
    # kernel).  `achieved` averages chains of GEMV_CHAIN back-to-back launches;
    # single_launch_* is one launch right after the GEMM between events;
    # cuda_core_best is the fastest CUDA-core kernel timed the same way.
    line["roofline_gemv"] = {"bound": "hbm", "achieved": round(gemv_n1_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                             "frac": round(gemv_n1_gbs / hbm_peak, 4),
                             "traffic": committed_traffic("gemv_bf16_34816x5120_n1"),
                             "peak_source": f"{peak_src} hbm_gbs", **gemv}
    if dist is not None:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return
    import oracle
    from bf16_gemm_skinny_gb300 import inputs

    oracle.build()
    A_h, B_h = inputs.gemm_operands(GEMM_M, GEMM_N, GEMM_K, "uniform")
    threads = oracle.max_threads()
    # size each step so that warm-up + timed steps take about `budget` seconds
    t0 = time.perf_counter()
    oracle.gemm_f16_colmajor(A_h, B_h, GEMM_M, GEMM_N, GEMM_K, cols=list(range(threads)))
    per_batch = time.perf_counter() - t0
    budget = 150.0
    batches = max(1, int(budget / max(per_batch, 1e-3) / (args.steps + args.warmup)))
    cols_per_step = batches * threads
    for w in range(args.warmup):
        oracle.gemm_f16_colmajor(A_h, B_h, GEMM_M, GEMM_N, GEMM_K, cols=[(w + i) % GEMM_N for i in range(threads)])
    times = []
    for s in range(args.steps):
        cols = [(s * 131 + i * 977) % GEMM_N for i in range(cols_per_step)]
        t0 = time.perf_counter()
        oracle.gemm_f16_colmajor(A_h, B_h, GEMM_M, GEMM_N, GEMM_K, cols=cols)
        times.append(time.perf_counter() - t0)
    flops_per_step = 2 * GEMM_M * GEMM_K * cols_per_step
    value = flops_per_step * len(times) / sum(times) / 1e12
    sample = (f"{cols_per_step} output columns of the 8192x8192x16384 GEMM per step "
              f"(each 8192x16384 FMAs in FP64)")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * statistics.fmean(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (seeded PCG64)",
        "config": {"workload": WORKLOAD, "gemm": [GEMM_M, GEMM_N, GEMM_K], "gemv": [GEMV_M, GEMV_K, list(GEMV_NS)],
                   "parallelism": "host cores"},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_case(args):
    """One kernel, one shape, `warmup + steps` launches, nothing else: the
    command the ncu summaries in profiles/ are taken with.
    Cases: gemm:MxNxK (FP16 column-major GEMM) or gemv:MxKxn (BF16 linear)."""
    import torch

    from bf16_gemm_skinny_gb300 import _native as bsk
    from bf16_gemm_skinny_gb300 import build as bsk_build
    from bf16_gemm_skinny_gb300 import inputs

    kind, shape = args.case.split(":")
    a, b, c = (int(v) for v in shape.lower().split("x"))
    bsk_build.build()
    for kv in args.opt or []:
        key, val = kv.split("=")
        bsk.set_option(key, int(val))
    dev = torch.device("cuda", 0)
    to_dev = lambda bits: torch.from_numpy(bits.view("int16")).to(dev)  # noqa: E731
    if kind == "gemm":
        A, B = inputs.gemm_operands(a, b, c, "uniform")
        Ad, Bd = to_dev(A), to_dev(B)
        C = torch.empty(a * b, dtype=torch.int16, device=dev)
        if args.layout:
            order, ta, tb, mode = (int(v) for v in args.layout.split(","))
            M, N, K = a, b, c
            lda = (K if ta else M) if order == 0 else (M if ta else K)
            ldb = (N if tb else K) if order == 0 else (K if tb else N)
            ldc = M if order == 0 else N
            bias = to_dev(inputs.to_f16_bits(inputs.draw("uniform", max(M, N), 41))) if mode else None
            call = lambda: bsk.gemm_f16_enqueue(order, ta, tb, Ad, lda, Bd, ldb, C, ldc, M, N, K,  # noqa: E731
                                                bias, mode)
        else:
            call = lambda: bsk.gemm_f16_colmajor_enqueue(Ad, Bd, C, a, b, c)  # noqa: E731
        work, unit = 2.0 * a * b * c, "TFLOP/s"
    elif kind == "fp8":
        # fp8:MxNxK -> E4M3 A (K-major), B (K-major), BF16 C
        A, B = inputs.fp8_operands(a, b, c, "normal1", "e4m3")
        Ad, Bd = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
        C = torch.empty(a * b, dtype=torch.int16, device=dev)
        call = lambda: bsk.gemm_fp8_enqueue(bsk.FP8_E4M3, Ad, c, Bd, c, C, a, bsk.OUT_BF16,  # noqa: E731
                                            a, b, c, 1.0)
        work, unit = 2.0 * a * b * c, "TFLOP/s"
    elif kind == "gemv":
        W, x = inputs.linear_operands(a, b, c, "normal0.02", "normal1")
        Wd, xd = to_dev(W), to_dev(x)
        y = torch.empty(a * c, dtype=torch.int16, device=dev)
        call = lambda: bsk.gemv_bf16_enqueue(Wd, xd, y, a, b, c)  # noqa: E731
        work, unit = 2.0 * (a * b + c * b + c * a), "GB/s"
    elif kind == "attn":
        # attn:L x segments x 0 -> 16 query / 4 KV heads, head_dim 256, 784-token pages
        L, segs = a, b
        nqh, nkv, hd, bs = 16, 4, 256, 784
        nb = -(-L // bs)
        n = nb * bs * nkv * hd
        kd = to_dev(inputs.to_bf16_bits(inputs.draw("normal1", n, 31)))
        vd = to_dev(inputs.to_bf16_bits(inputs.draw("normal1", n, 32)))
        qd = to_dev(inputs.to_bf16_bits(inputs.draw("normal1", nqh * hd, 33)))
        btd = torch.arange(nb, dtype=torch.int32, device=dev)
        sld = torch.tensor([L], dtype=torch.int32, device=dev)
        od = torch.empty(nqh * hd, dtype=torch.int16, device=dev)
        call = lambda: bsk.decode_attention_bf16_enqueue(  # noqa: E731
            qd, kd, vd, btd, sld, od, 1, nqh, nkv, hd, bs, nb, nb, L, 1.0 / 16.0, segs)
        work, unit = float(L * nkv * hd * 4), "GB/s"
    else:
        raise SystemExit(f"unknown case {args.case}")
    for _ in range(args.warmup):
        call()
    bsk.stream_check()
    if args.sustained:
        # back to back for `sustained` seconds (the power-capped regime), SM
        # clock sampled during the run
        torch.cuda.synchronize()
        sampler = ClockSampler(0)
        sampler.start()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        launches, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < args.sustained:
            for _ in range(50):
                call()
            launches += 50
            torch.cuda.synchronize()
        e1.record()
        torch.cuda.synchronize()
        clocks = sampler.stop()
        bsk.stream_check()
        ms = e0.elapsed_time(e1) / launches
        rate = work / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
        print(json.dumps({"case": args.case, "opt": args.opt or [], "sustained_s": args.sustained, "launches": launches,
                          "ms": round(ms, 4), unit: round(rate, 1), "clocks": clocks}), flush=True)
        return
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        call()
    e1.record()
    bsk.stream_check()
    ms = e0.elapsed_time(e1) / max(1, args.steps)
    rate = work / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
    print(json.dumps({"case": args.case, "ms": round(ms, 4), unit: round(rate, 1)}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="oracle CPU-baseline budget for the headline GEMM (about 2.5 s more per other workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip timing the 256^3, ragged and prefill workloads after the step")
    ap.add_argument("--case", help="profile mode: one kernel only, e.g. gemm:8192x8192x8192 or gemv:34816x5120x1")
    ap.add_argument("--opt", action="append", help="profile mode: library option name=value (repeatable)")
    ap.add_argument("--layout", help="profile mode, gemm case: run gemm_f16 with order,transa,transb,bias_mode "
                                     "(e.g. 0,0,1,2) instead of gemm_f16_colmajor")
    ap.add_argument("--sustained", type=float, default=0.0,
                    help="profile mode: run the case back to back for this many seconds, sampling the SM clock")
    args = ap.parse_args(argv)
    if args.case:
        run_case(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
