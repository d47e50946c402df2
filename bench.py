"""SGEMM throughput bench (GFLOP/s and % of the GB300 FP32 FFMA peak).

python bench.py [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME | --shape MxNxK] [--config ID]
                [--op-a 0|1] [--op-b 0|1] [--alpha X] [--beta Y] [--batch B]
                [--extra-workloads NAME,...] [--noalloc] [--probe-fma]

A step is one C = A . B product of the workload (default: the 4096-cube,
N(0,1) inputs, seed 2) through the library's C ABI, inputs resident in HBM.
W untimed steps, then exactly K timed steps bracketed by a device
synchronisation; value = 2*M*N*K*K_steps / time. The library runs on one GPU:
a multi-rank launch (WORLD_SIZE > 1, or --gpus N > 1) prints an
"unavailable" line and measures nothing.

Also reported on the same JSON line:
  e2e           the same metric through the same call with host buffers:
                pinned host A, B copied in, C copied out, inside the timing
                (steps pipelined over two buffer sets and three streams; the
                serial figure is reported beside it);
  roofline      the main kernel's achieved FP32 FLOP/s (CUDA events on its
                stream) against the FFMA peak SMs x 128 lanes x 2 FLOP x max
                SM clock ("alu"-bound: the intensity is far above the HBM
                ridge), with DRAM traffic from the committed ncu record
                (profiles/ffma_tma_sq4096.json);
  cpu_baseline  the FP64 CPU oracle timed on this host's cores (count and CPU
                model stated): the whole product when it takes under ~30 s,
                else the sampled rows and columns the parity tests check,
                else a bounded row sample (--cpu-threads 1 gives the
                single-core figure);
  step_ms       median, best and mean device time of the timed steps;
  warm          for workloads that fit in L2 (timed with an L2 flush before
                every step), the same steps back to back without the flush;
  clocks        nvidia-smi samples taken during the timed region;
  workloads     the other named workloads (256^3, 1024^3, 4097x3001x2049,
                16384^3 by default with the 4096-cube headline), each timed
                the same way over at least min(K, 10) steps and half a
                second, with its own clock samples.
--impl reference times that oracle alone as the reference arm.

--probe-fma builds bench_fma_peak.cu and prints the FP32 FMA rate of one SM
(scalar FFMA and paired FFMA2, loop-invariant operands) against the nominal
128 lanes x 2 FLOP per clock, then exits.

With --op-a/--op-b/--alpha/--beta/--batch the step is instead one call of
the general form C_b = alpha * op(A_b) . op(B_b) + beta * C_b over `batch`
copies of the workload's operands (stored transposed where op = 1), FLOPs
batch * 2*M*N*K; the step includes any packing pass the call makes. The
host-buffer, tensor-core, CPU and extra-workload legs are then left out.
"""

from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time
import uuid

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

FP32_LANES_PER_SM = 128          # FP32 FMA units per SM (4 partitions x 32)
DEFAULT_SM_MAX_MHZ = 2070.0      # GB300 maximum SM clock
HEADLINE_WORKLOAD = "sq4096"
EXTRA_WORKLOADS = ("sq256", "sq1024", "rect4097x3001x2049", "sq16384")
L2_BYTES = 126.5 * 2 ** 20       # GB300 L2 capacity
# Machine-readable record of the ncu capture of the headline product kernel.
PROFILE_RECORD = os.path.join(ROOT, "profiles", "ffma_tma_sq4096.json")
# The separately reported tensor-core path: 3xTF32 on tcgen05, clusters of
# two CTAs sharing each B tile by TMA multicast.
TENSOR_CONFIG = "tf32x3_pair_128x256_k16_s4"
TENSOR_FALLBACK_CONFIG = "tf32x3_128x256_k16_s4"
KERNEL_SOURCES = [os.path.join(ROOT, "dense_fp32_matrix_07_gb300", "csrc", f)
                  for f in ("ffma_tma.cuh", "kernels_ffma_tma.cu", "kernels_ffma_tma_ktail.cu",
                            "kernels_ffma_tma_dep.cu", "ptx.cuh", "schedule.cuh", "schedule.cu")]


def product_flops(M: int, N: int, K: int) -> float:
    """2MNK: one multiply and one add per term of every output's dot product
    (Chapter 9: Optimised Matrix Multiplication, section 9.1: 2N^3 for N x N)."""
    return 2.0 * M * N * K


def compulsory_bytes(M: int, N: int, K: int) -> float:
    """4(MK + KN + MN): each FP32 element of A and B read once, C written once
    (section 9.1 counts 3N^2 elements, 12N^2 bytes, for N x N)."""
    return 4.0 * (M * K + K * N + M * N)


def intensity(M: int, N: int, K: int) -> float:
    """Arithmetic intensity in FLOP/byte (section 9.1: N/6 for N x N)."""
    return product_flops(M, N, K) / compulsory_bytes(M, N, K)


def job_gflops(flops_per_step: float, steps: int, seconds: float) -> float:
    """Throughput of `steps` products of `flops_per_step` FLOPs in `seconds`."""
    return flops_per_step * steps / seconds / 1e9


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code: `//` comments, trailing blanks and
    blank lines are left out, so a comment edit keeps the profiled DRAM
    figure valid while any code change drops it."""
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, encoding="utf-8") as f:
            for line in f:
                if '"' not in line:
                    line = line.split("//", 1)[0]
                line = line.rstrip()
                if line:
                    h.update(line.encode("utf-8") + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic(config_name: str):
    """DRAM bytes per launch of the headline product kernel from the
    committed ncu record, or None when the record is missing, is for another
    kernel configuration, or predates the current kernel source."""
    try:
        with open(PROFILE_RECORD) as f:
            rec = json.load(f)
        src, cfg, val = rec["kernel_source_sha256"], rec["kernel_config"], rec["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError, TypeError):
        return None
    if src != kernel_source_hash() or cfg != config_name or val is None:
        return None
    return float(val)


def call_launches(sg, cfg, M, N, K, lda, ldb, ldc, a, b, c, num_sms, config=-1, op_a=0, op_b=0,
                  alpha=1.0, beta=0.0, sa=0, sb=0, sc=0, batch=1):
    """(kernels of the library one sgemm_general_ex() call launches, as the
    library itself plans them; what runs beside the product, in words)."""
    rc, n = sg.sgemm_general_plan_launches(op_a, op_b, M, N, K, alpha, lda, sa, ldb, sb, beta, ldc, sc, batch,
                                           a, b, c, num_sms, config)
    if rc != 0:
        raise RuntimeError(f"plan: {sg.sgemm_error_string(rc)}")
    if not sg.sgemm_config_name(cfg).startswith("ffma"):
        return n, ([f"{2 * batch} 3xTF32 split passes ({batch} entries, one product launch each)"]
                   if sg.sgemm_config_name(cfg).startswith("tf32") else [])
    tail = sg.sgemm_plan_row_tail(cfg, M, N, K, batch)[1] > 0
    other = ["the layout pass (operand copies, counter zeroing)"] if n - 1 - tail > 0 else []
    return n, other + (["the last-rows kernel"] if tail else [])


def measured_tf32_tflops() -> tuple:
    """(TF32 dense tensor peak in TFLOP/s, basis): the measured BF16 burst
    peak scaled by the nominal TF32/BF16 ratio 1.1/2.25, else the profiling
    recipe's fallback BF16 figure (1.9 PFLOP/s) scaled the same way."""
    ratio = 1.1 / 2.25
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16 = float(json.load(f)["bf16_tflops"])
        return bf16 * ratio, f"measured BF16 {bf16:.1f} TF x 1.1/2.25 (nominal TF32/BF16)"
    except (OSError, KeyError, ValueError):
        return 1900.0 * ratio, "fallback BF16 1900 TF x 1.1/2.25 (nominal TF32/BF16)"


def measured_sm_max_mhz() -> float:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["sm_max_mhz"])
    except (OSError, KeyError, ValueError):
        return DEFAULT_SM_MAX_MHZ


class ClockSampler:
    """nvidia-smi sampling of the SM clock and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None
        self.t_start = self.t_end = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu=timestamp,{self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", self.gpu_id, "-lms", "10"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, start: bool):
        if start:
            self.t_start = time.time()
        else:
            self.t_end = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return parse_clock_samples(lines, self.t_start, self.t_end)


def parse_clock_samples(lines, t_start, t_end):
    """Summary of nvidia-smi CSV samples (the ClockSampler query fields):
    median SM clock and max SM clock over the samples inside [t_start,
    t_end] (host and nvidia-smi share the wall clock), plus every throttle
    reason seen active; the two samples nearest the window when the window
    was shorter than the sampling period; None without samples."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        # timestamp, index, clocks.sm, clocks.max.sm, power.draw, active,
        # hw_slowdown, hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
        if len(parts) < 10:
            continue
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            rows.append({"t": ts, "sm": float(parts[2]), "max": float(parts[3]),
                         "hw": parts[6], "hw_thermal": parts[7], "sw_thermal": parts[8],
                         "sw_power": parts[9]})
        except ValueError:
            continue
    if not rows:
        return None
    inside = [r for r in rows if t_start - 0.03 <= r["t"] <= t_end + 0.03]
    if not inside:
        mid = 0.5 * (t_start + t_end)
        inside = sorted(rows, key=lambda r: abs(r["t"] - mid))[:2]
    reasons = set()
    for r in inside:
        for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
            if r[key].lower().startswith("active"):
                reasons.add(name)
    return {"sm_mhz": statistics.median(r["sm"] for r in inside),
            "sm_max_mhz": max(r["max"] for r in inside),
            "samples": len(inside), "reasons": sorted(reasons)}


def nvsmi_gpu_id(dev, local: int) -> str:
    """nvidia-smi's id of this process's GPU (its UUID when torch knows it)."""
    import torch
    try:
        raw = torch.cuda.get_device_properties(dev).uuid
        b = raw.bytes if hasattr(raw, "bytes") else None
        u = str(uuid.UUID(bytes=bytes(b))) if b is not None and len(b) == 16 else str(raw)
        if re.fullmatch(r"(GPU-)?[0-9a-fA-F-]{36}", u):
            return u if u.startswith("GPU-") else "GPU-" + u
    except (AttributeError, RuntimeError, ValueError, TypeError):
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [p for p in vis.split(",") if p.strip()]
    return parts[local].strip() if local < len(parts) else str(local)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def host_cores() -> int:
    """CPU cores this process may run on (a launcher's OMP_NUM_THREADS=1 does
    not limit the oracle: the timing runs alone on rank 0)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


def run_reference(args, world, rank):
    """The reference arm: the FP64 CPU oracle over bounded samples of rows."""
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    w = shape_workload(args.shape) if args.shape else workloads.WORKLOADS[args.workload]
    oracle.build()
    oracle.set_num_threads(args.cpu_threads if args.cpu_threads > 0 else host_cores())
    A, B = workloads.make_workload(w)
    An, Bn = A.numpy(), B.numpy()
    # Size the steps so the whole run (warm-up + timed) takes about 90 s of
    # oracle time on this host's cores, at most 3 s per step.
    probe_rows = np.arange(min(w.M, oracle.num_threads()), dtype=np.int64)
    t0 = time.perf_counter()
    oracle.sgemm_rows(w.M, w.N, w.K, An, w.lda, Bn, w.ldb, probe_rows, want_abs=False)
    dt = max(time.perf_counter() - t0, 1e-4) / len(probe_rows)
    per_step = min(3.0, 90.0 / (args.steps + args.warmup))
    rows_per_step = int(max(1, min(w.M, per_step / dt)))
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        oracle.sgemm_rows(w.M, w.N, w.K, An, w.lda, Bn, w.ldb,
                          np.sort(rng.choice(w.M, rows_per_step, replace=False)), want_abs=False)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.sgemm_rows(w.M, w.N, w.K, An, w.lda, Bn, w.ldb,
                          np.sort(rng.choice(w.M, rows_per_step, replace=False)), want_abs=False)
    elapsed = time.perf_counter() - t0
    value = job_gflops(product_flops(rows_per_step, w.N, w.K), args.steps, elapsed)
    sample = f"{rows_per_step} random full rows of C per step ({rows_per_step}x{w.N}x{w.K})"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, "cpu_oracle_f64", l2="host CPU: no GPU cache involved"),
        "cpu_baseline": {"value": round(value, 3), "unit": "GFLOP/s", "cores": oracle.num_threads(),
                         "cpu_model": cpu_model(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


METRIC = "SGEMM GFLOP/s at N=4096 FP32 and % of GB300 FP32 FFMA peak"


def workload_config(w, kernel, l2=None):
    total = 4 * (w.M * w.lda + w.K * w.ldb + w.M * w.ldc)
    if l2 is None:
        l2 = (f"A+B+C = {total / 1e6:.0f} MB > {L2_BYTES / 1e6:.0f} MB L2, no flush"
              if total > L2_BYTES else
              f"A+B+C = {total / 1e6:.1f} MB: L2 flushed between steps")
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "lda": w.lda, "ldb": w.ldb,
            "ldc": w.ldc, "dist": w.dist, "seed": w.seed, "kernel": kernel, "l2": l2}


def cpu_baseline(w, A, B, threads=0, budget_s=30.0, min_s=10.0):
    """The oracle on this host's cores. The unit of work is the whole
    product when that fits in about `budget_s` seconds; otherwise the rows
    and columns of C that the parity tests check on a sampled workload;
    otherwise a bounded sample of full rows. The unit is repeated until at
    least `min_s` seconds have been timed. `threads` > 0 pins the oracle's
    thread count."""
    import numpy as np
    import oracle
    oracle.build()
    oracle.set_num_threads(threads if threads > 0 else host_cores())
    An, Bn = A.numpy(), B.numpy()
    probe = np.arange(min(w.M, oracle.num_threads()), dtype=np.int64)
    t0 = time.perf_counter()
    oracle.sgemm_rows(w.M, w.N, w.K, An, w.lda, Bn, w.ldb, probe, want_abs=False)
    per_row = max(time.perf_counter() - t0, 1e-4) / len(probe)
    if per_row * w.M <= budget_s:
        def unit():
            oracle.sgemm(w.M, w.N, w.K, An, w.lda, Bn, w.ldb, want_abs=False)
        done = product_flops(w.M, w.N, w.K)
        what = f"the whole product ({w.M}x{w.N}x{w.K})"
    elif w.sampled and per_row * (256 * (1 + w.N / w.M)) <= budget_s:
        rows = workloads.sample_indices(w.M, 256, w.seed + 1000)
        cols = workloads.sample_indices(w.N, 256, w.seed + 2000)

        def unit():
            oracle.sgemm_rows(w.M, w.N, w.K, An, w.lda, Bn, w.ldb, rows, want_abs=False)
            oracle.sgemm_cols(w.M, w.N, w.K, An, w.lda, Bn, w.ldb, cols, want_abs=False)
        done = product_flops(len(rows), w.N, w.K) + product_flops(w.M, len(cols), w.K)
        what = (f"the {len(rows)} rows and {len(cols)} columns of C the parity test checks "
                f"({len(rows)}x{w.N}x{w.K} + {w.M}x{len(cols)}x{w.K})")
    else:
        nrows = int(max(oracle.num_threads(), min(w.M, (budget_s / 3) / per_row)))
        rows = workloads.sample_indices(w.M, nrows, 77)

        def unit():
            oracle.sgemm_rows(w.M, w.N, w.K, An, w.lda, Bn, w.ldb, rows, want_abs=False)
        done = product_flops(len(rows), w.N, w.K)
        what = f"{len(rows)} sampled full rows of C ({len(rows)}x{w.N}x{w.K})"
    reps, dt = 0, 0.0
    t0 = time.perf_counter()
    while dt < min_s or reps == 0:
        unit()
        reps += 1
        dt = time.perf_counter() - t0
    return {"value": round(job_gflops(done, reps, dt), 3), "unit": "GFLOP/s",
            "cores": oracle.num_threads(), "cpu_model": cpu_model(), "kind": "oracle",
            "sample": f"{what} x {reps}, {dt:.1f} s"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the
    platform's processor string)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine() or "unknown"


FMA_PEAK_SRC = os.path.join(ROOT, "bench_fma_peak.cu")
FMA_PEAK_LIB = os.path.join(ROOT, "_build", "libfma_peak.so")


def run_fma_peak():
    """bench_fma_peak.cu on every SM: FP32 FLOP per clock per SM of scalar
    FFMA and paired FFMA2 loops against the nominal 128 lanes x 2 FLOP; one
    JSON line. Built here on demand (the library build never compiles it)."""
    import ctypes
    from dense_fp32_matrix_07_gb300 import build as _b
    os.makedirs(os.path.dirname(FMA_PEAK_LIB), exist_ok=True)
    if not os.path.exists(FMA_PEAK_LIB) or os.path.getmtime(FMA_PEAK_LIB) < os.path.getmtime(FMA_PEAK_SRC):
        tmp = FMA_PEAK_LIB + f".tmp{os.getpid()}"
        subprocess.run([_b._nvcc(), *_b.NVCC_FLAGS, "-shared", "-cudart", "static", FMA_PEAK_SRC, "-o", tmp,
                        "-lpthread", "-ldl", "-lrt"], check=True)
        os.replace(tmp, FMA_PEAK_LIB)
    lib = ctypes.CDLL(FMA_PEAK_LIB)
    d = ctypes.c_double
    lib.fma_peak_run.restype = ctypes.c_int
    lib.fma_peak_run.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(d), ctypes.POINTER(d), ctypes.POINTER(d)]
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out = {}
    for paired, name in ((0, "ffma"), (1, "ffma2")):
        ms, mhz, flops = d(), d(), d()
        rc = lib.fma_peak_run(paired, 5, ctypes.byref(ms), ctypes.byref(mhz), ctypes.byref(flops))
        if rc != 0:
            raise RuntimeError(f"fma peak probe {name}: CUDA error {rc}")
        per_clk = flops.value / (ms.value * 1e-3) / (mhz.value * 1e6) / sms
        out[name] = {"best_ms": round(ms.value, 4), "sm_mhz": round(mhz.value, 1),
                     "tflops": round(flops.value / (ms.value * 1e-3) / 1e12, 2),
                     "flop_per_clk_per_sm": round(per_clk, 1), "frac_of_256": round(per_clk / 256.0, 4)}
    print(json.dumps({"probe": "fp32_fma_peak", "sms": sms, "nominal_flop_per_clk_per_sm": 256,
                      "results": out}), flush=True)
    return 0


def parse_shape(text: str):
    """"MxNxK" -> (M, N, K), each a positive integer."""
    parts = text.lower().split("x")
    if len(parts) != 3 or not all(p.isdigit() and int(p) > 0 for p in parts):
        raise ValueError(f"shape {text!r} is not MxNxK with positive integers")
    return tuple(int(p) for p in parts)


def shape_workload(text: str):
    """An ad-hoc workload of the given shape: tight strides, N(0,1) inputs
    from seed 0 (the named workloads' recipe)."""
    M, N, K = parse_shape(text)
    return workloads.Workload(f"shape_{M}x{N}x{K}", M, N, K, K, N, N, "normal", 0)


def unavailable_multi_gpu(world: int, gpus: int) -> dict:
    """The line a multi-rank launch of the library's arm prints: the library
    and its bench run on one GPU; nothing is measured."""
    n = max(world, gpus)
    return {"impl": "ours", "metric": METRIC, "n_gpus": n, "value": None, "unit": "GFLOP/s",
            "unavailable": f"single-GPU library: {n} GPUs requested; the product is one GPU's "
                           "SGEMM, run one process per GPU for independent products"}


def time_steps(step, stream, steps, warmup, flush=None, min_seconds=0.0, max_steps=None, sampler=None):
    """Runs `warmup` untimed steps, then at least `steps` timed steps (more,
    up to `max_steps`, until about `min_seconds` of device time), each
    bracketed by CUDA events on `stream`, with an L2 flush before each when
    `flush` is given. Returns the per-step device times in ms and the clock
    summary of `sampler` over the timed region."""
    import torch
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    n = steps
    if min_seconds > 0:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        one = max(e0.elapsed_time(e1) / 1e3, 1e-6)
        n = max(steps, int(min_seconds / one) + 1)
        if max_steps:
            n = min(n, max_steps)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(True)
    for i in range(n):
        if flush is not None:
            flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(False)
    clocks = sampler.stop() if sampler else None
    return [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)], clocks


def measure_extra_workload(sg, w, dev, stream, steps, warmup, peak_tflops, gpu_id):
    """One named workload through sgemm() with the automatic configuration:
    operands drawn by the workloads recipe, at least min(`steps`, 10) timed
    steps and half a second of device time (L2 flushed between steps when
    A + B + C fit in it), its own clock samples. Returns the workloads entry."""
    import torch
    A, B = workloads.make_workload(w)
    dA, dB = A.to(dev), B.to(dev)
    del A, B
    dC = torch.empty((w.M, w.ldc), dtype=torch.float32, device=dev)
    sh = stream.cuda_stream
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    _, cfg, pa, pb = sg.sgemm_plan(w.M, w.N, w.K, w.lda, w.ldb, w.ldc, dA.data_ptr(), dB.data_ptr(),
                                   dC.data_ptr(), num_sms)
    a_addr, b_addr, c_addr = dA.data_ptr(), dB.data_ptr(), dC.data_ptr()
    total = 4 * (w.M * w.lda + w.K * w.ldb + w.M * w.ldc)
    flush = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=dev) if total <= L2_BYTES else None

    def step():
        r = sg.sgemm(w.M, w.N, w.K, dA.data_ptr(), w.lda, dB.data_ptr(), w.ldb, dC.data_ptr(), w.ldc, sh)
        if r != 0:
            raise RuntimeError(f"{w.name}: {sg.sgemm_error_string(r)}")

    sampler = ClockSampler(gpu_id)
    sampler.start()
    ms, clocks = time_steps(step, stream, min(steps, 10), warmup, flush, min_seconds=0.5, max_steps=5000,
                            sampler=sampler)
    if sg.sgemm_check_status(sh) != 0:
        raise RuntimeError(f"device status after the {w.name} steps")
    flops = product_flops(w.M, w.N, w.K)
    value = job_gflops(flops, len(ms), sum(ms) / 1e3)
    best = flops / (min(ms) * 1e-3) / 1e9
    l2 = "flushed between steps" if flush is not None else "A+B+C > L2, no flush"
    del dA, dB, dC, flush
    torch.cuda.empty_cache()
    return {"value": round(value, 1), "unit": "GFLOP/s", "config": sg.sgemm_config_name(cfg),
            "fp32_peak_pct": round(100.0 * value / 1e3 / peak_tflops, 2),
            "best_step_fp32_peak_pct": round(100.0 * best / 1e3 / peak_tflops, 2),
            "steps": len(ms),
            "launches_per_step": call_launches(sg, cfg, w.M, w.N, w.K, w.lda, w.ldb, w.ldc, a_addr, b_addr,
                                               c_addr, num_sms)[0],
            "step_ms": {"median": round(statistics.median(ms), 4), "best": round(min(ms), 4),
                        "mean": round(statistics.mean(ms), 4)},
            "l2": l2,
            "shape": {"M": w.M, "N": w.N, "K": w.K, "lda": w.lda, "ldb": w.ldb, "ldc": w.ldc,
                      "dist": w.dist, "seed": w.seed},
            "clocks": clocks}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=HEADLINE_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--shape", default="", metavar="MxNxK",
                    help="time an ad-hoc MxNxK product (tight strides, N(0,1) inputs, seed 0) "
                         "instead of a named workload")
    ap.add_argument("--config", type=int, default=-1, help="force a kernel config id")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="steps of each e2e leg (default: the timed steps up to 30, or about 0.25 s of "
                         "device time if that is more, so the first copy in and the last copy out weigh little)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-copy legs")
    ap.add_argument("--no-tf32x3", action="store_true",
                    help="skip the separately reported 3xTF32 tensor-core measurement")
    ap.add_argument("--extra-workloads", default=None, metavar="NAME[,NAME...]",
                    help="other named workloads to time in the same run (default: "
                         f"{','.join(EXTRA_WORKLOADS)} with the {HEADLINE_WORKLOAD} headline, none "
                         "otherwise; an empty string: none)")
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="oracle threads for cpu_baseline (default: all host cores)")
    ap.add_argument("--op-a", type=int, choices=(0, 1), default=0,
                    help="general form: A stored transposed (K x M)")
    ap.add_argument("--op-b", type=int, choices=(0, 1), default=0,
                    help="general form: B stored transposed (N x K)")
    ap.add_argument("--alpha", type=float, default=1.0, help="general form: alpha")
    ap.add_argument("--beta", type=float, default=0.0, help="general form: beta (C is read when nonzero)")
    ap.add_argument("--batch", type=int, default=1, help="general form: strided batch of this many products")
    ap.add_argument("--noalloc", action="store_true",
                    help="time the allocation-free entry point sgemm_noalloc instead of sgemm_ex")
    ap.add_argument("--probe-fma", action="store_true",
                    help="run the FP32 FMA peak microbench (bench_fma_peak.cu) and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.shape:
        try:
            parse_shape(args.shape)
        except ValueError as e:
            ap.error(str(e))
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if world > 1 or args.gpus > 1:
        # One GPU per product: no rank of a multi-rank launch touches a GPU.
        if rank == 0:
            print(json.dumps(unavailable_multi_gpu(world, args.gpus)), flush=True)
        return 0
    if args.probe_fma:
        return run_fma_peak()
    extra = list(EXTRA_WORKLOADS) if args.extra_workloads is None else \
        [x for x in args.extra_workloads.split(",") if x]
    unknown = [x for x in extra if x not in workloads.WORKLOADS]
    if unknown:
        ap.error(f"unknown workloads {unknown}")
    return run_ours(args, local, extra)


def run_ours(args, local, extra):
    import torch
    import dense_fp32_matrix_07_gb300 as sg

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = shape_workload(args.shape) if args.shape else workloads.WORKLOADS[args.workload]
    A, B = workloads.make_workload(w)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    general = args.op_a or args.op_b or args.alpha != 1.0 or args.beta != 0.0 or args.batch > 1
    if general or args.noalloc:
        # The host-buffer, tensor-core, CPU and extra-workload legs belong to
        # the plain sgemm() workload.
        args.no_e2e = args.no_tf32x3 = args.no_cpu_baseline = True
    if general and args.noalloc:
        raise SystemExit("--noalloc times the plain form only")
    if general or args.noalloc or args.config >= 0 or args.shape or \
            (args.extra_workloads is None and w.name != HEADLINE_WORKLOAD):
        extra = []
    if not general:
        dA, dB = A.to(dev), B.to(dev)
        dC = torch.empty((w.M, w.ldc), dtype=torch.float32, device=dev)
        rc, cfg, pa, pb = sg.sgemm_plan(w.M, w.N, w.K, w.lda, w.ldb, w.ldc, dA.data_ptr(),
                                        dB.data_ptr(), dC.data_ptr(), num_sms)
        if args.noalloc and sg.sgemm_config_name(cfg).endswith("_ka"):
            # sgemm_noalloc makes the transposed copy of A in its fixed 16 Mi-float
            # array when it fits beside a packed B, else runs the twin that reads A
            # as stored.
            r32 = lambda x: (x + 31) // 32 * 32
            if w.K * r32(w.M) + (w.K * r32(w.N) if pb else 0) > (16 << 20):
                cfg = sg.config_ids()[sg.sgemm_config_name(cfg)[:-3]]
                pa = int(dA.data_ptr() % 16 != 0 or w.lda % 4 != 0)
        # sgemm_noalloc launches one pass per packed operand and the product
        # (its stream-K counters are zeroed by a memset); sgemm_ex() what the
        # library plans for the call.
        if args.noalloc:
            launches_per_step = 1 + pa + pb
            other_launches = [f"{pa + pb} operand layout pass(es)"] if pa + pb else []
        else:
            launches_per_step, other_launches = call_launches(sg, cfg, w.M, w.N, w.K, w.lda, w.ldb, w.ldc,
                                                              dA.data_ptr(), dB.data_ptr(), dC.data_ptr(),
                                                              num_sms, args.config)
        total_bytes = 4 * (w.M * w.lda + w.K * w.ldb + w.M * w.ldc)
        flops = product_flops(w.M, w.N, w.K)

        def step():
            if args.noalloc:
                r = sg.sgemm_noalloc(w.M, w.N, w.K, dA.data_ptr(), w.lda, dB.data_ptr(), w.ldb,
                                     dC.data_ptr(), w.ldc, sh)
            else:
                r = sg.sgemm_ex(w.M, w.N, w.K, dA.data_ptr(), w.lda, dB.data_ptr(), w.ldb,
                                dC.data_ptr(), w.ldc, args.config, sh)
            if r != 0:
                raise RuntimeError(sg.sgemm_error_string(r))
    else:
        # The general form C_b = alpha * op(A_b) . op(B_b) + beta * C_b over
        # `batch` copies of the workload's operands, stored as op asks (A as
        # K x M when op_a = 1, B as N x K when op_b = 1) with tight strides.
        gA = (A[:, :w.K].t() if args.op_a else A[:, :w.K]).contiguous()
        gB = (B[:, :w.N].t() if args.op_b else B[:, :w.N]).contiguous()
        lda_g, ldb_g, ldc_g = gA.shape[1], gB.shape[1], w.N
        sa, sb, sc = gA.numel(), gB.numel(), w.M * w.N
        dA = gA.reshape(1, -1).to(dev).repeat(args.batch, 1)
        dB = gB.reshape(1, -1).to(dev).repeat(args.batch, 1)
        dC = torch.ones((args.batch, w.M, w.N), dtype=torch.float32, device=dev)
        # The configuration and operand packs of the step, as the library chooses them.
        rc, cfg, pa, pb = sg.sgemm_general_plan(args.op_a, args.op_b, w.M, w.N, w.K, args.alpha, lda_g, sa, ldb_g,
                                                sb, args.beta, ldc_g, sc, args.batch, dA.data_ptr(),
                                                dB.data_ptr(), dC.data_ptr(), num_sms, args.config)
        if rc != 0:
            raise SystemExit(f"general form: {sg.sgemm_error_string(rc)}")
        launches_per_step, other_launches = call_launches(
            sg, cfg, w.M, w.N, w.K, lda_g, ldb_g, ldc_g, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), num_sms,
            args.config, args.op_a, args.op_b, args.alpha, args.beta, sa, sb, sc, args.batch)
        total_bytes = 4 * args.batch * (sa + sb + sc)
        flops = args.batch * product_flops(w.M, w.N, w.K)

        def step():
            r = sg.sgemm_general_ex(args.op_a, args.op_b, w.M, w.N, w.K, args.alpha, dA.data_ptr(), lda_g, sa,
                                    dB.data_ptr(), ldb_g, sb, args.beta, dC.data_ptr(), ldc_g, sc, args.batch,
                                    args.config, sh)
            if r != 0:
                raise RuntimeError(sg.sgemm_error_string(r))
    if args.config >= 0:
        cfg = args.config
    cfg_name = sg.sgemm_config_name(cfg)

    flush = None
    if total_bytes <= L2_BYTES:
        flush = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=dev)

    gpu_id = nvsmi_gpu_id(dev, local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    t0 = time.perf_counter()
    kernel_ms, clocks = time_steps(step, stream, args.steps, args.warmup, flush, sampler=sampler)
    elapsed_host = time.perf_counter() - t0
    if sg.sgemm_check_status(sh) != 0:
        raise RuntimeError("device status after the timed region")
    step_s = sum(kernel_ms) / 1e3   # device time of the timed steps (flush excluded)
    value = job_gflops(flops, args.steps, step_s)

    # An L2-resident workload is also timed warm: the same steps back to
    # back, operands left in L2 by the previous step.
    warm = None
    if flush is not None:
        warm_steps = min(args.steps, 200)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(warm_steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        if sg.sgemm_check_status(sh) != 0:
            raise RuntimeError("device status after the warm steps")
        warm_s = ev0.elapsed_time(ev1) / 1e3
        warm = {"value": round(job_gflops(flops, warm_steps, warm_s), 1), "unit": "GFLOP/s",
                "steps": warm_steps, "ms_per_step": round(warm_s / warm_steps * 1e3, 4),
                "note": "back-to-back steps, no L2 flush between them"}

    # ---- e2e: host buffers, copies inside the timing ----
    # Every step copies A and B in from pinned host memory, runs the product
    # through the C ABI and copies C back. "serial" does the three in order
    # on one stream; "pipelined" is how a caller streams independent steps:
    # two buffer sets and three streams, so the copies of one step overlap
    # the product of another.
    # Each leg starts with a copy in and ends with a copy out that overlap no
    # product (about 1 ms at 4096^3): spread over the timed steps (at most
    # 30), or over about a quarter second of device time if that is more.
    if args.e2e_steps is not None:
        e2e_steps = max(2, args.e2e_steps)
    else:
        e2e_steps = max(2, min(args.steps, 30), int(0.25 / max(statistics.median(kernel_ms) / 1e3, 1e-6)))
    if not args.no_e2e:
        hA = A.pin_memory()
        hB = B.pin_memory()
        hC = [torch.empty((w.M, w.ldc), dtype=torch.float32).pin_memory() for _ in range(2)]
        dA2, dB2 = torch.empty_like(dA), torch.empty_like(dB)
        dC2 = torch.empty_like(dC)
        sets = [(dA, dB, dC), (dA2, dB2, dC2)]

    def product(a, b, c, stream_handle):
        r = sg.sgemm_ex(w.M, w.N, w.K, a.data_ptr(), w.lda, b.data_ptr(), w.ldb,
                        c.data_ptr(), w.ldc, args.config, stream_handle)
        if r != 0:
            raise RuntimeError(sg.sgemm_error_string(r))

    def e2e_serial(n):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(n):
            dA.copy_(hA, non_blocking=True)
            dB.copy_(hB, non_blocking=True)
            product(dA, dB, dC, sh)
            hC[0].copy_(dC, non_blocking=True)
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) / 1e3

    s_in, s_mm, s_out = (torch.cuda.Stream(dev) for _ in range(3))

    def e2e_pipelined(n):
        done_in = [torch.cuda.Event() for _ in range(2)]
        done_mm = [torch.cuda.Event() for _ in range(2)]
        done_out = [torch.cuda.Event() for _ in range(2)]
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for s_ in (s_in, s_mm, s_out):
            s_.wait_event(ev0)
        for i in range(n):
            k = i % 2
            a, b, c = sets[k]
            if i >= 2:
                s_in.wait_event(done_mm[k])      # the product reading a, b is done
            with torch.cuda.stream(s_in):
                a.copy_(hA, non_blocking=True)
                b.copy_(hB, non_blocking=True)
            done_in[k].record(s_in)
            s_mm.wait_event(done_in[k])
            if i >= 2:
                s_mm.wait_event(done_out[k])     # C of two steps ago has been read
            product(a, b, c, s_mm.cuda_stream)
            done_mm[k].record(s_mm)
            s_out.wait_event(done_mm[k])
            with torch.cuda.stream(s_out):
                hC[k].copy_(c, non_blocking=True)
            done_out[k].record(s_out)
        stream.wait_stream(s_out)
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) / 1e3

    e2e_value = serial_value = None
    if not args.no_e2e:
        e2e_serial(2)
        e2e_pipelined(2)
        torch.cuda.synchronize()
        serial_s = e2e_serial(e2e_steps)
        e2e_s = e2e_pipelined(e2e_steps)
        if sg.sgemm_check_status(sh) != 0:
            raise RuntimeError("device status after the e2e steps")
        e2e_value = job_gflops(flops, e2e_steps, e2e_s)
        serial_value = job_gflops(flops, e2e_steps, serial_s)

    # ---- the optional 3xTF32 tensor-core path, reported separately ----
    tc = None
    if not args.no_tf32x3 and args.config < 0:
        tc_name = TENSOR_CONFIG
        tc_cfg = sg.config_ids()[tc_name]
        tc_fallback = None

        def tc_step():
            r = sg.sgemm_ex(w.M, w.N, w.K, dA.data_ptr(), w.lda, dB.data_ptr(), w.ldb,
                            dC.data_ptr(), w.ldc, tc_cfg, sh)
            if r != 0:
                raise RuntimeError(sg.sgemm_error_string(r))

        tc_step()
        if sg.sgemm_check_status(sh) == sg.SGEMM_ERR_LAUNCH:
            # The cluster kernel found itself launched without its cluster
            # (a profiler that drops the cluster shape of a cooperative
            # launch does this) and wrote nothing: time the single-CTA
            # kernel instead and say so.
            tc_fallback = f"{tc_name} reported a launch without its cluster"
            tc_name = TENSOR_FALLBACK_CONFIG
            tc_cfg = sg.config_ids()[tc_name]
        for _ in range(3):
            tc_step()
        torch.cuda.synchronize()
        tc_steps = max(3, min(args.steps, 50))
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(tc_steps):
            if flush is not None:
                flush.zero_()
            tc_step()
        ev1.record(stream)
        torch.cuda.synchronize()
        if sg.sgemm_check_status(sh) != 0:
            raise RuntimeError("device status after the 3xTF32 steps")
        tc_s = ev0.elapsed_time(ev1) / 1e3
        tc_value = job_gflops(flops, tc_steps, tc_s)
        tf32_peak, tf32_basis = measured_tf32_tflops()
        tensor_tflops = 3 * flops * tc_steps / tc_s / 1e12   # three TF32 products per FP32 product
        tc = {"value": round(tc_value, 1), "unit": "GFLOP/s", "config": tc_name, "fallback": tc_fallback,
              "steps": tc_steps, "launches_per_step": 3,
              "note": "FP32 result from three TF32 tensor-core products (hi.hi + hi.lo + lo.hi), "
                      "same 1e-4 * sum|A_ik B_kj| tolerance; includes the split pre-passes",
              "roofline": {"bound": "tensor", "achieved": round(tensor_tflops, 1),
                           "peak": round(tf32_peak, 1), "unit": "TFLOP/s",
                           "frac": round(tensor_tflops / tf32_peak, 4), "peak_basis": tf32_basis}}

    sm_max = measured_sm_max_mhz()
    peak_tflops = num_sms * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12

    # ---- the other named workloads, each timed the same way ----
    extra_out = None
    if extra:
        del s_in, s_mm, s_out
        if not args.no_e2e:
            del dA2, dB2, dC2, sets
        torch.cuda.empty_cache()
        extra_out = {name: measure_extra_workload(sg, workloads.WORKLOADS[name], dev, stream, args.steps,
                                                  args.warmup, peak_tflops, gpu_id)
                     for name in extra}

    avg_launch_s = statistics.mean(kernel_ms) / 1e3
    achieved_tflops = flops / avg_launch_s / 1e12
    traffic = None if general else profiled_traffic(cfg_name)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GFLOP/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_s / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": dict(workload_config(w, cfg_name), entry="sgemm_noalloc") if args.noalloc else
                  workload_config(w, cfg_name) if not general else dict(
            workload_config(w, cfg_name, l2=(f"A+B+C = {total_bytes / 1e6:.1f} MB"
                                             + (": L2 flushed between steps" if flush is not None else " > L2, no flush"))),
            form={"op_a": args.op_a, "op_b": args.op_b, "alpha": args.alpha, "beta": args.beta,
                  "batch": args.batch}),
        "fp32_peak_pct": round(100.0 * value / 1e3 / peak_tflops, 2),
        "e2e": None if e2e_value is None else {"value": round(e2e_value, 1), "unit": "GFLOP/s",
                "h2d_bytes_per_step": int(hA.numel() * 4 + hB.numel() * 4),
                "d2h_bytes_per_step": int(hC[0].numel() * 4),
                "steps": e2e_steps,
                "mode": "pipelined: 2 buffer sets, H2D / product / D2H on 3 streams",
                "serial_value": round(serial_value, 1)},
        "step_ms": {"median": round(statistics.median(kernel_ms), 4), "best": round(min(kernel_ms), 4),
                    "mean": round(statistics.mean(kernel_ms), 4)},
        "warm": warm,
        "gpu_launches": args.steps * launches_per_step,
        "roofline": {"bound": "alu", "achieved": round(achieved_tflops, 3),
                     "peak": round(peak_tflops, 3), "unit": "TFLOP/s",
                     "frac": round(achieved_tflops / peak_tflops, 4),
                     "traffic": traffic,
                     "peak_basis": f"{num_sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 FLOP x "
                                   f"{sm_max:.0f} MHz (max SM clock)",
                     "achieved_basis": ("2MNK / mean CUDA-event time of one call: the product kernel"
                                        + (" with " + " and ".join(other_launches)
                                           if other_launches else "")
                                        + ", on the launching stream")},
        "clocks": clocks,
        "host_elapsed_s": round(elapsed_host, 3),
        "tensor_core_3xtf32": tc,
        "workloads": extra_out,
    }
    if clocks and clocks.get("sm_mhz"):
        line["roofline"]["frac_at_sampled_clock"] = round(
            achieved_tflops / (peak_tflops * clocks["sm_mhz"] / sm_max), 4)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, A, B, args.cpu_threads)
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
