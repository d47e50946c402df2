"""SGEMM throughput bench (GFLOP/s and % of the GB300 FP32 FFMA peak).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME] [--config ID]

A step is one C = A . B product of the workload (default: the 4096-cube,
N(0,1) inputs, seed 2) through the library's C ABI, inputs resident in HBM.
W untimed steps, then exactly K timed steps bracketed by a barrier and a
device synchronisation; value = 2*M*N*K*K_steps*ranks / max-over-ranks time.
Multi-GPU runs are independent replicas (one per rank, no collective on the
data path): scaling is weak.

Also reported on the same JSON line:
  e2e           the same metric through the same call with host buffers:
                pinned host A, B copied in, C copied out, inside the timing;
  roofline      the main kernel's achieved FP32 FLOP/s (CUDA events on its
                stream) against the FFMA peak SMs x 128 lanes x 2 FLOP x max
                SM clock ("alu"-bound: the intensity is far above the HBM
                ridge), with DRAM traffic from the committed ncu summary;
  cpu_baseline  the FP64 CPU oracle timed on this host's cores over a bounded
                sample of C's rows;
  clocks        nvidia-smi samples taken during the timed region.
--impl reference times that oracle alone as the reference arm.
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
L2_BYTES = 126.5 * 2 ** 20       # GB300 L2 capacity
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "ffma_tma_sq4096.md")
KERNEL_SOURCES = [os.path.join(ROOT, "dense_fp32_matrix_07_gb300", "csrc", f)
                  for f in ("kernels_ffma_tma.cu", "ptx.cuh")]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(config_name: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    summary is missing, is for another kernel config, or predates the
    current kernel source."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    src = re.search(r"kernel_source_sha256:\s*(\w+)", text)
    cfg = re.search(r"kernel_config:\s*(\S+)", text)
    val = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (src and cfg and val):
        return None
    if src.group(1) != kernel_source_hash() or cfg.group(1) != config_name:
        return None
    return float(val.group(1))


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
                 "-i", self.gpu_id, "-lms", "50"],
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
        rows = []
        for line in open(self.path):
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
        os.unlink(self.path)
        if not rows:
            return None
        # Samples taken inside the timed region (host and nvidia-smi share the
        # clock); if the region was shorter than the sampling period, the
        # samples nearest to it.
        inside = [r for r in rows if self.t_start - 0.03 <= r["t"] <= self.t_end + 0.03]
        if not inside:
            mid = 0.5 * (self.t_start + self.t_end)
            inside = sorted(rows, key=lambda r: abs(r["t"] - mid))[:2]
        load = inside
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["max"] for r in load),
                "samples": len(load), "reasons": sorted(reasons)}


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


def run_reference(args, world, rank):
    """The reference arm: the FP64 CPU oracle over bounded samples of rows."""
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    w = workloads.WORKLOADS[args.workload]
    oracle.build()
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
    flops = 2.0 * rows_per_step * w.N * w.K * args.steps
    value = flops / elapsed / 1e9
    sample = f"{rows_per_step} random full rows of C per step ({rows_per_step}x{w.N}x{w.K})"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, "cpu_oracle_f64", l2="host CPU: no GPU cache involved"),
        "cpu_baseline": {"value": round(value, 3), "unit": "GFLOP/s", "cores": oracle.num_threads(),
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


def cpu_baseline(w, A, B):
    """The oracle on this host's cores over a bounded sample (~10 s) of rows."""
    import numpy as np
    import oracle
    oracle.build()
    An, Bn = A.numpy(), B.numpy()
    probe = np.arange(min(w.M, oracle.num_threads()), dtype=np.int64)
    t0 = time.perf_counter()
    oracle.sgemm_rows(w.M, w.N, w.K, An, w.lda, Bn, w.ldb, probe, want_abs=False)
    per_row = max(time.perf_counter() - t0, 1e-4) / len(probe)
    nrows = int(max(oracle.num_threads(), min(w.M, 10.0 / per_row)))
    rows = workloads.sample_indices(w.M, nrows, 77)
    t0 = time.perf_counter()
    oracle.sgemm_rows(w.M, w.N, w.K, An, w.lda, Bn, w.ldb, rows, want_abs=False)
    dt = time.perf_counter() - t0
    return {"value": round(2.0 * len(rows) * w.N * w.K / dt / 1e9, 3), "unit": "GFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{len(rows)} sampled full rows of C ({len(rows)}x{w.N}x{w.K}), {dt:.1f} s"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="sq4096", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--config", type=int, default=-1, help="force a kernel config id")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()

    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    import dense_fp32_matrix_07_gb300 as sg

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    def barrier():
        if pg is not None:
            pg.barrier()

    w = workloads.WORKLOADS[args.workload]
    A, B = workloads.make_workload(w)
    dA, dB = A.to(dev), B.to(dev)
    dC = torch.empty((w.M, w.ldc), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rc, cfg, pa, pb = sg.sgemm_plan(w.M, w.N, w.K, w.lda, w.ldb, w.ldc, dA.data_ptr(),
                                    dB.data_ptr(), dC.data_ptr(), num_sms)
    if args.config >= 0:
        cfg = args.config
    cfg_name = sg.sgemm_config_name(cfg)
    launches_per_step = 1 + pa + pb
    flops = 2.0 * w.M * w.N * w.K

    total_bytes = 4 * (w.M * w.lda + w.K * w.ldb + w.M * w.ldc)
    flush = None
    if total_bytes <= L2_BYTES:
        flush = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=dev)

    def step():
        r = sg.sgemm_ex(w.M, w.N, w.K, dA.data_ptr(), w.lda, dB.data_ptr(), w.ldb,
                        dC.data_ptr(), w.ldc, args.config, sh)
        if r != 0:
            raise RuntimeError(sg.sgemm_error_string(r))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if sg.sgemm_check_status(sh) != 0:
        raise RuntimeError("device status after warm-up")

    sampler = ClockSampler(nvsmi_gpu_id(dev, local))
    if rank == 0:
        sampler.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    sampler.mark(True)
    t0 = time.perf_counter()
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier()
    elapsed_host = time.perf_counter() - t0
    sampler.mark(False)
    clocks = sampler.stop() if rank == 0 else None
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    step_s = sum(kernel_ms) / 1e3   # device time of the timed steps (flush excluded)
    if flush is None:
        step_s = max(step_s, starts[0].elapsed_time(ends[-1]) / 1e3)
    if sg.sgemm_check_status(sh) != 0:
        raise RuntimeError("device status after the timed region")

    t_max = step_s
    if pg is not None:
        t = torch.tensor([step_s], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        t_max = float(t.item())
    value = flops * args.steps * world / t_max / 1e9

    # ---- e2e: host buffers, copies inside the timing ----
    hA = A.pin_memory()
    hB = B.pin_memory()
    hC = torch.empty((w.M, w.ldc), dtype=torch.float32).pin_memory()
    e2e_steps = max(1, min(args.e2e_steps, args.steps))

    def e2e_step():
        dA.copy_(hA, non_blocking=True)
        dB.copy_(hB, non_blocking=True)
        step()
        hC.copy_(dC, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    e2e_s = ev0.elapsed_time(ev1) / 1e3
    if pg is not None:
        t = torch.tensor([e2e_s], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        e2e_s = float(t.item())
    e2e_value = flops * e2e_steps * world / e2e_s / 1e9

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return 0

    sm_max = measured_sm_max_mhz()
    peak_tflops = num_sms * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    avg_launch_s = statistics.mean(kernel_ms) / 1e3
    achieved_tflops = flops / avg_launch_s / 1e12
    traffic = profiled_traffic(cfg_name)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_max / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(w, cfg_name),
        "fp32_peak_pct": round(100.0 * value / world / 1e3 / peak_tflops, 2),
        "e2e": {"value": round(e2e_value, 1), "unit": "GFLOP/s",
                "h2d_bytes_per_step": int(hA.numel() * 4 + hB.numel() * 4),
                "d2h_bytes_per_step": int(hC.numel() * 4)},
        "gpu_launches": args.steps * launches_per_step,
        "roofline": {"bound": "alu", "achieved": round(achieved_tflops, 3),
                     "peak": round(peak_tflops, 3), "unit": "TFLOP/s",
                     "frac": round(achieved_tflops / peak_tflops, 4),
                     "traffic": traffic,
                     "peak_basis": f"{num_sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 FLOP x "
                                   f"{sm_max:.0f} MHz (max SM clock)"},
        "clocks": clocks,
        "host_elapsed_s": round(elapsed_host, 3),
    }
    if clocks and clocks.get("sm_mhz"):
        line["roofline"]["frac_at_sampled_clock"] = round(
            achieved_tflops / (peak_tflops * clocks["sm_mhz"] / sm_max), 4)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, A, B)
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
