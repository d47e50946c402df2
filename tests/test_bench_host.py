"""Host logic of the bench (no GPU): the measurement arithmetic against the
figures the pages print, the refusal of multi-rank launches (a world-size-2
torchrun with gloo ranks on the CPU), nvidia-smi sample parsing, the gating
of the profiled traffic, and the shape and workload arguments."""

import datetime
import json
import os
import re
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "page_figures.json")))


@pytest.mark.parametrize("n", [1, 16, 256, 1024, 4096])
def test_flop_and_byte_counts_match_the_pages(n):
    assert GOLDEN["flops_square"]["value"] == "2*N^3"
    assert GOLDEN["compulsory_bytes_square"]["value"] == "12*N^2"
    assert bench.product_flops(n, n, n) == 2 * n ** 3
    assert bench.compulsory_bytes(n, n, n) == 12 * n ** 2
    assert bench.intensity(n, n, n) == pytest.approx(n / 6)


def test_intensity_at_4096_is_the_pages_683():
    assert round(bench.intensity(4096, 4096, 4096)) == GOLDEN["intensity_n4096"]["value"]


def test_rectangular_counts():
    # 2MNK FLOPs and 4(MK+KN+MN) bytes for the 4097 x 3001 x 2049 workload.
    assert bench.product_flops(4097, 3001, 2049) == 2 * 4097 * 3001 * 2049
    assert bench.compulsory_bytes(4097, 3001, 2049) == 4 * (4097 * 2049 + 2049 * 3001 + 4097 * 3001)


def test_simple_kernel_tile_footprint_is_the_pages_2176_bytes():
    # The predicated 16x16 kernel keeps the page's padded [16][17] tiles; its
    # static shared memory, as ptxas reports it, must be 2 * 16 * 17 * 4.
    from dense_fp32_matrix_07_gb300 import build as b
    src = os.path.join(b.CSRC, "kernels_basic.cu")
    r = subprocess.run([b._nvcc(), *b.NVCC_FLAGS, "-Xptxas", "-v", "-I", b.INCLUDE, "-c", src,
                        "-o", os.devnull], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    log = r.stdout + r.stderr
    block = log[log.index("sgemm_tiled_simple_kernel"):]
    smem = int(re.search(r"(\d+) bytes smem", block).group(1))
    assert smem == GOLDEN["padded_tile16_smem_bytes"]["value"]


def test_job_throughput():
    # 10 steps of 2 GFLOP in 1 s.
    assert bench.job_gflops(2e9, 10, 1.0) == pytest.approx(20.0)


def test_multi_rank_launch_measures_nothing(monkeypatch, capsys):
    # A world-size-2 launch of the library's arm prints one "unavailable" line
    # from rank 0 and returns before any device work, so no kernel of the
    # library (the cluster-pair tensor kernel included) can run on 2 GPUs.
    def no_device_work(*a, **k):
        raise AssertionError("a multi-rank launch reached the device path")

    monkeypatch.setattr(bench, "run_ours", no_device_work)
    monkeypatch.setattr(bench, "run_fma_peak", no_device_work)
    for rank in ("0", "1"):
        monkeypatch.setenv("WORLD_SIZE", "2")
        monkeypatch.setenv("RANK", rank)
        monkeypatch.setenv("LOCAL_RANK", rank)
        monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "2", "--steps", "3", "--warmup", "3"])
        assert bench.main() == 0
        out = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
        if rank == "0":
            assert len(out) == 1
            d = json.loads(out[0])
            assert d["value"] is None and d["n_gpus"] == 2 and "single-GPU" in d["unavailable"]
        else:
            assert out == []
    # --gpus 2 without a launcher is refused the same way.
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "2", "--probe-fma"])
    assert bench.main() == 0
    assert "unavailable" in capsys.readouterr().out


def test_two_rank_torchrun_launch_prints_one_line():
    # The launch the multi-GPU contract uses, on CPU gloo ranks: one line,
    # from rank 0, and neither rank loads the CUDA library.
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(29600 + os.getpid() % 300),
                        os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, cwd=ROOT, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1 and json.loads(lines[0])["unavailable"]
    assert "libsgemm" not in r.stderr


def _sample(ts, sm, active="Not Active", power_cap="Not Active"):
    stamp = datetime.datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{stamp}, 0, {sm}, 2070, 900.0, 0x0, {active}, Not Active, Not Active, {power_cap}\n"


def test_clock_samples_are_filtered_to_the_timed_window():
    t0 = 1_800_000_000.0
    lines = [_sample(t0 - 1.0, 1000),                      # before: idle
             _sample(t0 + 0.1, 2070), _sample(t0 + 0.2, 2050, power_cap="Active"),
             _sample(t0 + 0.3, 2070),
             _sample(t0 + 2.0, 900, active="Active")]     # after: ignored
    c = bench.parse_clock_samples(lines, t0, t0 + 0.35)
    assert c == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 3, "reasons": ["sw_power_cap"]}


def test_short_windows_take_the_nearest_samples():
    t0 = 1_800_000_000.0
    lines = [_sample(t0 - 0.2, 2000), _sample(t0 + 0.3, 2040), _sample(t0 + 5, 800)]
    c = bench.parse_clock_samples(lines, t0 + 0.1, t0 + 0.11)
    assert c["samples"] == 2 and c["sm_mhz"] == 2020.0
    assert bench.parse_clock_samples(["garbage\n"], t0, t0 + 1) is None


def test_profiled_traffic_is_reported_only_for_the_profiled_kernel(tmp_path, monkeypatch):
    rec = json.load(open(bench.PROFILE_RECORD))
    cfg, src = rec["kernel_config"], rec["kernel_source_sha256"]
    if src == bench.kernel_source_hash() and rec["dram_bytes_per_launch"] is not None:
        assert bench.profiled_traffic(cfg) > 0
    else:
        assert bench.profiled_traffic(cfg) is None     # stale record: no traffic claim
    assert bench.profiled_traffic("some_other_config") is None
    # A record of the current source gives its figure; a changed source drops it.
    fake = tmp_path / "rec.json"
    fake.write_text(json.dumps({"kernel_config": "k", "kernel_source_sha256": bench.kernel_source_hash(),
                                "dram_bytes_per_launch": 1.5e8}))
    monkeypatch.setattr(bench, "PROFILE_RECORD", str(fake))
    assert bench.profiled_traffic("k") == 1.5e8
    fake.write_text(json.dumps({"kernel_config": "k", "kernel_source_sha256": "0" * 16,
                                "dram_bytes_per_launch": 1.5e8}))
    assert bench.profiled_traffic("k") is None


def test_shape_argument_gives_a_tight_normal_workload():
    w = bench.shape_workload("2432x2048x16384")
    assert (w.M, w.N, w.K, w.lda, w.ldb, w.ldc, w.dist, w.seed) == (2432, 2048, 16384, 16384, 2048, 2048,
                                                                       "normal", 0)
    for bad in ("12x3", "0x4x4", "axbxc", "4x4x4x4"):
        with pytest.raises(ValueError):
            bench.parse_shape(bad)


def test_unknown_extra_workload_is_rejected_before_any_device_work():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--extra-workloads", "sq256,nope"],
                       capture_output=True, text=True, cwd=ROOT, timeout=300)
    assert r.returncode != 0 and "nope" in r.stderr


def test_cpu_model_is_named():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_gpu_launches_follow_the_library_plan():
    """bench.py counts the library's launches per step from the library's own
    host-only plan: the product, the layout pass (operands to lay out or
    counters to zero), the last-rows kernel; 3xTF32 two splits and the
    product per entry."""
    import dense_fp32_matrix_07_gb300 as sg

    def plain(M, N, K, lda, ldb, ldc, config=-1):
        _, cfg, _, _ = sg.sgemm_general_plan(0, 0, M, N, K, 1.0, lda, 0, ldb, 0, 0.0, ldc, 0, 1, 0, 0, 0, 152,
                                             config)
        return bench.call_launches(sg, cfg, M, N, K, lda, ldb, ldc, 0, 0, 0, 152, config)

    n, other = plain(4096, 4096, 4096, 4096, 4096, 4096)
    assert n == 2 and other == ["the layout pass (operand copies, counter zeroing)"]
    n, other = plain(4097, 3001, 2049, 2049, 3001, 3001)
    assert n == 3 and other[-1] == "the last-rows kernel"
    assert plain(1536, 1536, 1536, 1536, 1536, 1536) == (1, [])
    assert plain(256, 256, 256, 256, 256, 256) == (1, [])
    tf = sg.config_ids()["tf32x3_pair_128x256_k16_s4"]
    _, cfg, _, _ = sg.sgemm_general_plan(0, 0, 512, 512, 512, 1.0, 512, 512 * 512, 512, 512 * 512, 0.0, 512,
                                         512 * 512, 2, 0, 0, 0, 152, tf)
    n, other = bench.call_launches(sg, cfg, 512, 512, 512, 512, 512, 512, 0, 0, 0, 152, tf, sa=512 * 512,
                                   sb=512 * 512, sc=512 * 512, batch=2)
    assert n == 6 and "3xTF32 split passes" in other[0]
