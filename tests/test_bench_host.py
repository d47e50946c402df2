"""Host logic of the bench (no GPU): the measurement arithmetic against the
figures the pages print, the multi-rank aggregation on a world-size-2 gloo
group, nvidia-smi sample parsing, and the gating of the profiled traffic."""

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


def test_job_throughput_is_weak_scaling_over_ranks():
    # Two ranks each ran 10 steps of 2 GFLOP; the slower took 1 s.
    assert bench.job_gflops(2e9, 10, 2, 1.0) == pytest.approx(40.0)
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # Rank r measured (1 + r) s for the timed steps and (10 - r) s e2e.
        t = bench.max_over_ranks([1.0 + rank, 10.0 - rank], dist, "cpu")
        v = bench.job_gflops(4e9, 5, world, t[0])
        out.put((rank, t, v))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_on_a_two_rank_gloo_group():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in results:
        assert t == [2.0, 10.0], (rank, t)          # slowest rank's times everywhere
        assert v == pytest.approx(4e9 * 5 * 2 / 2.0 / 1e9)


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


def test_profiled_traffic_is_reported_only_for_the_profiled_kernel():
    text = open(bench.PROFILE_SUMMARY).read()
    cfg = re.search(r"kernel_config:\s*(\S+)", text).group(1)
    src = re.search(r"kernel_source_sha256:\s*(\w+)", text).group(1)
    if src == bench.kernel_source_hash():
        assert bench.profiled_traffic(cfg) > 0
    else:
        assert bench.profiled_traffic(cfg) is None     # stale summary: no traffic claim
    assert bench.profiled_traffic("some_other_config") is None


def test_config_comparison_rejects_unknown_names_before_any_device_work():
    # Runs on a host without a GPU: the names are checked first.
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--shapes", "64x64x64",
                        "--compare-configs", "ffma2_128x256_k32_s4_ka,no_such_config"],
                       capture_output=True, text=True, cwd=ROOT, timeout=300)
    assert r.returncode != 0
    assert "no_such_config" in r.stderr and "ffma2_128x256_k32_s4_ka" in r.stderr
