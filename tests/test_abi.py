"""C-ABI library: loads without a GPU, exports every declared symbol, and its
host-only logic (status strings, config table, the planner) behaves. No
compute call is made here."""

import ctypes
import os
import re

import pytest

import dense_fp32_matrix_07_gb300 as sg

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "sgemm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sgemm\w*)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_functions():
    assert declared_functions() == sorted(sg.EXPORTED)


def test_library_exports_every_declared_symbol(sgemm_lib):
    for name in declared_functions():
        assert hasattr(sgemm_lib, name), name
        assert isinstance(getattr(sgemm_lib, name), ctypes._CFuncPtr)


def test_library_links_no_cuda_driver_or_runtime_dynamically():
    # The CUDA runtime is linked statically and the driver is reached through
    # the runtime's entry-point query, so the library loads on any host.
    import subprocess
    out = subprocess.run(["ldd", sg.library_path()], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out and "libcudart" not in out, out


def test_error_strings():
    for code in range(8):
        s = sg.sgemm_error_string(code)
        assert s and s != "unknown sgemm status code"
    assert sg.sgemm_error_string(99) == "unknown sgemm status code"
    assert sg.sgemm_error_string(sg.SGEMM_ERR_TIMEOUT).startswith("SGEMM_ERR_TIMEOUT")


def test_config_table():
    n = sg.sgemm_num_configs()
    assert n >= 2
    names = [sg.sgemm_config_name(i) for i in range(n)]
    assert len(set(names)) == n and "?" not in names
    assert names[0] == "tiled16_simple"
    assert sg.sgemm_config_name(n) == "?" and sg.sgemm_config_name(-1) == "?"


@pytest.mark.parametrize("args,code", [
    ((-1, 4, 4, 4, 4, 4), sg.SGEMM_ERR_INVALID_VALUE),
    ((4, -1, 4, 4, 4, 4), sg.SGEMM_ERR_INVALID_VALUE),
    ((4, 4, -1, 4, 4, 4), sg.SGEMM_ERR_INVALID_VALUE),
    ((4, 4, 4, 3, 4, 4), sg.SGEMM_ERR_INVALID_VALUE),   # lda < K
    ((4, 4, 4, 4, 3, 4), sg.SGEMM_ERR_INVALID_VALUE),   # ldb < N
    ((4, 4, 4, 4, 4, 3), sg.SGEMM_ERR_INVALID_VALUE),   # ldc < N
    ((4, 4, 0, 0, 4, 4), sg.SGEMM_OK),                  # K = 0: lda, ldb unused
    ((0, 4, 4, 0, 0, 0), sg.SGEMM_OK),                  # M = 0: nothing to do
    ((2 ** 31, 4, 4, 4, 4, 4), sg.SGEMM_ERR_OVERFLOW),  # beyond 32-bit coordinates
    ((2 ** 30, 4, 4, 2 ** 62, 4, 4), sg.SGEMM_ERR_OVERFLOW),  # byte extent overflows
])
def test_plan_validates_sizes(args, code):
    rc, *_ = sg.sgemm_plan(*args, 0, 0, 0, 148)
    assert rc == code


def test_plan_packs_only_misaligned_operands():
    # Aligned operands with 16-byte rows: read in place by the row-major
    # 128x256 configuration (N below 2048)...
    rc, cfg, pa, pb = sg.sgemm_plan(65536, 1024, 1024, 1024, 1024, 1024, 0, 0, 0, 148)
    assert rc == 0 and sg.sgemm_config_name(cfg) == "ffma2_128x256_k32_s4" and (pa, pb) == (0, 0)
    # ...while the k-major configuration (N >= 2048) reads B in place and
    # transposes A into scratch.
    rc, cfg, pa, pb = sg.sgemm_plan(4096, 4096, 4096, 4096, 4096, 4096, 0, 0, 0, 148)
    assert rc == 0 and sg.sgemm_config_name(cfg) == "ffma2_128x256_k32_s4_ka" and (pa, pb) == (1, 0)
    # Rows that are not a multiple of 16 bytes (the 4097x3001x2049 workload).
    rc, cfg, pa, pb = sg.sgemm_plan(4097, 3001, 2049, 2049, 3001, 3001, 0, 0, 0, 148)
    assert rc == 0 and (pa, pb) == (1, 1)
    # A misaligned base address alone forces a pack of that operand.
    rc, cfg, pa, pb = sg.sgemm_plan(1024, 1024, 1024, 1024, 1024, 1024, 4, 0, 0, 148)
    assert rc == 0 and (pa, pb) == (1, 0)
    rc, cfg, pa, pb = sg.sgemm_plan(1024, 1024, 1024, 1024, 1024, 1024, 0, 8, 12, 148)
    assert rc == 0 and (pa, pb) == (0, 1)
    # The small-product kernel reads any layout in place.
    rc, cfg, pa, pb = sg.sgemm_plan(256, 256, 256, 256, 256, 256, 4, 8, 12, 148)
    assert rc == 0 and sg.sgemm_config_name(cfg) == "small_32x32_k256" and (pa, pb) == (0, 0)


@pytest.mark.parametrize("n,name", [
    (256, "small_32x32_k256"),          # small: no TMA set-up, 32x32 tiles, each K panel loaded at once
    (384, "small_32x32_k256"),
    (512, "ffma2_128x64_k32_s4"),       # 16 tiles of 128x128: the smallest TMA tiles
    (1024, "ffma2_128x128_k32_s4"),     # 64 tiles of 128x128 (>= a third of the SMs)
    (2048, "ffma2_128x128_k32_s4_ka"),  # 128 tiles of 128x256 < 148 SMs; N >= 2048: A k-major
    (4096, "ffma2_128x256_k32_s4_ka"),  # 512 tiles of 128x256, N >= 2048: A k-major
])
def test_plan_tile_size_follows_the_problem(n, name):
    rc, cfg, *_ = sg.sgemm_plan(n, n, n, n, n, n, 0, 0, 0, 148)
    assert rc == 0 and sg.sgemm_config_name(cfg) == name


@pytest.mark.parametrize("M,N,K,name", [
    (512, 512, 256, "small_32x32_k256"),            # C of 2^18, K 256: the small-product kernel
    (1024, 1024, 64, "ffma2_128x128_k32_s4"),       # C of 2^20: TMA tiles, although M*N*K = 2^26
    (256, 256, 1024, "ffma2_128x64_k32_s4"),        # K 1024: TMA tiles (stream-K), M*N*K = 2^26
    (2048, 2048, 512, "ffma2_128x128_k32_s4"),      # M*N*K = 2.1e9: the transpose pass would not pay
    (4096, 4096, 256, "ffma2_128x256_k32_s4"),      # 4.3e9: the same on 128x256 tiles
    (1536, 2048, 2048, "ffma2_128x128_k32_s4_ka"),  # 6.4e9 and N >= 2048: A k-major
    (4096, 1536, 4096, "ffma2_128x256_k32_s4"),     # N < 2048 at any size: A read as stored
])
def test_plan_takes_the_kmajor_pass_only_when_it_pays(M, N, K, name):
    rc, cfg, pa, _ = sg.sgemm_plan(M, N, K, K, N, N, 0, 0, 0, 152)
    assert rc == 0 and sg.sgemm_config_name(cfg) == name and pa == (1 if name.endswith("_ka") else 0)


def test_plan_long_k_skips_the_simple_kernel():
    # A tiny output with a long K goes to the stream-K kernel, not one small block.
    rc, cfg, *_ = sg.sgemm_plan(1, 1, 1 << 20, 1 << 20, 1, 1, 0, 0, 0, 148)
    assert rc == 0 and sg.sgemm_config_name(cfg).startswith("ffma")


def test_plan_rejects_nonpositive_sm_count():
    rc, *_ = sg.sgemm_plan(4, 4, 4, 4, 4, 4, 0, 0, 0, 0)
    assert rc == sg.SGEMM_ERR_INVALID_VALUE


def test_fma_peak_microbench_compiles_for_sm_103a():
    # bench.py --probe-fma builds it on a GPU machine; here it must at least
    # cross-compile (the library build never includes it).
    import subprocess
    from dense_fp32_matrix_07_gb300 import build as _b
    import bench
    r = subprocess.run([_b._nvcc(), *_b.NVCC_FLAGS, "-c", bench.FMA_PEAK_SRC, "-o", os.devnull],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_fail_next_allocs_hook_validates_its_count():
    assert sg.sgemm_test_fail_next_allocs(-1) == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_test_fail_next_allocs(2) == sg.SGEMM_OK
    assert sg.sgemm_test_fail_next_allocs(0) == sg.SGEMM_OK


def test_general_plan_follows_the_library_choice():
    name = lambda c: sg.sgemm_config_name(c) if c >= 0 else None
    plan = lambda *a, config=-1: sg.sgemm_general_plan(*a, 0, 0, 0, 152, config)
    # A transposed A (K x M, aligned) is read in place by the k-major configuration...
    rc, cfg, pa, pb = plan(1, 0, 4096, 4096, 4096, 1.0, 4096, 0, 4096, 0, 0.0, 4096, 0, 1)
    assert (rc, name(cfg), pa, pb) == (0, "ffma2_128x256_k32_s4_ka", 0, 0)
    # ...a plain A is transposed for it, and a transposed B is packed.
    rc, cfg, pa, pb = plan(0, 1, 4096, 4096, 4096, 1.0, 4096, 0, 4096, 0, 0.0, 4096, 0, 1)
    assert (rc, name(cfg), pa, pb) == (0, "ffma2_128x256_k32_s4_ka", 1, 1)
    # A transposed A on rows that are not a multiple of 4 floats is copied first.
    rc, cfg, pa, pb = plan(1, 0, 4096, 4096, 4096, 1.0, 4097, 0, 4096, 0, 0.0, 4096, 0, 1)
    assert (rc, pa, pb) == (0, 1, 0)
    # Below N = 2048 the row-major configuration reads an aligned strided batch in place.
    rc, cfg, pa, pb = plan(0, 0, 1024, 1024, 1024, 1.0, 1024, 1 << 20, 1024, 0, 0.0, 1024, 1 << 20, 16)
    assert (rc, name(cfg), pa, pb) == (0, "ffma2_128x128_k32_s4", 0, 0)
    # Tiny general products take the smallest TMA tiles, not the pages' ladder kernel.
    rc, cfg, pa, pb = plan(0, 0, 150, 200, 70, -1.5, 73, 150 * 73, 205, 70 * 205, 2.0, 202, 150 * 202, 3)
    assert (rc, name(cfg), pa, pb) == (0, "ffma2_128x64_k32_s4", 1, 1)
    # K == 0 only scales C: no product configuration.
    assert plan(0, 0, 150, 200, 0, 1.0, 1, 0, 200, 0, 2.0, 202, 0, 1)[:2] == (0, -1)
    # Status codes as sgemm_general_ex(): overlapping C entries, a plain-form-only forced configuration.
    assert plan(0, 0, 150, 200, 70, 1.0, 70, 0, 200, 0, 0.0, 202, 0, 3)[0] == sg.SGEMM_ERR_INVALID_VALUE
    ladder = sg.config_ids()["ladder_register_tiled_2x2"]
    assert plan(0, 0, 256, 256, 256, 1.0, 256, 0, 256, 0, 0.5, 256, 0, 1, config=ladder)[0] == \
        sg.SGEMM_ERR_UNSUPPORTED


@pytest.mark.parametrize("M,N,K,rows", [
    (4097, 3001, 2049, 1),      # the odd rectangle: one row past 32 block rows
    (4100, 3001, 2049, 4),
    (4104, 3001, 2049, 8),
    (4105, 3001, 2049, 0),      # 9 rows: the tiled product pads them
    (4096, 4096, 4096, 0),      # whole block rows
    (129, 129, 129, 0),         # M not past a block row, and a small product
    (1025, 1024, 1024, 0),      # round_up(N, BN) * K = 2^20: below the tail kernel's fixed cost
    (1025, 1024, 2048, 1),
])
def test_row_tail_decision(M, N, K, rows):
    rc, cfg, _, _ = sg.sgemm_plan(M, N, K, K, N, N, 0, 0, 0, 152)
    assert rc == 0
    assert sg.sgemm_plan_row_tail(cfg, M, N, K) == (0, rows)


def test_row_tail_only_on_tma_ffma_configurations():
    ids = sg.config_ids()
    for name in ("tiled16_simple", "ladder_register_tiled_2x2", "tf32x3_128x256_k16_s4", "tf32x3_pair_128x256_k16_s4"):
        assert sg.sgemm_plan_row_tail(ids[name], 4097, 3001, 2049) == (0, 0), name
    for name in ("ffma2_128x256_k32_s4", "ffma2_128x128_k32_s4_ka", "ffma2_128x64_k32_s4", "ffma_128x128_k32_s4"):
        assert sg.sgemm_plan_row_tail(ids[name], 4097, 3001, 2049) == (0, 1), name
    # Batches of up to 65535 entries (one grid dimension of the tail kernel).
    cfg = ids["ffma2_128x256_k32_s4"]
    assert sg.sgemm_plan_row_tail(cfg, 4097, 3001, 2049, 65535) == (0, 1)
    assert sg.sgemm_plan_row_tail(cfg, 4097, 3001, 2049, 65536) == (0, 0)
    assert sg.sgemm_plan_row_tail(-1, 4097, 3001, 2049)[0] == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_plan_row_tail(cfg, -1, 3001, 2049)[0] == sg.SGEMM_ERR_INVALID_VALUE


def test_general_plan_launches_counts_the_calls_kernels():
    """Host-only launch count of a call: the product, the layout pass (for an
    operand that goes through scratch, or for arrival counters to zero), the
    last-rows kernel; 3xTF32: two splits and the product per entry; only a
    scaling kernel when K == 0 or alpha == 0 (none when beta == 1)."""
    P = sg.sgemm_general_plan_launches

    def plain(M, N, K, lda, ldb, ldc, config=-1):
        return P(0, 0, M, N, K, 1.0, lda, 0, ldb, 0, 0.0, ldc, 0, 1, 0, 0, 0, 152, config)

    assert plain(4096, 4096, 4096, 4096, 4096, 4096) == (0, 2)     # A transposed, product
    assert plain(4097, 3001, 2049, 2049, 3001, 3001) == (0, 3)     # pass for A and B, product, last row
    assert plain(1024, 1024, 1024, 1024, 1024, 1024) == (0, 2)     # counters zeroed, product
    assert plain(1536, 1536, 1536, 1536, 1536, 1536) == (0, 1)     # whole tiles, aligned: product only
    assert plain(256, 256, 256, 256, 256, 256) == (0, 1)           # the small-product kernel
    dp = sg.config_ids()["ffma2_128x256_k32_s4_dp"]
    assert plain(129, 2048, 1024, 1024, 2051, 2048, dp) == (0, 3)  # pass for B, product, last row
    tf = sg.config_ids()["tf32x3_pair_128x256_k16_s4"]
    assert P(0, 0, 512, 512, 512, 1.0, 512, 512 * 512, 512, 512 * 512, 0.0, 512, 512 * 512, 3,
             0, 0, 0, 152, tf) == (0, 9)
    assert P(0, 0, 10, 10, 0, 1.0, 1, 0, 10, 0, 0.5, 10, 0, 1, 0, 0, 0, 152) == (0, 1)
    assert P(0, 0, 10, 10, 0, 1.0, 1, 0, 10, 0, 1.0, 10, 0, 1, 0, 0, 0, 152) == (0, 0)
    assert P(0, 0, -1, 10, 10, 1.0, 10, 0, 10, 0, 0.0, 10, 0, 1, 0, 0, 0, 152)[0] == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.load().sgemm_general_plan_launches(0, 0, 10, 10, 10, 1.0, 10, 0, 10, 0, 0.0, 10, 0, 1,
                                                 0, 0, 0, 152, -1, None) == sg.SGEMM_ERR_INVALID_VALUE
