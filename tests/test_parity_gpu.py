"""GPU parity: the CUDA library (through its C ABI) against the FP64 oracle.

Covers every kernel configuration on a shape sweep with ragged tails,
integer-valued inputs (bit-exact), strides beyond the row length, misaligned
pointers (the pack path), a NaN-prefilled C (C is never read), guard bands
(no write outside C's rows), the degenerate sizes, and the named workloads
at their full sizes (every element up to 4096^3 and 4097x3001x2049, float
and integer inputs; sampled rows and columns at 16384^3 only).
"""

import itertools

import numpy as np
import pytest
import torch

import dense_fp32_matrix_07_gb300 as sg
import workloads
from gpu_util import DeviceMatrix, assert_parity, check_untouched_padding, run

pytestmark = pytest.mark.gpu

CONFIGS = list(range(sg.sgemm_num_configs()))
CFG_IDS = [sg.sgemm_config_name(i) for i in CONFIGS]
EDGE = [1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 127, 128, 129, 255, 256, 257]


def _oracle_check(oracle, M, N, K, A, lda, B, ldb, C, exact, what):
    Cref, S = oracle.sgemm(M, N, K, A.numpy(), lda, B.numpy(), ldb)
    return assert_parity(C, Cref, S, exact, what)


def _shapes(seed, n):
    rng = np.random.default_rng(seed)
    out = {(1, 1, 1), (257, 257, 257), (129, 1, 33), (1, 257, 129), (33, 17, 1)}
    while len(out) < n:
        out.add(tuple(int(x) for x in rng.choice(EDGE, 3)))
    return sorted(out)


@pytest.mark.parametrize("config", CONFIGS, ids=CFG_IDS)
def test_shape_sweep_float(cuda_device, oracle, config):
    for n, (M, N, K) in enumerate(_shapes(1000 + config, 40)):
        A, B = workloads.make_operands(M, N, K, "uniform", n)
        rc, C, dC = run(M, N, K, A, K, B, N, config=config)
        assert rc == 0, (M, N, K, sg.sgemm_error_string(rc))
        _oracle_check(oracle, M, N, K, A, K, B, N, C, False, f"cfg {config} {M}x{N}x{K}")
        check_untouched_padding(dC, N)


FFMA_TMA = [i for i in CONFIGS if sg.sgemm_config_name(i).startswith("ffma")]


@pytest.mark.parametrize("config", FFMA_TMA, ids=[sg.sgemm_config_name(i) for i in FFMA_TMA])
def test_k_tail_both_kernels(cuda_device, oracle, config):
    """K = 64 + k_last on both sides of the point where the call stops
    trimming the last slab (k_last <= 3/8 of the slab depth: 12 of 32, 6 of
    16) and multiplies the whole zero-filled slab instead; integer inputs,
    so both kernels must match the oracle exactly, on a stream-K schedule
    (M, N give several tiles) and with a ragged last row block."""
    for n, k_last in enumerate((1, 6, 7, 12, 13, 31)):
        M, N, K = 300, 260, 64 + k_last
        A, B = workloads.make_operands(M, N, K, "int", 700 + n)
        rc, C, dC = run(M, N, K, A, K, B, N, config=config)
        assert rc == 0, (K, sg.sgemm_error_string(rc))
        _oracle_check(oracle, M, N, K, A, K, B, N, C, True, f"cfg {config} K={K}")
        check_untouched_padding(dC, N)


@pytest.mark.parametrize("config", CONFIGS, ids=CFG_IDS)
def test_shape_sweep_integer_exact(cuda_device, oracle, config):
    for n, (M, N, K) in enumerate(_shapes(2000 + config, 25)):
        A, B = workloads.make_operands(M, N, K, "int", 50 + n)
        rc, C, _ = run(M, N, K, A, K, B, N, config=config)
        assert rc == 0
        _oracle_check(oracle, M, N, K, A, K, B, N, C, True, f"cfg {config} {M}x{N}x{K}")


@pytest.mark.parametrize("config", CONFIGS, ids=CFG_IDS)
@pytest.mark.parametrize("shape", [(300, 200, 100), (517, 389, 1000), (1024, 1024, 1024)])
def test_multi_tile_ragged(cuda_device, oracle, config, shape):
    M, N, K = shape
    for dist, exact in (("normal", False), ("int", True)):
        A, B = workloads.make_operands(M, N, K, dist, 7)
        rc, C, dC = run(M, N, K, A, K, B, N, config=config)
        assert rc == 0
        _oracle_check(oracle, M, N, K, A, K, B, N, C, exact, f"cfg {config} {shape} {dist}")
        check_untouched_padding(dC, N)


@pytest.mark.parametrize("config", CONFIGS, ids=CFG_IDS)
def test_strides_beyond_row_length(cuda_device, oracle, config):
    M, N, K = 133, 70, 91
    for lda, ldb, ldc in [(K + 5, N + 3, N + 7), (K + 3, N + 10, N + 4), (128, 72, 96)]:
        A, B = workloads.make_operands(M, N, K, "uniform", 3, lda=lda, ldb=ldb)
        rc, C, dC = run(M, N, K, A, lda, B, ldb, ldc=ldc, config=config)
        assert rc == 0
        _oracle_check(oracle, M, N, K, A, lda, B, ldb, C, False, f"cfg {config} ld {lda},{ldb},{ldc}")
        check_untouched_padding(dC, N)


@pytest.mark.parametrize("config", CONFIGS, ids=CFG_IDS)
@pytest.mark.parametrize("offsets", [(1, 0, 0), (0, 2, 0), (0, 0, 3), (3, 1, 2)])
def test_misaligned_pointers(cuda_device, oracle, config, offsets):
    M, N, K = 100, 130, 70
    A, B = workloads.make_operands(M, N, K, "normal", 4)
    rc, C, dC = run(M, N, K, A, K, B, N, config=config, offsets=offsets)
    assert rc == 0
    _oracle_check(oracle, M, N, K, A, K, B, N, C, False, f"cfg {config} offsets {offsets}")
    check_untouched_padding(dC, N)


@pytest.mark.parametrize("config", CONFIGS, ids=CFG_IDS)
def test_nan_in_a_row_propagates(cuda_device, config):
    M, N, K = 160, 150, 140
    A, B = workloads.make_operands(M, N, K, "uniform", 5)
    A[37, 11] = float("nan")
    rc, C, _ = run(M, N, K, A, K, B, N, config=config, c_fill=0.0)
    assert rc == 0
    assert torch.isnan(C[37]).all()
    assert not torch.isnan(torch.cat([C[:37], C[38:]])).any()


def test_k_zero_writes_zeros(cuda_device):
    M, N = 37, 45
    rc, C, dC = run(M, N, 0, torch.zeros(1), 1, torch.zeros(1), N, ldc=N + 3)
    assert rc == 0
    assert bool((C == 0).all())
    check_untouched_padding(dC, N)


@pytest.mark.parametrize("M,N", [(0, 5), (5, 0), (0, 0)])
def test_empty_output_is_a_noop(cuda_device, M, N):
    dC = DeviceMatrix(None, 4, 8, 8)
    stream = torch.cuda.current_stream().cuda_stream
    assert sg.sgemm(M, N, 3, 0, 3, 0, max(N, 1), dC.ptr, max(N, 1), stream) == 0
    torch.cuda.synchronize()
    assert dC.guard_intact() and bool((dC.matrix() == 12345.678).all())


def test_invalid_arguments_launch_nothing(cuda_device):
    M, N, K = 8, 8, 8
    A, B = workloads.make_operands(M, N, K, "uniform", 1)
    dA, dB = DeviceMatrix(A, M, K, K), DeviceMatrix(B, K, N, N)
    dC = DeviceMatrix(None, M, N, N)
    s = torch.cuda.current_stream().cuda_stream
    E = sg.SGEMM_ERR_INVALID_VALUE
    cases = [
        ((-1, N, K, dA.ptr, K, dB.ptr, N, dC.ptr, N), E),
        ((M, N, K, dA.ptr, K - 1, dB.ptr, N, dC.ptr, N), E),
        ((M, N, K, dA.ptr, K, dB.ptr, N - 1, dC.ptr, N), E),
        ((M, N, K, dA.ptr, K, dB.ptr, N, dC.ptr, N - 1), E),
        ((M, N, K, 0, K, dB.ptr, N, dC.ptr, N), E),
        ((M, N, K, dA.ptr, K, 0, N, dC.ptr, N), E),
        ((M, N, K, dA.ptr, K, dB.ptr, N, 0, N), E),
        ((M, N, K, dA.ptr, K, dB.ptr, N, dA.ptr + 16, N), E),   # C overlaps A
        ((M, N, K, dA.ptr, K, dB.ptr, N, dB.ptr, N), E),        # C aliases B
        ((2 ** 31, N, K, dA.ptr, K, dB.ptr, N, dC.ptr, N), sg.SGEMM_ERR_OVERFLOW),
    ]
    for args, code in cases:
        assert sg.sgemm(*args, s) == code, args
    assert sg.sgemm_ex(M, N, K, dA.ptr, K, dB.ptr, N, dC.ptr, N, sg.sgemm_num_configs(), s) == E
    torch.cuda.synchronize()
    assert bool((dC.matrix() == 12345.678).all()), "a rejected call wrote C"
    assert sg.sgemm_check_status(s) == 0


# --------------------------------------------------------------------------
# The named workloads at their full sizes, through sgemm() (automatic config,
# the launch the bench times).
# --------------------------------------------------------------------------

def _run_workload(w, dist=None, config=-1):
    dist = dist or w.dist
    A, B = workloads.make_operands(w.M, w.N, w.K, dist, w.seed, w.lda, w.ldb)
    rc, C, dC = run(w.M, w.N, w.K, A, w.lda, B, w.ldb, ldc=w.ldc, c_fill=float("nan"), config=config)
    assert rc == 0
    check_untouched_padding(dC, w.N)
    return A, B, C


# The oracle's full product of a named workload, computed once per module
# (the same operands serve the FFMA and both tensor-core checks).
_FULL_REFERENCE = {}


def _full_reference(oracle, w, dist, A, B):
    key = (w.name, dist or w.dist)
    if key not in _FULL_REFERENCE:
        _FULL_REFERENCE[key] = oracle.sgemm(w.M, w.N, w.K, A.numpy(), w.lda, B.numpy(), w.ldb)
    return _FULL_REFERENCE[key]


def _full_check(oracle, w, dist, A, B, C, what):
    """Every element of C against the oracle (the course page, section 1:
    C_row,col is the dot product of row `row` of A and column `col` of B):
    within 1e-4 * sum|A_ik B_kj| for float inputs, bit-exact for integers."""
    Cref, S = _full_reference(oracle, w, dist, A, B)
    return assert_parity(C, Cref, S, (dist or w.dist) == "int", what)


@pytest.mark.parametrize("name,dist", [("sq256", None), ("sq256_int", None), ("sq1024", None),
                                       ("sq1024_int", None), ("rect4097x3001x2049", None),
                                       ("rect4097x3001x2049", "int"), ("sq4096", None), ("sq4096", "int")])
def test_workload_full_check(cuda_device, oracle, name, dist):
    w = workloads.WORKLOADS[name]
    A, B, C = _run_workload(w, dist)
    r = _full_check(oracle, w, dist, A, B, C, f"{name} {dist or w.dist}")
    print(f"{name} {dist or w.dist}: max |diff|/S = {r:.3e}")
    del A, B, C
    torch.cuda.empty_cache()


def _sampled_check(oracle, w, A, B, C, exact):
    rows = workloads.sample_indices(w.M, 256, w.seed + 1000)
    cols = workloads.sample_indices(w.N, 256, w.seed + 2000)
    Cr, Sr = oracle.sgemm_rows(w.M, w.N, w.K, A.numpy(), w.lda, B.numpy(), w.ldb, rows)
    Cc, Sc = oracle.sgemm_cols(w.M, w.N, w.K, A.numpy(), w.lda, B.numpy(), w.ldb, cols)
    r1 = assert_parity(C[torch.from_numpy(rows)], Cr, Sr, exact, f"{w.name} rows")
    r2 = assert_parity(C[:, torch.from_numpy(cols)], Cc, Sc, exact, f"{w.name} cols")
    return max(r1, r2)


@pytest.mark.parametrize("name,dist", [("sq16384", None), ("sq16384", "int")])
def test_workload_sampled_check(cuda_device, oracle, name, dist):
    """16384^3 only: 256 sampled rows and 256 sampled columns of C, every
    element of each (the full FP64 product would take the host minutes)."""
    w = workloads.WORKLOADS[name]
    A, B, C = _run_workload(w, dist)
    r = _sampled_check(oracle, w, A, B, C, dist == "int")
    print(f"{name} {dist or w.dist}: max |diff|/S = {r:.3e}")
    del A, B, C
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cfg_name", ["tf32x3_128x256_k16_s4", "tf32x3_pair_128x256_k16_s4"])
@pytest.mark.parametrize("name", ["rect4097x3001x2049", "sq4096", "sq16384"])
def test_tf32x3_tensor_core_path_at_full_size(cuda_device, oracle, name, cfg_name):
    """The 3xTF32 tcgen05 path at the full workload sizes (single CTAs, and
    clusters of two sharing B tiles), within 1e-4 * sum|A_ik B_kj| (float)
    and bit-exact (integers): every element below 16384^3, sampled rows and
    columns there."""
    w = workloads.WORKLOADS[name]
    cfg = sg.config_ids()[cfg_name]
    for dist in (None, "int"):
        A, B, C = _run_workload(w, dist, config=cfg)
        if w.sampled:
            r = _sampled_check(oracle, w, A, B, C, dist == "int")
        else:
            r = _full_check(oracle, w, dist, A, B, C, f"tf32x3 {name} {dist or w.dist}")
        print(f"tf32x3 {name} {dist or w.dist}: max |diff|/S = {r:.3e}")
        del A, B, C
        torch.cuda.empty_cache()


def test_status_is_clean_after_the_suite(cuda_device):
    assert sg.sgemm_check_status(torch.cuda.current_stream().cuda_stream) == sg.SGEMM_OK
