"""GB300 (sm_103a) single-precision GEMM: C = A . B on row-major FP32 matrices.

This package is a thin ctypes binding over the C ABI in ``include/sgemm.h``
(``_build/libsgemm.so``, compiled from ``csrc/`` by ``build.py``). Its
functions carry the same names and arguments as the C functions and only
marshal arguments: pointers are plain integers (device addresses, e.g. a
torch tensor's ``data_ptr()``), streams are integers (``cudaStream_t``,
e.g. ``torch.cuda.current_stream().cuda_stream``; 0 is the default stream).
Every step of the product runs in the library's CUDA kernels; there is no
CPU fallback, and loading fails loudly if the library cannot be built or
loaded.
"""

from __future__ import annotations

import ctypes
import threading

from . import build as _build

SGEMM_OK = 0
SGEMM_ERR_INVALID_VALUE = 1
SGEMM_ERR_OVERFLOW = 2
SGEMM_ERR_ALLOC = 3
SGEMM_ERR_LAUNCH = 4
SGEMM_ERR_TIMEOUT = 5
SGEMM_ERR_CUDA = 6
SGEMM_ERR_UNSUPPORTED = 7
SGEMM_ERR_SCRATCH_LIMIT = 8

# Every function declared in include/sgemm.h.
EXPORTED = ("sgemm", "sgemm_ex", "sgemm_check_status", "sgemm_error_string",
            "sgemm_num_configs", "sgemm_config_name", "sgemm_plan", "sgemm_noalloc",
            "sgemm_test_withhold_copy", "sgemm_test_schedule", "sgemm_plan_row_tail",
            "sgemm_test_fail_next_allocs", "sgemm_general", "sgemm_general_ex", "sgemm_general_plan",
            "sgemm_general_plan_launches")

_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


class SgemmError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {sgemm_error_string(code)} ({code})")
        self.code = code


def load(rebuild: bool = False):
    """Build (if needed) and load the library; raises if either fails."""
    global _lib
    with _lock:
        if _lib is None or rebuild:
            path = _build.build(force=rebuild)
            lib = ctypes.CDLL(path)
            lib.sgemm.restype = ctypes.c_int
            lib.sgemm.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]
            lib.sgemm_ex.restype = ctypes.c_int
            lib.sgemm_ex.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
                                     ctypes.c_int, _vp]
            lib.sgemm_noalloc.restype = ctypes.c_int
            lib.sgemm_noalloc.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]
            lib.sgemm_test_withhold_copy.restype = ctypes.c_int
            lib.sgemm_test_withhold_copy.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp,
                                                     _i64, ctypes.c_int, _vp]
            lib.sgemm_test_schedule.restype = ctypes.c_int
            lib.sgemm_test_schedule.argtypes = [_i64, _i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i64,
                                                ctypes.c_int, _i64, _vp, _i64, _vp, _vp]
            lib.sgemm_plan_row_tail.restype = ctypes.c_int
            lib.sgemm_plan_row_tail.argtypes = [ctypes.c_int, _i64, _i64, _i64, _i64, _vp]
            lib.sgemm_test_fail_next_allocs.restype = ctypes.c_int
            lib.sgemm_test_fail_next_allocs.argtypes = [ctypes.c_int]
            gen = [ctypes.c_int, ctypes.c_int, _i64, _i64, _i64, ctypes.c_float, _vp, _i64, _i64,
                   _vp, _i64, _i64, ctypes.c_float, _vp, _i64, _i64, _i64]
            lib.sgemm_general.restype = ctypes.c_int
            lib.sgemm_general.argtypes = gen + [_vp]
            lib.sgemm_general_ex.restype = ctypes.c_int
            lib.sgemm_general_ex.argtypes = gen + [ctypes.c_int, _vp]
            _pi = ctypes.POINTER(ctypes.c_int)
            lib.sgemm_general_plan.restype = ctypes.c_int
            lib.sgemm_general_plan.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64, _i64, ctypes.c_float,
                                               _i64, _i64, _i64, _i64, ctypes.c_float, _i64, _i64, _i64,
                                               ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int,
                                               ctypes.c_int, _pi, _pi, _pi]
            lib.sgemm_general_plan_launches.restype = ctypes.c_int
            lib.sgemm_general_plan_launches.argtypes = lib.sgemm_general_plan.argtypes[:19] + [_pi]
            lib.sgemm_check_status.restype = ctypes.c_int
            lib.sgemm_check_status.argtypes = [_vp]
            lib.sgemm_error_string.restype = ctypes.c_char_p
            lib.sgemm_error_string.argtypes = [ctypes.c_int]
            lib.sgemm_num_configs.restype = ctypes.c_int
            lib.sgemm_num_configs.argtypes = []
            lib.sgemm_config_name.restype = ctypes.c_char_p
            lib.sgemm_config_name.argtypes = [ctypes.c_int]
            lib.sgemm_plan.restype = ctypes.c_int
            lib.sgemm_plan.argtypes = [_i64, _i64, _i64, _i64, _i64, _i64,
                                       ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                       ctypes.c_int,
                                       ctypes.POINTER(ctypes.c_int),
                                       ctypes.POINTER(ctypes.c_int),
                                       ctypes.POINTER(ctypes.c_int)]
            _lib = lib
    return _lib


def library_path() -> str:
    return _build.LIB


def sgemm(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """C = A . B on device pointers; returns the status code (0 = OK)."""
    return load().sgemm(M, N, K, A, lda, B, ldb, C, ldc, stream)


def sgemm_ex(M, N, K, A, lda, B, ldb, C, ldc, config, stream=0) -> int:
    """sgemm() with a forced kernel configuration (-1 = automatic)."""
    return load().sgemm_ex(M, N, K, A, lda, B, ldb, C, ldc, config, stream)


def sgemm_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """sgemm() for callers that cannot allocate: misaligned operands are
    packed into the library's fixed 64 MiB scratch array instead of
    allocated scratch (SGEMM_ERR_SCRATCH_LIMIT if they would not fit), and
    stream-K partial sums go in a fixed 24 MiB array. All calls on a device
    share those arrays, so calls that overlap on the GPU race on them."""
    return load().sgemm_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream)


def sgemm_test_fail_next_allocs(n) -> int:
    """Test hook: the next `n` scratch allocations are treated as failed (host only)."""
    return load().sgemm_test_fail_next_allocs(n)


def sgemm_test_withhold_copy(M, N, K, A, lda, B, ldb, C, ldc, slab, stream=0) -> int:
    """Test hook: the 128x256 TMA product whose first CTA never issues the copy of its
    `slab`-th K slab, so the kernel's bounded waits expire (about a second)
    and sgemm_check_status() reports SGEMM_ERR_TIMEOUT."""
    return load().sgemm_test_withhold_copy(M, N, K, A, lda, B, ldb, C, ldc, slab, stream)


def sgemm_test_schedule(M, N, K, bm, bn, bk, slots, policy, batch=1):
    """Test hook (host only): the persistent kernels' work schedule. Returns
    (items, info): items an (n, 10) int64 array of CTA, tile, first slab, end
    slab, batch entry, tile row, tile column, and for a part of a split tile
    its first CTA, last CTA and partial-sum slot (-1 otherwise); info a dict
    of grid, tiles, dp_tiles, sk_ctas, nk, tiles_m, tiles_n."""
    import numpy as np
    count = ctypes.c_int64(0)
    info = np.zeros(7, dtype=np.int64)
    cap = 1024
    while True:
        items = np.zeros((cap, 10), dtype=np.int64)
        rc = load().sgemm_test_schedule(M, N, K, bm, bn, bk, slots, policy, batch,
                                        items.ctypes.data, cap, ctypes.addressof(count), info.ctypes.data)
        if rc == SGEMM_OK:
            keys = ("grid", "tiles", "dp_tiles", "sk_ctas", "nk", "tiles_m", "tiles_n")
            return items[: count.value], dict(zip(keys, (int(x) for x in info)))
        if count.value <= cap:
            raise SgemmError(rc, "sgemm_test_schedule")
        cap = int(count.value)


def sgemm_general(op_a, op_b, M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b,
                  beta, C, ldc, stride_c, batch, stream=0) -> int:
    """C_b = alpha * op(A_b) . op(B_b) + beta * C_b for b < batch."""
    return load().sgemm_general(op_a, op_b, M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b,
                                beta, C, ldc, stride_c, batch, stream)


def sgemm_general_ex(op_a, op_b, M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b,
                     beta, C, ldc, stride_c, batch, config, stream=0) -> int:
    """sgemm_general() with a forced kernel configuration (-1 = automatic)."""
    return load().sgemm_general_ex(op_a, op_b, M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b,
                                   beta, C, ldc, stride_c, batch, config, stream)


def sgemm_check_status(stream=0) -> int:
    """Waits for `stream`, reads and clears the device error word."""
    return load().sgemm_check_status(stream)


def sgemm_error_string(code: int) -> str:
    return load().sgemm_error_string(code).decode()


def sgemm_num_configs() -> int:
    return load().sgemm_num_configs()


def sgemm_config_name(config: int) -> str:
    return load().sgemm_config_name(config).decode()


def sgemm_plan(M, N, K, lda, ldb, ldc, a_addr, b_addr, c_addr, num_sms):
    """Host-only: (status, config, pack_a, pack_b) that sgemm() would use."""
    cfg, pa, pb = ctypes.c_int(-1), ctypes.c_int(-1), ctypes.c_int(-1)
    rc = load().sgemm_plan(M, N, K, lda, ldb, ldc, a_addr, b_addr, c_addr, num_sms,
                           ctypes.byref(cfg), ctypes.byref(pa), ctypes.byref(pb))
    return rc, cfg.value, pa.value, pb.value


def sgemm_plan_row_tail(config, M, N, K, batch=1):
    """Host-only: (status, rows) — the last rows of C that a call on this
    configuration computes with the row-tail kernel (0: none)."""
    rows = ctypes.c_int64(-1)
    rc = load().sgemm_plan_row_tail(config, M, N, K, batch, ctypes.addressof(rows))
    return rc, rows.value


def sgemm_general_plan(op_a, op_b, M, N, K, alpha, lda, stride_a, ldb, stride_b, beta, ldc, stride_c,
                       batch, a_addr, b_addr, c_addr, num_sms, config=-1):
    """Host-only: (status, config, pack_a, pack_b) that sgemm_general_ex() would use
    (config -1 when the call runs no product)."""
    cfg, pa, pb = ctypes.c_int(-1), ctypes.c_int(-1), ctypes.c_int(-1)
    rc = load().sgemm_general_plan(op_a, op_b, M, N, K, alpha, lda, stride_a, ldb, stride_b, beta, ldc,
                                   stride_c, batch, a_addr, b_addr, c_addr, num_sms, config,
                                   ctypes.byref(cfg), ctypes.byref(pa), ctypes.byref(pb))
    return rc, cfg.value, pa.value, pb.value


def sgemm_general_plan_launches(op_a, op_b, M, N, K, alpha, lda, stride_a, ldb, stride_b, beta, ldc, stride_c,
                                batch, a_addr, b_addr, c_addr, num_sms, config=-1):
    """Host-only: (status, kernels of this library that sgemm_general_ex() would launch)."""
    n = ctypes.c_int(-1)
    rc = load().sgemm_general_plan_launches(op_a, op_b, M, N, K, alpha, lda, stride_a, ldb, stride_b, beta, ldc,
                                            stride_c, batch, a_addr, b_addr, c_addr, num_sms, config,
                                            ctypes.byref(n))
    return rc, n.value


def config_ids() -> dict:
    """Map of configuration name -> id."""
    return {sgemm_config_name(i): i for i in range(sgemm_num_configs())}
