"""CPU oracle for FP32 SGEMM (C = A . B, row-major), FP64 accumulation.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this package; the CUDA library never
does, and this package never imports the library. It wraps the plain C
triple loop in ``sgemm_oracle.c`` (compiled here with gcc) through ctypes.

Definition followed: "Перемножение матриц: наивное и тайловое", section 1
(C_row,col is the dot product of row `row` of A and column `col` of B,
row-major offset row*n + col), and Chapter 9: Optimised Matrix
Multiplication, section 9.1 (2N^3 FLOPs). Each function returns the product
in float64 together with S = sum_k |A_ik * B_kj|, the scale of the FP32
tolerance |C_gpu - C_ref| <= 1e-4 * S.

Every function here is pinned by ``tests/test_oracle.py`` (identity,
closed forms, exact integer products, exact rational brute force, a float64
library cross-check, sampled-versus-full and transpose invariants) and by
``tests/test_oracle_mutants.py`` (planted mistakes must fail those pins).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_fp = ctypes.POINTER(ctypes.c_float)
_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_int64)


def compile_library(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle C source into a shared library with gcc."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           *extra_flags, src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build() -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        compile_library()
    return _LIB_PATH


def load_library(path: str):
    lib = ctypes.CDLL(path)
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_sgemm_f64.restype = ctypes.c_int
    lib.oracle_sgemm_f64.argtypes = [_i64, _i64, _i64, _fp, _i64, _fp, _i64,
                                     _dp, _i64, _dp, _i64]
    lib.oracle_sgemm_rows_f64.restype = ctypes.c_int
    lib.oracle_sgemm_rows_f64.argtypes = [_i64, _i64, _i64, _fp, _i64, _fp, _i64,
                                          _lp, _i64, _dp, _dp]
    lib.oracle_sgemm_general_f64.restype = ctypes.c_int
    lib.oracle_sgemm_general_f64.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64, _i64, ctypes.c_double,
                                             _fp, _i64, _i64, _fp, _i64, _i64,
                                             ctypes.c_double, _fp, _i64, _i64, _i64, _dp, _dp]
    lib.oracle_sgemm_cols_f64.restype = ctypes.c_int
    lib.oracle_sgemm_cols_f64.argtypes = [_i64, _i64, _i64, _fp, _i64, _fp, _i64,
                                          _lp, _i64, _dp, _dp]
    return lib


def _get():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


class Oracle:
    """ctypes front end over one compiled oracle library (the default one,
    or a variant compiled from another source, as the mutation tests do)."""

    def __init__(self, lib=None):
        self._lib_override = lib

    @property
    def lib(self):
        return self._lib_override if self._lib_override is not None else _get()

    # -- helpers ---------------------------------------------------------
    @staticmethod
    def _as_f32(x, rows, ld):
        x = np.asarray(x)
        if x.dtype != np.float32:
            raise TypeError("oracle operands are float32")
        x = np.ascontiguousarray(x)
        if x.size < (rows - 1) * ld + (0 if rows == 0 else 1) and rows > 0:
            raise ValueError("operand buffer too small for its shape/stride")
        return x

    @staticmethod
    def _ptr(x, typ):
        return x.ctypes.data_as(typ) if x is not None else None

    # -- API -------------------------------------------------------------
    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        self.lib.oracle_set_num_threads(int(n))

    def sgemm(self, M, N, K, A, lda, B, ldb, want_abs=True):
        """Full product. A: flat/2-D float32 with M rows of stride lda;
        B: K rows of stride ldb. Returns (C, S) as float64 (M, N) arrays
        (S is None when want_abs is False)."""
        M, N, K = int(M), int(N), int(K)
        A = self._as_f32(A, M if K > 0 else 0, lda)
        B = self._as_f32(B, K, ldb)
        C = np.empty((M, N), dtype=np.float64)
        S = np.empty((M, N), dtype=np.float64) if want_abs else None
        if M == 0 or N == 0:
            return C, S
        rc = self.lib.oracle_sgemm_f64(M, N, K, self._ptr(A, _fp), lda,
                                       self._ptr(B, _fp), ldb,
                                       self._ptr(C, _dp), N,
                                       self._ptr(S, _dp) if S is not None else None, N)
        if rc != 0:
            raise ValueError(f"oracle_sgemm_f64 rejected its arguments ({rc})")
        return C, S

    def sgemm_rows(self, M, N, K, A, lda, B, ldb, rows, want_abs=True):
        """Rows `rows` of C (and S) as float64 (len(rows), N) arrays."""
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        A = self._as_f32(A, M, lda)
        B = self._as_f32(B, K, ldb)
        C = np.empty((len(rows), N), dtype=np.float64)
        S = np.empty((len(rows), N), dtype=np.float64) if want_abs else None
        rc = self.lib.oracle_sgemm_rows_f64(M, N, K, self._ptr(A, _fp), lda,
                                            self._ptr(B, _fp), ldb,
                                            self._ptr(rows, _lp), len(rows),
                                            self._ptr(C, _dp),
                                            self._ptr(S, _dp) if S is not None else None)
        if rc != 0:
            raise ValueError(f"oracle_sgemm_rows_f64 rejected its arguments ({rc})")
        return C, S

    def sgemm_cols(self, M, N, K, A, lda, B, ldb, cols, want_abs=True):
        """Columns `cols` of C (and S) as float64 (M, len(cols)) arrays."""
        cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
        A = self._as_f32(A, M, lda)
        B = self._as_f32(B, K, ldb)
        C = np.empty((M, len(cols)), dtype=np.float64)
        S = np.empty((M, len(cols)), dtype=np.float64) if want_abs else None
        rc = self.lib.oracle_sgemm_cols_f64(M, N, K, self._ptr(A, _fp), lda,
                                            self._ptr(B, _fp), ldb,
                                            self._ptr(cols, _lp), len(cols),
                                            self._ptr(C, _dp),
                                            self._ptr(S, _dp) if S is not None else None)
        if rc != 0:
            raise ValueError(f"oracle_sgemm_cols_f64 rejected its arguments ({rc})")
        return C, S


    def sgemm_general(self, op_a, op_b, M, N, K, alpha, A, lda, sa, B, ldb, sb,
                      beta, Cin, ldc, sc, batch, want_abs=True):
        """alpha * op(A_b) . op(B_b) + beta * C_b for b < batch. A, B, Cin:
        flat float32 arrays (Cin may be None when beta == 0). Returns (C, S)
        as float64 (batch, M, N) arrays."""
        A = np.ascontiguousarray(np.asarray(A, dtype=np.float32).reshape(-1))
        B = np.ascontiguousarray(np.asarray(B, dtype=np.float32).reshape(-1))
        Cp = None
        if Cin is not None:
            Cp = np.ascontiguousarray(np.asarray(Cin, dtype=np.float32).reshape(-1))
        C = np.empty((batch, M, N), dtype=np.float64)
        S = np.empty((batch, M, N), dtype=np.float64) if want_abs else None
        rc = self.lib.oracle_sgemm_general_f64(op_a, op_b, M, N, K, float(alpha),
                                               self._ptr(A, _fp), lda, sa, self._ptr(B, _fp), ldb, sb,
                                               float(beta), self._ptr(Cp, _fp) if Cp is not None else None,
                                               ldc, sc, batch, self._ptr(C, _dp),
                                               self._ptr(S, _dp) if S is not None else None)
        if rc != 0:
            raise ValueError(f"oracle_sgemm_general_f64 rejected its arguments ({rc})")
        return C, S


_default = Oracle()
sgemm = _default.sgemm
sgemm_rows = _default.sgemm_rows
sgemm_cols = _default.sgemm_cols
sgemm_general = _default.sgemm_general
num_threads = _default.num_threads
set_num_threads = _default.set_num_threads
