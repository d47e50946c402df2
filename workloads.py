"""Seeded synthetic SGEMM workloads shared by the tests, the bench and smoke().

This module only draws random input matrices and names the workload shapes.
It holds none of the matrix-multiply arithmetic: the CPU oracle (``oracle/``)
and the CUDA library (``dense_fp32_matrix_07_gb300``) both take its arrays as
plain inputs and never import each other.

Recipe (the same for every consumer):

* ``g = torch.Generator('cpu').manual_seed(seed)``; A is drawn first, then B,
  from the same generator, on the CPU, as float32, row-major, tight strides.
* ``uniform``: ``torch.rand(...) * 2 - 1``, i.e. U[-1, 1) (exact in FP32).
* ``normal``: ``torch.randn(...)``, i.e. N(0, 1).
* ``int``: ``torch.randint(-4, 5, ...)`` cast to float32: integers in [-4, 4].
  Every partial sum of such a product stays below 16*K in magnitude, so for
  K <= 2**20 every FP32 partial sum in any order is exact.

The shapes are those of the FP32 SGEMM workloads the pages discuss: square
N x N products (the handbook's and the course's running example is N = 1024,
the book's intensity example is N = 4096), plus an odd rectangular shape
with non-tile-multiple sizes and leading dimensions that are not multiples of
four floats, and a 16384-cube large case.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One SGEMM problem C(MxN) = A(MxK) . B(KxN), row-major with strides."""

    name: str
    M: int
    N: int
    K: int
    lda: int
    ldb: int
    ldc: int
    dist: str          # 'uniform' | 'normal' | 'int'
    seed: int
    sampled: bool = False   # check only sampled rows/columns of C

    @property
    def flops(self) -> int:
        # 2MNK floating-point operations: one multiply and one add per term
        # (Chapter 9: Optimised Matrix Multiplication, section 9.1).
        return 2 * self.M * self.N * self.K


WORKLOADS = {
    "sq256": Workload("sq256", 256, 256, 256, 256, 256, 256, "uniform", 0),
    "sq256_int": Workload("sq256_int", 256, 256, 256, 256, 256, 256, "int", 0),
    "sq1024": Workload("sq1024", 1024, 1024, 1024, 1024, 1024, 1024, "uniform", 1),
    "sq1024_int": Workload("sq1024_int", 1024, 1024, 1024, 1024, 1024, 1024, "int", 1),
    "sq4096": Workload("sq4096", 4096, 4096, 4096, 4096, 4096, 4096, "normal", 2),
    "rect4097x3001x2049": Workload("rect4097x3001x2049", 4097, 3001, 2049,
                                   2049, 3001, 3001, "uniform", 3),
    "sq16384": Workload("sq16384", 16384, 16384, 16384, 16384, 16384, 16384,
                        "normal", 4, sampled=True),
}


def _draw(g: torch.Generator, rows: int, cols: int, dist: str) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(rows, cols, generator=g, dtype=torch.float32) * 2 - 1
    if dist == "normal":
        return torch.randn(rows, cols, generator=g, dtype=torch.float32)
    if dist == "int":
        return torch.randint(-4, 5, (rows, cols), generator=g).to(torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def make_operands(M: int, N: int, K: int, dist: str, seed: int,
                  lda: int | None = None, ldb: int | None = None):
    """Return (A, B) as CPU float32 tensors of shape (M, lda) and (K, ldb).

    Columns beyond K (resp. N) are padding that the product must never read;
    they are filled with NaN so that any read of them shows up as NaN in C.
    """
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    if lda < K or ldb < N:
        raise ValueError("leading dimension shorter than the row")
    g = torch.Generator("cpu").manual_seed(seed)
    a = _draw(g, M, K, dist)
    b = _draw(g, K, N, dist)
    if lda != K:
        A = torch.full((M, lda), float("nan"), dtype=torch.float32)
        A[:, :K] = a
    else:
        A = a
    if ldb != N:
        B = torch.full((K, ldb), float("nan"), dtype=torch.float32)
        B[:, :N] = b
    else:
        B = b
    return A.contiguous(), B.contiguous()


def make_workload(w: Workload):
    """Operands of a named workload (see the module docstring for the recipe)."""
    return make_operands(w.M, w.N, w.K, w.dist, w.seed, w.lda, w.ldb)


def sample_indices(n: int, count: int, seed: int) -> np.ndarray:
    """Sorted distinct indices into range(n): 0, n-1 and count-2 random others.

    Used to pick the rows and columns of C that are checked on the largest
    workload (a full check there is out of reach for a CPU oracle).
    """
    if count >= n:
        return np.arange(n, dtype=np.int64)
    g = torch.Generator("cpu").manual_seed(seed)
    inner = torch.randperm(n - 2, generator=g)[: count - 2] + 1
    idx = np.concatenate([[0, n - 1], inner.numpy()]).astype(np.int64)
    return np.unique(idx)


def special_matrix(kind: str, rows: int, cols: int) -> torch.Tensor:
    """Structured float32 matrices used by closed-form checks.

    kind: 'ones' (all ones), 'row_index' (entry = its row index),
    'col_index' (entry = its column index), 'identity', 'alt_sign_col'
    (entry = (-1)**col), 'col_plus1' (entry = col + 1), 'row_plus1'.
    """
    r = torch.arange(rows, dtype=torch.float32).view(rows, 1).expand(rows, cols)
    c = torch.arange(cols, dtype=torch.float32).view(1, cols).expand(rows, cols)
    if kind == "ones":
        return torch.ones(rows, cols, dtype=torch.float32)
    if kind == "row_index":
        return r.contiguous()
    if kind == "col_index":
        return c.contiguous()
    if kind == "row_plus1":
        return (r + 1).contiguous()
    if kind == "col_plus1":
        return (c + 1).contiguous()
    if kind == "identity":
        return torch.eye(rows, cols, dtype=torch.float32)
    if kind == "alt_sign_col":
        return (1 - 2 * (c.to(torch.int64) % 2)).to(torch.float32).contiguous()
    raise ValueError(kind)
