"""Pins for the CPU oracle: checks that tie it to something other than itself.

Each ``check_*`` function takes an ``oracle.Oracle`` instance and raises
AssertionError when the oracle disagrees with an independent fact:

* exact rational brute force on tiny shapes (Python ``fractions``),
* identity matrices (A.I = A and I.B = B, rectangular too),
* closed-form products of structured matrices,
* integer-valued inputs against exact int64 arithmetic,
* a float64 library matmul,
* strided (padded) operands against compact ones,
* sampled rows/columns against the full product,
* the transpose identity (A.B)^T = B^T.A^T,
* the absolute-sum S against the product of |A| and |B|,
* IEEE propagation of NaN, the empty sum (K = 0), rejected arguments.

The definition being pinned is C_ij = sum_k A_ik B_kj ("Перемножение матриц:
наивное и тайловое", section 1), with row-major storage at row*ld + col.
``tests/test_oracle.py`` runs every check on the real oracle;
``tests/test_oracle_mutants.py`` plants plausible mistakes in copies of the
oracle's C source and requires each to fail at least one check.
"""

from __future__ import annotations

import itertools
from fractions import Fraction

import numpy as np
import torch

import workloads


def _rand(rows, cols, dist, seed):
    A, _ = workloads.make_operands(rows, 1, cols, dist, seed)
    return A.numpy()


def _pair(M, N, K, dist, seed):
    A, B = workloads.make_operands(M, N, K, dist, seed)
    return A.numpy(), B.numpy()


def check_bruteforce_rational(o, max_dim=6, seed=11):
    """All M, N, K in 1..max_dim: exact rational sum of exact products."""
    rng = np.random.default_rng(seed)
    for M, N, K in itertools.product(range(1, max_dim + 1), repeat=3):
        # Mix magnitudes so that the double sum actually rounds.
        A = (rng.standard_normal((M, K)) * 2.0 ** rng.integers(-20, 20, (M, K))).astype(np.float32)
        B = (rng.standard_normal((K, N)) * 2.0 ** rng.integers(-20, 20, (K, N))).astype(np.float32)
        C, S = o.sgemm(M, N, K, A, K, B, N)
        for i in range(M):
            for j in range(N):
                exact = sum(Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
                            for k in range(K))
                sabs = sum(abs(Fraction(float(A[i, k])) * Fraction(float(B[k, j])))
                           for k in range(K))
                bound = Fraction(K, 2 ** 53) * sabs
                err = abs(Fraction(float(C[i, j])) - exact)
                assert err <= bound, (M, N, K, i, j, float(err), float(bound))
                assert Fraction(float(S[i, j])) >= sabs * (1 - Fraction(K, 2 ** 52)), (M, N, K, i, j)
                assert abs(Fraction(float(S[i, j])) - sabs) <= bound, (M, N, K, i, j)


def check_identity(o):
    """A.I = A and I.B = B exactly, with square and rectangular identities."""
    for (M, K, N) in [(5, 7, 7), (7, 5, 3), (3, 4, 9), (33, 17, 17), (1, 1, 1)]:
        A = _rand(M, K, "normal", 1)
        I = workloads.special_matrix("identity", K, N).numpy()
        C, _ = o.sgemm(M, N, K, A, K, I, N)
        want = np.zeros((M, N))
        w = min(K, N)
        want[:, :w] = A[:, :w].astype(np.float64)
        assert np.array_equal(C, want), (M, K, N)
        I2 = workloads.special_matrix("identity", M, K).numpy()
        B = _rand(K, N, "normal", 2)
        C2, _ = o.sgemm(M, N, K, I2, K, B, N)
        want2 = np.zeros((M, N))
        h = min(M, K)
        want2[:h, :] = B[:h, :].astype(np.float64)
        assert np.array_equal(C2, want2), (M, K, N)


def check_closed_forms(o):
    """Structured products with closed forms (all exact in double)."""
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (16, 9, 33), (40, 17, 129)]:
        sm = workloads.special_matrix
        i = np.arange(M, dtype=np.float64).reshape(M, 1)
        j = np.arange(N, dtype=np.float64).reshape(1, N)
        # all ones: every entry is K
        C, _ = o.sgemm(M, N, K, sm("ones", M, K).numpy(), K, sm("ones", K, N).numpy(), N)
        assert np.array_equal(C, np.full((M, N), float(K))), ("ones", M, N, K)
        # A_ik = 1, B_kj = k: sum_k k = K(K-1)/2
        C, _ = o.sgemm(M, N, K, sm("ones", M, K).numpy(), K, sm("row_index", K, N).numpy(), N)
        assert np.array_equal(C, np.full((M, N), K * (K - 1) / 2)), ("sum k", M, N, K)
        # A_ik = i, B_kj = j: C_ij = i * j * K
        C, _ = o.sgemm(M, N, K, sm("row_index", M, K).numpy(), K, sm("col_index", K, N).numpy(), N)
        assert np.array_equal(C, i * j * K), ("i*j*K", M, N, K)
        # A_ik = i, B_kj = k: C_ij = i * K(K-1)/2   (a transposed A would differ)
        C, _ = o.sgemm(M, N, K, sm("row_index", M, K).numpy(), K, sm("row_index", K, N).numpy(), N)
        assert np.array_equal(C, np.broadcast_to(i * (K * (K - 1) / 2), (M, N))), ("i*sum k", M, N, K)
        # A_ik = k + 1, B_kj = k + 1: sum of squares K(K+1)(2K+1)/6
        C, _ = o.sgemm(M, N, K, sm("col_plus1", M, K).numpy(), K, sm("row_plus1", K, N).numpy(), N)
        assert np.array_equal(C, np.full((M, N), K * (K + 1) * (2 * K + 1) / 6)), ("squares", M, N, K)
        # A_ik = (-1)^k, B = ones: K mod 2 (signs must cancel)
        C, S = o.sgemm(M, N, K, sm("alt_sign_col", M, K).numpy(), K, sm("ones", K, N).numpy(), N)
        assert np.array_equal(C, np.full((M, N), float(K % 2))), ("alt", M, N, K)
        assert np.array_equal(S, np.full((M, N), float(K))), ("alt abs", M, N, K)
        # A_ik = 1, B_kj = j: C_ij = K * j   (B must be read along its row)
        C, _ = o.sgemm(M, N, K, sm("ones", M, K).numpy(), K, sm("col_index", K, N).numpy(), N)
        assert np.array_equal(C, np.broadcast_to(K * j, (M, N))), ("K*j", M, N, K)


def check_integer_exact(o):
    """Integer inputs in [-4, 4]: equal to exact int64 matrix products."""
    for n, (M, N, K) in enumerate([(1, 1, 1), (7, 13, 5), (64, 48, 100), (31, 33, 257)]):
        A, B = _pair(M, N, K, "int", 100 + n)
        C, S = o.sgemm(M, N, K, A, K, B, N)
        Ai, Bi = A.astype(np.int64), B.astype(np.int64)
        assert np.array_equal(C, (Ai @ Bi).astype(np.float64)), (M, N, K)
        assert np.array_equal(S, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64)), (M, N, K)


def check_float64_library(o):
    """Random normal inputs: within 1e-12 * S of torch's float64 matmul."""
    for n, (M, N, K) in enumerate([(64, 64, 64), (100, 37, 300), (257, 129, 511)]):
        A, B = _pair(M, N, K, "normal", 200 + n)
        C, S = o.sgemm(M, N, K, A, K, B, N)
        ref = (torch.from_numpy(A).double() @ torch.from_numpy(B).double()).numpy()
        assert np.all(np.abs(C - ref) <= 1e-12 * S), (M, N, K)


def check_strides(o):
    """Padded leading dimensions give the compact result; padding is never read."""
    M, N, K = 19, 23, 29
    A, B = workloads.make_operands(M, N, K, "uniform", 7)
    Ap, Bp = workloads.make_operands(M, N, K, "uniform", 7, lda=K + 5, ldb=N + 3)
    C, S = o.sgemm(M, N, K, A.numpy(), K, B.numpy(), N)
    Cp, Sp = o.sgemm(M, N, K, Ap.numpy(), K + 5, Bp.numpy(), N + 3)
    assert not np.isnan(Cp).any()
    assert np.array_equal(C, Cp) and np.array_equal(S, Sp)


def check_sampled(o):
    """Sampled rows and columns equal the same rows/columns of the full product."""
    M, N, K = 37, 41, 53
    A, B = _pair(M, N, K, "normal", 9)
    C, S = o.sgemm(M, N, K, A, K, B, N)
    rows = workloads.sample_indices(M, 9, 1)
    cols = workloads.sample_indices(N, 9, 2)
    Cr, Sr = o.sgemm_rows(M, N, K, A, K, B, N, rows)
    Cc, Sc = o.sgemm_cols(M, N, K, A, K, B, N, cols)
    assert np.array_equal(Cr, C[rows]) and np.array_equal(Sr, S[rows])
    assert np.array_equal(Cc, C[:, cols]) and np.array_equal(Sc, S[:, cols])


def check_transpose(o):
    """(A.B)^T = B^T.A^T, element for element (same k order)."""
    M, N, K = 21, 14, 33
    A, B = _pair(M, N, K, "normal", 5)
    C, _ = o.sgemm(M, N, K, A, K, B, N)
    Bt = np.ascontiguousarray(B.T)
    At = np.ascontiguousarray(A.T)
    Ct, _ = o.sgemm(N, M, K, Bt, K, At, M)
    assert np.array_equal(C, Ct.T)


def check_abs_sum(o):
    """S(A, B) equals the product of |A| and |B|, and bounds |C|."""
    M, N, K = 17, 19, 65
    A, B = _pair(M, N, K, "normal", 6)
    C, S = o.sgemm(M, N, K, A, K, B, N)
    Cabs, _ = o.sgemm(M, N, K, np.abs(A), K, np.abs(B), N)
    assert np.array_equal(S, Cabs)
    assert np.all(np.abs(C) <= S)


def check_special_values(o):
    """NaN in row i of A makes row i of C NaN and nothing else; K=0 is zero."""
    M, N, K = 6, 5, 4
    A, B = _pair(M, N, K, "uniform", 3)
    A = A.copy()
    A[2, 1] = np.nan
    C, _ = o.sgemm(M, N, K, A, K, B, N)
    assert np.isnan(C[2]).all()
    assert not np.isnan(np.delete(C, 2, axis=0)).any()
    C0, S0 = o.sgemm(3, 4, 0, np.zeros(1, np.float32), 1, np.zeros(1, np.float32), 4)
    assert np.array_equal(C0, np.zeros((3, 4))) and np.array_equal(S0, np.zeros((3, 4)))
    Ce, _ = o.sgemm(0, 4, 3, np.zeros(1, np.float32), 3, np.zeros(12, np.float32), 4)
    assert Ce.shape == (0, 4)


def check_general_reduces_to_plain(o):
    """op = (as stored, as stored), alpha = 1, beta = 0, one entry: the
    general form is the plain product, bit for bit."""
    M, N, K = 23, 19, 37
    A, B = _pair(M, N, K, "normal", 31)
    C, S = o.sgemm(M, N, K, A, K, B, N)
    G, GS = o.sgemm_general(0, 0, M, N, K, 1.0, A, K, 0, B, N, 0, 0.0, None, N, 0, 1)
    assert np.array_equal(G[0], C) and np.array_equal(GS[0], S)


def check_general_transposes(o):
    """A stored transposed (K x M) with op_a = 1, B stored transposed (N x K)
    with op_b = 1, each give the same product as the plain layout."""
    M, N, K = 13, 17, 29
    A, B = _pair(M, N, K, "normal", 32)
    C, _ = o.sgemm(M, N, K, A, K, B, N)
    At, Bt = np.ascontiguousarray(A.T), np.ascontiguousarray(B.T)
    for op_a, op_b, a, lda, b, ldb in ((1, 0, At, M, B, N), (0, 1, A, K, Bt, K), (1, 1, At, M, Bt, K)):
        G, _ = o.sgemm_general(op_a, op_b, M, N, K, 1.0, a, lda, 0, b, ldb, 0, 0.0, None, N, 0, 1)
        assert np.array_equal(G[0], C), (op_a, op_b)


def check_general_alpha_beta(o):
    """All-ones A and B (C = K), times alpha, plus beta * C_in, exactly; beta
    = 0 never reads C_in (NaN there stays out)."""
    M, N, K = 5, 6, 7
    A = np.ones(M * K, np.float32)
    B = np.ones(K * N, np.float32)
    Cin = (np.arange(M * N, dtype=np.float32) - 9).reshape(M, N)
    for alpha, beta in ((2.0, 0.0), (-0.5, 3.0), (0.0, -1.0), (1.0, 1.0)):
        G, S = o.sgemm_general(0, 0, M, N, K, alpha, A, K, 0, B, N, 0, beta, Cin, N, 0, 1)
        want = alpha * K + beta * Cin.astype(np.float64)
        assert np.array_equal(G[0], want), (alpha, beta)
        assert np.array_equal(S[0], abs(alpha) * K + np.abs(beta * Cin.astype(np.float64))), (alpha, beta)
    nan_c = np.full((M, N), np.nan, np.float32)
    G, _ = o.sgemm_general(0, 0, M, N, K, 1.0, A, K, 0, B, N, 0, 0.0, nan_c, N, 0, 1)
    assert not np.isnan(G).any()


def check_general_batch(o):
    """Entry b of a strided batch equals the plain product of entry b;
    stride 0 shares one operand across the batch."""
    M, N, K, batch = 9, 11, 14, 4
    sa, sb, sc = M * K + 3, K * N + 5, M * N + 2
    rng = np.random.default_rng(33)
    A = rng.standard_normal(batch * sa).astype(np.float32)
    B = rng.standard_normal(batch * sb).astype(np.float32)
    Cin = rng.standard_normal(batch * sc).astype(np.float32)
    G, _ = o.sgemm_general(0, 0, M, N, K, 1.5, A, K, sa, B, N, sb, -2.0, Cin, N, sc, batch)
    Gs, _ = o.sgemm_general(0, 0, M, N, K, 1.0, A, K, sa, B, N, 0, 0.0, None, N, 0, batch)
    for b in range(batch):
        C, _ = o.sgemm(M, N, K, A[b * sa:], K, B[b * sb:], N)
        cin = Cin[b * sc: b * sc + M * N].reshape(M, N).astype(np.float64)
        assert np.array_equal(G[b], 1.5 * C - 2.0 * cin), b
        C0, _ = o.sgemm(M, N, K, A[b * sa:], K, B, N)
        assert np.array_equal(Gs[b], C0), b


def check_general_bruteforce_rational(o, seed=34):
    """Tiny shapes, both ops, alpha and beta: within the double rounding bound
    of the exact rational result."""
    rng = np.random.default_rng(seed)
    for M, N, K in itertools.product((1, 2, 3), (1, 3), (1, 2, 4)):
        for op_a, op_b in itertools.product((0, 1), repeat=2):
            alpha, beta = float(rng.choice([0.5, -3.0, 1.25])), float(rng.choice([0.0, 2.0, -0.75]))
            Ar = rng.standard_normal((K, M) if op_a else (M, K)).astype(np.float32)
            Br = rng.standard_normal((N, K) if op_b else (K, N)).astype(np.float32)
            Cin = rng.standard_normal((M, N)).astype(np.float32)
            G, S = o.sgemm_general(op_a, op_b, M, N, K, alpha, Ar, Ar.shape[1], 0, Br, Br.shape[1], 0,
                                   beta, Cin, N, 0, 1)
            for i in range(M):
                for j in range(N):
                    acc = sum(Fraction(float(Ar[k, i] if op_a else Ar[i, k])) *
                              Fraction(float(Br[j, k] if op_b else Br[k, j])) for k in range(K))
                    sab = sum(abs(Fraction(float(Ar[k, i] if op_a else Ar[i, k])) *
                                  Fraction(float(Br[j, k] if op_b else Br[k, j]))) for k in range(K))
                    exact = Fraction(alpha) * acc + Fraction(beta) * Fraction(float(Cin[i, j]))
                    scale = abs(Fraction(alpha)) * sab + abs(Fraction(beta) * Fraction(float(Cin[i, j])))
                    bound = Fraction(K + 3, 2 ** 52) * scale
                    assert abs(Fraction(float(G[0, i, j])) - exact) <= bound, (M, N, K, op_a, op_b, i, j)


ALL_CHECKS = [
    check_bruteforce_rational,
    check_identity,
    check_closed_forms,
    check_integer_exact,
    check_float64_library,
    check_strides,
    check_sampled,
    check_transpose,
    check_abs_sum,
    check_special_values,
    check_general_reduces_to_plain,
    check_general_transposes,
    check_general_alpha_beta,
    check_general_batch,
    check_general_bruteforce_rational,
]
