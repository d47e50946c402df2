"""Planted mistakes in the oracle must fail at least one pin (CPU only).

Each mutant is a textual edit of a copy of oracle/sgemm_oracle.c (a dropped
term, a wrong sign, a transposed or mis-strided operand, a lost
initialisation, reduced precision, a wrong sampled index, a wrong absolute
sum). The copy is compiled to a temporary library and the full pin suite of
tests/oracle_pins.py is run against it; the test passes only if some pin
rejects the mutant. The real oracle source is never modified.
"""

import os

import pytest

import oracle as oracle_pkg
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle_pkg.__file__), "sgemm_oracle.c")

MUTANTS = {
    "drop_last_k_term": ("for (int64_t k = 0; k < K; ++k) {\n        const double a",
                         "for (int64_t k = 0; k < K - 1; ++k) {\n        const double a"),
    "wrong_sign": ("\n            crow[j] += p;", "\n            crow[j] -= p;"),
    "transposed_B": ("const double p = a * (double)brow[j];",
                     "const double p = a * (double)B[(j < K ? j : 0) * ldb + (k < N ? k : 0)];"),
    "ignores_lda": ("oracle_row(N, K, K > 0 ? A + i * lda : A,",
                    "oracle_row(N, K, K > 0 ? A + i * K : A,"),
    "ignores_ldb": ("const float *brow = B + k * ldb;", "const float *brow = B + k * N;"),
    "no_init": ("\n        crow[j] = 0.0;\n", "\n        crow[j] = (j == 0) ? 1.0 : 0.0;\n"),
    "float_accumulate": ("\n            crow[j] += p;", "\n            crow[j] = (float)(crow[j] + p);"),
    "shifted_k_index": ("const double a = (double)arow[k];",
                        "const double a = (double)arow[k > 0 ? k - 1 : 0];"),
    "abs_without_abs": ("\n            if (srow) srow[j] += fabs(p);", "\n            if (srow) srow[j] += p;"),
    "rows_wrong_index": ("oracle_row(N, K, A + rows[r] * lda,", "oracle_row(N, K, A + r * lda,"),
    "cols_wrong_index": ("Bsel[k * ncols + c] = B[k * ldb + cols[c]];",
                         "Bsel[k * ncols + c] = B[k * ldb + c];"),
    "general_transposed_a_index": ("A[b * sa + i * lda + k] : A[b * sa + k * lda + i]",
                                   "A[b * sa + i * lda + k] : A[b * sa + i * lda + k]"),
    "general_transposed_b_index": ("B[b * sb + k * ldb + j] : B[b * sb + j * ldb + k]",
                                   "B[b * sb + k * ldb + j] : B[b * sb + k * ldb + j]"),
    "general_no_alpha": ("crow[j] = alpha * crow[j] + beta * c;", "crow[j] = crow[j] + beta * c;"),
    "general_beta_sign": ("crow[j] = alpha * crow[j] + beta * c;", "crow[j] = alpha * crow[j] - beta * c;"),
    "general_ignores_batch_stride_b": ("B[b * sb + k * ldb + j] :", "B[k * ldb + j] :"),
    "general_abs_without_alpha": ("srow[j] = fabs(alpha) * srow[j] + fabs(beta * c);",
                                  "srow[j] = srow[j] + fabs(beta * c);"),
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    src = tmp_path / f"{name}.c"
    src.write_text(source.replace(old, new))
    lib_path = oracle_pkg.compile_library(str(src), str(tmp_path / f"lib{name}.so"))
    mutant = oracle_pkg.Oracle(oracle_pkg.load_library(lib_path))
    failures = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(mutant)
        except (AssertionError, ValueError):
            failures.append(check.__name__)
    assert failures, f"mutant {name} passed every pin"
