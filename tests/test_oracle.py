"""The CPU oracle against its pins (no GPU). See tests/oracle_pins.py."""

import numpy as np
import pytest

import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(oracle, check):
    check(oracle)


def test_oracle_rejects_bad_arguments(oracle):
    A = np.zeros(64, np.float32)
    with pytest.raises(ValueError):
        oracle.sgemm(4, 4, 4, A, 3, A, 4)          # lda < K
    with pytest.raises(ValueError):
        oracle.sgemm(4, 4, 4, A, 4, A, 3)          # ldb < N
    with pytest.raises(ValueError):
        oracle.sgemm_rows(4, 4, 4, A, 4, A, 4, [4])  # row out of range
    with pytest.raises(ValueError):
        oracle.sgemm_cols(4, 4, 4, A, 4, A, 4, [-1])  # column out of range


def test_oracle_threads(oracle):
    assert oracle.num_threads() >= 1
