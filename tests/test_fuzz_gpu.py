"""Seeded random cases of the general form C_b = alpha * op(A_b) . op(B_b) +
beta * C_b against the oracle's general function: shapes with ragged tails,
padded leading dimensions (some not multiples of four floats, so operands
are packed), odd batch strides, both operand orientations, alpha/beta,
shared operands, on every TMA configuration family and the automatic
choice. Integer-valued cases must be bit-exact."""

import numpy as np
import pytest
import torch

import dense_fp32_matrix_07_gb300 as sg

pytestmark = pytest.mark.gpu

IDS = sg.config_ids()
FAMILIES = [-1, IDS["ffma2_128x64_k32_s4"], IDS["ffma2_128x128_k32_s4_sk"], IDS["ffma2_128x256_k32_s4"],
            IDS["ffma2_128x256_k32_s4_ka"], IDS["ffma2_128x128_k32_s4_ka"], IDS["ffma_128x128_k32_s4"],
            IDS["tf32x3_128x256_k16_s4"], IDS["tf32x3_pair_128x256_k16_s4"]]
CASES_PER_FAMILY = 10


def _case(rng):
    M, N, K = (int(x) for x in rng.integers(1, 300, 3))
    op_a, op_b = (int(x) for x in rng.integers(0, 2, 2))
    batch = int(rng.integers(1, 4))
    a_rows, a_cols = (K, M) if op_a else (M, K)
    b_rows, b_cols = (N, K) if op_b else (K, N)
    lda, ldb, ldc = (c + int(rng.integers(0, 6)) for c in (a_cols, b_cols, N))
    shared_a, shared_b = rng.random() < 0.2, rng.random() < 0.2
    sa = 0 if (shared_a and batch > 1) else a_rows * lda + int(rng.integers(0, 5))
    sb = 0 if (shared_b and batch > 1) else b_rows * ldb + int(rng.integers(0, 5))
    sc = M * ldc + int(rng.integers(0, 5))
    alpha = float(rng.choice([1.0, -1.0, 0.5, 2.0]))
    beta = float(rng.choice([0.0, 0.0, 1.0, -0.5]))
    exact = rng.random() < 0.3
    return M, N, K, op_a, op_b, batch, lda, ldb, ldc, sa, sb, sc, alpha, beta, exact


def _buffer(rng, n, exact):
    if exact:
        return rng.integers(-4, 5, n).astype(np.float32)
    return (rng.random(n, dtype=np.float32) * 2 - 1).astype(np.float32)


@pytest.mark.parametrize("config", FAMILIES, ids=["auto" if c < 0 else sg.sgemm_config_name(c) for c in FAMILIES])
def test_random_general_cases(cuda_device, oracle, config):
    rng = np.random.default_rng(9000 + config)
    s = torch.cuda.current_stream().cuda_stream
    for case in range(CASES_PER_FAMILY):
        M, N, K, op_a, op_b, batch, lda, ldb, ldc, sa, sb, sc, alpha, beta, exact = _case(rng)
        a_rows = K if op_a else M
        b_rows = N if op_b else K
        na = (batch - 1) * sa + a_rows * lda
        nb = (batch - 1) * sb + b_rows * ldb
        nc = (batch - 1) * sc + M * ldc
        A, B, Cin = _buffer(rng, na, exact), _buffer(rng, nb, exact), _buffer(rng, nc, exact)
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        dC = torch.from_numpy(Cin).cuda()
        what = f"case {case}: {M}x{N}x{K} op {op_a}{op_b} batch {batch} ld {lda},{ldb},{ldc} " \
               f"strides {sa},{sb},{sc} alpha {alpha} beta {beta} exact {exact}"
        rc = sg.sgemm_general_ex(op_a, op_b, M, N, K, alpha, dA.data_ptr(), lda, sa, dB.data_ptr(), ldb, sb,
                                 beta, dC.data_ptr(), ldc, sc, batch, config, s)
        assert rc == sg.SGEMM_OK, (what, sg.sgemm_error_string(rc))
        assert sg.sgemm_check_status(s) == sg.SGEMM_OK, what
        out = dC.cpu().numpy()
        Cref, S = oracle.sgemm_general(op_a, op_b, M, N, K, alpha, A, lda, sa, B, ldb, sb,
                                       beta, Cin if beta != 0 else None, ldc, sc, batch)
        live = np.zeros(nc, dtype=bool)
        for b in range(batch):
            got = np.stack([out[b * sc + r * ldc: b * sc + r * ldc + N] for r in range(M)]).astype(np.float64)
            for r in range(M):
                live[b * sc + r * ldc: b * sc + r * ldc + N] = True
            if exact:
                assert np.array_equal(got, Cref[b].astype(np.float32).astype(np.float64)), what
            else:
                assert np.all(np.abs(got - Cref[b]) <= 1e-4 * S[b]), what
        assert np.array_equal(out[~live], Cin[~live]), what + ": a float outside C's entries changed"
