"""GPU parity of the general form C_b = alpha * op(A_b) . op(B_b) + beta * C_b
(sgemm_general) against the oracle's general function: both operand
orientations, alpha/beta, strided and shared (stride 0) batches, across the
FFMA and 3xTF32 configurations, including forced stream-K splits."""

import numpy as np
import pytest
import torch

import dense_fp32_matrix_07_gb300 as sg
import workloads

pytestmark = pytest.mark.gpu

IDS = sg.config_ids()
CONFIGS = [-1, IDS["ffma2_128x128_k32_s4"], IDS["ffma2_128x256_k32_s4_sk"], IDS["ffma2_128x256_k32_s4_ka"],
           IDS["ffma2_128x128_k32_s4_sk"],
           IDS["ffma_128x128_k32_s4"], IDS["tf32x3_128x256_k16_s4"], IDS["tf32x3_128x256_k16_s4_sk"],
           IDS["tf32x3_pair_128x256_k16_s4"]]
CFG_IDS = ["auto" if c < 0 else sg.sgemm_config_name(c) for c in CONFIGS]


def _entries(rows, cols, ld, stride, batch, dist, seed, pad_fill=float("nan")):
    """A flat float32 buffer holding `batch` rows x cols matrices (leading
    dimension ld, batch stride `stride`; stride 0 = one shared matrix)."""
    n = (batch - 1) * stride + (rows - 1) * ld + cols if rows and cols else 1
    buf = torch.full((max(n, 1),), pad_fill, dtype=torch.float32)
    for b in range(batch if stride else 1):
        m, _ = workloads.make_operands(rows, 1, cols, dist, seed + b)
        view = buf[b * stride: b * stride + (rows - 1) * ld + cols]
        for r in range(rows):
            view[r * ld: r * ld + cols] = m[r]
    return buf


def _run(op_a, op_b, M, N, K, alpha, beta, batch, config, dist="uniform", seed=0,
         pad=(3, 5, 2), extra_stride=(7, 0, 9), shared=(False, False)):
    a_rows, a_cols = (K, M) if op_a else (M, K)
    b_rows, b_cols = (N, K) if op_b else (K, N)
    lda, ldb, ldc = a_cols + pad[0], b_cols + pad[1], N + pad[2]
    sa = 0 if shared[0] else a_rows * lda + extra_stride[0]
    sb = 0 if shared[1] else b_rows * ldb + extra_stride[1]
    sc = M * ldc + extra_stride[2]
    A = _entries(a_rows, a_cols, lda, sa, batch, dist, seed)
    B = _entries(b_rows, b_cols, ldb, sb, batch, dist, seed + 100)
    Cin = _entries(M, N, ldc, sc, batch, dist, seed + 200, pad_fill=7.0)
    if beta == 0.0:
        for b in range(batch):   # C must not be read: poison the live entries
            for r in range(M):
                Cin[b * sc + r * ldc: b * sc + r * ldc + N] = float("nan")
    dA, dB, dC = A.cuda(), B.cuda(), Cin.clone().cuda()
    s = torch.cuda.current_stream().cuda_stream
    rc = sg.sgemm_general_ex(op_a, op_b, M, N, K, alpha, dA.data_ptr(), lda, sa, dB.data_ptr(), ldb, sb,
                             beta, dC.data_ptr(), ldc, sc, batch, config, s)
    torch.cuda.synchronize()
    assert sg.sgemm_check_status(s) == 0
    out = dC.cpu()
    return rc, A, B, Cin, out, (lda, ldb, ldc, sa, sb, sc)


def _check(oracle, op_a, op_b, M, N, K, alpha, beta, batch, A, B, Cin, out, lds, exact):
    lda, ldb, ldc, sa, sb, sc = lds
    Cref, S = oracle.sgemm_general(op_a, op_b, M, N, K, alpha, A.numpy(), lda, sa, B.numpy(), ldb, sb,
                                   beta, Cin.numpy() if beta != 0 else None, ldc, sc, batch)
    for b in range(batch):
        got = np.stack([out[b * sc + r * ldc: b * sc + r * ldc + N].numpy() for r in range(M)]).astype(np.float64)
        if exact:
            assert np.array_equal(got, Cref[b].astype(np.float32).astype(np.float64)), b
        else:
            bad = np.abs(got - Cref[b]) > 1e-4 * S[b]
            assert not bad.any(), (b, np.argwhere(bad)[:3])
    # Every float outside the live M x N entries (row padding, gaps between
    # batch entries) is left as it was.
    live = torch.zeros(out.numel(), dtype=torch.bool)
    for b in range(batch):
        for r in range(M):
            live[b * sc + r * ldc: b * sc + r * ldc + N] = True
    assert torch.equal(out[~live], Cin[~live])

@pytest.mark.parametrize("config", CONFIGS, ids=CFG_IDS)
@pytest.mark.parametrize("op_a,op_b", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_ops_alpha_beta_batch(cuda_device, oracle, config, op_a, op_b):
    M, N, K, batch = 150, 200, 70, 3
    for alpha, beta in ((1.0, 0.0), (-1.5, 0.0), (0.75, 2.0)):
        rc, A, B, Cin, out, lds = _run(op_a, op_b, M, N, K, alpha, beta, batch, config, seed=op_a * 2 + op_b)
        assert rc == 0, sg.sgemm_error_string(rc)
        _check(oracle, op_a, op_b, M, N, K, alpha, beta, batch, A, B, Cin, out, lds, exact=False)


@pytest.mark.parametrize("config", CONFIGS, ids=CFG_IDS)
def test_integer_exact_with_alpha_beta(cuda_device, oracle, config):
    M, N, K, batch = 257, 129, 300, 2
    rc, A, B, Cin, out, lds = _run(1, 0, M, N, K, 2.0, -1.0, batch, config, dist="int", seed=5)
    assert rc == 0
    _check(oracle, 1, 0, M, N, K, 2.0, -1.0, batch, A, B, Cin, out, lds, exact=True)


@pytest.mark.parametrize("config", [-1, IDS["ffma2_128x256_k32_s4"], IDS["ffma2_128x256_k32_s4_ka"],
                                    IDS["tf32x3_128x256_k16_s4"]],
                         ids=["auto", "ffma2_128x256", "ffma2_128x256_ka", "tf32x3"])
@pytest.mark.parametrize("shared", [(True, False), (False, True)], ids=["shared_A", "shared_B"])
def test_shared_operand_across_the_batch(cuda_device, oracle, config, shared):
    M, N, K, batch = 300, 260, 130, 4
    rc, A, B, Cin, out, lds = _run(0, 0, M, N, K, 1.0, 0.0, batch, config, shared=shared, pad=(0, 0, 0),
                                   extra_stride=(0, 0, 0))
    assert rc == 0
    _check(oracle, 0, 0, M, N, K, 1.0, 0.0, batch, A, B, Cin, out, lds, exact=False)


def test_aligned_batch_runs_in_place_and_many_small_entries(cuda_device, oracle):
    # 16-byte-aligned strides: no packing; 40 small entries share one launch.
    M, N, K, batch = 64, 96, 48, 40
    rc, A, B, Cin, out, lds = _run(0, 0, M, N, K, 1.0, 1.0, batch, -1, pad=(0, 0, 0), extra_stride=(0, 0, 0))
    assert rc == 0
    _check(oracle, 0, 0, M, N, K, 1.0, 1.0, batch, A, B, Cin, out, lds, exact=False)


def test_alpha_zero_scales_c_without_reading_a_or_b(cuda_device):
    M, N, batch, ldc, sc = 33, 40, 2, 45, 33 * 45 + 3
    Cin = torch.randn(batch * sc)
    for beta in (0.0, 1.0, -2.5):
        dC = Cin.clone().cuda()
        s = torch.cuda.current_stream().cuda_stream
        assert sg.sgemm_general(0, 0, M, N, 17, 0.0, 0, 17, 0, 0, N, 0, beta, dC.data_ptr(), ldc, sc, batch, s) == 0
        torch.cuda.synchronize()
        out = dC.cpu()
        for b in range(batch):
            for r in range(M):
                o = b * sc + r * ldc
                want = Cin[o:o + N] * beta if beta != 0 else torch.zeros(N)
                assert torch.equal(out[o:o + N], want)
                assert torch.equal(out[o + N:o + ldc], Cin[o + N:o + ldc])


def test_rejected_general_arguments(cuda_device):
    dA = torch.zeros(4096, device="cuda")
    dC = torch.zeros(4096, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    E = sg.SGEMM_ERR_INVALID_VALUE
    p, c = dA.data_ptr(), dC.data_ptr()
    assert sg.sgemm_general(2, 0, 8, 8, 8, 1.0, p, 8, 0, p, 8, 0, 0.0, c, 8, 64, 1, s) == E       # bad op
    assert sg.sgemm_general(0, 0, 8, 8, 8, 1.0, p, 8, -1, p, 8, 0, 0.0, c, 8, 64, 2, s) == E      # negative stride
    assert sg.sgemm_general(0, 0, 8, 8, 8, 1.0, p, 8, 0, p, 8, 0, 0.0, c, 8, 63, 2, s) == E       # C entries overlap
    assert sg.sgemm_general(1, 0, 8, 9, 4, 1.0, p, 7, 0, p, 9, 0, 0.0, c, 9, 72, 1, s) == E       # lda < M for op_a=1
    assert sg.sgemm_general_ex(0, 0, 8, 8, 8, 2.0, p, 8, 0, p, 8, 0, 0.0, c, 8, 64, 1,
                               IDS["tiled16_simple"], s) == sg.SGEMM_ERR_UNSUPPORTED
    assert sg.sgemm_general(0, 0, 8, 8, 8, 1.0, p, 8, 0, p, 8, 0, 0.0, c, 8, 64, 0, s) == sg.SGEMM_OK  # empty batch
    torch.cuda.synchronize()
    assert bool((dC == 0).all())


@pytest.mark.parametrize("M,N,K", [(1024, 1024, 64), (2048, 2560, 64)], ids=["128x128_tiles", "128x256_tiles"])
def test_transposed_a_read_in_place_by_the_kmajor_configurations(cuda_device, oracle, M, N, K):
    # Large enough for the automatic choice to take 128x128 or 128x256 tiles;
    # for an A stored transposed on aligned rows (lda = M, a multiple of 4,
    # tight batch stride) that means a k-major configuration reading it in
    # place, with no pack. Integer inputs, so the result is exact.
    batch = 2
    rc, A, B, Cin, out, lds = _run(1, 0, M, N, K, 1.0, 0.0, batch, -1, dist="int", seed=9, pad=(0, 0, 0),
                                   extra_stride=(0, 0, 0))
    assert rc == 0
    _check(oracle, 1, 0, M, N, K, 1.0, 0.0, batch, A, B, Cin, out, lds, exact=True)
