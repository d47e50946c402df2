"""GPU parity of the row-tail path: for M = 128 q + r (1 <= r <= 8) the TMA
configurations run the tiled product on the first M - r rows and a
kernel on the last r rows (CTAs that split K, the last of each column
block adding the parts in order). Every case is checked against the FP64
oracle over all of C (float inputs within 1e-4 * sum|A_ik B_kj|, integer
inputs bit-exact), with the planner confirming that the tail kernel runs."""

import pytest
import torch

import dense_fp32_matrix_07_gb300 as sg
import workloads
from gpu_util import assert_parity, check_untouched_padding, run

pytestmark = pytest.mark.gpu

FFMA_TMA = [n for n in (sg.sgemm_config_name(i) for i in range(sg.sgemm_num_configs())) if n.startswith("ffma")]


def _tail_rows(cfg, M, N, K, batch=1):
    rc, rows = sg.sgemm_plan_row_tail(cfg, M, N, K, batch)
    assert rc == 0
    return rows


@pytest.mark.parametrize("r", [1, 2, 5, 8])
@pytest.mark.parametrize("dist", ["normal", "int"])
def test_row_tail_automatic_choice(cuda_device, oracle, r, dist):
    # Ragged N and K too, and lda / ldb that are not multiples of 4 (packed B).
    M, N, K = 256 + r, 1003, 2101
    rc, cfg, _, _ = sg.sgemm_plan(M, N, K, K, N, N + 3, 0, 0, 0, torch.cuda.get_device_properties(0).multi_processor_count)
    assert rc == 0 and _tail_rows(cfg, M, N, K) == r
    A, B = workloads.make_operands(M, N, K, dist, 40 + r)
    rc, C, dC = run(M, N, K, A, K, B, N, ldc=N + 3)
    assert rc == 0
    Cref, S = oracle.sgemm(M, N, K, A.numpy(), K, B.numpy(), N)
    assert_parity(C, Cref, S, dist == "int", f"tail {r} {dist}")
    check_untouched_padding(dC, N)


@pytest.mark.parametrize("name", FFMA_TMA)
def test_row_tail_under_every_ffma_configuration(cuda_device, oracle, name):
    cfg = sg.config_ids()[name]
    M, N, K = 387, 1536, 1400          # 3 block rows + 3 rows
    assert _tail_rows(cfg, M, N, K) == 3
    for dist, exact in (("uniform", False), ("int", True)):
        A, B = workloads.make_operands(M, N, K, dist, 9)
        rc, C, dC = run(M, N, K, A, K, B, N, config=cfg, offsets=(1, 0, 0))
        assert rc == 0
        Cref, S = oracle.sgemm(M, N, K, A.numpy(), K, B.numpy(), N)
        assert_parity(C, Cref, S, exact, f"{name} {dist}")
        check_untouched_padding(dC, N)


def test_row_tail_of_the_odd_rectangle_shape(cuda_device, oracle):
    # 4097 x 3001 x 2049 runs 4096 rows tiled and one row in the tail kernel
    # (the named workload's full check covers it too; this one uses integers).
    w = workloads.WORKLOADS["rect4097x3001x2049"]
    rc, cfg, _, _ = sg.sgemm_plan(w.M, w.N, w.K, w.lda, w.ldb, w.ldc, 0, 0, 0,
                                  torch.cuda.get_device_properties(0).multi_processor_count)
    assert rc == 0 and _tail_rows(cfg, w.M, w.N, w.K) == 1
    A, B = workloads.make_operands(w.M, w.N, w.K, "int", 77, w.lda, w.ldb)
    rc, C, _ = run(w.M, w.N, w.K, A, w.lda, B, w.ldb, ldc=w.ldc)
    assert rc == 0
    Cref, S = oracle.sgemm(w.M, w.N, w.K, A.numpy(), w.lda, B.numpy(), w.ldb)
    assert_parity(C, Cref, S, True, "rect int")


@pytest.mark.parametrize("op_a,op_b,alpha,beta,batch", [
    (0, 0, 1.0, 0.0, 3),
    (1, 0, -0.5, 0.0, 2),
    (0, 1, 2.0, 1.5, 2),
    (1, 1, 1.0, -1.0, 3),
])
def test_row_tail_in_the_general_form(cuda_device, oracle, op_a, op_b, alpha, beta, batch):
    M, N, K = 262, 1100, 2000          # 2 block rows + 6 rows
    cfg = sg.config_ids()["ffma2_128x256_k32_s4"]
    assert _tail_rows(cfg, M, N, K, batch) == 6
    g = torch.Generator().manual_seed(5 + op_a + 2 * op_b)
    A = torch.randint(-4, 5, (batch, K, M) if op_a else (batch, M, K), generator=g).float()
    B = torch.randint(-4, 5, (batch, N, K) if op_b else (batch, K, N), generator=g).float()
    C0 = torch.randint(-4, 5, (batch, M, N), generator=g).float()
    dA, dB, dC = A.cuda(), B.cuda(), C0.cuda()
    lda, ldb = A.shape[2], B.shape[2]
    s = torch.cuda.current_stream().cuda_stream
    rc = sg.sgemm_general_ex(op_a, op_b, M, N, K, alpha, dA.data_ptr(), lda, A[0].numel(),
                             dB.data_ptr(), ldb, B[0].numel(), beta, dC.data_ptr(), N, M * N, batch, cfg, s)
    assert rc == 0
    torch.cuda.synchronize()
    assert sg.sgemm_check_status(s) == sg.SGEMM_OK
    C = dC.cpu()
    for b in range(batch):
        Ab = A[b].t() if op_a else A[b]
        Bb = B[b].t() if op_b else B[b]
        Cref, S = oracle.sgemm(M, N, K, Ab.contiguous().numpy(), K, Bb.contiguous().numpy(), N)
        want = alpha * Cref + beta * C0[b].double().numpy()
        # Integer inputs, alpha and beta exact in FP32: the result is exact.
        assert_parity(C[b], want, S, True, f"entry {b}")


@pytest.mark.parametrize("M,N,K", [(131, 300, 8000), (4097, 1024, 20000), (261, 2000, 12345)])
def test_row_tail_with_k_split_across_ctas(cuda_device, oracle, M, N, K):
    # Few column blocks, or a long K: up to 16 CTAs per column block split K
    # and the last to finish adds their sums in chunk order.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rc, cfg, _, _ = sg.sgemm_plan(M, N, K, K, N, N, 0, 0, 0, sms)
    assert rc == 0 and _tail_rows(cfg, M, N, K) == M % 128
    for dist, exact in (("normal", False), ("int", True)):
        A, B = workloads.make_operands(M, N, K, dist, 21)
        rc, C, dC = run(M, N, K, A, K, B, N)
        assert rc == 0
        Cref, S = oracle.sgemm(M, N, K, A.numpy(), K, B.numpy(), N)
        assert_parity(C, Cref, S, exact, f"{M}x{N}x{K} {dist}")
        check_untouched_padding(dC, N)


def test_row_tail_behind_layout_pass_with_idle_sms(cuda_device, oracle):
    # The tail kernel reads the copy of B that the call's layout pass writes.
    # Here B's rows are not 16-byte aligned (ldb = 2051), so the pass copies
    # B, and the forced whole-tile 128x256 configuration runs only 8 product
    # CTAs: most SMs stay free for the tail kernel the moment the product
    # lets it in. It must not read B's copy before the pass has completed.
    # Each repetition draws a new B, so a stale copy from the repetition
    # before (the pool hands back the same scratch) would show in row 128.
    cfg = sg.config_ids()["ffma2_128x256_k32_s4_dp"]
    M, N, K, ldb = 129, 2048, 1024, 2051
    rc, _, pa, pb = sg.sgemm_general_plan(0, 0, M, N, K, 1.0, K, 0, ldb, 0, 0.0, N, 0, 1, 0, 0, 0,
                                          torch.cuda.get_device_properties(0).multi_processor_count, cfg)
    assert rc == 0 and (pa, pb) == (0, 1) and _tail_rows(cfg, M, N, K) == 1
    for rep in range(20):
        A, B = workloads.make_operands(M, N, K, "int", 300 + rep, ldb=ldb)
        rc, C, dC = run(M, N, K, A, K, B, ldb, config=cfg)
        assert rc == 0
        Cref, S = oracle.sgemm(M, N, K, A.numpy(), K, B.numpy(), ldb)
        assert_parity(C, Cref, S, True, f"rep {rep}")
        check_untouched_padding(dC, N)
