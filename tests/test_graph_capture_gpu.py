"""sgemm calls captured in a CUDA graph and replayed: the library's work on a
stream (pool scratch, the layout pass and the product queued behind it with
programmatic serialization, the row-tail kernel behind the product, cluster
launches) must be capturable, and a replay must compute the product of the
inputs present at replay time. Checked against the oracle."""

import numpy as np
import pytest
import torch

import dense_fp32_matrix_07_gb300 as sg
import workloads

pytestmark = pytest.mark.gpu

IDS = sg.config_ids()


def _capture_and_replay(oracle, M, N, K, config):
    dA = torch.empty((M, K), device="cuda")
    dB = torch.empty((K, N), device="cuda")
    dC = torch.full((M, N), float("nan"), device="cuda")
    side = torch.cuda.Stream()
    # Warm-up outside the capture: per-device set-up happens on the first call.
    A0, B0 = workloads.make_operands(M, N, K, "int", 1)
    dA.copy_(A0)
    dB.copy_(B0)
    with torch.cuda.stream(side):
        assert sg.sgemm_ex(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N, config,
                           side.cuda_stream) == sg.SGEMM_OK
    side.synchronize()
    assert sg.sgemm_check_status(side.cuda_stream) == sg.SGEMM_OK

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        rc = sg.sgemm_ex(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N, config,
                         side.cuda_stream)
    assert rc == sg.SGEMM_OK, sg.sgemm_error_string(rc)

    for seed, dist in ((2, "int"), (3, "uniform"), (4, "int")):
        A, B = workloads.make_operands(M, N, K, dist, seed)
        dA.copy_(A)
        dB.copy_(B)
        dC.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert sg.sgemm_check_status(side.cuda_stream) == sg.SGEMM_OK
        Cref, S = oracle.sgemm(M, N, K, A.numpy(), K, B.numpy(), N)
        C = dC.cpu().numpy().astype(np.float64)
        if dist == "int":
            assert np.array_equal(C, Cref.astype(np.float32).astype(np.float64)), seed
        else:
            assert np.all(np.abs(C - Cref) <= 1e-4 * S), seed


@pytest.mark.parametrize("config_name", [None, "ffma2_128x256_k32_s4_sk", "ffma2_128x256_k32_s4_ka",
                                         "ffma2_128x128_k32_s4", "tf32x3_pair_128x256_k16_s4"])
def test_captured_products_replay_correctly(cuda_device, oracle, config_name):
    # Several tiles, ragged edges (K = 515 also trims the last slab), the
    # layout pass of the k-major configuration, the stream-K tail.
    _capture_and_replay(oracle, 700, 900, 515, -1 if config_name is None else IDS[config_name])


@pytest.mark.parametrize("M,N,K", [(385, 1024, 2048), (1153, 2048, 2560), (200, 300, 150)])
def test_captured_launch_chains_replay_correctly(cuda_device, oracle, M, N, K):
    # The automatic choice: the one-block counter zeroing, the product behind
    # it and the row-tail kernel behind the product (385 rows; 1153 rows with
    # the k-major layout pass first), and the small-product kernel.
    _capture_and_replay(oracle, M, N, K, -1)


def test_captured_general_form_with_packing(cuda_device, oracle):
    # A stored transposed with an odd leading dimension (packed into pool
    # scratch inside the graph), alpha/beta, a batch of two.
    M, N, K, batch = 300, 260, 130, 2
    lda, ldb, ldc = M + 3, N, N + 1
    sa, sb, sc = K * lda, K * ldb, M * ldc
    dA = torch.empty(batch * sa, device="cuda")
    dB = torch.empty(batch * sb, device="cuda")
    dC = torch.empty(batch * sc, device="cuda")
    side = torch.cuda.Stream()

    def call():
        return sg.sgemm_general(1, 0, M, N, K, -0.5, dA.data_ptr(), lda, sa, dB.data_ptr(), ldb, sb, 2.0,
                                dC.data_ptr(), ldc, sc, batch, side.cuda_stream)

    with torch.cuda.stream(side):
        assert call() == sg.SGEMM_OK
    side.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        assert call() == sg.SGEMM_OK
    g = torch.Generator("cpu").manual_seed(7)
    A = torch.randint(-4, 5, (batch * sa,), generator=g).float()
    B = torch.randint(-4, 5, (batch * sb,), generator=g).float()
    C0 = torch.randint(-4, 5, (batch * sc,), generator=g).float()
    dA.copy_(A)
    dB.copy_(B)
    dC.copy_(C0)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert sg.sgemm_check_status(side.cuda_stream) == sg.SGEMM_OK
    Cref, _ = oracle.sgemm_general(1, 0, M, N, K, -0.5, A.numpy(), lda, sa, B.numpy(), ldb, sb, 2.0,
                                   C0.numpy(), ldc, sc, batch)
    out = dC.cpu().numpy()
    for b in range(batch):
        got = np.stack([out[b * sc + r * ldc: b * sc + r * ldc + N] for r in range(M)])
        assert np.array_equal(got, Cref[b].astype(np.float32)), b
