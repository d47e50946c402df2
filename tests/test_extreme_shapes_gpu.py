"""Degenerate and extreme shapes on the GPU against the oracle: a 4M-long dot
product (one tile split over every CTA by stream-K), tall and wide skinny
products, and the largest row and column counts the library accepts
(2^31 - 1), which exercise its 64-bit index arithmetic.

The giant operands are generated on the device in chunks from an integer
hash of the element index, v(i) = ((i * 2654435761) mod 2^32) mod 17 - 8
(integers in [-8, 8]); the oracle gets the same values for the sampled rows
or columns by evaluating that formula on the host. All products are of
integer-valued inputs whose sums stay below 2^24 in magnitude, so every
checked element must be bit-exact."""

import numpy as np
import pytest
import torch

import dense_fp32_matrix_07_gb300 as sg
import workloads

pytestmark = pytest.mark.gpu

SENTINEL = 12345.0


def _hash_values(idx: np.ndarray) -> np.ndarray:
    return (((idx.astype(np.uint64) * np.uint64(2654435761)) % np.uint64(2 ** 32)) % np.uint64(17)).astype(
        np.int64) - 8


def _fill_hashed(dst: torch.Tensor, count: int, stride: int = 1, chunk: int = 1 << 27):
    """dst[i * stride] = v(i) for i < count, on the device, chunk by chunk."""
    for start in range(0, count, chunk):
        n = min(chunk, count - start)
        i = torch.arange(start, start + n, dtype=torch.int64, device=dst.device)
        v = (((i * 2654435761) % (2 ** 32)) % 17 - 8).to(torch.float32)
        dst[start * stride: (start + n - 1) * stride + 1: stride] = v
        del i, v


def _status_ok():
    assert sg.sgemm_check_status(torch.cuda.current_stream().cuda_stream) == sg.SGEMM_OK


def test_long_k_dot_product(cuda_device, oracle):
    K = 1 << 22
    g = torch.Generator("cpu").manual_seed(11)
    a = torch.randint(-1, 2, (1, K), generator=g).to(torch.float32)
    b = torch.randint(-1, 2, (K, 1), generator=g).to(torch.float32)
    dA, dB = a.cuda(), b.cuda()
    Cref, _ = oracle.sgemm(1, 1, K, a.numpy(), K, b.numpy(), 1)
    for ldb in (1, 4):                                  # packed B, then B read in place
        dBl = torch.zeros((K, ldb), device="cuda")
        dBl[:, 0] = dB[:, 0]
        dC = torch.full((1, 1), float("nan"), device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        assert sg.sgemm(1, 1, K, dA.data_ptr(), K, dBl.data_ptr(), ldb, dC.data_ptr(), 1, s) == sg.SGEMM_OK
        _status_ok()
        assert float(dC.item()) == float(np.float32(Cref[0, 0])), ldb


@pytest.mark.parametrize("M,N,K", [((1 << 20) + 3, 3, 5), (3, (1 << 20) + 7, 5), (5000, 4, 300)])
def test_skinny_products(cuda_device, oracle, M, N, K):
    A, B = workloads.make_operands(M, N, K, "int", 21)
    dA, dB = A.cuda(), B.cuda()
    dC = torch.full((M, N), float("nan"), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert sg.sgemm(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N, s) == sg.SGEMM_OK
    _status_ok()
    Cref, _ = oracle.sgemm(M, N, K, A.numpy(), K, B.numpy(), N)
    assert np.array_equal(dC.cpu().numpy(), Cref.astype(np.float32))


def _sample(n, count, seed):
    # Random indices plus both ends, drawn without materialising range(n).
    idx = np.random.default_rng(seed).integers(0, n, count, dtype=np.int64)
    return np.unique(np.concatenate([idx, np.arange(8), np.arange(n - 8, n)]))


@pytest.mark.parametrize("config_name", [None, "tf32x3_pair_128x256_k16_s4"])
def test_largest_column_count(cuda_device, oracle, config_name):
    # M = 1, K = 1, N = 2^31 - 1: C row 0 = A00 * B row 0. ldc = 2^31 (C rows
    # 16-byte aligned: vector stores up to the last full group of columns).
    N = (1 << 31) - 1
    ldc = 1 << 31
    a00 = 3.0
    dA = torch.full((1, 1), a00, device="cuda")
    dB = torch.empty(N, device="cuda")
    _fill_hashed(dB, N)
    dC = torch.full((ldc,), SENTINEL, device="cuda")
    config = -1 if config_name is None else sg.config_ids()[config_name]
    s = torch.cuda.current_stream().cuda_stream
    rc = sg.sgemm_ex(1, N, 1, dA.data_ptr(), 1, dB.data_ptr(), N, dC.data_ptr(), ldc, config, s)
    assert rc == sg.SGEMM_OK, sg.sgemm_error_string(rc)
    _status_ok()
    cols = _sample(N, 2000, 31)
    got = dC[torch.from_numpy(cols).cuda()].cpu().numpy()
    Bs = _hash_values(cols).astype(np.float32).reshape(1, -1)
    Cref, _ = oracle.sgemm(1, len(cols), 1, np.array([[a00]], dtype=np.float32), 1, Bs, len(cols))
    assert np.array_equal(got, Cref[0].astype(np.float32))
    assert float(dC[N].item()) == SENTINEL            # the padding column stays untouched
    del dA, dB, dC
    torch.cuda.empty_cache()


def test_largest_row_count(cuda_device, oracle):
    # M = 2^31 - 1, N = 1, K = 1, lda = 4 (A read in place): C[i] = A[i] * B00.
    M = (1 << 31) - 1
    b00 = -2.0
    dA = torch.zeros((M - 1) * 4 + 1, device="cuda")
    _fill_hashed(dA, M, stride=4)
    dB = torch.full((1, 1), b00, device="cuda")
    dC = torch.full((M,), SENTINEL, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = sg.sgemm(M, 1, 1, dA.data_ptr(), 4, dB.data_ptr(), 1, dC.data_ptr(), 1, s)
    assert rc == sg.SGEMM_OK, sg.sgemm_error_string(rc)
    _status_ok()
    rows = _sample(M, 2000, 41)
    got = dC[torch.from_numpy(rows).cuda()].cpu().numpy()
    As = _hash_values(rows).astype(np.float32).reshape(-1, 1)
    Cref, _ = oracle.sgemm(len(rows), 1, 1, As, 1, np.array([[b00]], dtype=np.float32), 1)
    assert np.array_equal(got, Cref[:, 0].astype(np.float32))
    del dA, dB, dC
    torch.cuda.empty_cache()
