"""sgemm_noalloc(): the entry point for callers that cannot allocate device
memory (their device memory belongs to another allocator or a fixed arena,
or their loop may not take the driver's allocation path).

It must give the same product as sgemm() — within the tolerance every parity
test here uses, |diff| <= 1e-4 * sum_k |A_ik B_kj| — including when operands
need packing (which sgemm() does in allocated scratch and sgemm_noalloc()
does in the library's fixed 64 MiB array), on two calls in a row that reuse
that array, and it must refuse work whose packed operands would not fit.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process.
"""

import pytest
import torch

import dense_fp32_matrix_07_gb300 as sg
import workloads
from gpu_util import SENTINEL, TOL, DeviceMatrix, assert_parity

pytestmark = pytest.mark.gpu


def _both(oracle, M, N, K, lda, ldb, ldc, offsets, dist, seed):
    A, B = workloads.make_operands(M, N, K, dist, seed, lda, ldb)
    dA = DeviceMatrix(A, M, K, lda, offsets[0])
    dB = DeviceMatrix(B, K, N, ldb, offsets[1])
    dC_ref = DeviceMatrix(None, M, N, ldc, offsets[2])
    dC_new = DeviceMatrix(None, M, N, ldc, offsets[2])
    s = torch.cuda.current_stream().cuda_stream
    assert sg.sgemm(M, N, K, dA.ptr, lda, dB.ptr, ldb, dC_ref.ptr, ldc, s) == sg.SGEMM_OK
    assert sg.sgemm_noalloc(M, N, K, dA.ptr, lda, dB.ptr, ldb, dC_new.ptr, ldc, s) == sg.SGEMM_OK
    torch.cuda.synchronize()
    assert sg.sgemm_check_status(s) == sg.SGEMM_OK
    assert dC_new.guard_intact(), "sgemm_noalloc wrote outside C"
    if ldc > N:
        assert bool((dC_new.matrix()[:, N:] == SENTINEL).all())
    c_ref = dC_ref.matrix()[:, :N]
    c_new = dC_new.matrix()[:, :N]
    _, S = oracle.sgemm(M, N, K, A.numpy(), lda, B.numpy(), ldb)
    diff = (c_new.double() - c_ref.double()).abs().numpy()
    assert (diff <= TOL * S).all(), f"sgemm_noalloc differs from sgemm beyond 1e-4*S ({M}x{N}x{K})"
    return A, B, c_new, S


# (M, N, K, lda, ldb, ldc, pointer offsets in floats): both operands packed,
# only A packed (odd base address), nothing packed.
CASES = [
    (517, 389, 1000, 1003, 391, 389, (0, 0, 0)),
    (300, 257, 129, 129, 257, 257, (1, 0, 2)),
    (256, 256, 256, 256, 256, 256, (0, 0, 0)),
]


@pytest.mark.parametrize("case", CASES, ids=["pack_AB", "pack_A", "aligned"])
def test_noalloc_matches_sgemm_on_two_calls_in_a_row(cuda_device, oracle, case):
    M, N, K, lda, ldb, ldc, offs = case
    # Two calls in a row share the scratch array; the second uses other data.
    for call, seed in enumerate((11, 12)):
        dist = "uniform" if call == 0 else "int"
        A, B, c_new, S = _both(oracle, M, N, K, lda, ldb, ldc, offs, dist, seed)
        Cref, S = oracle.sgemm(M, N, K, A.numpy(), lda, B.numpy(), ldb)
        assert_parity(c_new, Cref, S, dist == "int", f"noalloc call {call}")


@pytest.mark.parametrize("shape", [(1024, 2048, 2944), (8192, 2048, 2052)], ids=["kmajor_copy", "twin"])
def test_noalloc_kmajor_choice(cuda_device, oracle, shape):
    # N >= 2048 and M*N*K >= 6e9: sgemm() takes a k-major configuration and
    # transposes A into pool scratch. sgemm_noalloc() makes that copy in its
    # fixed array when it fits (1024 x 2048 x 2944: 2944 x 1024 floats), else
    # runs the twin that reads A as stored (8192 x 2048 x 2052: the copy
    # would be 2052 x 8192 floats, over 16 Mi, while A's rows, 2052 floats,
    # need no pack). Integer inputs: both give the exact product.
    M, N, K = shape
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rc, cfg, pa, _ = sg.sgemm_plan(M, N, K, K, N, N, 0, 0, 0, sms)
    assert rc == 0 and sg.sgemm_config_name(cfg).endswith("_ka") and pa == 1
    for call, seed in enumerate((31, 32) if M * N * K < 1 << 32 else (31,)):
        A, B, c_new, S = _both(oracle, M, N, K, K, N, N, (0, 0, 0), "int", seed)
        Cref, S = oracle.sgemm(M, N, K, A.numpy(), K, B.numpy(), N)
        assert_parity(c_new, Cref, S, True, f"noalloc {shape} call {call}")


def test_noalloc_back_to_back_calls_with_shrinking_operands(cuda_device, oracle):
    # A large packed call leaves data in the whole array; a smaller one right
    # after it on the same stream must only see its own operands.
    _both(oracle, 2049, 1001, 2047, 2049, 1003, 1001, (0, 0, 0), "normal", 21)
    _both(oracle, 65, 33, 17, 19, 35, 33, (3, 1, 0), "normal", 22)


def test_noalloc_refuses_operands_beyond_its_scratch(cuda_device):
    # A with 4097 x 4097 and lda = 4097 packs into 4097 * 4128 floats > 16 Mi.
    M = K = 4097
    N = 8
    dA = DeviceMatrix(None, M, K, K, fill=1.0)
    dB = DeviceMatrix(None, K, N, N, fill=1.0)
    dC = DeviceMatrix(None, M, N, N)
    s = torch.cuda.current_stream().cuda_stream
    rc = sg.sgemm_noalloc(M, N, K, dA.ptr, K, dB.ptr, N, dC.ptr, N, s)
    assert rc == sg.SGEMM_ERR_SCRATCH_LIMIT
    assert "64 MiB" in sg.sgemm_error_string(rc)
    torch.cuda.synchronize()
    assert bool((dC.matrix() == SENTINEL).all()), "a refused call wrote C"
    # The same operands through sgemm() (allocated scratch) work.
    assert sg.sgemm(M, N, K, dA.ptr, K, dB.ptr, N, dC.ptr, N, s) == sg.SGEMM_OK
    torch.cuda.synchronize()
    assert bool((dC.matrix() == float(K)).all())
