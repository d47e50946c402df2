"""Failure detection on the GPU without a fault: a copy that is never issued
makes the kernel's bounded waits expire; the kernel reports a timeout through
the device error word and exits, and the context stays usable. A scratch
allocation that fails (made to, by a host-side test hook) sends an automatic
k-major choice to its row-major twin."""

import time

import numpy as np
import pytest
import torch

import dense_fp32_matrix_07_gb300 as sg
import workloads
from gpu_util import DeviceMatrix, assert_parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("slab", [0, 5])
def test_withheld_copy_times_out_and_the_context_survives(cuda_device, oracle, slab):
    M, N, K = 256, 256, 512          # 16 K slabs; two 128x256 tiles, whole-tile schedule
    A, B = workloads.make_operands(M, N, K, "int", 3)
    dA, dB = DeviceMatrix(A, M, K, K), DeviceMatrix(B, K, N, N)
    dC = DeviceMatrix(None, M, N, N)
    s = torch.cuda.current_stream().cuda_stream
    assert sg.sgemm_check_status(s) == sg.SGEMM_OK
    t0 = time.perf_counter()
    assert sg.sgemm_test_withhold_copy(M, N, K, dA.ptr, K, dB.ptr, N, dC.ptr, N, slab, s) == sg.SGEMM_OK
    assert sg.sgemm_check_status(s) == sg.SGEMM_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 0.5 < elapsed < 20.0, elapsed            # the waits gave up after about a second
    assert sg.sgemm_check_status(s) == sg.SGEMM_OK   # the word was cleared
    # The same context still computes correct products.
    assert sg.sgemm(M, N, K, dA.ptr, K, dB.ptr, N, dC.ptr, N, s) == sg.SGEMM_OK
    assert sg.sgemm_check_status(s) == sg.SGEMM_OK
    Cref, S = oracle.sgemm(M, N, K, A.numpy(), K, B.numpy(), N)
    assert_parity(dC.matrix(), Cref, S, True, "after the timeout")


def test_negative_slab_is_a_plain_product(cuda_device, oracle):
    M, N, K = 200, 300, 100
    A, B = workloads.make_operands(M, N, K, "uniform", 4)
    dA, dB = DeviceMatrix(A, M, K, K), DeviceMatrix(B, K, N, N)
    dC = DeviceMatrix(None, M, N, N)
    s = torch.cuda.current_stream().cuda_stream
    assert sg.sgemm_test_withhold_copy(M, N, K, dA.ptr, K, dB.ptr, N, dC.ptr, N, -1, s) == sg.SGEMM_OK
    assert sg.sgemm_check_status(s) == sg.SGEMM_OK
    Cref, S = oracle.sgemm(M, N, K, A.numpy(), K, B.numpy(), N)
    assert_parity(dC.matrix(), Cref, S, False, "slab -1")


@pytest.mark.parametrize("shape", [(600, 513, 257), (1000, 1000, 1000)])
def test_cluster_pair_split_tiles_need_no_cooperative_launch(cuda_device, oracle, shape):
    # Shapes whose pair-kernel schedule splits the leftover tiles in K (the
    # first is smoke()'s): the launch carries only its cluster shape, the
    # last part of each split tile reduces it, and the product is exact.
    M, N, K = shape
    A, B = workloads.make_operands(M, N, K, "int", 6)
    dA, dB = DeviceMatrix(A, M, K, K), DeviceMatrix(B, K, N, N)
    dC = DeviceMatrix(None, M, N, N)
    s = torch.cuda.current_stream().cuda_stream
    pair = sg.config_ids()["tf32x3_pair_128x256_k16_s4"]
    Cref, S = oracle.sgemm(M, N, K, A.numpy(), K, B.numpy(), N)
    for _ in range(2):
        assert sg.sgemm_ex(M, N, K, dA.ptr, K, dB.ptr, N, dC.ptr, N, pair, s) == sg.SGEMM_OK
        assert sg.sgemm_check_status(s) == sg.SGEMM_OK
        assert_parity(dC.matrix(), Cref, S, True, f"pair kernel {shape}")


def test_kmajor_choice_falls_back_when_its_scratch_cannot_be_had(cuda_device, oracle):
    # N >= 2048, M*N*K >= 6e9 and enough 128x128 tiles: the automatic choice
    # is a k-major configuration, which needs scratch for the transposed A.
    # With that allocation failing, the row-major twin runs the product
    # instead.
    M, N, K = 1024, 2048, 2944
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rc, cfg, pa, _ = sg.sgemm_plan(M, N, K, K, N, N, 0, 0, 0, sms)
    assert rc == 0 and sg.sgemm_config_name(cfg).endswith("_ka") and pa == 1
    A, B = workloads.make_operands(M, N, K, "int", 11)
    dA, dB = DeviceMatrix(A, M, K, K), DeviceMatrix(B, K, N, N)
    dC = DeviceMatrix(None, M, N, N)
    s = torch.cuda.current_stream().cuda_stream
    Cref, S = oracle.sgemm(M, N, K, A.numpy(), K, B.numpy(), N)
    try:
        assert sg.sgemm_test_fail_next_allocs(1) == sg.SGEMM_OK
        assert sg.sgemm(M, N, K, dA.ptr, K, dB.ptr, N, dC.ptr, N, s) == sg.SGEMM_OK
        assert sg.sgemm_check_status(s) == sg.SGEMM_OK
        assert_parity(dC.matrix(), Cref, S, True, "row-major twin after the failed allocation")
        # Forced, the k-major configuration has nowhere to go: it reports the
        # failure and enqueues nothing (C keeps its sentinel).
        dC2 = DeviceMatrix(None, M, N, N)
        before = dC2.matrix().clone()
        assert sg.sgemm_test_fail_next_allocs(1) == sg.SGEMM_OK
        assert sg.sgemm_ex(M, N, K, dA.ptr, K, dB.ptr, N, dC2.ptr, N, cfg, s) == sg.SGEMM_ERR_ALLOC
        torch.cuda.synchronize()
        assert torch.equal(dC2.matrix().view(torch.int32), before.view(torch.int32))
    finally:
        sg.sgemm_test_fail_next_allocs(0)
    # With no failure pending, the k-major configuration itself runs.
    assert sg.sgemm_ex(M, N, K, dA.ptr, K, dB.ptr, N, dC.ptr, N, cfg, s) == sg.SGEMM_OK
    assert sg.sgemm_check_status(s) == sg.SGEMM_OK
    assert_parity(dC.matrix(), Cref, S, True, "k-major")
