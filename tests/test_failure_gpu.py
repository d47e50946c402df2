"""Failure detection on the GPU without a fault: a copy that is never issued
makes the kernel's bounded waits expire; the kernel reports a timeout through
the device error word and exits, and the context stays usable."""

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
