"""Failure detection on the GPU without a fault: a copy that is never issued
makes the kernel's bounded waits expire; the kernel reports a timeout through
the device error word and exits, and the context stays usable. A cluster
kernel launched without its cluster notices before it touches anything and
reports a launch error."""

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


@pytest.mark.parametrize("n", [512, 1000])
def test_cluster_kernel_refuses_a_launch_without_its_cluster(cuda_device, oracle, n):
    # 512^3: whole tiles; 1000^3: ragged edges. In both the check comes first.
    A, B = workloads.make_operands(n, n, n, "int", 6)
    dA, dB = DeviceMatrix(A, n, n, n), DeviceMatrix(B, n, n, n)
    sentinel = torch.full((n, n), 7.0)
    dC = DeviceMatrix(sentinel, n, n, n)
    s = torch.cuda.current_stream().cuda_stream
    assert sg.sgemm_check_status(s) == sg.SGEMM_OK
    assert sg.sgemm_test_launch_without_cluster(n, n, n, dA.ptr, n, dB.ptr, n, dC.ptr, n, s) == sg.SGEMM_OK
    assert sg.sgemm_check_status(s) == sg.SGEMM_ERR_LAUNCH
    assert torch.equal(dC.matrix(), sentinel)        # nothing was written
    assert sg.sgemm_check_status(s) == sg.SGEMM_OK   # the word was cleared
    # The same configuration with its cluster computes the exact product.
    pair = sg.config_ids()["tf32x3_pair_128x256_k16_s4"]
    assert sg.sgemm_ex(n, n, n, dA.ptr, n, dB.ptr, n, dC.ptr, n, pair, s) == sg.SGEMM_OK
    assert sg.sgemm_check_status(s) == sg.SGEMM_OK
    Cref, S = oracle.sgemm(n, n, n, A.numpy(), n, B.numpy(), n)
    assert_parity(dC.matrix(), Cref, S, True, "pair kernel after the refused launch")
