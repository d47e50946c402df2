"""Concurrent calls from several host threads, each on its own stream: the
per-device state, the scratch pool, the tensor-map encoder and the stream-K
workspaces must not interfere. ctypes releases the GIL for the duration of
each library call, so the calls overlap in the library and on the GPU. Every
product uses integer-valued inputs and must match the oracle bit for bit."""

import threading

import numpy as np
import pytest
import torch

import dense_fp32_matrix_07_gb300 as sg
import workloads

pytestmark = pytest.mark.gpu

IDS = sg.config_ids()


def test_concurrent_calls_on_separate_streams(cuda_device, oracle):
    # (M, N, K, lda, config): packed and in-place operands, stream-K tails,
    # the simple kernel and the 3xTF32 cluster-pair kernel.
    jobs = [
        (517, 389, 1000, 1003, -1),
        (1024, 1024, 1024, 1024, IDS["ffma2_128x128_k32_s4_sk"]),
        (300, 257, 129, 129, -1),
        (700, 900, 515, 515, IDS["tf32x3_pair_128x256_k16_s4"]),
        (640, 520, 300, 301, IDS["ffma2_128x256_k32_s4_ka"]),
    ]
    inputs, refs = [], []
    for n, (M, N, K, lda, _) in enumerate(jobs):
        A, B = workloads.make_operands(M, N, K, "int", 60 + n, lda=lda)
        inputs.append((A, B))
        Cref, _ = oracle.sgemm(M, N, K, A.numpy(), lda, B.numpy(), N)
        refs.append(Cref.astype(np.float32))
    errors = []
    results = [None] * len(jobs)

    def worker(n):
        try:
            M, N, K, lda, config = jobs[n]
            A, B = inputs[n]
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                dA, dB = A.cuda(), B.cuda()
                dC = torch.full((M, N), float("nan"), device="cuda")
                for _ in range(20):
                    rc = sg.sgemm_ex(M, N, K, dA.data_ptr(), lda, dB.data_ptr(), N, dC.data_ptr(), N, config,
                                     stream.cuda_stream)
                    if rc != sg.SGEMM_OK:
                        errors.append((n, sg.sgemm_error_string(rc)))
                        return
            stream.synchronize()
            results[n] = dC.cpu().numpy()
        except Exception as e:        # surfaced by the assertion below
            errors.append((n, repr(e)))

    threads = [threading.Thread(target=worker, args=(n,)) for n in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert sg.sgemm_check_status(torch.cuda.current_stream().cuda_stream) == sg.SGEMM_OK
    for n in range(len(jobs)):
        assert np.array_equal(results[n], refs[n]), n
