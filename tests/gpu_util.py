"""Helpers of the GPU parity tests: device buffers with pointer offsets and
guard bands, one library call through the C ABI, and the parity bar.

The parity bar (the SGEMM tolerance):
  * float inputs: every checked element satisfies
        |C_gpu - C_ref| <= 1e-4 * S,   S = sum_k |A_ik * B_kj|
    with C_ref and S from the FP64 oracle;
  * integer-valued inputs whose partial sums stay below 2^24 in magnitude:
    C_gpu equals float32(C_ref) exactly (compared as values, so +0 == -0).
"""

from __future__ import annotations

import numpy as np
import torch

import dense_fp32_matrix_07_gb300 as sg

TOL = 1e-4
GUARD = 64            # floats of guard band after each buffer
SENTINEL = 12345.678  # value of the guard band and of C's untouched entries


class DeviceMatrix:
    """rows x cols matrix with leading dimension ld inside a flat device
    buffer, starting `offset` floats after the (256-byte-aligned) allocation
    and followed by a guard band."""

    def __init__(self, host: torch.Tensor | None, rows: int, cols: int, ld: int,
                 offset: int = 0, fill: float = SENTINEL):
        self.rows, self.cols, self.ld, self.offset = rows, cols, ld, offset
        self.extent = rows * ld if rows > 0 else 0
        self.buf = torch.full((offset + self.extent + GUARD,), fill,
                              dtype=torch.float32, device="cuda")
        if host is not None and self.extent > 0:
            flat = host.reshape(-1)[: self.extent]
            self.buf[offset: offset + flat.numel()] = flat.to("cuda")

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr() + 4 * self.offset

    def matrix(self) -> torch.Tensor:
        """The rows x ld view (CPU copy)."""
        return self.buf[self.offset: self.offset + self.extent].view(self.rows, self.ld).cpu()

    def guard_intact(self) -> bool:
        g = self.buf[self.offset + self.extent:]
        pre = self.buf[: self.offset]
        return bool((g == SENTINEL).all()) and bool((pre == SENTINEL).all())


def run(M, N, K, A, lda, B, ldb, ldc=None, config=-1, offsets=(0, 0, 0), c_fill=float("nan")):
    """One sgemm_ex() call. A: (M, lda) CPU tensor, B: (K, ldb).

    C starts filled with `c_fill` inside its rows (columns < N) and with the
    sentinel in the columns between N and ldc and in the guard band.
    Returns (rc, C as an (M, N) CPU tensor, dC) with dC the device matrix.
    """
    ldc = N if ldc is None else ldc
    dA = DeviceMatrix(A, M, K, lda, offsets[0])
    dB = DeviceMatrix(B, K, N, ldb, offsets[1])
    dC = DeviceMatrix(None, M, N, ldc, offsets[2])
    if M > 0 and N > 0:
        dC.buf[offsets[2]: offsets[2] + M * ldc].view(M, ldc)[:, :N] = c_fill
    stream = torch.cuda.current_stream().cuda_stream
    rc = sg.sgemm_ex(M, N, K, dA.ptr, lda, dB.ptr, ldb, dC.ptr, ldc, config, stream)
    torch.cuda.synchronize()
    st = sg.sgemm_check_status(stream)
    assert st == sg.SGEMM_OK, sg.sgemm_error_string(st)
    assert dA.guard_intact() and dB.guard_intact(), "input buffers were modified"
    C = dC.matrix()[:, :N] if M > 0 else torch.empty(0, N)
    return rc, C, dC


def check_untouched_padding(dC, N):
    """Columns N..ldc of C and the guard band must still hold the sentinel."""
    assert dC.guard_intact(), "write past the end of C"
    if dC.ld > N and dC.rows > 0:
        pad = dC.matrix()[:, N:]
        assert bool((pad == SENTINEL).all()), "write into the columns between N and ldc"


def assert_parity(C_gpu: torch.Tensor, C_ref: np.ndarray, S: np.ndarray, exact: bool, what=""):
    """Applies the parity bar; returns the largest |diff| / S."""
    c = C_gpu.numpy().astype(np.float64)
    assert c.shape == C_ref.shape, (c.shape, C_ref.shape)
    if exact:
        want = C_ref.astype(np.float32).astype(np.float64)
        bad = np.argwhere(c != want)
        assert bad.size == 0, f"{what}: {len(bad)} integer results differ, first at {bad[0]}: " \
                              f"{c[tuple(bad[0])]} vs {want[tuple(bad[0])]}"
        return 0.0
    assert not np.isnan(c).any() or np.isnan(C_ref).any(), f"{what}: NaN in the GPU result"
    diff = np.abs(c - C_ref)
    ok = diff <= TOL * S
    if not ok.all():
        i = np.argwhere(~ok)[0]
        raise AssertionError(f"{what}: {int((~ok).sum())} elements outside 1e-4*S; first at "
                             f"{tuple(i)}: gpu {c[tuple(i)]} ref {C_ref[tuple(i)]} S {S[tuple(i)]}")
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(S > 0, diff / S, 0.0)
    return float(r.max()) if r.size else 0.0
