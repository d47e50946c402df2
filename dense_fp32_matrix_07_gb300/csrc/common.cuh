// Shared definitions of the SGEMM library's CUDA translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sgemm_gb300 {

// Arguments of one product C = A . B (row-major, FP32, device pointers).
struct GemmArgs {
    int64_t M, N, K;
    const float *A;
    int64_t lda;
    const float *B;
    int64_t ldb;
    float *C;
    int64_t ldc;
    unsigned int *status;  // device error word of the current device
    int num_sms;           // streaming multiprocessors of the current device
};

// Bits of the device error word.
enum : unsigned int {
    kStatusTimeout = 1u,   // a bounded wait gave up
};

// Spin limit of every device-side wait. Each failed try_wait sleeps up to
// ~256 ns, so the limit corresponds to roughly a second or two of waiting,
// orders of magnitude above any legitimate wait in these kernels.
constexpr unsigned int kSpinLimit = 1u << 23;

// Device address of the current device's error word.
cudaError_t device_status_word(unsigned int **out);

// Launchers (each returns the launch's cudaGetLastError()).
cudaError_t launch_zero_fill(float *C, int64_t M, int64_t N, int64_t ldc,
                             cudaStream_t stream);
cudaError_t launch_pack(const float *src, int64_t rows, int64_t cols,
                        int64_t ld_src, float *dst, int64_t ld_dst,
                        cudaStream_t stream);
cudaError_t launch_tiled_simple(const GemmArgs &g, cudaStream_t stream);

}  // namespace sgemm_gb300
