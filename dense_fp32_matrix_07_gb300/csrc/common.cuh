// Shared definitions of the SGEMM library's CUDA translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sgemm_gb300 {

// How the TMA kernels divide the output tiles among their CTAs.
enum SchedPolicy : int {
    kSchedAuto = 0,          // whole tiles, or stream-K when the last wave is short
    kSchedDataParallel = 1,  // whole tiles only (needs no workspace)
    kSchedStreamK = 2,       // every tile's K slabs shared out evenly (tests)
    kSchedTailSplit = 3      // whole tiles for full waves; each leftover tile
                             // split into equal K parts that run in lockstep
};

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
    int sched = kSchedDataParallel;
    void *workspace = nullptr;     // stream-K partial sums and flags, or null
    size_t workspace_bytes = 0;
    int withhold_it = -1;          // test hook: CTA 0's producer skips this copy
};

// Bits of the device error word.
enum : unsigned int {
    kStatusTimeout = 1u,   // a bounded wait gave up
};

// Probe-count backstop of the device-side waits. Their primary bound is wall
// clock (about a second of %globaltimer time, orders of magnitude above any
// legitimate wait in these kernels); this caps the number of probe rounds in
// case the timer were not to advance.
constexpr unsigned int kSpinLimit = 1u << 20;

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
