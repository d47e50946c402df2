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
    void *workspace = nullptr;     // stream-K partial sums and arrival counters, or null
    size_t workspace_bytes = 0;
    int withhold_it = -1;          // test hook: CTA 0's producer skips this copy
    // General form: C_b = alpha * A_b . B_b + beta * C_b for b < batch, with
    // batch strides in elements (a stride of 0 shares one operand).
    float alpha = 1.0f, beta = 0.0f;
    int64_t batch = 1;
    int64_t stride_a = 0, stride_b = 0, stride_c = 0;
    // Operand storage: 0 as multiplied (A: M x K, B: K x N), 1 transposed
    // (A stored K x M, B stored N x K). Only kernels that read the operands
    // themselves (the 3xTF32 split) see 1; the others get packed copies.
    int op_a = 0, op_b = 0;
    // Set when this call's layout pass (launch_pack_pair) was queued right
    // before the product and has zeroed the stream-K arrival counters at the
    // start of `workspace`: the product then skips its own zeroing and, for K
    // a multiple of the slab depth, launches with programmatic stream
    // serialization, its threads waiting for the pass to complete before
    // they touch global memory.
    bool behind_pack = false;
    // Set when the caller has zeroed the stream-K arrival counters at the
    // start of `workspace` (the layout pass or one memset of the call).
    bool counters_zeroed = false;
};

// Bits of the device error word.
enum : unsigned int {
    kStatusTimeout = 1u,        // a bounded wait gave up
    kStatusLaunchConfig = 2u,   // a kernel found its launch shape wrong and did nothing
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
// One operand's layout pass: entry b of src (rows x cols, ld_src, batch
// stride s_src) to dst (ld_dst, batch stride s_dst), copied as it is or
// transposed (dst[b][c][r] = src[b][r][c]), by `blocks` blocks of 256 threads.
struct PackJob {
    const float *src;
    int64_t rows, cols, ld_src, s_src;
    float *dst;
    int64_t ld_dst, s_dst, batch;
    int transpose;
    int64_t blocks;
};
PackJob pack_job(const float *src, int64_t rows, int64_t cols, int64_t ld_src, int64_t s_src, float *dst,
                 int64_t ld_dst, int64_t s_dst, int64_t batch, bool transpose);
// Jobs a and b (either may have 0 blocks) in one launch, which also zeroes
// zero_bytes at `zero` (null: nothing) and lets a kernel queued behind it with
// programmatic stream serialization start while its last blocks run.
cudaError_t launch_pack_pair(const PackJob &a, const PackJob &b, unsigned int *zero, size_t zero_bytes,
                             cudaStream_t stream);
// One transposing layout pass on its own (the allocation-free entry point).
cudaError_t launch_pack_transpose_batched(const float *src, int64_t rows, int64_t cols,
                                          int64_t ld_src, int64_t s_src, float *dst,
                                          int64_t ld_dst, int64_t s_dst, int64_t batch,
                                          cudaStream_t stream);
// C_b = beta * C_b (beta == 0 writes zeros without reading C).
cudaError_t launch_scale(float *C, int64_t M, int64_t N, int64_t ldc, int64_t stride_c,
                         int64_t batch, float beta, cudaStream_t stream);
cudaError_t launch_tiled_simple(const GemmArgs &g, cudaStream_t stream);

}  // namespace sgemm_gb300
