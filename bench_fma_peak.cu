// FP32 FMA peak microbench: how many FP32 multiply-adds one GB300 SM retires
// per clock when nothing but the FMA pipe limits it. The main kernel's
// roofline is the nominal rate, 128 FMA lanes x 2 FLOP per clock per SM
// (Chapter 9: Optimised Matrix Multiplication, section 9.5, counts the FP32
// lanes of an SM the same way); this shows that rate is reachable, with
// scalar FFMA and with paired FFMA2 (two FP32 FMAs per instruction).
//
// Measurement only: bench.py --probe-fma builds it on demand; the library
// never links it. One block of 512 threads per SM (4 warps per SM
// sub-partition), each thread 16 independent accumulator chains with
// loop-invariant multiplicands, so no load, branch or dependency stall can
// hide behind the FMA pipe. Block 0 records clock64 and %globaltimer around
// its loop, which gives the SM clock the launch actually ran at.
#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr int kThreads = 512;
constexpr int kChains = 16;   // FP32 accumulators per thread

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

template <bool PAIRED>
__global__ void __launch_bounds__(kThreads, 1)
fma_peak_kernel(float *out, int iters, float x, float y, unsigned long long *clk)
{
    const long long c0 = clock64();
    const unsigned long long t0 = globaltimer_ns();
    float acc[kChains];
#pragma unroll
    for (int j = 0; j < kChains; ++j) acc[j] = (float)(threadIdx.x + j);
    if constexpr (PAIRED) {
        const float2 a = make_float2(x, x), b = make_float2(y, -y);
        float2 *p = reinterpret_cast<float2 *>(acc);
        for (int i = 0; i < iters; ++i) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
#pragma unroll
                for (int j = 0; j < kChains / 2; ++j) p[j] = __ffma2_rn(a, b, p[j]);
        }
    } else {
        for (int i = 0; i < iters; ++i) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
#pragma unroll
                for (int j = 0; j < kChains; ++j) acc[j] = fmaf(x, y, acc[j]);
        }
    }
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < kChains; ++j) s += acc[j];
    out[blockIdx.x * kThreads + threadIdx.x] = s;   // keeps the loop alive
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        clk[0] = (unsigned long long)(clock64() - c0);
        clk[1] = globaltimer_ns() - t0;
    }
}

}  // namespace

extern "C" {

// Runs the FFMA (paired = 0) or FFMA2 (paired = 1) loop `reps` times on
// every SM of the current device. Outputs: the best launch time in ms (CUDA
// events), the SM clock in MHz measured by block 0 during that launch, and
// the FP32 FLOPs one launch performs (2 per multiply-add). Returns 0 or the
// CUDA error code.
int fma_peak_run(int paired, int reps, double *best_ms, double *sm_mhz, double *flops)
{
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return (int)e;
    const int iters = 1 << 14;
    float *out = nullptr;
    unsigned long long *clk = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if ((e = cudaMalloc(&out, (size_t)sms * kThreads * sizeof(float))) != cudaSuccess) return (int)e;
    if ((e = cudaMalloc(&clk, 2 * sizeof(unsigned long long))) != cudaSuccess) {
        cudaFree(out);
        return (int)e;
    }
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    double best = 1e30, mhz = 0.0;
    for (int r = 0; r < reps + 1 && e == cudaSuccess; ++r) {
        cudaEventRecord(e0);
        if (paired)
            fma_peak_kernel<true><<<sms, kThreads>>>(out, iters, 1.0001f, 0.9999f, clk);
        else
            fma_peak_kernel<false><<<sms, kThreads>>>(out, iters, 1.0001f, 0.9999f, clk);
        cudaEventRecord(e1);
        if ((e = cudaEventSynchronize(e1)) != cudaSuccess) break;
        float ms = 0.0f;
        cudaEventElapsedTime(&ms, e0, e1);
        unsigned long long h[2] = {0, 0};
        if ((e = cudaMemcpy(h, clk, sizeof(h), cudaMemcpyDeviceToHost)) != cudaSuccess) break;
        if (r > 0 && ms < best) {   // the first launch warms up
            best = ms;
            mhz = h[1] > 0 ? (double)h[0] / (double)h[1] * 1e3 : 0.0;
        }
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaFree(out);
    cudaFree(clk);
    if (e != cudaSuccess) return (int)e;
    *best_ms = best;
    *sm_mhz = mhz;
    *flops = 2.0 * (double)sms * kThreads * (double)iters * 8 * kChains;
    return 0;
}

}  // extern "C"
