// FP32 FMA throughput probes: what the FP32 pipe of one GB300 SM sustains
// for the instruction patterns an SGEMM mainloop is made of. They bound the
// main kernel's roofline from the inside (the nominal peak is 128 FMA lanes
// x 2 FLOP per clock per SM; Chapter 9: Optimised Matrix Multiplication,
// section 9.5, counts the per-SM FP32 lanes the same way).
//
// Every probe runs one block per SM, touches only its own output slot and a
// shared-memory tile it fills itself, and has no waits; it measures its own
// SM clock (clock64 over %globaltimer) so FLOP per clock per SM follows.
//
//   0  FFMA, loop-invariant multiplicands, 16 independent chains per thread
//   1  FFMA2 (paired FP32 FMA), loop-invariant multiplicands
//   2  FFMA, 8 x 8 outer product from registers (a[i] * b[j] into acc[i][j])
//   3  FFMA2, 8 x 8 outer product from registers, a[i] broadcast to both
//      lanes, fixed operand registers
//   4  as 3, with the operand registers rotated every k
//   5  SGEMM inner loop from shared memory: 8 x 8 thread tiles, 128 x 128
//      block, A rows 128-byte swizzled (LDS.128 of 4 k), B read as float4
//   6  as 5 with 8 x 16 thread tiles (128 x 256 block): the main kernel's tile
//   7  as 5 with 12 warps (3 per SM sub-partition), 192 x 128 block
//   8  as 3 with the multiplicands swapped: ffma2(b pair, broadcast a, acc)
//   9  as 6 with the multiplicands swapped
//  10  8 x 8 outer product from registers with a held as true pairs (a, a)
//      (not a broadcast), b pairs reused across the inner loop (b outer)
//  11  as 10 with a pairs reused across the inner loop (a outer)
// The order of the FFMA2s of one k step (ORDER below): 0 row-major (for each
// row i, every b pair q: the row change swaps both multiplicands), 1 row
// serpentine (q runs backwards on odd rows, so consecutive FFMA2s always
// share a multiplicand), 2 column serpentine (b pair outer, rows alternate).
//  12  8 x 8 outer product from registers, broadcast a, row serpentine
//  13  as 12, column serpentine
//  14  8 x 16 outer product from registers, broadcast a, row-major
//  15  as 14, row serpentine
//  16  as 14, column serpentine
//  17  as 6 (8 x 16 from shared memory), row serpentine
//  18  as 6, column serpentine
//  19  as 5 (8 x 8 from shared memory), row serpentine
//  20  as 5, column serpentine
//  21  as 6, zigzag down strips of two b pairs (each FFMA2 shares a
//      multiplicand with the one before)
//  22  as 6, column serpentine over each half of the rows in turn
//  23  as 6, column serpentine, b pairs in reverse order on odd k
//  24  8 x 16 loop with the A slab k-major (one LDS.128 gives 4 rows at
//      one k), column serpentine
//  25  as 24, row-major order
//  26  the 8 x 8 loop (128 x 128 block) with the A slab k-major, column
//      serpentine
//  27  as 24 in the main kernel's launch shape: 384 threads, the third
//      warpgroup leaving after setmaxnreg hands 232 registers to the others
//  28  as 18 (row-major A slab, column serpentine), the 8 A values of one
//      k read by 8 scalar shared loads in place of 4-k LDS.128 per row
//  29  as 28, row-major order
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

namespace {

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record(unsigned long long *clk, long long c0, unsigned long long t0)
{
    const long long c1 = clock64();
    const unsigned long long t1 = global_ns();
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        clk[0] = (unsigned long long)(c1 - c0);
        clk[1] = t1 - t0;
    }
}

// 0 / 1: loop-invariant multiplicands.
template <bool PAIRED>
__global__ void __launch_bounds__(256) peak_kernel(float *out, int iters, float x, float y, unsigned long long *clk)
{
    float2 a[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = make_float2(threadIdx.x * 1e-3f + j, j * 0.5f);
    const float2 x2 = make_float2(x, x), y2 = make_float2(y, y);
    const long long c0 = clock64();
    const unsigned long long t0 = global_ns();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (PAIRED) {
                a[j] = __ffma2_rn(a[j], x2, y2);
            } else {
                a[j].x = fmaf(a[j].x, x, y);
                a[j].y = fmaf(a[j].y, x, y);
            }
        }
    }
    record(clk, c0, t0);
    float s = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += a[j].x + a[j].y;
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// 2 / 3 / 4 / 10 / 11: 8 x 8 outer products from registers, 32 k per iteration.
template <int MODE, bool SWAP = false>
__global__ void __launch_bounds__(256, 1) outer_kernel(float *out, int iters, unsigned long long *clk)
{
    float a[8], bs[8];
    float2 b[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        a[i] = threadIdx.x * 1e-3f + i;
        bs[i] = i * 0.3f;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) b[q] = make_float2(q * 0.5f, q * 0.25f + threadIdx.x * 1e-4f);
    // True pairs (a, a + z) with an opaque zero z: the compiler cannot fold
    // them back into a broadcast of one register.
    unsigned zbits;
    asm volatile("mov.u32 %0, 0;" : "=r"(zbits));
    const float z = __uint_as_float(zbits);
    float2 a2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a2[i] = make_float2(a[i], a[i] + z);
    float2 acc[8][4];
    float accs[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) accs[i][j] = 0.f;
    }
    const long long c0 = clock64();
    const unsigned long long t0 = global_ns();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            if (MODE == 10) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i][q] = __ffma2_rn(a2[i], b[q], acc[i][q]);
                continue;
            }
            if (MODE == 11) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[i][q] = __ffma2_rn(a2[i], b[q], acc[i][q]);
                continue;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (MODE == 2) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) accs[i][j] = fmaf(a[i], bs[j], accs[i][j]);
                } else if (MODE == 3) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        acc[i][q] = SWAP ? __ffma2_rn(b[q], make_float2(a[i], a[i]), acc[i][q])
                                         : __ffma2_rn(make_float2(a[i], a[i]), b[q], acc[i][q]);
                } else {
                    const float av = a[(i + k) & 7];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        acc[i][q] = __ffma2_rn(make_float2(av, av), b[(q + k) & 3], acc[i][q]);
                }
            }
        }
    }
    record(clk, c0, t0);
    float s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int q = 0; q < 4; ++q) s += acc[i][q].x + acc[i][q].y;
#pragma unroll
        for (int j = 0; j < 8; ++j) s += accs[i][j];
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// One k step of a TM x (2 NP) outer product: acc[i][q] += a[i] * b[q], the
// scalar a[i] broadcast to both lanes of the FFMA2, in the given ORDER.
template <int ORDER, int TM, int NP>
__device__ __forceinline__ void outer_step(float2 (&acc)[TM][NP], const float (&a)[TM], const float2 (&b)[NP],
                                           int kk = 0)
{
    if constexpr (ORDER == 3) {
        // zigzag down strips of two b pairs: (i,p) (i,p+1) (i+1,p+1) (i+1,p) ...
#pragma unroll
        for (int p0 = 0; p0 < NP; p0 += 2)
#pragma unroll
            for (int ii = 0; ii < TM; ++ii) {
                const int i = (p0 & 2) ? TM - 1 - ii : ii;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int q = p0 + ((ii & 1) ? 1 - e : e);
                    acc[i][q] = __ffma2_rn(make_float2(a[i], a[i]), b[q], acc[i][q]);
                }
            }
    } else if constexpr (ORDER == 4) {
        // column serpentine over each half of the rows in turn
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int q = 0; q < NP; ++q)
#pragma unroll
                for (int ii = 0; ii < TM / 2; ++ii) {
                    const int i = h * (TM / 2) + ((q & 1) ? TM / 2 - 1 - ii : ii);
                    acc[i][q] = __ffma2_rn(make_float2(a[i], a[i]), b[q], acc[i][q]);
                }
    } else if constexpr (ORDER == 5) {
        // column serpentine with the b pairs taken in reverse on odd k
#pragma unroll
        for (int qq = 0; qq < NP; ++qq) {
            const int q = (kk & 1) ? NP - 1 - qq : qq;
#pragma unroll
            for (int ii = 0; ii < TM; ++ii) {
                const int i = (qq & 1) ? TM - 1 - ii : ii;
                acc[i][q] = __ffma2_rn(make_float2(a[i], a[i]), b[q], acc[i][q]);
            }
        }
    } else if constexpr (ORDER == 2) {
#pragma unroll
        for (int q = 0; q < NP; ++q)
#pragma unroll
            for (int ii = 0; ii < TM; ++ii) {
                const int i = (q & 1) ? TM - 1 - ii : ii;
                acc[i][q] = __ffma2_rn(make_float2(a[i], a[i]), b[q], acc[i][q]);
            }
    } else {
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int qq = 0; qq < NP; ++qq) {
                const int q = (ORDER == 1 && (i & 1)) ? NP - 1 - qq : qq;
                acc[i][q] = __ffma2_rn(make_float2(a[i], a[i]), b[q], acc[i][q]);
            }
    }
}

// 12 - 16: 8 x (2 NP) outer products from registers in a given order, 32 k
// per iteration, fixed operand registers.
template <int NP, int ORDER>
__global__ void __launch_bounds__(256, 1) ordered_outer_kernel(float *out, int iters, unsigned long long *clk)
{
    float a[8];
    float2 b[NP];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = threadIdx.x * 1e-3f + i;
#pragma unroll
    for (int q = 0; q < NP; ++q) b[q] = make_float2(q * 0.5f, q * 0.25f + threadIdx.x * 1e-4f);
    float2 acc[8][NP];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < NP; ++q) acc[i][q] = make_float2(0.f, 0.f);
    const long long c0 = clock64();
    const unsigned long long t0 = global_ns();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int k = 0; k < 32; ++k) outer_step<ORDER>(acc, a, b);
    }
    record(clk, c0, t0);
    float s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < NP; ++q) s += acc[i][q].x + acc[i][q].y;
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

namespace {

// 5 / 6: the SGEMM inner loop on one 32-deep slab held in shared memory.
// 8 warps as 2 x 4, each 8 x 4 threads with TM x TN thread tiles: block
// 128 x (16 TN). A is [128][32] floats with 16-byte chunk c of row r stored
// at chunk c ^ (r & 7); B is [32][BN] floats. Each thread loads 4 k of A per
// row with one LDS.128 and TN/4 float4 of B per k, then issues TM * TN / 2
// broadcast FFMA2 per k.
template <int TN, int WM = 2, bool SWAP = false, int ORDER = -1, bool SCALAR_A = false>
__global__ void __launch_bounds__(WM * 4 * 32, 1) inner_kernel(float *out, int iters, unsigned long long *clk)
{
    constexpr int TM = 8, TR = 8, TC = 4, WN = 4;
    constexpr int BM = WM * TR * TM, BN = WN * TC * TN, NT = WM * WN * 32;
    extern __shared__ __align__(1024) unsigned char smem[];
    float *sA = reinterpret_cast<float *>(smem);
    float *sB = reinterpret_cast<float *>(smem + BM * 128);
    for (int e = threadIdx.x; e < BM * 32; e += NT) sA[e] = (e % 7) * 0.25f - 0.5f;
    for (int e = threadIdx.x; e < BN * 32; e += NT) sB[e] = (e % 5) * 0.125f - 0.25f;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wm = (warp / WN) * TR * TM, wn = (warp % WN) * TC * TN;
    const int ty = lane / TC, tx = lane % TC;
    const char *As = reinterpret_cast<const char *>(sA) + (wm + ty) * 128;
    const char *Bs = reinterpret_cast<const char *>(sB) + (wn + tx * 4) * 4;
    float2 acc[TM][TN / 2];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);
    const long long c0 = clock64();
    const unsigned long long t0 = global_ns();
    for (int it = 0; it < iters; ++it) {
        // An opaque zero offset keeps the compiler from hoisting the shared
        // loads out of the iteration loop.
        unsigned z;
        asm volatile("mov.u32 %0, 0;" : "=r"(z));
        const char *Ai = As + z, *Bi = Bs + z;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
            float a[TM][4];
#pragma unroll
            for (int i = 0; i < TM && !SCALAR_A; ++i) {
                const int r = ty + TR * i;    // (wm + r) & 7 == r & 7
                const float4 v =
                    *reinterpret_cast<const float4 *>(Ai + TR * i * 128 + (((unsigned)kb ^ (unsigned)(r & 7)) << 4));
                a[i][0] = v.x;
                a[i][1] = v.y;
                a[i][2] = v.z;
                a[i][3] = v.w;
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int k = kb * 4 + kk;
                float4 b[TN / 4];
#pragma unroll
                for (int g = 0; g < TN / 4; ++g)
                    b[g] = *reinterpret_cast<const float4 *>(Bi + k * BN * 4 + g * TC * 16);
                if constexpr (ORDER >= 0) {
                    float ak[TM];
                    float2 b2[TN / 2];
                    if constexpr (SCALAR_A) {
                        // One 4-byte shared load per row at this k: row
                        // ty + 8i, 16-byte chunk kb ^ ty, word kk. The 8 rows
                        // of a warp's distinct ty fall in 8 distinct chunks,
                        // so the loads are conflict-free; inline PTX keeps
                        // them from being merged into the 16-byte loads.
                        const unsigned base = (unsigned)__cvta_generic_to_shared(Ai) +
                                              ((((unsigned)kb ^ (unsigned)(ty & 7)) << 4) | (unsigned)(kk * 4));
#pragma unroll
                        for (int i = 0; i < TM; ++i)
                            asm("ld.shared.f32 %0, [%1];" : "=f"(ak[i]) : "r"(base + (unsigned)(TR * i * 128)));
                    } else {
#pragma unroll
                        for (int i = 0; i < TM; ++i) ak[i] = a[i][kk];
                    }
#pragma unroll
                    for (int g = 0; g < TN / 4; ++g) {
                        b2[2 * g] = make_float2(b[g].x, b[g].y);
                        b2[2 * g + 1] = make_float2(b[g].z, b[g].w);
                    }
                    outer_step<ORDER>(acc, ak, b2, kk);
                    continue;
                }
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    const float2 aa = make_float2(a[i][kk], a[i][kk]);
#pragma unroll
                    for (int g = 0; g < TN / 4; ++g) {
                        if (SWAP) {
                            acc[i][2 * g] = __ffma2_rn(make_float2(b[g].x, b[g].y), aa, acc[i][2 * g]);
                            acc[i][2 * g + 1] = __ffma2_rn(make_float2(b[g].z, b[g].w), aa, acc[i][2 * g + 1]);
                        } else {
                            acc[i][2 * g] = __ffma2_rn(aa, make_float2(b[g].x, b[g].y), acc[i][2 * g]);
                            acc[i][2 * g + 1] = __ffma2_rn(aa, make_float2(b[g].z, b[g].w), acc[i][2 * g + 1]);
                        }
                    }
                }
            }
        }
    }
    record(clk, c0, t0);
    float s = 0;
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) s += acc[i][j].x + acc[i][j].y;
    out[blockIdx.x * NT + threadIdx.x] = s;
}

template <int TN, int WM = 2>
constexpr int inner_smem() { return WM * 64 * 128 + 4 * 4 * TN * 128; }

// 24 / 25: the 8 x 16 loop with the A slab stored k-major, [32][128]
// floats (M contiguous). Thread row ty owns rows 4ty..4ty+3 and
// 32+4ty..32+4ty+3 of its warp's 64, so per k two conflict-free LDS.128
// give its 8 A values in consecutive registers (with the row-major slab,
// the 8 values of one k sit 4 registers apart). B as in 6.
template <int ORDER, int TN = 16, bool SPLIT = false>
__global__ void __launch_bounds__(SPLIT ? 384 : 256, 1) inner_kmajor_kernel(float *out, int iters,
                                                                            unsigned long long *clk)
{
    constexpr int BM = 128, BN = 16 * TN, NT = 256;
    extern __shared__ __align__(1024) unsigned char smem[];
    float *sA = reinterpret_cast<float *>(smem);                 // [32][BM]
    float *sB = reinterpret_cast<float *>(smem + 32 * BM * 4);   // [32][BN]
    if (threadIdx.x < NT) {
        for (int e = threadIdx.x; e < BM * 32; e += NT) sA[e] = (e % 7) * 0.25f - 0.5f;
        for (int e = threadIdx.x; e < BN * 32; e += NT) sB[e] = (e % 5) * 0.125f - 0.25f;
    }
    __syncthreads();
    if constexpr (SPLIT) {
        // The main kernel's launch shape: a third warpgroup hands its
        // registers to the two computing ones (40 / 232 of the 168 each
        // thread was launched with) and leaves.
        if (threadIdx.x >= NT) {
            asm volatile("setmaxnreg.dec.sync.aligned.u32 40;");
            return;
        }
        asm volatile("setmaxnreg.inc.sync.aligned.u32 232;");
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wm = (warp / 4) * 64, wn = (warp % 4) * 4 * TN;
    const int ty = lane / 4, tx = lane % 4;
    const char *As = reinterpret_cast<const char *>(sA) + (wm + 4 * ty) * 4;
    const char *Bs = reinterpret_cast<const char *>(sB) + (wn + tx * 4) * 4;
    float2 acc[8][TN / 2];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);
    const long long c0 = clock64();
    const unsigned long long t0 = global_ns();
    for (int it = 0; it < iters; ++it) {
        unsigned z;
        asm volatile("mov.u32 %0, 0;" : "=r"(z));
        const char *Ai = As + z, *Bi = Bs + z;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const float4 lo = *reinterpret_cast<const float4 *>(Ai + k * BM * 4);
            const float4 hi = *reinterpret_cast<const float4 *>(Ai + k * BM * 4 + 128);
            const float ak[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
            float2 b2[TN / 2];
#pragma unroll
            for (int g = 0; g < TN / 4; ++g) {
                const float4 v = *reinterpret_cast<const float4 *>(Bi + k * BN * 4 + g * 64);
                b2[2 * g] = make_float2(v.x, v.y);
                b2[2 * g + 1] = make_float2(v.z, v.w);
            }
            outer_step<ORDER>(acc, ak, b2, k);
        }
    }
    record(clk, c0, t0);
    float s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) s += acc[i][j].x + acc[i][j].y;
    out[blockIdx.x * NT + threadIdx.x] = s;
}

}  // namespace

extern "C" {

// Number of probe kinds (see the list at the top of this file).
int fma_probe_count(void) { return 30; }

// Runs probe `kind` on one block per SM: one warm-up launch, then `reps`
// timed launches (CUDA events); returns the best launch time, the SM clock
// the kernel measured (MHz) and the FP32 operations of one launch (FMA = 2).
// Returns 0, or a cudaError_t value. Allocates and frees its own small
// buffers; synchronises the device.
int fma_probe_run(int kind, int reps, double *best_ms, double *sm_mhz, double *flops)
{
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return (int)e;
    if (kind < 0 || kind > 29 || reps < 1) return (int)cudaErrorInvalidValue;
    float *out = nullptr;
    unsigned long long *clk = nullptr;
    if ((e = cudaMalloc(&out, sizeof(float) * 384 * (size_t)sms)) != cudaSuccess) return (int)e;
    if ((e = cudaMalloc(&clk, 2 * sizeof(unsigned long long))) != cudaSuccess) {
        cudaFree(out);
        return (int)e;
    }
    const int peak_iters = 1 << 16, loop_iters = 2048;
    double f = 0;
    auto launch = [&]() {
        switch (kind) {
        case 0: peak_kernel<false><<<sms, 256>>>(out, peak_iters, 0.999f, 0.001f, clk); break;
        case 1: peak_kernel<true><<<sms, 256>>>(out, peak_iters, 0.999f, 0.001f, clk); break;
        case 2: outer_kernel<2><<<sms, 256>>>(out, loop_iters, clk); break;
        case 3: outer_kernel<3><<<sms, 256>>>(out, loop_iters, clk); break;
        case 4: outer_kernel<4><<<sms, 256>>>(out, loop_iters, clk); break;
        case 5: inner_kernel<8><<<sms, 256, inner_smem<8>()>>>(out, loop_iters, clk); break;
        case 6: inner_kernel<16><<<sms, 256, inner_smem<16>()>>>(out, loop_iters, clk); break;
        case 7: inner_kernel<8, 3><<<sms, 384, inner_smem<8, 3>()>>>(out, loop_iters, clk); break;
        case 8: outer_kernel<3, true><<<sms, 256>>>(out, loop_iters, clk); break;
        case 10: outer_kernel<10><<<sms, 256>>>(out, loop_iters, clk); break;
        case 11: outer_kernel<11><<<sms, 256>>>(out, loop_iters, clk); break;
        case 12: ordered_outer_kernel<4, 1><<<sms, 256>>>(out, loop_iters, clk); break;
        case 13: ordered_outer_kernel<4, 2><<<sms, 256>>>(out, loop_iters, clk); break;
        case 14: ordered_outer_kernel<8, 0><<<sms, 256>>>(out, loop_iters, clk); break;
        case 15: ordered_outer_kernel<8, 1><<<sms, 256>>>(out, loop_iters, clk); break;
        case 16: ordered_outer_kernel<8, 2><<<sms, 256>>>(out, loop_iters, clk); break;
        case 17: inner_kernel<16, 2, false, 1><<<sms, 256, inner_smem<16>()>>>(out, loop_iters, clk); break;
        case 18: inner_kernel<16, 2, false, 2><<<sms, 256, inner_smem<16>()>>>(out, loop_iters, clk); break;
        case 19: inner_kernel<8, 2, false, 1><<<sms, 256, inner_smem<8>()>>>(out, loop_iters, clk); break;
        case 20: inner_kernel<8, 2, false, 2><<<sms, 256, inner_smem<8>()>>>(out, loop_iters, clk); break;
        case 21: inner_kernel<16, 2, false, 3><<<sms, 256, inner_smem<16>()>>>(out, loop_iters, clk); break;
        case 22: inner_kernel<16, 2, false, 4><<<sms, 256, inner_smem<16>()>>>(out, loop_iters, clk); break;
        case 23: inner_kernel<16, 2, false, 5><<<sms, 256, inner_smem<16>()>>>(out, loop_iters, clk); break;
        case 24: inner_kmajor_kernel<2><<<sms, 256, inner_smem<16>()>>>(out, loop_iters, clk); break;
        case 25: inner_kmajor_kernel<0><<<sms, 256, inner_smem<16>()>>>(out, loop_iters, clk); break;
        case 26: inner_kmajor_kernel<2, 8><<<sms, 256, inner_smem<8>()>>>(out, loop_iters, clk); break;
        case 27: inner_kmajor_kernel<2, 16, true><<<sms, 384, inner_smem<16>()>>>(out, loop_iters, clk); break;
        case 28: inner_kernel<16, 2, false, 2, true><<<sms, 256, inner_smem<16>()>>>(out, loop_iters, clk); break;
        case 29: inner_kernel<16, 2, false, 0, true><<<sms, 256, inner_smem<16>()>>>(out, loop_iters, clk); break;
        default: inner_kernel<16, 2, true><<<sms, 256, inner_smem<16>()>>>(out, loop_iters, clk); break;
        }
    };
    if (kind <= 1) f = 2.0 * 16 * peak_iters * 256.0 * sms;
    else if (kind <= 4 || kind == 8 || (kind >= 10 && kind <= 13)) f = 2.0 * 64 * 32 * (double)loop_iters * 256.0 * sms;
    else if (kind >= 14 && kind <= 16) f = 2.0 * 128 * 32 * (double)loop_iters * 256.0 * sms;
    else if (kind == 5 || kind == 19 || kind == 20 || kind == 26) f = 2.0 * 128 * 128 * 32 * (double)loop_iters * sms;
    else if (kind == 6 || kind == 9 || (kind >= 17 && kind <= 25) || kind >= 27) f = 2.0 * 128 * 256 * 32 * (double)loop_iters * sms;
    else f = 2.0 * 192 * 128 * 32 * (double)loop_iters * sms;
    e = cudaFuncSetAttribute(inner_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, inner_smem<8>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inner_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, inner_smem<16>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inner_kernel<8, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 inner_smem<8, 3>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inner_kernel<16, 2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 inner_smem<16>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inner_kernel<16, 2, false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 inner_smem<16>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inner_kernel<16, 2, false, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 inner_smem<16>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inner_kernel<16, 2, false, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 inner_smem<16>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inner_kernel<16, 2, false, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 inner_smem<16>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inner_kernel<16, 2, false, 5>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 inner_smem<16>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inner_kmajor_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 inner_smem<16>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inner_kmajor_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 inner_smem<16>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inner_kmajor_kernel<2, 16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 inner_smem<16>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inner_kernel<16, 2, false, 2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 inner_smem<16>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inner_kernel<16, 2, false, 0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 inner_smem<16>());
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (e == cudaSuccess) e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    std::vector<float> ms;
    if (e == cudaSuccess) {
        launch();
        e = cudaDeviceSynchronize();
    }
    for (int r = 0; r < reps && e == cudaSuccess; ++r) {
        cudaEventRecord(e0);
        launch();
        cudaEventRecord(e1);
        e = cudaEventSynchronize(e1);
        float t = 0;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&t, e0, e1);
        ms.push_back(t);
    }
    unsigned long long c[2] = {0, 0};
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaMemcpy(c, clk, sizeof(c), cudaMemcpyDeviceToHost);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaFree(out);
    cudaFree(clk);
    if (e != cudaSuccess) return (int)e;
    *best_ms = *std::min_element(ms.begin(), ms.end());
    *sm_mhz = c[1] ? (double)c[0] / (double)c[1] * 1e3 : 0.0;
    *flops = f;
    return 0;
}

}  // extern "C"

// L2 sharing probe: every block reads the whole of one `n4`-float4 buffer
// (all blocks at about the same time) and writes one sum. The DRAM bytes of
// a cold launch, against the buffer's size, show how many times the L2
// fetches data that every SM reads.
namespace {

__global__ void __launch_bounds__(1024) l2_shared_read_kernel(const float4 *__restrict__ buf, int64_t n4,
                                                              float *__restrict__ out)
{
    float s = 0.0f;
    for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = buf[i];
        s += v.x + v.y + v.z + v.w;
    }
    __shared__ float red[32];
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
        out[blockIdx.x] = t;
    }
}

}  // namespace

extern "C" {

// One block of 1024 threads per SM reads the same `mib` MiB buffer; runs
// `reps` launches (the buffer is written once, before them) and returns the
// best launch time. Returns 0 or a cudaError_t value.
int l2_probe_shared_read(int mib, int reps, double *best_ms)
{
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return (int)e;
    if (mib < 1 || mib > 4096 || reps < 1) return (int)cudaErrorInvalidValue;
    const int64_t n4 = (int64_t)mib * (1 << 20) / 16;
    float4 *buf = nullptr;
    float *out = nullptr;
    if ((e = cudaMalloc(&buf, (size_t)n4 * 16)) != cudaSuccess) return (int)e;
    if ((e = cudaMalloc(&out, sizeof(float) * (size_t)sms)) != cudaSuccess) {
        cudaFree(buf);
        return (int)e;
    }
    e = cudaMemset(buf, 0, (size_t)n4 * 16);
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (e == cudaSuccess) e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    float best = 0.0f;
    for (int r = 0; r < reps && e == cudaSuccess; ++r) {
        cudaEventRecord(e0);
        l2_shared_read_kernel<<<sms, 1024>>>(buf, n4, out);
        cudaEventRecord(e1);
        e = cudaEventSynchronize(e1);
        float t = 0.0f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&t, e0, e1);
        if (r == 0 || t < best) best = t;
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaFree(buf);
    cudaFree(out);
    if (e != cudaSuccess) return (int)e;
    *best_ms = best;
    return 0;
}

}  // extern "C"
