// The pages' own kernel ladder, rebuilt for sm_103a so their speed-ups can be
// measured on GB300 next to the TMA kernel. Each follows its page's design
// (thread mapping, tiling, reuse); unlike the pages' listings, every access
// is predicated, so any M, N, K and leading dimension work.
#include "common.cuh"
#include "configs.cuh"

namespace sgemm_gb300 {

namespace {

// Chapter 9: Optimised Matrix Multiplication, section 9.2 (Stage 0): one
// thread per output with threadIdx.x running down a column of C, i.e. the
// row index — consecutive lanes read A and write C a full row apart.
__global__ void ladder_naive_kernel(int64_t M, int64_t N, int64_t K, const float *__restrict__ A,
                                    int64_t lda, const float *__restrict__ B, int64_t ldb,
                                    float *__restrict__ C, int64_t ldc)
{
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;   // row of C
    const int64_t j = blockIdx.y * (int64_t)blockDim.y + threadIdx.y;   // column of C
    if (i >= M || j >= N) return;
    float sum = 0.0f;
    for (int64_t k = 0; k < K; ++k) sum = fmaf(A[i * lda + k], B[k * ldb + j], sum);
    C[i * ldc + j] = sum;
}

// Section 9.3 (Stage 1) and "Перемножение матриц: наивное и тайловое",
// section 1: threadIdx.x runs along a row of C, so B loads and C stores are
// coalesced and the A element is one broadcast per warp.
__global__ void ladder_coalesced_kernel(int64_t M, int64_t N, int64_t K, const float *__restrict__ A,
                                        int64_t lda, const float *__restrict__ B, int64_t ldb,
                                        float *__restrict__ C, int64_t ldc)
{
    const int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;   // column of C
    const int64_t i = blockIdx.y * (int64_t)blockDim.y + threadIdx.y;   // row of C
    if (i >= M || j >= N) return;
    float sum = 0.0f;
    for (int64_t k = 0; k < K; ++k) sum = fmaf(A[i * lda + k], B[k * ldb + j], sum);
    C[i * ldc + j] = sum;
}

// The CUDA Handbook, ch.17, section 17.3 (Cache Blocking), as a design: a
// thread computes a TM x TN block of C wholly in registers, reading A and B
// straight from global memory without shared memory, and the caches capture
// the reuse: threads of a warp take side-by-side blocks, so their B reads
// share cache lines and their A values are the same few rows. Here the
// blocks are dealt out by one flat index over a 1-D grid, consecutive
// indices running along a row of blocks; rows and columns past the edge of
// C are clamped to the last valid ones while reading and skipped when
// storing, so no load needs a predicate.
template <int TM, int TN>
__global__ void __launch_bounds__(256)
ladder_cache_blocked_kernel(int64_t M, int64_t N, int64_t K, const float *__restrict__ A, int64_t lda,
                            const float *__restrict__ B, int64_t ldb, float *__restrict__ C, int64_t ldc)
{
    const int64_t blocks_n = (N + TN - 1) / TN;
    const int64_t blocks = ((M + TM - 1) / TM) * blocks_n;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t blk = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; blk < blocks; blk += step) {
        const int64_t r0 = (blk / blocks_n) * TM, c0 = (blk % blocks_n) * TN;
        int64_t arow[TM], bcol[TN];
#pragma unroll
        for (int i = 0; i < TM; ++i) arow[i] = (r0 + i < M ? r0 + i : M - 1) * lda;
#pragma unroll
        for (int j = 0; j < TN; ++j) bcol[j] = c0 + j < N ? c0 + j : N - 1;
        float acc[TM][TN];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;
        const float *bk = B;
        for (int64_t k = 0; k < K; ++k, bk += ldb) {
            float bv[TN];
#pragma unroll
            for (int j = 0; j < TN; ++j) bv[j] = bk[bcol[j]];
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const float av = A[arow[i] + k];
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(av, bv[j], acc[i][j]);
            }
        }
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            if (r0 + i >= M) break;
            float *crow = C + (r0 + i) * ldc;
#pragma unroll
            for (int j = 0; j < TN; ++j)
                if (c0 + j < N) crow[c0 + j] = acc[i][j];
        }
    }
}

// Section 9.5 (Stage 3, register tiling) with section 9.6's launch bounds:
// a block of (T/RN) x (T/RM) threads computes a T x T tile of C; each thread
// loads an RM x RN patch of the padded A and B tiles and keeps an RM x RN
// micro-tile, so each shared value feeds RM*RN multiply-adds. The B patch
// is read at column col0 + c, where col0 already includes the thread's
// column offset (the page's warning about counting tx*RN twice).
template <int T, int RM, int RN, int MIN_BLOCKS>
__global__ void __launch_bounds__((T / RM) * (T / RN), MIN_BLOCKS)
ladder_register_tiled_kernel(int64_t M, int64_t N, int64_t K, const float *__restrict__ A, int64_t lda,
                             const float *__restrict__ B, int64_t ldb, float *__restrict__ C, int64_t ldc)
{
    __shared__ float sA[T][T + 1];
    __shared__ float sB[T][T + 1];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int64_t tiles_n = (N + T - 1) / T;
    const int64_t tiles = ((M + T - 1) / T) * tiles_n;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t row0 = (t / tiles_n) * T + ty * RM;
        const int64_t col0 = (t % tiles_n) * T + tx * RN;
        float acc[RM][RN];
#pragma unroll
        for (int r = 0; r < RM; ++r)
#pragma unroll
            for (int c = 0; c < RN; ++c) acc[r][c] = 0.0f;
        for (int64_t k0 = 0; k0 < K; k0 += T) {
#pragma unroll
            for (int r = 0; r < RM; ++r)
#pragma unroll
                for (int c = 0; c < RN; ++c) {
                    const int64_t ka = k0 + tx * RN + c;
                    sA[ty * RM + r][tx * RN + c] =
                        (row0 + r < M && ka < K) ? A[(row0 + r) * lda + ka] : 0.0f;
                    const int64_t kb = k0 + ty * RM + r;
                    sB[ty * RM + r][tx * RN + c] =
                        (kb < K && col0 + c < N) ? B[kb * ldb + col0 + c] : 0.0f;
                }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < T; ++k) {
                float a[RM], b[RN];
#pragma unroll
                for (int r = 0; r < RM; ++r) a[r] = sA[ty * RM + r][k];
#pragma unroll
                for (int c = 0; c < RN; ++c) b[c] = sB[k][tx * RN + c];
#pragma unroll
                for (int r = 0; r < RM; ++r)
#pragma unroll
                    for (int c = 0; c < RN; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
            }
            __syncthreads();
        }
#pragma unroll
        for (int r = 0; r < RM; ++r)
#pragma unroll
            for (int c = 0; c < RN; ++c)
                if (row0 + r < M && col0 + c < N) C[(row0 + r) * ldc + col0 + c] = acc[r][c];
    }
}

unsigned clamp_grid(int64_t blocks, int64_t cap)
{
    if (blocks < 1) blocks = 1;
    return (unsigned)(blocks < cap ? blocks : cap);
}

}  // namespace

cudaError_t launch_ladder(int kernel, const GemmArgs &g, cudaStream_t stream)
{
    switch (kernel) {
    case kKernLadderNaive: {
        // 16 x 16 blocks, x over rows (the stage-0 mapping); grid.y <= 65535.
        const dim3 block(16, 16);
        const int64_t gx = (g.M + 15) / 16, gy = (g.N + 15) / 16;
        if (gx > 0x7fffffff || gy > 65535) return cudaErrorInvalidConfiguration;
        ladder_naive_kernel<<<dim3((unsigned)gx, (unsigned)gy), block, 0, stream>>>(
            g.M, g.N, g.K, g.A, g.lda, g.B, g.ldb, g.C, g.ldc);
        break;
    }
    case kKernLadderCoalesced: {
        const dim3 block(16, 16);
        const int64_t gx = (g.N + 15) / 16, gy = (g.M + 15) / 16;
        if (gx > 0x7fffffff || gy > 65535) return cudaErrorInvalidConfiguration;
        ladder_coalesced_kernel<<<dim3((unsigned)gx, (unsigned)gy), block, 0, stream>>>(
            g.M, g.N, g.K, g.A, g.lda, g.B, g.ldb, g.C, g.ldc);
        break;
    }
    case kKernLadderCacheBlocked8x8: {
        // One 8 x 8 block of C per thread, 256 threads a CTA, at most 16
        // CTAs per SM's worth of blocks at once (grid-stride beyond that).
        const int64_t blocks = ((g.M + 7) / 8) * ((g.N + 7) / 8);
        ladder_cache_blocked_kernel<8, 8><<<clamp_grid((blocks + 255) / 256, (int64_t)g.num_sms * 16), 256, 0,
                                            stream>>>(g.M, g.N, g.K, g.A, g.lda, g.B, g.ldb, g.C, g.ldc);
        break;
    }
    case kKernLadderRegisterTiled2x2: {
        constexpr int T = 16;
        const int64_t tiles = ((g.M + T - 1) / T) * ((g.N + T - 1) / T);
        ladder_register_tiled_kernel<T, 2, 2, 16><<<clamp_grid(tiles, (int64_t)g.num_sms * 256),
                                                   dim3(T / 2, T / 2), 0, stream>>>(
            g.M, g.N, g.K, g.A, g.lda, g.B, g.ldb, g.C, g.ldc);
        break;
    }
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace sgemm_gb300
