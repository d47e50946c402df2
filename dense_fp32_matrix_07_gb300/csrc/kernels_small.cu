// Small products: C = A . B for up to about 400^3 (M*N*K <= 2^26, K <= 1024),
// where one tile per CTA cannot fill the GPU with work and the time goes to
// launch and memory latency rather than to the FP32 pipe.
//
// The pages' register-tiled kernel (Chapter 9, section 9.5) walks K in
// 16-deep tiles, each a global load, a barrier and 16 k of FMAs, so a 256^3
// product waits on 16 round trips to memory in a row. This kernel asks for
// all of its K panel at once instead: a CTA owns a 32 x 32 tile of C, and
// for each chunk of up to 256 k its 256 threads load the A panel (32 rows)
// and the B panel (32 columns) together, one barrier, then multiply the
// whole chunk from shared memory; a product with K <= 256 waits on memory
// once. Each thread computes 2 x 2 outputs: per 4 k it reads its two A rows
// as float4 (rows padded to 260 floats, so the 4 rows a warp reads hit
// distinct bank groups) and 4 float2 of B, for 16 FMAs.
//
// Any layout: rows of A and B are read as float4 when both operands are
// 16-byte aligned with leading dimensions that are multiples of 4, else one
// float at a time; reads past M, N or K give zero, and only entries inside C
// are written.
#include "common.cuh"
#include "configs.cuh"

namespace sgemm_gb300 {

namespace {

constexpr int kSmallTile = 32;                     // C tile: 32 x 32
constexpr int kSmallThreads = 256;                 // 16 x 16 threads, 2 x 2 outputs each
constexpr int kSmallChunk = 256;                   // k per chunk
constexpr int kSmallARow = kSmallChunk + 4;        // floats per A row in shared memory
constexpr size_t kSmallSmem = (size_t)(kSmallTile * kSmallARow + kSmallChunk * kSmallTile) * sizeof(float);

template <bool VEC>
__global__ void __launch_bounds__(kSmallThreads)
sgemm_small_kernel(int64_t M, int64_t N, int64_t K, const float *__restrict__ A, int64_t lda,
                   const float *__restrict__ B, int64_t ldb, float *__restrict__ C, int64_t ldc)
{
    extern __shared__ float4 small_smem[];
    float *sA = reinterpret_cast<float *>(small_smem);      // [32][kSmallARow]
    float *sB = sA + kSmallTile * kSmallARow;               // [kSmallChunk][32]
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int64_t tiles_n = (N + kSmallTile - 1) / kSmallTile;
    const int64_t row0 = (int64_t)(blockIdx.x / tiles_n) * kSmallTile;
    const int64_t col0 = (int64_t)(blockIdx.x % tiles_n) * kSmallTile;

    float acc[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};
    for (int64_t k0 = 0; k0 < K; k0 += kSmallChunk) {
        const int kc = (int)(K - k0 < kSmallChunk ? K - k0 : kSmallChunk);
        const int kc4 = (kc + 3) & ~3;      // the chunk rounded up to whole groups of 4 k
        // A panel: 32 rows x kc4 k as float4 groups, all issued before the
        // first store to shared memory.
        if constexpr (VEC) {
            constexpr int per = kSmallTile * kSmallChunk / 4 / kSmallThreads;   // 8 float4 a thread
            float4 va[per], vb[per];
#pragma unroll
            for (int j = 0; j < per; ++j) {
                const int e = tid + j * kSmallThreads;     // float4 index in the [32][64] panel
                const int r = e / (kSmallChunk / 4), c4 = e % (kSmallChunk / 4);
                const int64_t row = row0 + r, k = k0 + 4 * c4;
                va[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (4 * c4 < kc4 && row < M) {
                    if (k + 3 < K) {
                        va[j] = __ldg(reinterpret_cast<const float4 *>(A + row * lda + k));
                    } else {
                        const float *p = A + row * lda + k;
                        va[j].x = p[0];
                        if (k + 1 < K) va[j].y = p[1];
                        if (k + 2 < K) va[j].z = p[2];
                    }
                }
                // B panel: kc rows x 32 columns, 8 float4 per row.
                const int kr = e / (kSmallTile / 4), n4 = e % (kSmallTile / 4);
                const int64_t kb = k0 + kr, col = col0 + 4 * n4;
                vb[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (kr < kc4 && kb < K) {
                    if (col + 3 < N) {
                        vb[j] = __ldg(reinterpret_cast<const float4 *>(B + kb * ldb + col));
                    } else if (col < N) {
                        const float *p = B + kb * ldb + col;
                        vb[j].x = p[0];
                        if (col + 1 < N) vb[j].y = p[1];
                        if (col + 2 < N) vb[j].z = p[2];
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < per; ++j) {
                const int e = tid + j * kSmallThreads;
                const int r = e / (kSmallChunk / 4), c4 = e % (kSmallChunk / 4);
                *reinterpret_cast<float4 *>(sA + r * kSmallARow + 4 * c4) = va[j];
                const int kr = e / (kSmallTile / 4), n4 = e % (kSmallTile / 4);
                *reinterpret_cast<float4 *>(sB + kr * kSmallTile + 4 * n4) = vb[j];
            }
        } else {
            // One float at a time (misaligned operands); 32 of A and 32 of B
            // a thread, loaded before they are stored.
            constexpr int per = kSmallTile * kSmallChunk / kSmallThreads;      // 32
            float va[per], vb[per];
#pragma unroll
            for (int j = 0; j < per; ++j) {
                const int e = tid + j * kSmallThreads;
                const int r = e / kSmallChunk, c = e % kSmallChunk;
                const int64_t row = row0 + r, k = k0 + c;
                va[j] = (c < kc4 && row < M && k < K) ? A[row * lda + k] : 0.0f;
                const int kr = e / kSmallTile, n = e % kSmallTile;
                const int64_t kb = k0 + kr, col = col0 + n;
                vb[j] = (kr < kc4 && kb < K && col < N) ? B[kb * ldb + col] : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < per; ++j) {
                const int e = tid + j * kSmallThreads;
                sA[(e / kSmallChunk) * kSmallARow + e % kSmallChunk] = va[j];
                sB[(e / kSmallTile) * kSmallTile + e % kSmallTile] = vb[j];
            }
        }
        __syncthreads();
        // Rows 2ty, 2ty + 1 and columns 2tx, 2tx + 1 of the tile; the chunk's
        // k in groups of 4 (k past K hold zeros in both panels).
        const float *a0 = sA + (2 * ty) * kSmallARow, *a1 = a0 + kSmallARow;
        const float *b = sB + 2 * tx;
#pragma unroll 4
        for (int k = 0; k < kc4; k += 4) {
            const float4 x0 = *reinterpret_cast<const float4 *>(a0 + k);
            const float4 x1 = *reinterpret_cast<const float4 *>(a1 + k);
            const float xa[2][4] = {{x0.x, x0.y, x0.z, x0.w}, {x1.x, x1.y, x1.z, x1.w}};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 y = *reinterpret_cast<const float2 *>(b + (k + u) * kSmallTile);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    acc[r][0] = fmaf(xa[r][u], y.x, acc[r][0]);
                    acc[r][1] = fmaf(xa[r][u], y.y, acc[r][1]);
                }
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int64_t row = row0 + 2 * ty + r;
        if (row >= M) break;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int64_t col = col0 + 2 * tx + c;
            if (col < N) C[row * ldc + col] = acc[r][c];
        }
    }
}

}  // namespace

cudaError_t prepare_small()
{
    cudaError_t e = cudaFuncSetAttribute(sgemm_small_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmallSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(sgemm_small_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmallSmem);
}

cudaError_t launch_small(const GemmArgs &g, cudaStream_t stream)
{
    const int64_t tiles = ((g.M + kSmallTile - 1) / kSmallTile) * ((g.N + kSmallTile - 1) / kSmallTile);
    if (tiles < 1 || tiles > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const bool vec = ((reinterpret_cast<uintptr_t>(g.A) | reinterpret_cast<uintptr_t>(g.B)) & 15u) == 0 &&
                     g.lda % 4 == 0 && g.ldb % 4 == 0;
    if (vec)
        sgemm_small_kernel<true><<<(unsigned)tiles, kSmallThreads, kSmallSmem, stream>>>(
            g.M, g.N, g.K, g.A, g.lda, g.B, g.ldb, g.C, g.ldc);
    else
        sgemm_small_kernel<false><<<(unsigned)tiles, kSmallThreads, kSmallSmem, stream>>>(
            g.M, g.N, g.K, g.A, g.lda, g.B, g.ldb, g.C, g.ldc);
    return cudaGetLastError();
}

}  // namespace sgemm_gb300
