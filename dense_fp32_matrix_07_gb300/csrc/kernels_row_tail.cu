// The last few rows of C, apart from the tiled product.
//
// The TMA kernels cover C with 128-row block rows, so an M just past a
// multiple of 128 (4097 = 32 * 128 + 1) pads a whole block row of tiles
// for a handful of real rows: 3 % of the FMAs at 4097 x 3001 x 2049. The
// library then runs the tiled product on the first M - r rows only and this
// kernel on the last r <= 8: each row is the course page's dot product of a
// row of A with every column of B ("Перемножение матриц: наивное и
// тайловое", section 1), here r rows at a time against one streamed pass
// over B.
//
// Layout of the work: a CTA owns 128 columns (a float4 of B per lane) and a
// contiguous chunk of K; its 8 warps split that chunk again. Clusters of ks
// CTAs (ks <= 8) span all of K for the same columns. Each CTA adds its 8
// warps' sums in warp order in shared memory; after a cluster barrier, rank
// 0 reads the other CTAs' sums through distributed shared memory and adds
// them in rank order, so the result is deterministic (integer-valued inputs
// stay exact) and no global scratch, counter or memset is needed. A second
// cluster barrier keeps every CTA's shared memory alive until rank 0 is done.
//
// The kernel runs right after the tiled product, which reads and writes
// nothing of its rows: it is launched with programmatic stream
// serialization, so its CTAs take SMs as the product's persistent CTAs
// finish (the product signals its dependents at its start), and it waits
// for the product's completion only at its very end.
#include "common.cuh"
#include "configs.cuh"
#include "ptx.cuh"

namespace sgemm_gb300 {

namespace {

constexpr int kTailThreads = 256;          // 8 warps
constexpr int kTailWarps = kTailThreads / 32;
constexpr int kTailCols = 128;             // columns per CTA: 32 lanes x float4

constexpr int kTailBatch = 16;             // k per batch of loads in flight

// R: rows of the tail (the template keeps the inner loops branch-free).
template <int R>
__global__ void __launch_bounds__(kTailThreads)
row_tail_kernel(const RowTailArgs t)
{
    __shared__ float4 part[kTailWarps][R][32];
    __shared__ float4 cta_sum[R][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t rank = ptx::cluster_ctarank(), ks = ptx::cluster_nctarank();
    const int64_t b = blockIdx.z;
    const int64_t col = (int64_t)blockIdx.x * kTailCols + 4 * lane;
    // This CTA's chunk of K (its cluster rank), then this warp's share.
    const int64_t c0 = t.K * rank / ks, c1 = t.K * (rank + 1) / ks;
    const int64_t k0 = c0 + (c1 - c0) * w / kTailWarps, k1 = c0 + (c1 - c0) * (w + 1) / kTailWarps;
    const float *Ab = t.A + b * t.stride_a + t.m0 * t.a_row_stride;
    const float *Bb = t.B + b * t.stride_b;

    float4 acc[R];
#pragma unroll
    for (int i = 0; i < R; ++i) acc[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    auto fma4 = [](float4 &c, float a, const float4 &v) {
        c.x = fmaf(a, v.x, c.x);
        c.y = fmaf(a, v.y, c.y);
        c.z = fmaf(a, v.z, c.z);
        c.w = fmaf(a, v.w, c.w);
    };
    if (col + 3 < t.N) {
        // B rows are 16-byte aligned (the TMA path's operand), so a lane's
        // four columns are one float4. Loads go out kTailBatch k at a time
        // before their multiply-adds, so that many are in flight per lane.
        int64_t k = k0;
        for (; k + kTailBatch <= k1; k += kTailBatch) {
            float4 bv[kTailBatch];
            float av[R][kTailBatch];
#pragma unroll
            for (int u = 0; u < kTailBatch; ++u)
                bv[u] = __ldg(reinterpret_cast<const float4 *>(Bb + (k + u) * t.ldb + col));
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
                for (int u = 0; u < kTailBatch; ++u) av[i][u] = __ldg(Ab + i * t.a_row_stride + (k + u) * t.a_k_stride);
#pragma unroll
            for (int u = 0; u < kTailBatch; ++u)
#pragma unroll
                for (int i = 0; i < R; ++i) fma4(acc[i], av[i][u], bv[u]);
        }
        for (; k < k1; ++k) {
            const float4 bv = __ldg(reinterpret_cast<const float4 *>(Bb + k * t.ldb + col));
#pragma unroll
            for (int i = 0; i < R; ++i) fma4(acc[i], __ldg(Ab + i * t.a_row_stride + k * t.a_k_stride), bv);
        }
    } else if (col < t.N) {
        // The last columns: only those below N are read.
        for (int64_t k = k0; k < k1; ++k) {
            const float *bp = Bb + k * t.ldb + col;
            float4 bv = make_float4(bp[0], 0.0f, 0.0f, 0.0f);
            if (col + 1 < t.N) bv.y = bp[1];
            if (col + 2 < t.N) bv.z = bp[2];
#pragma unroll
            for (int i = 0; i < R; ++i) fma4(acc[i], Ab[i * t.a_row_stride + k * t.a_k_stride], bv);
        }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) part[w][i][lane] = acc[i];
    __syncthreads();
    if (w == 0) {
#pragma unroll
        for (int i = 0; i < R; ++i) {
            float4 s = part[0][i][lane];
            for (int v = 1; v < kTailWarps; ++v) {
                const float4 p = part[v][i][lane];
                s.x += p.x;
                s.y += p.y;
                s.z += p.z;
                s.w += p.w;
            }
            cta_sum[i][lane] = s;
        }
    }
    // Every CTA's sums are in its shared memory.
    ptx::cluster_sync_all();
    if (rank == 0 && w == 0 && col < t.N) {
        const uint32_t base = ptx::smem_addr(&cta_sum[0][0]);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            float4 s = cta_sum[i][lane];
            for (uint32_t q = 1; q < ks; ++q) {
                const float4 p = ptx::ld_shared_cluster_f4(base + (uint32_t)(i * 32 + lane) * 16u, q);
                s.x += p.x;
                s.y += p.y;
                s.z += p.z;
                s.w += p.w;
            }
            float *crow = t.C + b * t.stride_c + (t.m0 + i) * t.ldc + col;
            const float v[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (col + e < t.N) {
                    const float y = t.alpha * v[e];
                    crow[e] = t.beta != 0.0f ? fmaf(t.beta, crow[e], y) : y;
                }
        }
    }
    // No CTA leaves (releasing its shared memory) before rank 0 has read it.
    ptx::cluster_sync_all();
    // Launched behind the tiled product with programmatic serialization,
    // this grid may run while that one finishes; it does not complete before
    // that grid has, so whatever the stream runs next sees both.
    ptx::grid_dependency_wait();
}

using RowTailKernel = void (*)(const RowTailArgs);
constexpr RowTailKernel kRowTailKernels[kRowTailMax] = {
    row_tail_kernel<1>, row_tail_kernel<2>, row_tail_kernel<3>, row_tail_kernel<4>,
    row_tail_kernel<5>, row_tail_kernel<6>, row_tail_kernel<7>, row_tail_kernel<8>};

}  // namespace

cudaError_t launch_row_tail(const RowTailArgs &t, int num_sms, cudaStream_t stream)
{
    if (t.r < 1 || t.r > kRowTailMax || t.N < 1 || t.K < 1 || t.batch < 1 || t.batch > 65535)
        return cudaErrorInvalidValue;
    const int64_t col_blocks = (t.N + kTailCols - 1) / kTailCols;
    if (col_blocks > 0x7fffffff) return cudaErrorInvalidValue;
    // Clusters of ks CTAs split K: enough CTAs to cover the SMs about once
    // and a half, at least 4 k per warp.
    int ks = 1;
    while (ks < 8 && col_blocks * ks * t.batch * 2 < 3 * (int64_t)num_sms &&
           t.K >= (int64_t)ks * 2 * kTailWarps * 4)
        ks *= 2;
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)ks;
    attr[0].val.clusterDim.z = 1;
    // It may start on SMs that the tiled product (which signals its
    // dependents at its start) leaves before the whole grid has finished.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    lc.gridDim = dim3((unsigned)col_blocks, (unsigned)ks, (unsigned)t.batch);
    lc.blockDim = dim3(kTailThreads);
    lc.dynamicSmemBytes = 0;
    lc.stream = stream;
    lc.attrs = attr;
    lc.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&lc, kRowTailKernels[t.r - 1], t);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sgemm_gb300
