// The last few rows of C, apart from the tiled product.
//
// The TMA kernels cover C with 128-row block rows, so an M just past a
// multiple of 128 (4097 = 32 * 128 + 1) pads a whole block row of tiles
// for a handful of real rows: 3 % of the FMAs at 4097 x 3001 x 2049. The
// library then runs the tiled product on the first M - r rows and this
// kernel on the last r <= 8: each row is the course page's dot product of a
// row of A with every column of B ("Перемножение матриц: наивное и
// тайловое", section 1), here r rows at a time against one streamed pass
// over B.
//
// Layout of the work: a CTA owns 128 columns (a float4 of B per lane) and a
// contiguous chunk of K (one of ks, its blockIdx.y); its 8 warps split that
// chunk again. Each CTA adds its 8 warps' sums in warp order in shared
// memory. With ks > 1 it writes that sum to a slot of its own and counts
// itself in its column block's arrival counter; the CTA that completes the
// count adds the ks slots in chunk order and stores C, so the result is
// deterministic (integer-valued inputs stay exact) and no CTA waits for
// another. The CTAs need no cluster, so each can start on the first SM the
// product leaves.
//
// The kernel runs right after the tiled product, which reads and writes
// nothing of its rows: it is launched with programmatic stream
// serialization, so its CTAs take SMs as the product's persistent CTAs
// finish, and it waits for the product's completion only at its very end.
#include "common.cuh"
#include "configs.cuh"
#include "ptx.cuh"
#include "schedule.cuh"

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
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int ks = (int)gridDim.y, chunk = (int)blockIdx.y;
    const int64_t b = blockIdx.z, cb = blockIdx.x;
    const int64_t col = cb * kTailCols + 4 * lane;
    // This CTA's chunk of K, then this warp's share.
    const int64_t c0 = t.K * chunk / ks, c1 = t.K * (chunk + 1) / ks;
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
        float4 s[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            s[i] = part[0][i][lane];
            for (int v = 1; v < kTailWarps; ++v) {
                const float4 p = part[v][i][lane];
                s[i].x += p.x;
                s[i].y += p.y;
                s[i].z += p.z;
                s[i].w += p.w;
            }
        }
        bool store = ks == 1;
        if (!store) {
            // Publish this chunk's sum, then count it; the chunk that
            // completes the count adds all ks sums in chunk order.
            const int64_t blk = b * gridDim.x + cb;
            float4 *slots = reinterpret_cast<float4 *>(t.slots) + blk * (ks * R * 32);
#pragma unroll
            for (int i = 0; i < R; ++i) slots[(chunk * R + i) * 32 + lane] = s[i];
            __threadfence();
            __syncwarp();
            unsigned before = 0;
            if (lane == 0) before = atomic_inc_acq_rel_gpu(t.counters + blk);
            store = __shfl_sync(0xffffffffu, before, 0) == (unsigned)(ks - 1);
            if (store) {
                (void)ld_acquire_gpu(t.counters + blk);
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    s[i] = slots[i * 32 + lane];
                    for (int q = 1; q < ks; ++q) {
                        const float4 p = slots[(q * R + i) * 32 + lane];
                        s[i].x += p.x;
                        s[i].y += p.y;
                        s[i].z += p.z;
                        s[i].w += p.w;
                    }
                }
            }
        }
        if (store && col < t.N) {
#pragma unroll
            for (int i = 0; i < R; ++i) {
                float *crow = t.C + b * t.stride_c + (t.m0 + i) * t.ldc + col;
                const float v[4] = {s[i].x, s[i].y, s[i].z, s[i].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (col + e < t.N) {
                        const float y = t.alpha * v[e];
                        crow[e] = t.beta != 0.0f ? fmaf(t.beta, crow[e], y) : y;
                    }
            }
        }
    }
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

int row_tail_splits(int64_t r, int64_t N, int64_t K, int64_t batch, int num_sms)
{
    // Enough CTAs to cover the SMs about three times over, at least 4 k per
    // warp, at most 16 chunks for one row and 8 for more (the chunk sums
    // the last CTA adds grow with the rows; same-box A/B of 16 against 8:
    // 4097 x 3001 x 2049 778.4 against 779.4 us, 1025 x 1024 x 2048 81.3
    // against 83.0 us, but 4100 x 3001 x 2049 787.5 against 783.4 us).
    const int max_splits = r == 1 ? 16 : 8;
    const int64_t col_blocks = (N + kTailCols - 1) / kTailCols;
    int ks = 1;
    while (ks < max_splits && col_blocks * ks * 2 * batch <= 3 * (int64_t)num_sms &&
           K >= (int64_t)ks * 2 * kTailWarps * 4)
        ks *= 2;
    return ks;
}

size_t row_tail_counter_bytes(int64_t r, int64_t N, int64_t K, int64_t batch, int num_sms)
{
    if (row_tail_splits(r, N, K, batch, num_sms) == 1) return 0;
    const size_t n = (size_t)((N + kTailCols - 1) / kTailCols) * (size_t)batch * sizeof(unsigned);
    return (n + 255) / 256 * 256;
}

size_t row_tail_slot_bytes(int64_t r, int64_t N, int64_t K, int64_t batch, int num_sms)
{
    const int ks = row_tail_splits(r, N, K, batch, num_sms);
    if (ks == 1) return 0;
    return (size_t)((N + kTailCols - 1) / kTailCols) * (size_t)batch * ks * r * kTailCols * sizeof(float);
}

cudaError_t launch_row_tail(const RowTailArgs &t, int num_sms, cudaStream_t stream)
{
    if (t.r < 1 || t.r > kRowTailMax || t.N < 1 || t.K < 1 || t.batch < 1 || t.batch > 65535)
        return cudaErrorInvalidValue;
    const int64_t col_blocks = (t.N + kTailCols - 1) / kTailCols;
    if (col_blocks > 0x7fffffff) return cudaErrorInvalidValue;
    const int ks = row_tail_splits(t.r, t.N, t.K, t.batch, num_sms);
    if (ks > 1 && (t.counters == nullptr || t.slots == nullptr)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attr[1];
    // It may start on SMs that the tiled product leaves before the whole
    // grid has finished.
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.gridDim = dim3((unsigned)col_blocks, (unsigned)ks, (unsigned)t.batch);
    lc.blockDim = dim3(kTailThreads);
    lc.dynamicSmemBytes = 0;
    lc.stream = stream;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&lc, kRowTailKernels[t.r - 1], t);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sgemm_gb300
