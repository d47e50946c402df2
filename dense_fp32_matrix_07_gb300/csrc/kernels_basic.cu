// General-purpose kernels: the predicated shared-memory tiled product (any
// shape, stride and alignment), the zero fill used when K == 0, and the
// operand pack that gives misaligned operands 16-byte-aligned rows.
#include "common.cuh"

namespace sgemm_gb300 {

// ---------------------------------------------------------------------------
// Shared-memory tiled product, one thread per element of C.
//
// Chapter 9: Optimised Matrix Multiplication, section 9.4 (shared-memory
// tiling): a T x T block of threads computes a T x T tile of C, marching K in
// steps of T; each step stages a T x T tile of A and of B in shared memory,
// padded by one column so the column walk is free of bank conflicts, behind
// a barrier before the tile is read and another before it is overwritten
// ("Перемножение матриц: наивное и тайловое", section 2, on why both
// barriers are needed). Unlike the pages' listing, every global access is
// predicated, so M, N, K need not be multiples of T and any leading dimension
// and alignment is accepted; out-of-range tile entries are zero.
// ---------------------------------------------------------------------------
template <int T>
__global__ void __launch_bounds__(T * T)
sgemm_tiled_simple_kernel(int64_t M, int64_t N, int64_t K,
                          const float *__restrict__ A, int64_t lda,
                          const float *__restrict__ B, int64_t ldb,
                          float *__restrict__ C, int64_t ldc)
{
    __shared__ float sA[T][T + 1];
    __shared__ float sB[T][T + 1];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int64_t tiles_n = (N + T - 1) / T;
    const int64_t tiles = ((M + T - 1) / T) * tiles_n;

    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t row = (t / tiles_n) * T + ty;
        const int64_t col = (t % tiles_n) * T + tx;
        float acc = 0.0f;
        for (int64_t k0 = 0; k0 < K; k0 += T) {
            sA[ty][tx] = (row < M && k0 + tx < K) ? A[row * lda + k0 + tx] : 0.0f;
            sB[ty][tx] = (k0 + ty < K && col < N) ? B[(k0 + ty) * ldb + col] : 0.0f;
            __syncthreads();
#pragma unroll
            for (int k = 0; k < T; ++k) acc = fmaf(sA[ty][k], sB[k][tx], acc);
            __syncthreads();
        }
        if (row < M && col < N) C[row * ldc + col] = acc;
    }
}

cudaError_t launch_tiled_simple(const GemmArgs &g, cudaStream_t stream)
{
    constexpr int T = 16;
    const int64_t tiles = ((g.M + T - 1) / T) * ((g.N + T - 1) / T);
    const int64_t cap = (int64_t)g.num_sms * 64;
    const unsigned grid = (unsigned)(tiles < cap ? tiles : cap);
    sgemm_tiled_simple_kernel<T><<<grid, dim3(T, T), 0, stream>>>(
        g.M, g.N, g.K, g.A, g.lda, g.B, g.ldb, g.C, g.ldc);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Zero fill of an M x N block of C (the empty sum, K == 0).
// ---------------------------------------------------------------------------
__global__ void zero_fill_kernel(float *__restrict__ C, int64_t M, int64_t N,
                                 int64_t ldc)
{
    const int64_t total = M * N;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = e / N, j = e % N;
        C[i * ldc + j] = 0.0f;
    }
}

cudaError_t launch_zero_fill(float *C, int64_t M, int64_t N, int64_t ldc,
                             cudaStream_t stream)
{
    const int64_t total = M * N;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    zero_fill_kernel<<<(unsigned)blocks, 256, 0, stream>>>(C, M, N, ldc);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Pack: dst[r * ld_dst + c] = src[r * ld_src + c] for r < rows, c < cols.
// Each warp copies one row segment per iteration, so both the 4-byte reads
// (of a possibly misaligned source) and the writes are coalesced. Entries of
// dst beyond `cols` are left as they are: the product never reads them (its
// tensor maps describe only `cols` columns and fill the rest with zero).
// ---------------------------------------------------------------------------
__global__ void pack_kernel(const float *__restrict__ src, int64_t rows,
                            int64_t cols, int64_t ld_src,
                            float *__restrict__ dst, int64_t ld_dst)
{
    const int64_t segs = (cols + 255) / 256;       // 256-column segments per row
    const int64_t work = rows * segs;
    const int warps = blockDim.x / 32;
    const int lane = threadIdx.x & 31;
    for (int64_t w = blockIdx.x * (int64_t)warps + threadIdx.x / 32; w < work;
         w += (int64_t)gridDim.x * warps) {
        const int64_t r = w / segs;
        const int64_t c0 = (w % segs) * 256;
        const float *s = src + r * ld_src;
        float *d = dst + r * ld_dst;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int64_t c = c0 + q * 32 + lane;
            if (c < cols) d[c] = s[c];
        }
    }
}

cudaError_t launch_pack(const float *src, int64_t rows, int64_t cols,
                        int64_t ld_src, float *dst, int64_t ld_dst,
                        cudaStream_t stream)
{
    const int64_t work = rows * ((cols + 255) / 256);
    int64_t blocks = (work + 7) / 8;
    if (blocks > 8192) blocks = 8192;
    if (blocks < 1) blocks = 1;
    pack_kernel<<<(unsigned)blocks, 256, 0, stream>>>(src, rows, cols, ld_src,
                                                     dst, ld_dst);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Batched layout kernels of the general form alpha * op(A) . op(B) + beta * C.
// ---------------------------------------------------------------------------

// dst[b * s_dst + r * ld_dst + c] = src[b * s_src + r * ld_src + c].
__global__ void pack_batched_kernel(const float *__restrict__ src, int64_t rows, int64_t cols,
                                    int64_t ld_src, int64_t s_src, float *__restrict__ dst,
                                    int64_t ld_dst, int64_t s_dst, int64_t batch)
{
    const int64_t segs = (cols + 255) / 256;
    const int64_t work = batch * rows * segs;
    const int warps = blockDim.x / 32;
    const int lane = threadIdx.x & 31;
    for (int64_t w = blockIdx.x * (int64_t)warps + threadIdx.x / 32; w < work;
         w += (int64_t)gridDim.x * warps) {
        const int64_t seg = w % segs, rb = w / segs;
        const int64_t r = rb % rows, b = rb / rows;
        const float *sr = src + b * s_src + r * ld_src;
        float *dr = dst + b * s_dst + r * ld_dst;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int64_t c = seg * 256 + q * 32 + lane;
            if (c < cols) dr[c] = sr[c];
        }
    }
}

// dst[b * s_dst + c * ld_dst + r] = src[b * s_src + r * ld_src + c], through
// 64 x 64 shared-memory tiles (padded by one column): 32 x 8 threads, each
// moving 16 elements per tile, so reads (along c) and writes (along r) are
// both 128-byte warp segments.
__global__ void __launch_bounds__(256)
pack_transpose_batched_kernel(const float *__restrict__ src, int64_t rows, int64_t cols,
                              int64_t ld_src, int64_t s_src, float *__restrict__ dst,
                              int64_t ld_dst, int64_t s_dst, int64_t batch)
{
    __shared__ float tile[64][65];
    const int tx = threadIdx.x, ty = threadIdx.y;   // 32 x 8 threads
    const int64_t tiles_c = (cols + 63) / 64;
    const int64_t per_entry = ((rows + 63) / 64) * tiles_c;
    for (int64_t t = blockIdx.x; t < batch * per_entry; t += gridDim.x) {
        const int64_t b = t / per_entry, tt = t % per_entry;
        const int64_t r0 = (tt / tiles_c) * 64, c0 = (tt % tiles_c) * 64;
        const float *sb = src + b * s_src;
        float *db = dst + b * s_dst;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t r = r0 + ty + 8 * i;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t c = c0 + tx + 32 * h;
                tile[ty + 8 * i][tx + 32 * h] = (r < rows && c < cols) ? sb[r * ld_src + c] : 0.0f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t c = c0 + ty + 8 * i;   // output row
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t r = r0 + tx + 32 * h;
                if (c < cols && r < rows) db[c * ld_dst + r] = tile[tx + 32 * h][ty + 8 * i];
            }
        }
        __syncthreads();
    }
}

// C_b = beta * C_b; beta == 0 writes zeros without reading C.
__global__ void scale_batched_kernel(float *__restrict__ C, int64_t M, int64_t N, int64_t ldc,
                                     int64_t stride_c, int64_t batch, float beta)
{
    const int64_t total = batch * M * N;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = e % N, ib = e / N;
        const int64_t i = ib % M, b = ib / M;
        float *p = C + b * stride_c + i * ldc + j;
        *p = beta != 0.0f ? beta * *p : 0.0f;
    }
}

namespace {
unsigned grid_for(int64_t work, int64_t per_block, int64_t cap)
{
    int64_t g = (work + per_block - 1) / per_block;
    if (g < 1) g = 1;
    return (unsigned)(g < cap ? g : cap);
}
}  // namespace

cudaError_t launch_pack_batched(const float *src, int64_t rows, int64_t cols, int64_t ld_src,
                                int64_t s_src, float *dst, int64_t ld_dst, int64_t s_dst,
                                int64_t batch, cudaStream_t stream)
{
    pack_batched_kernel<<<grid_for(batch * rows * ((cols + 255) / 256), 8, 8192), 256, 0, stream>>>(
        src, rows, cols, ld_src, s_src, dst, ld_dst, s_dst, batch);
    return cudaGetLastError();
}

cudaError_t launch_pack_transpose_batched(const float *src, int64_t rows, int64_t cols,
                                          int64_t ld_src, int64_t s_src, float *dst,
                                          int64_t ld_dst, int64_t s_dst, int64_t batch,
                                          cudaStream_t stream)
{
    const int64_t tiles = batch * ((rows + 63) / 64) * ((cols + 63) / 64);
    pack_transpose_batched_kernel<<<grid_for(tiles, 1, 8192), dim3(32, 8), 0, stream>>>(
        src, rows, cols, ld_src, s_src, dst, ld_dst, s_dst, batch);
    return cudaGetLastError();
}

cudaError_t launch_scale(float *C, int64_t M, int64_t N, int64_t ldc, int64_t stride_c,
                         int64_t batch, float beta, cudaStream_t stream)
{
    scale_batched_kernel<<<grid_for(batch * M * N, 256, 4096), 256, 0, stream>>>(C, M, N, ldc, stride_c,
                                                                               batch, beta);
    return cudaGetLastError();
}

}  // namespace sgemm_gb300
