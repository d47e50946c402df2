// General-purpose kernels: the predicated shared-memory tiled product (any
// shape, stride and alignment), the zero fill used when K == 0, and the
// operand pack that gives misaligned operands 16-byte-aligned rows.
#include "common.cuh"
#include "ptx.cuh"

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
// Batched layout kernels of the general form alpha * op(A) . op(B) + beta * C.
// ---------------------------------------------------------------------------

// dst[b * s_dst + r * ld_dst + c] = src[b * s_src + r * ld_src + c]: each
// warp copies 256-column segments of rows, block `blk` of `nblk` (256
// threads) taking every nblk-th group of 8 segments, so the 4-byte reads (of
// a possibly misaligned source) and the writes are coalesced. Entries of dst
// beyond `cols` are left as they are: the product never reads them (its
// tensor maps describe only `cols` columns and fill the rest with zero).
__device__ __forceinline__ void copy_rows(const PackJob &j, int64_t blk, int64_t nblk)
{
    const int64_t segs = (j.cols + 255) / 256;
    const int64_t work = j.batch * j.rows * segs;
    const int lane = threadIdx.x & 31;
    for (int64_t w = blk * 8 + threadIdx.x / 32; w < work; w += nblk * 8) {
        const int64_t seg = w % segs, rb = w / segs;
        const int64_t r = rb % j.rows, b = rb / j.rows;
        const float *sr = j.src + b * j.s_src + r * j.ld_src;
        float *dr = j.dst + b * j.s_dst + r * j.ld_dst;
        // All eight loads go out before the first store (source and
        // destination never overlap), so they are in flight together.
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int64_t c = seg * 256 + q * 32 + lane;
            v[q] = c < j.cols ? __ldg(sr + c) : 0.0f;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int64_t c = seg * 256 + q * 32 + lane;
            if (c < j.cols) dr[c] = v[q];
        }
    }
}

// dst[b * s_dst + c * ld_dst + r] = src[b * s_src + r * ld_src + c], through
// 64 x 64 shared-memory tiles (padded by one column): 256 threads as 32 x 8,
// each moving 16 elements per tile, so reads (along c) and writes (along r)
// are both 128-byte warp segments.
__device__ __forceinline__ void transpose_tiles(const PackJob &j, int64_t blk, int64_t nblk,
                                                float (*tile)[65])
{
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int64_t tiles_c = (j.cols + 63) / 64;
    const int64_t per_entry = ((j.rows + 63) / 64) * tiles_c;
    for (int64_t t = blk; t < j.batch * per_entry; t += nblk) {
        const int64_t b = t / per_entry, tt = t % per_entry;
        const int64_t r0 = (tt / tiles_c) * 64, c0 = (tt % tiles_c) * 64;
        const float *sb = j.src + b * j.s_src;
        float *db = j.dst + b * j.s_dst;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t r = r0 + ty + 8 * i;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t c = c0 + tx + 32 * h;
                tile[ty + 8 * i][tx + 32 * h] = (r < j.rows && c < j.cols) ? __ldg(sb + r * j.ld_src + c) : 0.0f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t c = c0 + ty + 8 * i;   // output row
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t r = r0 + tx + 32 * h;
                if (c < j.cols && r < j.rows) db[c * j.ld_dst + r] = tile[tx + 32 * h][ty + 8 * i];
            }
        }
        __syncthreads();
    }
}

__device__ __forceinline__ void run_pack_job(const PackJob &j, int64_t blk, float (*tile)[65])
{
    if (j.transpose)
        transpose_tiles(j, blk, j.blocks, tile);
    else
        copy_rows(j, blk, j.blocks);
}

__global__ void __launch_bounds__(256) pack_transpose_batched_kernel(const PackJob j)
{
    __shared__ float tile[64][65];
    transpose_tiles(j, blockIdx.x, gridDim.x, tile);
}

// Both operands' layout passes of one product in one launch: blocks
// [0, a.blocks) run job a, the next b.blocks run job b, and one more block
// zeroes `zero_words` words (the arrival counters of the product's stream-K
// region and of the row-tail kernel; with no job, that block is the whole
// launch). Every
// block first allows a kernel queued behind this one with programmatic
// serialization (the product, which waits for this grid's completion before
// it reads anything) to start taking SMs as this grid's last blocks run.
// At most 40 registers a thread, so six blocks fit an SM (same-box A/B: a
// hair faster than 48 registers and five on 4097 x 3001 x 2049).
__global__ void __launch_bounds__(256, 6)
pack_pair_kernel(const PackJob a, const PackJob b, unsigned int *zero, int64_t zero_words)
{
    __shared__ float tile[64][65];
    ptx::grid_launch_dependents();
    const int64_t blk = blockIdx.x;
    if (blk < a.blocks) {
        run_pack_job(a, blk, tile);
    } else if (blk < a.blocks + b.blocks) {
        run_pack_job(b, blk - a.blocks, tile);
    } else {
        for (int64_t w = threadIdx.x; w < zero_words; w += blockDim.x) zero[w] = 0u;
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

PackJob pack_job(const float *src, int64_t rows, int64_t cols, int64_t ld_src, int64_t s_src, float *dst,
                 int64_t ld_dst, int64_t s_dst, int64_t batch, bool transpose)
{
    PackJob j{src, rows, cols, ld_src, s_src, dst, ld_dst, s_dst, batch, transpose ? 1 : 0, 0};
    j.blocks = transpose ? grid_for(batch * ((rows + 63) / 64) * ((cols + 63) / 64), 1, 8192)
                         : grid_for(batch * rows * ((cols + 255) / 256), 8, 8192);
    return j;
}

cudaError_t launch_pack_transpose_batched(const float *src, int64_t rows, int64_t cols,
                                          int64_t ld_src, int64_t s_src, float *dst,
                                          int64_t ld_dst, int64_t s_dst, int64_t batch,
                                          cudaStream_t stream)
{
    const PackJob j = pack_job(src, rows, cols, ld_src, s_src, dst, ld_dst, s_dst, batch, true);
    pack_transpose_batched_kernel<<<(unsigned)j.blocks, 256, 0, stream>>>(j);
    return cudaGetLastError();
}

cudaError_t launch_pack_pair(const PackJob &a, const PackJob &b, unsigned int *zero, size_t zero_bytes,
                             cudaStream_t stream)
{
    const int64_t zero_words = zero ? (int64_t)(zero_bytes / sizeof(unsigned int)) : 0;
    const int64_t blocks = a.blocks + b.blocks + (zero_words > 0 ? 1 : 0);
    if (blocks < 1 || blocks > 0x7fffffff) return cudaErrorInvalidValue;
    pack_pair_kernel<<<(unsigned)blocks, 256, 0, stream>>>(a, b, zero, zero_words);
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
