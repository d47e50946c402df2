// sgemm_noalloc(): the product for callers that cannot allocate device memory.
//
// sgemm() takes scratch from a stream-ordered memory pool when an operand has
// to be packed (its base is not 16-byte aligned or its rows are not a
// multiple of 4 floats). This entry point packs into a fixed array that lives
// in this file instead, and calls no allocator of any kind: the array is
// reserved when the library's device code is loaded on a GPU and is held by
// that GPU until the process exits.
//
// Set-up: the first call on each device (with that device current) looks up
// the array's device address with cudaGetSymbolAddress(), the error word's
// address, the SM count and the kernels' shared-memory limits, and caches
// them; later calls on the device reuse the cache. Make that first call
// before any stream capture begins.
//
// A second fixed array, 48 MiB, holds the stream-K partial sums and arrival
// counters of the product's schedule (at most two 128 x 256 tiles per SM:
// about 38 MiB on 152 SMs); a schedule that would need more runs whole tiles
// instead.
//
// Where sgemm() would take a k-major configuration (one that reads A as a
// transposed copy), this entry point makes that copy in its fixed array when
// it fits there (K * round_up(M, 32) floats, beside a packed B), and
// otherwise runs the configuration's twin, which reads A as stored.
//
// Sharing: every call on a device uses the same arrays, which keep whatever
// the last call left in them. Nothing in it has to start at zero (each call
// rewrites every packed entry the product reads, the padding at the end of
// packed rows is never read, and the stream-K arrival counters are zeroed by
// a memset on the call's stream before its product). Calls whose work overlaps on the
// GPU (different streams, or different host threads) race on the array and
// must be ordered by the caller.
#include "../../include/sgemm.h"
#include "common.cuh"
#include "configs.cuh"

#include <mutex>

namespace sgemm_gb300 {

// 16 Mi floats = 64 MiB: room for both packed operands of, e.g., a
// 4097 x 3001 x 2049 product (about 14.7 Mi floats).
constexpr int64_t kNoAllocScratchFloats = int64_t(16) << 20;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

// 48 MiB for the stream-K partial sums and arrival counters: two 128 x 256
// FP32 tiles (2 x 128 KiB) per CTA slot for up to 190 SMs, with room for the
// counters.
constexpr size_t kNoAllocWorkspaceBytes = size_t(48) << 20;

static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoAllocWorkspaceBytes];

namespace {

constexpr int kMaxDevices = 64;

struct NoAllocDevice {
    bool ready = false;
    int num_sms = 0;
    unsigned int *status = nullptr;   // device error word
    float *scratch = nullptr;         // device address of g_noalloc_scratch
    unsigned char *workspace = nullptr;   // device address of g_noalloc_workspace
};

std::mutex g_na_mutex;
NoAllocDevice g_na_devices[kMaxDevices];

int noalloc_device(NoAllocDevice **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_na_mutex);
    NoAllocDevice &d = g_na_devices[dev];
    if (!d.ready) {
        int sms = 0;
        unsigned int *status = nullptr;
        void *scratch = nullptr, *workspace = nullptr;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms <= 0 || device_status_word(&status) != cudaSuccess ||
            configs_prepare_device() != cudaSuccess ||
            cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || !scratch ||
            cudaGetSymbolAddress(&workspace, g_noalloc_workspace) != cudaSuccess || !workspace) {
            cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        d.num_sms = sms;
        d.status = status;
        d.scratch = static_cast<float *>(scratch);
        d.workspace = static_cast<unsigned char *>(workspace);
        d.ready = true;
    }
    *out = &d;
    return SGEMM_OK;
}

int64_t round_up32(int64_t x) { return (x + 31) / 32 * 32; }

// SGEMM_ERR_LAUNCH after clearing the failed launch's error, so the caller's
// next cudaGetLastError() does not report it again.
int launch_failed()
{
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
}

int64_t extent_elems(int64_t rows, int64_t cols, int64_t ld)
{
    return (rows == 0 || cols == 0) ? 0 : (rows - 1) * ld + cols;
}

bool ranges_overlap(uint64_t a, int64_t na, uint64_t b, int64_t nb)
{
    if (na == 0 || nb == 0) return false;
    return (__int128)a < (__int128)b + (__int128)nb * 4 && (__int128)b < (__int128)a + (__int128)na * 4;
}

// Copies a rows x cols matrix (leading dimension ld_src) into the scratch
// array at `offset`, with leading dimension ld_dst. One warp per 256-column
// row segment, so reads and writes are coalesced.
__global__ void pack_into_scratch_kernel(const float *__restrict__ src, int64_t rows, int64_t cols,
                                         int64_t ld_src, int64_t offset, int64_t ld_dst)
{
    float *dst = g_noalloc_scratch + offset;
    const int64_t segs = (cols + 255) / 256;
    const int64_t work = rows * segs;
    const int warps = blockDim.x / 32;
    const int lane = threadIdx.x & 31;
    for (int64_t w = blockIdx.x * (int64_t)warps + threadIdx.x / 32; w < work;
         w += (int64_t)gridDim.x * warps) {
        const int64_t r = w / segs;
        const int64_t c0 = (w % segs) * 256;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int64_t c = c0 + q * 32 + lane;
            if (c < cols) dst[r * ld_dst + c] = src[r * ld_src + c];
        }
    }
}

cudaError_t pack_into_scratch(const float *src, int64_t rows, int64_t cols, int64_t ld_src,
                              int64_t offset, int64_t ld_dst, cudaStream_t stream)
{
    int64_t blocks = (rows * ((cols + 255) / 256) + 7) / 8;
    if (blocks > 8192) blocks = 8192;
    if (blocks < 1) blocks = 1;
    pack_into_scratch_kernel<<<(unsigned)blocks, 256, 0, stream>>>(src, rows, cols, ld_src, offset,
                                                                   ld_dst);
    return cudaGetLastError();
}

}  // namespace
}  // namespace sgemm_gb300

using namespace sgemm_gb300;

extern "C" int sgemm_noalloc(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                             const float *B, int64_t ldb, float *C, int64_t ldc,
                             cudaStream_t stream)
{
    const uint64_t a = (uint64_t)(uintptr_t)A, b = (uint64_t)(uintptr_t)B,
                   c = (uint64_t)(uintptr_t)C;
    // Size and stride validation exactly as sgemm() does it (host only).
    int rc = sgemm_plan(M, N, K, lda, ldb, ldc, a, b, c, 1, nullptr, nullptr, nullptr);
    if (rc != SGEMM_OK) return rc;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (C == nullptr) return SGEMM_ERR_INVALID_VALUE;
    if (K > 0 && (A == nullptr || B == nullptr)) return SGEMM_ERR_INVALID_VALUE;
    const int64_t c_elems = extent_elems(M, N, ldc);
    if (K > 0 && (ranges_overlap(c, c_elems, a, extent_elems(M, K, lda)) ||
                  ranges_overlap(c, c_elems, b, extent_elems(K, N, ldb))))
        return SGEMM_ERR_INVALID_VALUE;

    NoAllocDevice *dev = nullptr;
    rc = noalloc_device(&dev);
    if (rc != SGEMM_OK) return rc;

    if (K == 0) return launch_zero_fill(C, M, N, ldc, stream) == cudaSuccess ? SGEMM_OK : launch_failed();

    int cfg = -1, pack_a = 0, pack_b = 0;
    rc = sgemm_plan(M, N, K, lda, ldb, ldc, a, b, c, dev->num_sms, &cfg, &pack_a, &pack_b);
    if (rc != SGEMM_OK) return rc;
    // A configuration that takes A k-major reads a transposed copy of A
    // (K rows of round_up(M, 32) floats): made in the fixed array when it fits
    // there beside a packed B, else the twin that reads A as stored runs.
    const int64_t ldb_p = round_up32(N);
    const int64_t b_floats = pack_b ? K * ldb_p : 0;
    const bool a_kmajor = kConfigTable[cfg].a_kmajor && K * round_up32(M) + b_floats <= kNoAllocScratchFloats;
    if (kConfigTable[cfg].a_kmajor && !a_kmajor) {
        cfg = cfg == kCfgFfma2_128x128_ka ? kCfgFfma2_128x128 : kCfgFfma2_128x256;
        pack_a = ((a & 15u) != 0 || lda % 4 != 0) ? 1 : 0;
    }
    const int64_t lda_p = a_kmajor ? round_up32(M) : round_up32(K);
    const int64_t a_floats = a_kmajor ? K * lda_p : (pack_a ? M * lda_p : 0);
    if (a_floats > kNoAllocScratchFloats || b_floats > kNoAllocScratchFloats ||
        a_floats + b_floats > kNoAllocScratchFloats)
        return SGEMM_ERR_SCRATCH_LIMIT;

    GemmArgs g{M, N, K, A, lda, B, ldb, C, ldc, dev->status, dev->num_sms};
    // The stream-K partial sums and counters go in the fixed workspace array
    // when they fit (they always do on GPUs of up to 190 SMs); otherwise the
    // product runs whole tiles, which need no workspace.
    g.sched = kSchedAuto;
    const size_t ws_bytes = config_workspace_bytes(cfg, g);
    if (ws_bytes > 0 && ws_bytes <= kNoAllocWorkspaceBytes) {
        g.workspace = dev->workspace;
        g.workspace_bytes = ws_bytes;
    } else {
        g.sched = kSchedDataParallel;
    }
    if (a_kmajor) {
        // The transposed copy, K x M with rows of lda_p floats.
        if (launch_pack_transpose_batched(A, M, K, lda, 0, dev->scratch, lda_p, K * lda_p, 1, stream) !=
            cudaSuccess)
            return launch_failed();
        g.A = dev->scratch;
        g.lda = lda_p;
        g.op_a = 1;
    } else if (pack_a) {
        if (pack_into_scratch(A, M, K, lda, 0, lda_p, stream) != cudaSuccess) return launch_failed();
        g.A = dev->scratch;
        g.lda = lda_p;
    }
    if (pack_b) {
        // a_floats is a multiple of 32 floats, so B's copy starts 128-byte aligned.
        if (pack_into_scratch(B, K, N, ldb, a_floats, ldb_p, stream) != cudaSuccess)
            return launch_failed();
        g.B = dev->scratch + a_floats;
        g.ldb = ldb_p;
    }
    return launch_config(cfg, g, stream) == cudaSuccess ? SGEMM_OK : launch_failed();
}
