// C ABI of the SGEMM library: argument validation, per-device state, the
// tile-configuration selector and kernel dispatch. The exported functions and
// their contracts are declared in include/sgemm.h.
#include "../../include/sgemm.h"
#include "common.cuh"
#include "configs.cuh"

#include <cstdlib>
#include <cstring>
#include <mutex>

namespace sgemm_gb300 {

// Device error word: kernels OR status bits into it (kStatusTimeout), and
// sgemm_check_status() reads and clears it. One copy exists per device.
__device__ unsigned int g_status_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    unsigned int *status = nullptr;   // device address of g_status_word
    cudaMemPool_t pool = nullptr;     // scratch for packed operands
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

// Per-device state, created on the first call that runs on the device.
int device_state(DeviceState **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &s = g_devices[dev];
    if (!s.ready) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms <= 0) {
            cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        void *status = nullptr;
        if (cudaGetSymbolAddress(&status, g_status_word) != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        if (configs_prepare_device() != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        // Keep up to 4 GiB of freed scratch in the pool between calls, so a
        // steady stream of calls does not map and unmap memory every time.
        uint64_t keep = 4ull << 30;
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        s.num_sms = sms;
        s.status = static_cast<unsigned int *>(status);
        s.pool = pool;
        s.ready = true;
    }
    *out = &s;
    return SGEMM_OK;
}

bool is_aligned16(uint64_t addr) { return (addr & 15u) == 0; }

// Extent in elements of a rows x cols matrix with leading dimension ld, or -1
// on overflow of the byte size.
int64_t extent(int64_t rows, int64_t cols, int64_t ld)
{
    if (rows == 0 || cols == 0) return 0;
    const __int128 e = (__int128)(rows - 1) * ld + cols;
    if (e * 4 > (__int128)INT64_MAX) return -1;
    return (int64_t)e;
}

bool overlaps(uint64_t a, int64_t a_elems, uint64_t b, int64_t b_elems)
{
    if (a_elems == 0 || b_elems == 0) return false;
    const __int128 a0 = a, a1 = (__int128)a + (__int128)a_elems * 4;
    const __int128 b0 = b, b1 = (__int128)b + (__int128)b_elems * 4;
    return a0 < b1 && b0 < a1;
}

// Size checks shared by sgemm_plan() and sgemm_ex() (no pointers involved).
int check_sizes(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (ldc < N || ldc < 1) return SGEMM_ERR_INVALID_VALUE;
    if (K > 0 && (lda < K || ldb < N)) return SGEMM_ERR_INVALID_VALUE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return SGEMM_ERR_OVERFLOW;
    if (extent(M, N, ldc) < 0) return SGEMM_ERR_OVERFLOW;
    if (K > 0 && (extent(M, K, lda) < 0 || extent(K, N, ldb) < 0)) return SGEMM_ERR_OVERFLOW;
    return SGEMM_OK;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

}  // namespace

// Device address of this device's error word (no allocation involved).
cudaError_t device_status_word(unsigned int **out)
{
    return cudaGetSymbolAddress(reinterpret_cast<void **>(out), g_status_word);
}

// Operand of a product that the TMA path reads in place only when its base
// is 16-byte aligned and its rows are a multiple of 16 bytes long.
static bool needs_pack(uint64_t addr, int64_t ld) { return !is_aligned16(addr) || (ld % 4) != 0; }

}  // namespace sgemm_gb300

using namespace sgemm_gb300;

extern "C" {

int sgemm_num_configs(void) { return kNumConfigs; }

const char *sgemm_config_name(int config)
{
    if (config < 0 || config >= kNumConfigs) return "?";
    return kConfigTable[config].name;
}

const char *sgemm_error_string(int code)
{
    switch (code) {
    case SGEMM_OK: return "SGEMM_OK: success";
    case SGEMM_ERR_INVALID_VALUE: return "SGEMM_ERR_INVALID_VALUE: invalid size, leading dimension, pointer, overlap or config";
    case SGEMM_ERR_OVERFLOW: return "SGEMM_ERR_OVERFLOW: an index or byte offset would overflow";
    case SGEMM_ERR_ALLOC: return "SGEMM_ERR_ALLOC: scratch allocation failed";
    case SGEMM_ERR_LAUNCH: return "SGEMM_ERR_LAUNCH: kernel launch failed";
    case SGEMM_ERR_TIMEOUT: return "SGEMM_ERR_TIMEOUT: a device-side wait hit its spin limit";
    case SGEMM_ERR_CUDA: return "SGEMM_ERR_CUDA: CUDA runtime failure";
    case SGEMM_ERR_UNSUPPORTED: return "SGEMM_ERR_UNSUPPORTED: the forced config cannot run this problem";
    case SGEMM_ERR_SCRATCH_LIMIT: return "SGEMM_ERR_SCRATCH_LIMIT: packed operands exceed sgemm_noalloc's 64 MiB scratch array";
    default: return "unknown sgemm status code";
    }
}

int sgemm_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
               uint64_t a_addr, uint64_t b_addr, uint64_t c_addr, int num_sms,
               int *out_config, int *out_pack_a, int *out_pack_b)
{
    const int rc = check_sizes(M, N, K, lda, ldb, ldc);
    if (rc != SGEMM_OK) return rc;
    if (num_sms <= 0) return SGEMM_ERR_INVALID_VALUE;
    const ProblemShape p{M, N, K, lda, ldb, ldc, a_addr, b_addr, c_addr, num_sms};
    const int cfg = select_config(p);
    const bool packs = kConfigTable[cfg].packs;
    if (out_config) *out_config = cfg;
    if (out_pack_a) *out_pack_a = (packs && needs_pack(a_addr, lda)) ? 1 : 0;
    if (out_pack_b) *out_pack_b = (packs && needs_pack(b_addr, ldb)) ? 1 : 0;
    return SGEMM_OK;
}

}  // extern "C"

namespace sgemm_gb300 {

// sgemm_ex() with two test-only knobs: a forced schedule policy (-1: the
// configuration's own) and a copy for CTA 0's producer to withhold (-1: none).
static int sgemm_impl(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                      const float *B, int64_t ldb, float *C, int64_t ldc, int config,
                      int sched_override, int withhold_it, cudaStream_t stream)
{
    if (config < -1 || config >= kNumConfigs) return SGEMM_ERR_INVALID_VALUE;
    int rc = check_sizes(M, N, K, lda, ldb, ldc);
    if (rc != SGEMM_OK) return rc;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (C == nullptr) return SGEMM_ERR_INVALID_VALUE;
    if (K > 0 && (A == nullptr || B == nullptr)) return SGEMM_ERR_INVALID_VALUE;

    const uint64_t a = (uint64_t)(uintptr_t)A, b = (uint64_t)(uintptr_t)B,
                   c = (uint64_t)(uintptr_t)C;
    const int64_t c_elems = extent(M, N, ldc);
    if (K > 0 && (overlaps(c, c_elems, a, extent(M, K, lda)) ||
                  overlaps(c, c_elems, b, extent(K, N, ldb))))
        return SGEMM_ERR_INVALID_VALUE;

    DeviceState *dev = nullptr;
    rc = device_state(&dev);
    if (rc != SGEMM_OK) return rc;

    if (K == 0) {
        if (launch_zero_fill(C, M, N, ldc, stream) != cudaSuccess) return SGEMM_ERR_LAUNCH;
        return SGEMM_OK;
    }

    const ProblemShape p{M, N, K, lda, ldb, ldc, a, b, c, dev->num_sms};
    const int cfg = config < 0 ? select_config(p) : config;
    if (!config_supports(cfg, p)) return SGEMM_ERR_UNSUPPORTED;

    GemmArgs g{M, N, K, A, lda, B, ldb, C, ldc, dev->status, dev->num_sms};
    g.sched = sched_override >= 0 ? sched_override : kConfigTable[cfg].sched;
    g.withhold_it = withhold_it;
    // One scratch allocation, carved into: packed A, packed B (rows padded to
    // a multiple of 32 floats = 128 bytes), then the stream-K workspace.
    const bool packs = kConfigTable[cfg].packs;
    const bool pa = packs && needs_pack(a, lda), pb = packs && needs_pack(b, ldb);
    const int64_t lda_p = round_up(K, 32), ldb_p = round_up(N, 32);
    const size_t a_bytes = pa ? (size_t)(M * lda_p) * 4 : 0;
    const size_t b_bytes = pb ? (size_t)(K * ldb_p) * 4 : 0;
    const size_t ws_off = (a_bytes + b_bytes + 255) / 256 * 256;
    const size_t ws_bytes = config_workspace_bytes(cfg, g);
    const size_t total = ws_off + ws_bytes;
    uint8_t *scratch = nullptr;
    if (total > 0) {
        if (cudaMallocFromPoolAsync((void **)&scratch, total, dev->pool, stream) != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_ALLOC;
        }
        if (pa) {
            float *dst = reinterpret_cast<float *>(scratch);
            if (launch_pack(A, M, K, lda, dst, lda_p, stream) != cudaSuccess) {
                cudaFreeAsync(scratch, stream);
                return SGEMM_ERR_LAUNCH;
            }
            g.A = dst;
            g.lda = lda_p;
        }
        if (pb) {
            float *dst = reinterpret_cast<float *>(scratch + a_bytes);
            if (launch_pack(B, K, N, ldb, dst, ldb_p, stream) != cudaSuccess) {
                cudaFreeAsync(scratch, stream);
                return SGEMM_ERR_LAUNCH;
            }
            g.B = dst;
            g.ldb = ldb_p;
        }
        if (ws_bytes > 0) {
            g.workspace = scratch + ws_off;
            g.workspace_bytes = ws_bytes;
        }
    }

    const cudaError_t err = launch_config(cfg, g, stream);
    if (scratch) cudaFreeAsync(scratch, stream);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
}

}  // namespace sgemm_gb300

extern "C" {

int sgemm_ex(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
             const float *B, int64_t ldb, float *C, int64_t ldc, int config,
             cudaStream_t stream)
{
    return sgemm_impl(M, N, K, A, lda, B, ldb, C, ldc, config, -1, -1, stream);
}

int sgemm(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
          const float *B, int64_t ldb, float *C, int64_t ldc, cudaStream_t stream)
{
    return sgemm_impl(M, N, K, A, lda, B, ldb, C, ldc, -1, -1, -1, stream);
}

int sgemm_test_withhold_copy(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                             const float *B, int64_t ldb, float *C, int64_t ldc, int slab,
                             cudaStream_t stream)
{
    // Whole tiles: no stream-K waits between CTAs, only the withheld copy.
    return sgemm_impl(M, N, K, A, lda, B, ldb, C, ldc, -1, kSchedDataParallel,
                      slab < 0 ? -1 : slab, stream);
}

int sgemm_check_status(cudaStream_t stream)
{
    DeviceState *dev = nullptr;
    const int rc = device_state(&dev);
    if (rc != SGEMM_OK) return rc;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    unsigned int word = 0;
    if (cudaMemcpyAsync(&word, dev->status, sizeof(word), cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    if (word != 0) {
        if (cudaMemsetAsync(dev->status, 0, sizeof(word), stream) != cudaSuccess ||
            cudaStreamSynchronize(stream) != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        if (word & kStatusTimeout) return SGEMM_ERR_TIMEOUT;
    }
    return SGEMM_OK;
}

}  // extern "C"
