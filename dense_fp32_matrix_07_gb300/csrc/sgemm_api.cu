// C ABI of the SGEMM library: argument validation, per-device state, the
// tile-configuration selector and kernel dispatch. The exported functions and
// their contracts are declared in include/sgemm.h.
#include "../../include/sgemm.h"
#include "common.cuh"
#include "configs.cuh"
#include "schedule.cuh"

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace sgemm_gb300 {

// Device error word: kernels OR status bits into it (kStatusTimeout,
// kStatusLaunchConfig), and sgemm_check_status() reads and clears it. One
// copy exists per device.
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

// Test hook (sgemm_test_fail_next_allocs): scratch allocations still to fail.
std::atomic<int> g_fail_allocs{0};

// One pending test failure, if any is left to take.
bool take_test_alloc_failure()
{
    int n = g_fail_allocs.load();
    while (n > 0)
        if (g_fail_allocs.compare_exchange_weak(n, n - 1)) return true;
    return false;
}

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
    case SGEMM_ERR_LAUNCH: return "SGEMM_ERR_LAUNCH: a kernel launch failed, or a kernel found its launch shape wrong and did nothing";
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
    // A k-major configuration always transposes the caller's M x K A.
    if (out_pack_a) *out_pack_a = (packs && (kConfigTable[cfg].a_kmajor || needs_pack(a_addr, lda))) ? 1 : 0;
    if (out_pack_b) *out_pack_b = (packs && needs_pack(b_addr, ldb)) ? 1 : 0;
    return SGEMM_OK;
}

}  // extern "C"

namespace sgemm_gb300 {

// One call of the general form alpha * op(A_b) . op(B_b) + beta * C_b.
struct Call {
    int op_a, op_b;
    int64_t M, N, K;
    float alpha;
    const float *A;
    int64_t lda, sa;
    const float *B;
    int64_t ldb, sb;
    float beta;
    float *C;
    int64_t ldc, sc;
    int64_t batch;
    int config;          // -1: automatic
    int sched_override;  // -1: the configuration's policy (test knob)
    int withhold_it;     // -1: none (test knob)
};

// Elements spanned by `batch` entries of extent `e` at stride `s`, or -1.
static int64_t batch_extent(int64_t e, int64_t s, int64_t batch)
{
    if (e <= 0) return e;
    const __int128 t = (__int128)(batch - 1) * s + e;
    if (t * 4 > (__int128)INT64_MAX) return -1;
    return (int64_t)t;
}

// Status of validate_call() for a call with no output entries (not exported).
constexpr int kNothingToDo = -1;

// Argument checks of a general-form call: SGEMM_OK, kNothingToDo (no output
// entries), or the status code the call returns. Null pointers and C
// overlapping A or B are checked only with `pointers` set: the plan takes
// operand addresses for their alignment alone.
static int validate_call(const Call &c, bool pointers)
{
    if (c.config < -1 || c.config >= kNumConfigs) return SGEMM_ERR_INVALID_VALUE;
    if ((c.op_a != 0 && c.op_a != 1) || (c.op_b != 0 && c.op_b != 1)) return SGEMM_ERR_INVALID_VALUE;
    if (c.M < 0 || c.N < 0 || c.K < 0 || c.batch < 0) return SGEMM_ERR_INVALID_VALUE;
    if (c.sa < 0 || c.sb < 0 || c.sc < 0) return SGEMM_ERR_INVALID_VALUE;
    if (c.batch == 0 || c.M == 0 || c.N == 0) return kNothingToDo;
    // Stored shapes: A is M x K (op 0) or K x M (op 1); B is K x N or N x K.
    const int64_t a_rows = c.op_a ? c.K : c.M, a_cols = c.op_a ? c.M : c.K;
    const int64_t b_rows = c.op_b ? c.N : c.K, b_cols = c.op_b ? c.K : c.N;
    const bool reads_ab = c.K > 0 && c.alpha != 0.0f;
    if (c.ldc < c.N || c.ldc < 1) return SGEMM_ERR_INVALID_VALUE;
    if (reads_ab && (c.lda < a_cols || c.ldb < b_cols || c.lda < 1 || c.ldb < 1)) return SGEMM_ERR_INVALID_VALUE;
    if (c.M > kMaxDim || c.N > kMaxDim || c.K > kMaxDim) return SGEMM_ERR_OVERFLOW;
    const int64_t c_one = extent(c.M, c.N, c.ldc);
    if (c_one < 0) return SGEMM_ERR_OVERFLOW;
    if (c.batch > 1 && c.sc < c_one) return SGEMM_ERR_INVALID_VALUE;   // C entries must not overlap
    const int64_t c_all = batch_extent(c_one, c.sc, c.batch);
    if (c_all < 0) return SGEMM_ERR_OVERFLOW;
    if (pointers && c.C == nullptr) return SGEMM_ERR_INVALID_VALUE;
    if (reads_ab) {
        if (pointers && (c.A == nullptr || c.B == nullptr)) return SGEMM_ERR_INVALID_VALUE;
        const int64_t a_one = extent(a_rows, a_cols, c.lda), b_one = extent(b_rows, b_cols, c.ldb);
        if (a_one < 0 || b_one < 0) return SGEMM_ERR_OVERFLOW;
        const int64_t a_all = batch_extent(a_one, c.sa, c.batch);
        const int64_t b_all = batch_extent(b_one, c.sb, c.batch);
        if (a_all < 0 || b_all < 0) return SGEMM_ERR_OVERFLOW;
        const uint64_t a = (uint64_t)(uintptr_t)c.A, b = (uint64_t)(uintptr_t)c.B, cp = (uint64_t)(uintptr_t)c.C;
        if (pointers && (overlaps(cp, c_all, a, a_all) || overlaps(cp, c_all, b, b_all)))
            return SGEMM_ERR_INVALID_VALUE;
    }
    return SGEMM_OK;
}

// The configuration of a validated call that reads A and B (K > 0, alpha
// != 0), automatic or forced, and whether A and B go through scratch first.
// Returns SGEMM_OK or SGEMM_ERR_UNSUPPORTED.
static int plan_call(const Call &c, int num_sms, int *out_cfg, bool *out_pa, bool *out_pb)
{
    const uint64_t a = (uint64_t)(uintptr_t)c.A, b = (uint64_t)(uintptr_t)c.B, cp = (uint64_t)(uintptr_t)c.C;
    const bool plain = c.op_a == 0 && c.op_b == 0 && c.alpha == 1.0f && c.beta == 0.0f && c.batch == 1;
    const ProblemShape p{c.M, c.N, c.K, c.lda, c.ldb, c.ldc, a, b, cp, num_sms};
    int cfg = c.config < 0 ? select_config(p) : c.config;
    // The automatic choice for small products is a plain-form-only kernel;
    // the general form takes the smallest TMA tiles instead.
    if (c.config < 0 && !plain && !kConfigTable[cfg].uses_tma) cfg = kCfgFfma2_128x64;
    // An A stored transposed (K x M) is what the k-major configurations read
    // in place, with no transposing pack: take them whenever their row-major
    // twins would run.
    if (c.config < 0 && c.op_a == 1 && cfg == kCfgFfma2_128x256) cfg = kCfgFfma2_128x256_ka;
    if (c.config < 0 && c.op_a == 1 && cfg == kCfgFfma2_128x128) cfg = kCfgFfma2_128x128_ka;
    if (!config_supports(cfg, p)) return SGEMM_ERR_UNSUPPORTED;
    // Kernels without TMA (the simple and ladder kernels) run the plain form only.
    if (!plain && !kConfigTable[cfg].uses_tma) return SGEMM_ERR_UNSUPPORTED;
    // TMA FFMA configurations read A (M x K) and B (K x N) in place when the
    // rows and batch strides are 16-byte multiples on a 16-byte-aligned base;
    // anything else (a transposed operand included) is packed into scratch,
    // rows padded to 32 floats. A shared operand (batch stride 0) is packed once.
    // A k-major configuration takes A stored K x M instead: in place when the
    // caller stores it so (op_a 1) on those terms, else transposed (a plain
    // A) or copied (a misaligned transposed one) into scratch.
    const bool packs = kConfigTable[cfg].packs;
    const bool akm = kConfigTable[cfg].a_kmajor;
    auto stride_ok = [&](int64_t s, int64_t one) { return c.batch <= 1 || s == 0 || (s % 4 == 0 && s >= one); };
    *out_pa = packs && (akm ? (c.op_a == 0 || needs_pack(a, c.lda) || !stride_ok(c.sa, c.K * c.lda))
                            : (c.op_a == 1 || needs_pack(a, c.lda) || !stride_ok(c.sa, c.M * c.lda)));
    *out_pb = packs && (c.op_b == 1 || needs_pack(b, c.ldb) || !stride_ok(c.sb, c.K * c.ldb));
    *out_cfg = cfg;
    return SGEMM_OK;
}

// The host-side plan of a call that computes a product (K > 0, alpha != 0):
// its configuration, the operands its layout pass packs, the scratch layout
// [packed A | packed B | the row-tail kernel's arrival counters | the
// product's stream-K workspace (its counters first) | the row-tail kernel's
// chunk sums], and how many of this library's kernels it launches. Both
// kinds of counter form one contiguous range, zeroed once before the
// product. `g` holds the caller's pointers; the packed ones and the
// workspace are set once the scratch exists.
struct CallPlan {
    int cfg = -1;
    bool pa = false, pb = false, akm = false;
    int64_t tail = 0, Mm = 0;
    int64_t a_rows = 0, a_cols = 0, a_rows_p = 0, lda_p = 0, ldb_p = 0, a_entries = 1, b_entries = 1;
    size_t a_bytes = 0, b_bytes = 0, ws_off = 0, ws_bytes = 0, tail_cnt_bytes = 0, tail_slot_bytes = 0;
    size_t sk_off = 0, slot_off = 0, total = 0, zero_bytes = 0;
    GemmArgs g{};
    int launches = 0;
};

static int plan_product(const Call &c, int num_sms, unsigned int *status, CallPlan &p)
{
    const int rc = plan_call(c, num_sms, &p.cfg, &p.pa, &p.pb);
    if (rc != SGEMM_OK) return rc;
    // The last `tail` rows (M just past a multiple of the block height) go
    // to the row-tail kernel; the tiled product covers the first Mm rows.
    p.tail = row_tail_rows(p.cfg, c.M, c.N, c.K, c.batch);
    p.Mm = c.M - p.tail;
    // Stored shape of the part of A the tiled product reads.
    p.a_rows = c.op_a ? c.K : p.Mm;
    p.a_cols = c.op_a ? p.Mm : c.K;

    GemmArgs &g = p.g;
    g = GemmArgs{p.Mm, c.N, c.K, c.A, c.lda, c.B, c.ldb, c.C, c.ldc, status, num_sms};
    g.sched = c.sched_override >= 0 ? c.sched_override : kConfigTable[p.cfg].sched;
    g.withhold_it = c.withhold_it;
    g.alpha = c.alpha;
    g.beta = c.beta;
    g.batch = c.batch;
    g.stride_a = c.batch > 1 ? c.sa : 0;
    g.stride_b = c.batch > 1 ? c.sb : 0;
    g.stride_c = c.batch > 1 ? c.sc : 0;
    g.op_a = c.op_a;
    g.op_b = c.op_b;

    p.akm = kConfigTable[p.cfg].a_kmajor;
    p.a_rows_p = p.akm ? c.K : p.Mm;                        // rows of the packed A
    p.lda_p = round_up(p.akm ? p.Mm : c.K, 32);
    p.ldb_p = round_up(c.N, 32);
    p.a_entries = (c.batch > 1 && c.sa != 0) ? c.batch : 1;
    p.b_entries = (c.batch > 1 && c.sb != 0) ? c.batch : 1;
    p.a_bytes = p.pa ? (size_t)(p.a_entries * p.a_rows_p * p.lda_p) * 4 : 0;
    p.b_bytes = p.pb ? (size_t)(p.b_entries * c.K * p.ldb_p) * 4 : 0;
    p.ws_off = (p.a_bytes + p.b_bytes + 255) / 256 * 256;
    if (p.pa) g.op_a = p.akm ? 1 : 0;
    if (p.pb) g.op_b = 0;
    p.ws_bytes = config_workspace_bytes(p.cfg, g);
    p.tail_cnt_bytes = p.tail > 0 ? row_tail_counter_bytes(p.tail, c.N, c.K, c.batch, num_sms) : 0;
    p.tail_slot_bytes = p.tail > 0 ? row_tail_slot_bytes(p.tail, c.N, c.K, c.batch, num_sms) : 0;
    p.sk_off = p.ws_off + p.tail_cnt_bytes;
    p.slot_off = p.sk_off + (p.ws_bytes + 255) / 256 * 256;
    p.total = (p.ws_bytes + p.tail_cnt_bytes + p.tail_slot_bytes) > 0 ? p.slot_off + p.tail_slot_bytes : p.ws_off;
    g.workspace_bytes = p.ws_bytes;
    // The counters to zero before the product: the tail kernel's, then the
    // stream-K ones at the start of the product's workspace.
    p.zero_bytes = p.tail_cnt_bytes + config_counter_bytes(p.cfg, g);
    if (!kConfigTable[p.cfg].uses_tma) {
        p.launches = 1;                                       // the simple and ladder kernels
    } else if (!kConfigTable[p.cfg].packs) {
        p.launches = 3 * (int)(c.batch > 1 ? c.batch : 1);   // 3xTF32: two splits and the product per entry
    } else {
        p.launches = 1 + ((p.pa || p.pb || p.zero_bytes > 0) ? 1 : 0) + (p.tail > 0 ? 1 : 0);
    }
    return SGEMM_OK;
}

static int sgemm_call(const Call &c, cudaStream_t stream)
{
    int rc = validate_call(c, true);
    if (rc == kNothingToDo) return SGEMM_OK;
    if (rc != SGEMM_OK) return rc;
    const bool reads_ab = c.K > 0 && c.alpha != 0.0f;

    DeviceState *dev = nullptr;
    rc = device_state(&dev);
    if (rc != SGEMM_OK) return rc;

    if (!reads_ab) {
        // The empty sum (K == 0) or alpha == 0: C = beta * C.
        if (c.beta == 1.0f) return SGEMM_OK;
        if (launch_scale(c.C, c.M, c.N, c.ldc, c.sc, c.batch, c.beta, stream) != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_LAUNCH;
        }
        return SGEMM_OK;
    }

    CallPlan p;
    rc = plan_product(c, dev->num_sms, dev->status, p);
    if (rc != SGEMM_OK) return rc;
    GemmArgs &g = p.g;
    uint8_t *scratch = nullptr;
    if (p.total > 0) {
        if (take_test_alloc_failure() ||
            cudaMallocFromPoolAsync((void **)&scratch, p.total, dev->pool, stream) != cudaSuccess) {
            cudaGetLastError();
            // An automatic k-major choice needs scratch for the whole
            // transposed A; when that cannot be had, the row-major twin
            // (which reads an aligned A as stored) runs the product instead.
            if (c.config < 0 && p.akm && c.op_a == 0) {
                Call twin = c;
                twin.config = p.cfg == kCfgFfma2_128x128_ka ? kCfgFfma2_128x128 : kCfgFfma2_128x256;
                return sgemm_call(twin, stream);
            }
            return SGEMM_ERR_ALLOC;
        }
        if (p.ws_bytes > 0) g.workspace = scratch + p.sk_off;
        unsigned int *const zero = reinterpret_cast<unsigned int *>(scratch + p.ws_off);
        if (p.pa || p.pb) {
            // Both layout passes in one launch, which also zeroes the
            // counters; the product is queued right behind it and (K a
            // multiple of the slab depth) may start while its last blocks run.
            PackJob ja{}, jb{};
            if (p.pa) {
                float *dst = reinterpret_cast<float *>(scratch);
                const bool transpose = p.akm ? c.op_a == 0 : c.op_a == 1;
                ja = pack_job(c.A, p.a_rows, p.a_cols, c.lda, c.sa, dst, p.lda_p, p.a_rows_p * p.lda_p,
                              p.a_entries, transpose);
                g.A = dst;
                g.lda = p.lda_p;
                g.stride_a = p.a_entries > 1 ? p.a_rows_p * p.lda_p : 0;
            }
            if (p.pb) {
                float *dst = reinterpret_cast<float *>(scratch + p.a_bytes);
                jb = c.op_b == 1
                         ? pack_job(c.B, c.N, c.K, c.ldb, c.sb, dst, p.ldb_p, c.K * p.ldb_p, p.b_entries, true)
                         : pack_job(c.B, c.K, c.N, c.ldb, c.sb, dst, p.ldb_p, c.K * p.ldb_p, p.b_entries, false);
                g.B = dst;
                g.ldb = p.ldb_p;
                g.stride_b = p.b_entries > 1 ? c.K * p.ldb_p : 0;
            }
            if (launch_pack_pair(ja, jb, p.zero_bytes > 0 ? zero : nullptr, p.zero_bytes, stream) != cudaSuccess) {
                cudaGetLastError();
                cudaFreeAsync(scratch, stream);
                return SGEMM_ERR_LAUNCH;
            }
            g.behind_pack = true;
            g.counters_zeroed = true;
        } else if (p.zero_bytes > 0) {
            // No operand to lay out: the same launch, one block, zeroes the
            // counters, and the product is queued behind it as above. This is
            // cheaper than a memset followed by an ordinary launch (same-box
            // A/B: 1024^3 48.6 against 50.2 us, 512 x 512 x 2048 36.6 against
            // 38.6 us, 1024 x 2048 x 2048 144.9 against 146.5 us).
            if (launch_pack_pair(PackJob{}, PackJob{}, zero, p.zero_bytes, stream) != cudaSuccess) {
                cudaGetLastError();
                cudaFreeAsync(scratch, stream);
                return SGEMM_ERR_LAUNCH;
            }
            g.behind_pack = true;
            g.counters_zeroed = true;
        }
    }

    cudaError_t err = launch_config(p.cfg, g, stream);
    if (err == cudaSuccess && p.tail > 0) {
        // The tail rows, from the caller's A and the B the product read.
        RowTailArgs t{};
        t.A = c.A;
        t.a_row_stride = c.op_a ? 1 : c.lda;
        t.a_k_stride = c.op_a ? c.lda : 1;
        t.stride_a = c.batch > 1 ? c.sa : 0;
        t.B = g.B;
        t.ldb = g.ldb;
        t.stride_b = g.stride_b;
        t.C = c.C;
        t.ldc = c.ldc;
        t.stride_c = c.batch > 1 ? c.sc : 0;
        t.m0 = p.Mm;
        t.r = (int)p.tail;
        t.N = c.N;
        t.K = c.K;
        t.batch = c.batch;
        t.alpha = c.alpha;
        t.beta = c.beta;
        t.counters = p.tail_cnt_bytes > 0 ? reinterpret_cast<unsigned int *>(scratch + p.ws_off) : nullptr;
        t.slots = p.tail_slot_bytes > 0 ? reinterpret_cast<float *>(scratch + p.slot_off) : nullptr;
        err = launch_row_tail(t, dev->num_sms, stream);
    }
    if (scratch) cudaFreeAsync(scratch, stream);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
}

static int sgemm_impl(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B, int64_t ldb,
                      float *C, int64_t ldc, int config, int sched_override, int withhold_it, cudaStream_t stream)
{
    const Call c{0, 0, M, N, K, 1.0f, A, lda, 0, B, ldb, 0, 0.0f, C, ldc, 0, 1,
                 config, sched_override, withhold_it};
    return sgemm_call(c, stream);
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
    // The 128x256 TMA kernel (whatever the size) on whole tiles: no stream-K
    // waits between CTAs, only the withheld copy.
    return sgemm_impl(M, N, K, A, lda, B, ldb, C, ldc, kCfgFfma2_128x256, kSchedDataParallel,
                      slab < 0 ? -1 : slab, stream);
}

int sgemm_test_fail_next_allocs(int n)
{
    if (n < 0) return SGEMM_ERR_INVALID_VALUE;
    g_fail_allocs.store(n);
    return SGEMM_OK;
}

int sgemm_test_schedule(int64_t M, int64_t N, int64_t K, int bm, int bn, int bk, int64_t slots, int policy,
                        int64_t batch, int64_t *items, int64_t capacity, int64_t *count, int64_t *info)
{
    if (M <= 0 || N <= 0 || K <= 0 || bm <= 0 || bn <= 0 || bk <= 0 || slots <= 0 || batch <= 0 ||
        policy < kSchedAuto || policy > kSchedTailSplit || capacity < 0 || !count || !info)
        return SGEMM_ERR_INVALID_VALUE;
    const Schedule s = plan_schedule(M, N, K, bm, bn, bk, slots, policy, true, batch);
    info[0] = s.grid;
    info[1] = s.tiles;
    info[2] = s.dp_tiles;
    info[3] = s.sk_ctas;
    info[4] = s.nk;
    info[5] = s.tiles_m;
    info[6] = s.tiles_n;
    int64_t n = 0;
    for (int g = 0; g < s.grid; ++g) {
        Cursor cur = cursor_init(s, g);
        Item it;
        while (next_item(s, cur, it)) {
            if (n < capacity) {
                int b, tm, tn;
                tile_coords_b(s, it.tile, b, tm, tn);
                const bool split = it.kb0 > 0 || it.kb1 < s.nk;
                int64_t *r = items + 10 * n;
                r[0] = g;
                r[1] = it.tile;
                r[2] = it.kb0;
                r[3] = it.kb1;
                r[4] = b;
                r[5] = tm;
                r[6] = tn;
                r[7] = split ? sk_first_cta(s, it.tile) : -1;
                r[8] = split ? sk_last_cta(s, it.tile) : -1;
                r[9] = split ? sk_slot(g, it.kb0) : -1;
            }
            ++n;
        }
    }
    *count = n;
    return n <= capacity ? SGEMM_OK : SGEMM_ERR_INVALID_VALUE;
}

int sgemm_general_ex(int op_a, int op_b, int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                     int64_t lda, int64_t stride_a, const float *B, int64_t ldb, int64_t stride_b, float beta,
                     float *C, int64_t ldc, int64_t stride_c, int64_t batch, int config, cudaStream_t stream)
{
    const Call c{op_a, op_b, M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b, beta, C, ldc, stride_c, batch,
                 config, -1, -1};
    return sgemm_call(c, stream);
}

int sgemm_general(int op_a, int op_b, int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                  int64_t stride_a, const float *B, int64_t ldb, int64_t stride_b, float beta, float *C,
                  int64_t ldc, int64_t stride_c, int64_t batch, cudaStream_t stream)
{
    return sgemm_general_ex(op_a, op_b, M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b, beta, C, ldc,
                            stride_c, batch, -1, stream);
}

int sgemm_general_plan(int op_a, int op_b, int64_t M, int64_t N, int64_t K, float alpha, int64_t lda,
                       int64_t stride_a, int64_t ldb, int64_t stride_b, float beta, int64_t ldc, int64_t stride_c,
                       int64_t batch, uint64_t a_addr, uint64_t b_addr, uint64_t c_addr, int num_sms, int config,
                       int *out_config, int *out_pack_a, int *out_pack_b)
{
    if (out_config) *out_config = -1;
    if (out_pack_a) *out_pack_a = 0;
    if (out_pack_b) *out_pack_b = 0;
    if (num_sms <= 0) return SGEMM_ERR_INVALID_VALUE;
    const Call c{op_a, op_b, M, N, K, alpha,
                 reinterpret_cast<const float *>((uintptr_t)a_addr), lda, stride_a,
                 reinterpret_cast<const float *>((uintptr_t)b_addr), ldb, stride_b, beta,
                 reinterpret_cast<float *>((uintptr_t)c_addr), ldc, stride_c, batch, config, -1, -1};
    int rc = validate_call(c, false);
    if (rc == kNothingToDo) return SGEMM_OK;
    if (rc != SGEMM_OK) return rc;
    if (K == 0 || alpha == 0.0f) return SGEMM_OK;   // no product: C = beta * C only
    int cfg = -1;
    bool pa = false, pb = false;
    rc = plan_call(c, num_sms, &cfg, &pa, &pb);
    if (rc != SGEMM_OK) return rc;
    if (out_config) *out_config = cfg;
    if (out_pack_a) *out_pack_a = pa ? 1 : 0;
    if (out_pack_b) *out_pack_b = pb ? 1 : 0;
    return SGEMM_OK;
}

int sgemm_general_plan_launches(int op_a, int op_b, int64_t M, int64_t N, int64_t K, float alpha, int64_t lda,
                                int64_t stride_a, int64_t ldb, int64_t stride_b, float beta, int64_t ldc,
                                int64_t stride_c, int64_t batch, uint64_t a_addr, uint64_t b_addr, uint64_t c_addr,
                                int num_sms, int config, int *out_launches)
{
    if (!out_launches) return SGEMM_ERR_INVALID_VALUE;
    *out_launches = 0;
    if (num_sms <= 0) return SGEMM_ERR_INVALID_VALUE;
    const Call c{op_a, op_b, M, N, K, alpha,
                 reinterpret_cast<const float *>((uintptr_t)a_addr), lda, stride_a,
                 reinterpret_cast<const float *>((uintptr_t)b_addr), ldb, stride_b, beta,
                 reinterpret_cast<float *>((uintptr_t)c_addr), ldc, stride_c, batch, config, -1, -1};
    int rc = validate_call(c, false);
    if (rc == kNothingToDo) return SGEMM_OK;
    if (rc != SGEMM_OK) return rc;
    if (K == 0 || alpha == 0.0f) {                      // C = beta * C only
        *out_launches = beta == 1.0f ? 0 : 1;
        return SGEMM_OK;
    }
    CallPlan p;
    rc = plan_product(c, num_sms, nullptr, p);
    if (rc != SGEMM_OK) return rc;
    *out_launches = p.launches;
    return SGEMM_OK;
}

int sgemm_plan_row_tail(int config, int64_t M, int64_t N, int64_t K, int64_t batch, int64_t *out_rows)
{
    if (!out_rows) return SGEMM_ERR_INVALID_VALUE;
    *out_rows = 0;
    if (config < 0 || config >= kNumConfigs || M < 0 || N < 0 || K < 0 || batch < 0) return SGEMM_ERR_INVALID_VALUE;
    *out_rows = row_tail_rows(config, M, N, K, batch);
    return SGEMM_OK;
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
        if (word & kStatusLaunchConfig) return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
}

}  // extern "C"
