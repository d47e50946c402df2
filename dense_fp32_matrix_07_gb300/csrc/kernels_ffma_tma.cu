// The main SGEMM kernel: CUDA-core FP32 multiply-adds with block, warp and
// thread register tiling, fed by TMA through a multi-stage shared-memory ring.
//
// Lineage on the pages, and what changes on sm_103a:
//  * The CUDA Handbook, ch.17, section 17.3 (Cache Blocking) and Figure 17-2:
//    a thread block owns a BM x BN tile of C and marches K in BK-deep slabs;
//    each thread keeps a TM x TN micro-tile of accumulators in registers
//    (8 x 8 was the best there), so one loaded strip of A and of B feeds 64
//    multiply-adds.
//  * Chapter 9: Optimised Matrix Multiplication, sections 9.4-9.6: slabs are
//    staged in shared memory once per block and reused, bank conflicts are
//    designed out, and registers per thread are traded against occupancy by
//    launch bounds. "Перемножение матриц: наивное и тайловое", section 2:
//    a slab may be read only after it is fully loaded, and overwritten only
//    after every thread is done with it.
// Here the copy engine (TMA) fills a ring of STAGES slabs; one producer warp
// issues the copies and each slab has a "full" mbarrier (read-after-write:
// the copy's bytes have landed) and an "empty" mbarrier (write-after-read:
// every consumer warp has finished with it), which replace the pages' two
// __syncthreads() per phase. The A slab uses the TMA 128-byte (BK 32) or
// 64-byte (BK 16) swizzle instead of the pages' +1 padding column, which
// TMA cannot produce. The grid is persistent (one CTA per SM) and walks the
// output tiles in groups of 8 block rows so concurrently running CTAs share
// A and B panels in L2. Zero fill of out-of-range boxes by TMA handles the
// M, N and K tails; the epilogue predicates its stores.
//
// Every mbarrier wait is bounded in time (about a second): on giving up, the
// thread sets the device error word (read by sgemm_check_status()) and
// returns; the producer first waits (bounded as well) for every copy it has
// issued, so no copy can land in the shared memory of an exited CTA.
#include "common.cuh"
#include "configs.cuh"
#include "ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <atomic>

namespace sgemm_gb300 {

namespace {

// Wall-clock limit of one bounded wait, in nanoseconds.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for phase `parity` of the mbarrier at `bar`; false after kWaitLimitNs.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 0; n < kSpinLimit; ++n) {
#pragma unroll 1
        for (int r = 0; r < 16; ++r)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
    return false;
}

template <int BM_, int BN_, int BK_, int STAGES_, bool PAIRED_, int MIN_BLOCKS_>
struct FfmaTmaCfg {
    static constexpr int BM = BM_, BN = BN_, BK = BK_, STAGES = STAGES_;
    static constexpr bool PAIRED = PAIRED_;   // FFMA2 (two FP32 FMAs per instruction)
    static constexpr int MIN_BLOCKS = MIN_BLOCKS_;
    // Warp tile 64 x 32 as 8 x 4 threads, thread tile 8 x 8.
    static constexpr int WM = 64, WN = 32, TM = 8, TN = 8;
    static constexpr int TROWS = WM / TM, TCOLS = WN / TN;
    static constexpr int WARPS_M = BM / WM, WARPS_N = BN / WN;
    static constexpr int CONSUMERS = WARPS_M * WARPS_N;
    static constexpr int THREADS = (CONSUMERS + 1) * 32;
    static constexpr int A_ROW_BYTES = BK * 4;
    static constexpr int A_BYTES = BM * BK * 4;
    static constexpr int B_ROW_BYTES = BN * 4;
    static constexpr int B_BYTES = BK * BN * 4;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 2 * STAGES * 8;
    // Row r of the A slab has its 16-byte chunk c stored at chunk c ^ swz(r),
    // swz(r) = r & 7 for 128-byte rows, (r >> 1) & 3 for 64-byte rows.
    static constexpr CUtensorMapSwizzle A_SWIZZLE =
        BK == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    static_assert(TROWS == 8 && TCOLS == 4, "thread layout is 8 x 4 per warp");
    static_assert(BM % WM == 0 && BN % WN == 0, "block tile must hold whole warp tiles");
    static_assert(BK == 32 || BK == 16, "BK is 16 or 32");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "stage buffers stay 1024-aligned");
    static_assert(BN <= 256 && BM <= 256, "TMA box dimensions are at most 256");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// Output tile of linear index t: groups of 8 block rows, column-major inside
// a group, so the CTAs running at the same time touch few A and B panels.
__device__ __forceinline__ void tile_coords(int64_t t, int tiles_m, int tiles_n, int &tm, int &tn)
{
    constexpr int G = 8;
    const int64_t per_group = (int64_t)G * tiles_n;
    const int64_t group = t / per_group;
    const int first_m = (int)(group * G);
    const int rows = min(tiles_m - first_m, G);
    const int64_t local = t - group * per_group;
    tm = first_m + (int)(local % rows);
    tn = (int)(local / rows);
}

template <class Cfg, bool VEC_C>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MIN_BLOCKS)
sgemm_ffma_tma_kernel(const __grid_constant__ CUtensorMap mapA,
                      const __grid_constant__ CUtensorMap mapB,
                      float *__restrict__ C, int64_t ldc, int M, int N, int K,
                      unsigned int *status)
{
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const base_ptr = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + STAGES * Cfg::A_BYTES;
    const uint32_t bars = sB + STAGES * Cfg::B_BYTES;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
    const int64_t tiles = (int64_t)tiles_m * tiles_n;
    const int nk = (K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), Cfg::CONSUMERS);
        }
        ptx::mbar_init_fence();
    }
    __syncthreads();

    if (warp == Cfg::CONSUMERS) {
        // ------------------------------ producer ------------------------------
        if (lane != 0) return;
        ptx::prefetch_tensormap(&mapA);
        ptx::prefetch_tensormap(&mapB);
        const uint64_t policy = ptx::policy_evict_last();
        int last_round[STAGES];
#pragma unroll
        for (int s = 0; s < STAGES; ++s) last_round[s] = -1;
        uint32_t it = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
            int tm, tn;
            tile_coords(t, tiles_m, tiles_n, tm, tn);
            for (int kb = 0; kb < nk; ++kb, ++it) {
                const int s = (int)(it % STAGES);
                const int round = (int)(it / STAGES);
                if (!wait_phase(empty_bar(s), (round & 1) ^ 1)) {
                    atomicOr(status, kStatusTimeout);
                    ok = false;
                    break;
                }
                ptx::mbar_arrive_expect_tx(full_bar(s), Cfg::STAGE_BYTES);
                ptx::tma_load_2d(sA + s * Cfg::A_BYTES, &mapA, full_bar(s), kb * BK, tm * BM, policy);
                ptx::tma_load_2d(sB + s * Cfg::B_BYTES, &mapB, full_bar(s), tn * BN, kb * BK, policy);
                last_round[s] = round;
            }
        }
        // Every issued copy must land before this CTA's shared memory goes away.
        for (int s = 0; s < STAGES; ++s) {
            if (last_round[s] >= 0 && !wait_phase(full_bar(s), last_round[s] & 1)) {
                atomicOr(status, kStatusTimeout);
            }
        }
        return;
    }

    // ------------------------------ consumers ------------------------------
    const int wm = (warp / Cfg::WARPS_N) * Cfg::WM;
    const int wn = (warp % Cfg::WARPS_N) * Cfg::WN;
    const int ty = lane / Cfg::TCOLS;   // 0..7: thread row (rows wm + ty + 8i)
    const int tx = lane % Cfg::TCOLS;   // 0..3: thread column (cols wn + 4tx + 16g + e)
    const uint32_t a_row_off = (uint32_t)(wm + ty) * Cfg::A_ROW_BYTES;
    const uint32_t a_xor = (BK == 32) ? (uint32_t)(ty & 7) : (uint32_t)((ty >> 1) & 3);
    const uint32_t b_col_off = (uint32_t)(wn + tx * 4) * 4;

    uint32_t it = 0;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        int tm, tn;
        tile_coords(t, tiles_m, tiles_n, tm, tn);

        float acc[8][8];
        float2 accp[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
#pragma unroll
            for (int q = 0; q < 4; ++q) accp[i][q] = make_float2(0.0f, 0.0f);
        }

        for (int kb = 0; kb < nk; ++kb, ++it) {
            const int s = (int)(it % STAGES);
            if (!wait_phase(full_bar(s), (it / STAGES) & 1)) {
                atomicOr(status, kStatusTimeout);
                return;
            }
            const uint8_t *As = base_ptr + s * Cfg::A_BYTES + a_row_off;
            const uint8_t *Bs = base_ptr + STAGES * Cfg::A_BYTES + s * Cfg::B_BYTES + b_col_off;
#pragma unroll
            for (int kg = 0; kg < BK / 4; ++kg) {
                // A fragment: rows wm+ty+8i, columns 4kg..4kg+3 of the slab.
                float4 a[8];
                const uint32_t chunk = ((uint32_t)kg ^ a_xor) << 4;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    a[i] = *reinterpret_cast<const float4 *>(As + i * 8 * Cfg::A_ROW_BYTES + chunk);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const int k = kg * 4 + kk;
                    const float4 b0 = *reinterpret_cast<const float4 *>(Bs + k * Cfg::B_ROW_BYTES);
                    const float4 b1 = *reinterpret_cast<const float4 *>(Bs + k * Cfg::B_ROW_BYTES + 64);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
                        if constexpr (Cfg::PAIRED) {
                            const float2 aa = make_float2(av, av);
                            accp[i][0] = __ffma2_rn(aa, make_float2(b0.x, b0.y), accp[i][0]);
                            accp[i][1] = __ffma2_rn(aa, make_float2(b0.z, b0.w), accp[i][1]);
                            accp[i][2] = __ffma2_rn(aa, make_float2(b1.x, b1.y), accp[i][2]);
                            accp[i][3] = __ffma2_rn(aa, make_float2(b1.z, b1.w), accp[i][3]);
                        } else {
                            acc[i][0] = fmaf(av, b0.x, acc[i][0]);
                            acc[i][1] = fmaf(av, b0.y, acc[i][1]);
                            acc[i][2] = fmaf(av, b0.z, acc[i][2]);
                            acc[i][3] = fmaf(av, b0.w, acc[i][3]);
                            acc[i][4] = fmaf(av, b1.x, acc[i][4]);
                            acc[i][5] = fmaf(av, b1.y, acc[i][5]);
                            acc[i][6] = fmaf(av, b1.z, acc[i][6]);
                            acc[i][7] = fmaf(av, b1.w, acc[i][7]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty_bar(s));
        }

        // Epilogue: rows wm+ty+8i, two runs of 4 columns per row.
        if constexpr (Cfg::PAIRED) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                acc[i][0] = accp[i][0].x; acc[i][1] = accp[i][0].y;
                acc[i][2] = accp[i][1].x; acc[i][3] = accp[i][1].y;
                acc[i][4] = accp[i][2].x; acc[i][5] = accp[i][2].y;
                acc[i][6] = accp[i][3].x; acc[i][7] = accp[i][3].y;
            }
        }
        const int64_t row0 = (int64_t)tm * BM + wm + ty;
        const int col0 = tn * BN + wn + tx * 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t row = row0 + 8 * i;
            if (row >= M) break;
            float *crow = C + row * ldc;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const int col = col0 + 16 * g;
                if (VEC_C && col + 3 < N) {
                    *reinterpret_cast<float4 *>(crow + col) =
                        make_float4(acc[i][4 * g], acc[i][4 * g + 1], acc[i][4 * g + 2], acc[i][4 * g + 3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (col + e < N) crow[col + e] = acc[i][4 * g + e];
                }
            }
        }
    }
}

using CfgFfma128x128k32s4 = FfmaTmaCfg<128, 128, 32, 4, false, 1>;
using CfgFfma2_128x128k32s4 = FfmaTmaCfg<128, 128, 32, 4, true, 1>;
using CfgFfma2_128x128k16s8 = FfmaTmaCfg<128, 128, 16, 8, true, 1>;
using CfgFfma2_128x64k32s4 = FfmaTmaCfg<128, 64, 32, 4, true, 2>;

std::atomic<PFN_cuTensorMapEncodeTiled_v12000> g_encode{nullptr};

cudaError_t get_encoder(PFN_cuTensorMapEncodeTiled_v12000 *out)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = g_encode.load();
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                               cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !p) return cudaErrorNotSupported;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        g_encode.store(fn);
    }
    *out = fn;
    return cudaSuccess;
}

// Row-major rows x cols FP32 matrix with leading dimension ld (elements),
// read in boxes of box_rows x box_cols.
cudaError_t encode_2d(CUtensorMap *map, const float *ptr, int64_t rows, int64_t cols, int64_t ld,
                      int box_rows, int box_cols, CUtensorMapSwizzle swizzle)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    const cudaError_t e = get_encoder(&encode);
    if (e != cudaSuccess) return e;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(ptr), dims,
                              strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <class Cfg>
cudaError_t set_smem_limit()
{
    cudaError_t e = cudaFuncSetAttribute(sgemm_ffma_tma_kernel<Cfg, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(sgemm_ffma_tma_kernel<Cfg, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
}

template <class Cfg>
cudaError_t launch(const GemmArgs &g, cudaStream_t stream)
{
    CUtensorMap mapA, mapB;
    cudaError_t e = encode_2d(&mapA, g.A, g.M, g.K, g.lda, Cfg::BM, Cfg::BK, Cfg::A_SWIZZLE);
    if (e != cudaSuccess) return e;
    e = encode_2d(&mapB, g.B, g.K, g.N, g.ldb, Cfg::BK, Cfg::BN, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    const int64_t tiles = ((g.M + Cfg::BM - 1) / Cfg::BM) * ((g.N + Cfg::BN - 1) / Cfg::BN);
    const int64_t slots = (int64_t)g.num_sms * Cfg::MIN_BLOCKS;
    const unsigned grid = (unsigned)(tiles < slots ? tiles : slots);
    const bool vec = ((reinterpret_cast<uintptr_t>(g.C) & 15u) == 0) && (g.ldc % 4 == 0);
    if (vec)
        sgemm_ffma_tma_kernel<Cfg, true><<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(
            mapA, mapB, g.C, g.ldc, (int)g.M, (int)g.N, (int)g.K, g.status);
    else
        sgemm_ffma_tma_kernel<Cfg, false><<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(
            mapA, mapB, g.C, g.ldc, (int)g.M, (int)g.N, (int)g.K, g.status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t prepare_ffma_tma()
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    cudaError_t e = get_encoder(&encode);
    if (e != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma128x128k32s4>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x128k32s4>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x128k16s8>()) != cudaSuccess) return e;
    return set_smem_limit<CfgFfma2_128x64k32s4>();
}

cudaError_t launch_ffma_tma(int cfg, const GemmArgs &g, cudaStream_t stream)
{
    switch (cfg) {
    case kCfgFfma128x128k32s4: return launch<CfgFfma128x128k32s4>(g, stream);
    case kCfgFfma2_128x128k32s4: return launch<CfgFfma2_128x128k32s4>(g, stream);
    case kCfgFfma2_128x128k16s8: return launch<CfgFfma2_128x128k16s8>(g, stream);
    case kCfgFfma2_128x64k32s4: return launch<CfgFfma2_128x64k32s4>(g, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace sgemm_gb300
