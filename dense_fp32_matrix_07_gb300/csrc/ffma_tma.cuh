// The main SGEMM kernel: CUDA-core FP32 multiply-adds with block, warp and
// thread register tiling, fed by TMA through a multi-stage shared-memory ring.
// This header holds the kernel template, its configurations and launcher;
// kernels_ffma_tma.cu instantiates the kernels for K a multiple of BK and
// kernels_ffma_tma_ktail.cu those that trim the last K slab, so the two
// halves compile in parallel.
//
// Lineage on the pages, and what changes on sm_103a:
//  * The CUDA Handbook, ch.17, section 17.3 (Cache Blocking) and Figure 17-2:
//    a thread block owns a BM x BN tile of C and marches K in BK-deep slabs;
//    each thread keeps a TM x TN micro-tile of accumulators in registers
//    (8 x 8 was the best there), so one loaded strip of A and of B feeds
//    TM*TN multiply-adds.
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
// TMA cannot produce. The k-major configurations read A stored K x M
// instead (a transposed copy, or the caller's transposed A): their slab is
// [BK][BM], M contiguous, unswizzled, and one LDS.128 gives a thread 4 of
// its rows at one k, in consecutive registers, which the FFMA2 loop issues
// faster than values 4 registers apart. Zero fill of out-of-range boxes by
// TMA handles the M, N and K tails; the epilogue predicates its stores.
//
// Work schedule (persistent grid, at most one CTA per SM and resident slot):
// output tiles are numbered in groups of 8 block rows (so CTAs running at the
// same time share A and B panels in L2). Tiles [0, dp_tiles) are whole-tile
// work, dealt round-robin. The remaining tiles form a stream-K region: their
// K-slab iterations, taken tile after tile, are cut into sk_ctas contiguous,
// equal ranges, one per CTA, which evens out the last waves. A tile whose
// slabs fall in several ranges is finished by the part that arrives last:
// every other part writes its partial sum to a slot of its own and bumps the
// tile's arrival counter (one per consumer warp, each warp handling its own
// fragment, so no CTA-wide barrier is involved); the part that completes the
// count adds all parts in CTA order (a fixed, deterministic order) and
// stores the tile. The CTA holding the tile's first slab usually arrives
// last; it looks at the counter first and, when every other part is in,
// adds them straight to its registers. No CTA waits for another.
//
// Every mbarrier wait is bounded in time (about a
// second): on giving up, the thread sets the device error word (read by
// sgemm_check_status()) and gives up its work; the producer first waits
// (bounded as well) for every copy it has issued, so no copy can land in the
// shared memory of an exited CTA.
#pragma once

#include "common.cuh"
#include "configs.cuh"
#include "ptx.cuh"
#include "schedule.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <atomic>

namespace sgemm_gb300 {

namespace {

template <int BM_, int BN_, int BK_, int STAGES_, int TN_, bool PAIRED_, int MIN_BLOCKS_, bool A_KMAJOR_ = false>
struct FfmaTmaCfg {
    static constexpr int BM = BM_, BN = BN_, BK = BK_, STAGES = STAGES_;
    static constexpr bool PAIRED = PAIRED_;   // FFMA2 (two FP32 FMAs per instruction)
    static constexpr int MIN_BLOCKS = MIN_BLOCKS_;
    // A stored K x M (k-major: the slab is [BK][BM], M contiguous) instead of
    // M x K. One LDS.128 then gives a thread 4 of its rows at one k in
    // consecutive registers.
    static constexpr bool A_KMAJOR = A_KMAJOR_;
    // Thread tile TM x TN; warp = 8 x 4 threads, so warp tile 64 x 4*TN.
    static constexpr int TM = 8, TN = TN_, G = TN / 4;
    static constexpr int TROWS = 8, TCOLS = 4;
    static constexpr int WM = TROWS * TM, WN = TCOLS * TN;
    static constexpr int WARPS_M = BM / WM, WARPS_N = BN / WN;
    static constexpr int CONSUMERS = WARPS_M * WARPS_N;
    static constexpr int CONSUMER_THREADS = CONSUMERS * 32;
    // Producer: one warp, or (wide thread tiles) a whole warpgroup that hands
    // registers to the consumer warpgroups with setmaxnreg: each SM
    // sub-partition's register file then holds 1 producer warp at
    // PRODUCER_REGS and 2 consumer warps at CONSUMER_REGS.
    static constexpr bool REG_SPLIT = TN > 8;
    // Stream-K fix-up shortcut for the part holding a split tile's first
    // slab (see the fix-up in the kernel): 8 x 8 thread tiles only.
    static constexpr bool OWNER_PEEK = !REG_SPLIT;
    static constexpr int PRODUCER_WARPS = REG_SPLIT ? 4 : 1;
    static constexpr int THREADS = CONSUMER_THREADS + 32 * PRODUCER_WARPS;
    static constexpr int LAUNCH_REGS = (65536 / THREADS) / 8 * 8;
    static constexpr int PRODUCER_REGS = 40;
    static constexpr int CONSUMER_REGS =
        ((LAUNCH_REGS * THREADS - PRODUCER_REGS * 32 * PRODUCER_WARPS) / CONSUMER_THREADS) / 8 * 8;
    static constexpr int A_ROW_BYTES = A_KMAJOR ? BM * 4 : BK * 4;   // one row of the smem slab
    static constexpr int A_BYTES = BM * BK * 4;
    static constexpr int B_ROW_BYTES = BN * 4;
    static constexpr int B_BYTES = BK * BN * 4;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 2 * STAGES * 8;
    // Row r of the A slab has its 16-byte chunk c stored at chunk c ^ swz(r),
    // swz(r) = r & 7 for 128-byte rows, (r >> 1) & 3 for 64-byte rows.
    // A k-major slab is read along its rows without conflicts and needs none.
    static constexpr CUtensorMapSwizzle A_SWIZZLE =
        A_KMAJOR ? CU_TENSOR_MAP_SWIZZLE_NONE
                 : (BK == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
    static_assert(TN % 4 == 0 && TN >= 8 && TN <= 16, "thread tile columns: 8, 12 or 16");
    static_assert(BM % WM == 0 && BN % WN == 0, "block tile must hold whole warp tiles");
    static_assert(BK == 32 || BK == 16, "BK is 16 or 32");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "stage buffers stay 1024-aligned");
    static_assert(BN <= 256 && BM <= 256, "TMA box dimensions are at most 256");
    static_assert(!A_KMAJOR || (PAIRED && WM == 64), "k-major A: FFMA2 and 64-row warp tiles");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
    static_assert(BM * BN == CONSUMER_THREADS * TM * TN, "one partial sum per accumulator");
    static_assert(!REG_SPLIT || (CONSUMERS % 4 == 0 && CONSUMER_REGS <= 255), "whole consumer warpgroups");
    // The split may not ask for more registers than the CTA was launched with.
    static_assert(!REG_SPLIT || PRODUCER_REGS * 32 * PRODUCER_WARPS + CONSUMER_REGS * CONSUMER_THREADS <=
                                    LAUNCH_REGS * THREADS,
                  "register split exceeds the launch allocation");
};

// Output side of a launch: C_b = alpha * acc + beta * C_b (C read only when
// beta != 0) for batch entry b at C + b * stride_c; a_bz / b_bz are 1 when A
// / B advance with the batch entry (their tensor maps' third coordinate)
// and 0 when one operand is shared by every entry.
struct Epilogue {
    float *C;
    int64_t ldc, stride_c;
    int M, N;
    float alpha, beta;
    int a_bz, b_bz;
};

// DEP: the instance launched behind the call's layout pass with
// programmatic serialization (kernels_ffma_tma_dep.cu).
template <class Cfg, bool VEC_C, bool K_TAIL, bool DEP = false>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MIN_BLOCKS)
sgemm_ffma_tma_kernel(const __grid_constant__ CUtensorMap mapA,
                      const __grid_constant__ CUtensorMap mapB,
                      const Epilogue ep, const Schedule sched, unsigned int *status, int withhold_it)
{
    const int M = ep.M, N = ep.N;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr int TN = Cfg::TN, G = Cfg::G;
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
    const int g = blockIdx.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), Cfg::CONSUMERS);
        }
        ptx::mbar_init_fence();
        // A kernel queued behind this one with programmatic serialization
        // (the last-rows kernel, which reads nothing this grid writes) may
        // take SMs as soon as this persistent grid's CTAs leave them.
        if constexpr (!DEP) ptx::grid_launch_dependents();
    }
    __syncthreads();
    if constexpr (DEP) {
        // Queued behind the call's layout pass with programmatic
        // serialization, this grid may start while that pass still runs: no
        // thread touches global memory before the pass has completed. Only
        // the DEP instances carry the wait: in the others, where it would be
        // a no-op, it still cost time (same-box A/B, 4096 x 3001 x 2048 with A
        // stored transposed, no layout pass: 744.4 against 742.9 us). The
        // last-rows kernel behind this grid reads the pass's copy of B, so it
        // is let in only once the pass is complete.
        ptx::grid_dependency_wait();
        if (threadIdx.x == 0) ptx::grid_launch_dependents();
    }

    if (warp >= Cfg::CONSUMERS) {
        // ------------------------------ producer ------------------------------
        if constexpr (Cfg::REG_SPLIT) ptx::setmaxnreg_dec<Cfg::PRODUCER_REGS>();
        if (warp != Cfg::CONSUMERS || lane != 0) return;
        ptx::prefetch_tensormap(&mapA);
        ptx::prefetch_tensormap(&mapB);
        const uint64_t policy = ptx::policy_evict_last();
        int last_round[STAGES];
#pragma unroll
        for (int s = 0; s < STAGES; ++s) last_round[s] = -1;
        uint32_t it = 0;
        bool ok = true;
        Cursor cur = cursor_init(sched, g);
        Item item;
        while (ok && next_item(sched, cur, item)) {
            int bt, tm, tn;
            tile_coords_b(sched, item.tile, bt, tm, tn);
            for (int kb = item.kb0; kb < item.kb1; ++kb, ++it) {
                const int s = (int)(it % STAGES);
                const int round = (int)(it / STAGES);
                if (!ptx::wait_phase(empty_bar(s), (round & 1) ^ 1)) {
                    atomicOr(status, kStatusTimeout);
                    ok = false;
                    break;
                }
                // Test hook (sgemm_test_withhold_copy): this copy is never
                // issued, so the consumers' wait for it must time out.
                if (g == 0 && (int)it == withhold_it) continue;
                ptx::mbar_arrive_expect_tx(full_bar(s), Cfg::STAGE_BYTES);
                if constexpr (Cfg::A_KMAJOR)
                    ptx::tma_load_3d(sA + s * Cfg::A_BYTES, &mapA, full_bar(s), tm * BM, kb * BK,
                                     bt * ep.a_bz, policy);
                else
                    ptx::tma_load_3d(sA + s * Cfg::A_BYTES, &mapA, full_bar(s), kb * BK, tm * BM,
                                     bt * ep.a_bz, policy);
                ptx::tma_load_3d(sB + s * Cfg::B_BYTES, &mapB, full_bar(s), tn * BN, kb * BK, bt * ep.b_bz,
                                 policy);
                last_round[s] = round;
            }
        }
        // Every issued copy must land before this CTA's shared memory goes away.
        for (int s = 0; s < STAGES; ++s) {
            if (last_round[s] >= 0 && !ptx::wait_phase(full_bar(s), last_round[s] & 1)) {
                atomicOr(status, kStatusTimeout);
            }
        }
        return;
    }

    // ------------------------------ consumers ------------------------------
    if constexpr (Cfg::REG_SPLIT) ptx::setmaxnreg_inc<Cfg::CONSUMER_REGS>();
    const int wm = (warp / Cfg::WARPS_N) * Cfg::WM;
    const int wn = (warp % Cfg::WARPS_N) * Cfg::WN;
    const int ty = lane / Cfg::TCOLS;   // 0..7: thread row (rows wm + ty + 8i)
    const int tx = lane % Cfg::TCOLS;   // 0..3: thread column (cols wn + 4tx + 16q + e)
    // Row-major A slab: this thread's rows wm+ty+8i start at row wm+ty;
    // k-major slab: its rows are wm+4ty+i and wm+32+4ty+i (i < 4), at byte
    // (wm+4ty)*4 (and 128 bytes on) of every k row.
    const uint32_t a_row_off =
        Cfg::A_KMAJOR ? (uint32_t)(wm + 4 * ty) * 4 : (uint32_t)(wm + ty) * Cfg::A_ROW_BYTES;
    const uint32_t a_xor = (BK == 32) ? (uint32_t)(ty & 7) : (uint32_t)((ty >> 1) & 3);
    const uint32_t b_col_off = (uint32_t)(wn + tx * 4) * 4;
    const int ct = warp * 32 + lane;    // consumer thread index (partial-sum layout)

    uint32_t it = 0;
    Cursor cur = cursor_init(sched, g);
    Item item;
    while (next_item(sched, cur, item)) {
        int bt, tm, tn;
        tile_coords_b(sched, item.tile, bt, tm, tn);

        // acc[i][4q + e] holds C[row i][column group q, element e]; accp is
        // the same tile as FFMA2 pairs (e = 0,1 and e = 2,3).
        float acc[8][TN];
        float2 accp[8][TN / 2];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;
#pragma unroll
            for (int j = 0; j < TN / 2; ++j) accp[i][j] = make_float2(0.0f, 0.0f);
        }

        for (int kb = item.kb0; kb < item.kb1; ++kb, ++it) {
            const int s = (int)(it % STAGES);
            if (!ptx::wait_phase_warp(full_bar(s), (it / STAGES) & 1)) {
                if (lane == 0) atomicOr(status, kStatusTimeout);
                return;
            }
            const uint8_t *As = base_ptr + s * Cfg::A_BYTES + a_row_off;
            const uint8_t *Bs = base_ptr + STAGES * Cfg::A_BYTES + s * Cfg::B_BYTES + b_col_off;
            if constexpr (K_TAIL) {
                if (kb == sched.nk - 1) {
                    // The last slab of a K that is not a multiple of BK: only
                    // its first k_last k hold data (TMA zero-filled the
                    // rest), so only those are multiplied. One k at a time,
                    // in the main loop's FFMA2 order.
#pragma unroll 1
                    for (int k = 0; k < sched.k_last; ++k) {
                        float av[8];
                        if constexpr (Cfg::A_KMAJOR) {
                            const float4 lo = *reinterpret_cast<const float4 *>(As + k * Cfg::A_ROW_BYTES);
                            const float4 hi = *reinterpret_cast<const float4 *>(As + k * Cfg::A_ROW_BYTES + 128);
                            av[0] = lo.x; av[1] = lo.y; av[2] = lo.z; av[3] = lo.w;
                            av[4] = hi.x; av[5] = hi.y; av[6] = hi.z; av[7] = hi.w;
                        } else {
                            // Column k of the swizzled slab: 16-byte chunk k / 4.
                            const uint32_t off = ((((uint32_t)k >> 2) ^ a_xor) << 4) + ((uint32_t)k & 3u) * 4;
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                av[i] = *reinterpret_cast<const float *>(As + i * 8 * Cfg::A_ROW_BYTES + off);
                        }
                        float4 b[G];
#pragma unroll
                        for (int q = 0; q < G; ++q)
                            b[q] = *reinterpret_cast<const float4 *>(Bs + k * Cfg::B_ROW_BYTES + 64 * q);
                        if constexpr (Cfg::PAIRED) {
#pragma unroll
                            for (int p = 0; p < TN / 2; ++p) {
                                const float4 &bq = b[p / 2];
                                const float2 bp = (p & 1) ? make_float2(bq.z, bq.w) : make_float2(bq.x, bq.y);
#pragma unroll
                                for (int ii = 0; ii < 8; ++ii) {
                                    const int i = (p & 1) ? 7 - ii : ii;
                                    accp[i][p] = __ffma2_rn(make_float2(av[i], av[i]), bp, accp[i][p]);
                                }
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 8; ++i)
#pragma unroll
                                for (int q = 0; q < G; ++q) {
                                    acc[i][4 * q + 0] = fmaf(av[i], b[q].x, acc[i][4 * q + 0]);
                                    acc[i][4 * q + 1] = fmaf(av[i], b[q].y, acc[i][4 * q + 1]);
                                    acc[i][4 * q + 2] = fmaf(av[i], b[q].z, acc[i][4 * q + 2]);
                                    acc[i][4 * q + 3] = fmaf(av[i], b[q].w, acc[i][4 * q + 3]);
                                }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(empty_bar(s));
                    continue;
                }
            }
            if constexpr (Cfg::A_KMAJOR) {
                // Per k: rows wm+4ty..+3 and wm+32+4ty..+3 as two float4.
#pragma unroll
                for (int k = 0; k < BK; ++k) {
                    const float4 lo = *reinterpret_cast<const float4 *>(As + k * Cfg::A_ROW_BYTES);
                    const float4 hi = *reinterpret_cast<const float4 *>(As + k * Cfg::A_ROW_BYTES + 128);
                    const float av[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                    float4 b[G];
#pragma unroll
                    for (int q = 0; q < G; ++q)
                        b[q] = *reinterpret_cast<const float4 *>(Bs + k * Cfg::B_ROW_BYTES + 64 * q);
                    // Column-serpentine order, as below.
#pragma unroll
                    for (int p = 0; p < TN / 2; ++p) {
                        const float4 &bq = b[p / 2];
                        const float2 bp = (p & 1) ? make_float2(bq.z, bq.w) : make_float2(bq.x, bq.y);
#pragma unroll
                        for (int ii = 0; ii < 8; ++ii) {
                            const int i = (p & 1) ? 7 - ii : ii;
                            accp[i][p] = __ffma2_rn(make_float2(av[i], av[i]), bp, accp[i][p]);
                        }
                    }
                }
            } else {
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
                        float4 b[G];
#pragma unroll
                        for (int q = 0; q < G; ++q)
                            b[q] = *reinterpret_cast<const float4 *>(Bs + k * Cfg::B_ROW_BYTES + 64 * q);
                        if constexpr (Cfg::PAIRED) {
                            // Column-serpentine order: each b pair meets the 8
                            // rows in turn, odd pairs walking the rows upwards, so
                            // consecutive FFMA2s always share a multiplicand
                            // register (87.9 % of the FP32 pipe for this loop
                            // measured alone, against 83.7 % row by row).
#pragma unroll
                            for (int p = 0; p < TN / 2; ++p) {
                                const float4 &bq = b[p / 2];
                                const float2 bp = (p & 1) ? make_float2(bq.z, bq.w) : make_float2(bq.x, bq.y);
#pragma unroll
                                for (int ii = 0; ii < 8; ++ii) {
                                    const int i = (p & 1) ? 7 - ii : ii;
                                    const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
                                    accp[i][p] = __ffma2_rn(make_float2(av, av), bp, accp[i][p]);
                                }
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
#pragma unroll
                                for (int q = 0; q < G; ++q) {
                                    acc[i][4 * q + 0] = fmaf(av, b[q].x, acc[i][4 * q + 0]);
                                    acc[i][4 * q + 1] = fmaf(av, b[q].y, acc[i][4 * q + 1]);
                                    acc[i][4 * q + 2] = fmaf(av, b[q].z, acc[i][4 * q + 2]);
                                    acc[i][4 * q + 3] = fmaf(av, b[q].w, acc[i][4 * q + 3]);
                                }
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty_bar(s));
        }

        if constexpr (Cfg::PAIRED) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < TN / 2; ++j) {
                    acc[i][2 * j] = accp[i][j].x;       // accp[i][j] = columns 2j, 2j+1
                    acc[i][2 * j + 1] = accp[i][j].y;
                }
        }

        if (item.kb0 > 0 || item.kb1 < sched.nk) {
            // A part of a split tile. Each consumer warp handles its own
            // fragment of the tile: slot layout float4 v of consumer thread
            // ct at index v * CONSUMER_THREADS + ct, so accesses coalesce.
            const int first = sk_first_cta(sched, item.tile);
            const int last = sk_last_cta(sched, item.tile);
            const unsigned others = (unsigned)(last - first);
            unsigned *ctr = sched.counters + (item.tile - sched.dp_tiles) * Cfg::CONSUMERS + warp;
            float *const parts = sched.partials;
            // With 8 x 8 thread tiles (the small-product configurations) the
            // CTA holding the first slab, which usually finishes its part
            // last, looks at the counter first: if every other part is in,
            // it adds them straight to its registers. The 8 x 16 tiles skip
            // that shortcut: the mainloop compiles without spills then, and
            // measured faster overall.
            bool reduce = false;
            if constexpr (Cfg::OWNER_PEEK) {
                if (g == first) {
                    unsigned seen = 0;
                    if (lane == 0) seen = ld_acquire_gpu(ctr);
                    reduce = __shfl_sync(0xffffffffu, seen, 0) == others;
                }
            }
            int h = first + 1;
            if (!reduce) {
                // Publish this part, then count it; the part that completes
                // the count sums every part from the slots (this one too).
                float4 *mine = reinterpret_cast<float4 *>(parts + sk_part_slot(g, first) * (BM * BN));
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int q = 0; q < G; ++q) {
                        mine[(i * G + q) * Cfg::CONSUMER_THREADS + ct] =
                            make_float4(acc[i][4 * q], acc[i][4 * q + 1], acc[i][4 * q + 2], acc[i][4 * q + 3]);
                        acc[i][4 * q] = acc[i][4 * q + 1] = acc[i][4 * q + 2] = acc[i][4 * q + 3] = 0.0f;
                    }
                __threadfence();
                __syncwarp();
                unsigned before = 0;
                if (lane == 0) before = atomic_inc_acq_rel_gpu(ctr);
                if (__shfl_sync(0xffffffffu, before, 0) != others) continue;   // not the last part
                h = first;
            }
            // Every part has been published: each lane acquires them itself,
            // then adds them in CTA order first, first + 1, ..., last (a
            // fixed order: results are deterministic).
            (void)ld_acquire_gpu(ctr);
            for (; h <= last; ++h) {
                const float4 *ph = reinterpret_cast<const float4 *>(parts + sk_part_slot(h, first) * (BM * BN));
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int q = 0; q < G; ++q) {
                        const float4 v = ph[(i * G + q) * Cfg::CONSUMER_THREADS + ct];
                        acc[i][4 * q] += v.x;
                        acc[i][4 * q + 1] += v.y;
                        acc[i][4 * q + 2] += v.z;
                        acc[i][4 * q + 3] += v.w;
                    }
            }
        }

        // Epilogue: rows wm+ty+8i (k-major A: wm+4ty+i, then wm+32+4ty+i-4),
        // G runs of 4 columns per row; rows rise with i either way.
        const int64_t row0 = (int64_t)tm * BM + wm + (Cfg::A_KMAJOR ? 4 * ty : ty);
        const int col0 = tn * BN + wn + tx * 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t row = row0 + (Cfg::A_KMAJOR ? (i < 4 ? i : 28 + i) : 8 * i);
            if (row >= M) break;
            float *crow = ep.C + (int64_t)bt * ep.stride_c + row * ep.ldc;
#pragma unroll
            for (int q = 0; q < G; ++q) {
                const int col = col0 + 16 * q;
                if (VEC_C && col + 3 < N) {
                    float4 *p = reinterpret_cast<float4 *>(crow + col);
                    float4 v = make_float4(ep.alpha * acc[i][4 * q], ep.alpha * acc[i][4 * q + 1],
                                           ep.alpha * acc[i][4 * q + 2], ep.alpha * acc[i][4 * q + 3]);
                    if (ep.beta != 0.0f) {
                        const float4 o = *p;
                        v.x = fmaf(ep.beta, o.x, v.x);
                        v.y = fmaf(ep.beta, o.y, v.y);
                        v.z = fmaf(ep.beta, o.z, v.z);
                        v.w = fmaf(ep.beta, o.w, v.w);
                    }
                    *p = v;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (col + e < N) {
                            float v = ep.alpha * acc[i][4 * q + e];
                            if (ep.beta != 0.0f) v = fmaf(ep.beta, crow[col + e], v);
                            crow[col + e] = v;
                        }
                }
            }
        }
    }
}

// Configurations: <BM, BN, BK, STAGES, TN, PAIRED, MIN_BLOCKS>.
using CfgFfma128x128k32s4 = FfmaTmaCfg<128, 128, 32, 4, 8, false, 1>;
using CfgFfma2_128x128k32s4 = FfmaTmaCfg<128, 128, 32, 4, 8, true, 1>;
using CfgFfma2_128x128k32s4ka = FfmaTmaCfg<128, 128, 32, 4, 8, true, 1, true>;
using CfgFfma2_128x128k16s8 = FfmaTmaCfg<128, 128, 16, 8, 8, true, 1>;
using CfgFfma2_128x64k32s4 = FfmaTmaCfg<128, 64, 32, 4, 8, true, 2>;
using CfgFfma2_128x256k32s4 = FfmaTmaCfg<128, 256, 32, 4, 16, true, 1>;
using CfgFfma2_128x256k32s4ka = FfmaTmaCfg<128, 256, 32, 4, 16, true, 1, true>;

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

// A batch of `batch` row-major rows x cols FP32 matrices, leading dimension
// ld and batch stride `stride` (elements), read in boxes of box_rows x
// box_cols of one entry. batch 1 (or a shared operand) uses stride rows*ld.
cudaError_t encode_3d(CUtensorMap *map, const float *ptr, int64_t rows, int64_t cols, int64_t ld,
                      int64_t batch, int64_t stride, int box_rows, int box_cols, CUtensorMapSwizzle swizzle)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    const cudaError_t e = get_encoder(&encode);
    if (e != cudaSuccess) return e;
    if (batch <= 1) {
        batch = 1;
        stride = rows * ld;
    }
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)ld * 4, (cuuint64_t)stride * 4};
    const cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(ptr), dims,
                              strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <class Cfg, bool K_TAIL, bool DEP = false>
cudaError_t set_smem_limit()
{
    cudaError_t e = cudaFuncSetAttribute(sgemm_ffma_tma_kernel<Cfg, true, K_TAIL, DEP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(sgemm_ffma_tma_kernel<Cfg, false, K_TAIL, DEP>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
}

// The schedule of a product; `with_sk` false gives whole tiles only.
template <class Cfg>
Schedule make_schedule(const GemmArgs &g, bool with_sk)
{
    return plan_schedule(g.M, g.N, g.K, Cfg::BM, Cfg::BN, Cfg::BK, g.num_sms * Cfg::MIN_BLOCKS, g.sched,
                         with_sk, g.batch);
}

template <class Cfg>
size_t workspace_bytes(const Schedule &s)
{
    return schedule_workspace_bytes(s, Cfg::CONSUMERS, Cfg::BM, Cfg::BN);
}

// Bytes at the start of the workspace that must be zero when the product
// starts (its stream-K arrival counters; 0 for whole tiles).
template <class Cfg>
size_t counter_bytes(const GemmArgs &g)
{
    if (g.workspace_bytes == 0) return 0;
    const Schedule s = make_schedule<Cfg>(g, true);
    return g.workspace_bytes >= workspace_bytes<Cfg>(s) ? schedule_counter_bytes(s, Cfg::CONSUMERS) : 0;
}

// Launches the product; K_TAIL selects the kernel that trims the last slab
// (for K not a multiple of BK), DEP the launch behind the call's layout pass.
template <class Cfg, bool K_TAIL, bool DEP = false>
cudaError_t launch(const GemmArgs &g, cudaStream_t stream)
{
    CUtensorMap mapA, mapB;
    // An operand with batch stride 0 is one matrix shared by every entry.
    const int a_bz = (g.batch > 1 && g.stride_a != 0) ? 1 : 0;
    const int b_bz = (g.batch > 1 && g.stride_b != 0) ? 1 : 0;
    // A is M x K, or K x M for a k-major configuration (boxes of BK rows of BM).
    cudaError_t e = Cfg::A_KMAJOR
                        ? encode_3d(&mapA, g.A, g.K, g.M, g.lda, a_bz ? g.batch : 1, g.stride_a, Cfg::BK, Cfg::BM,
                                    Cfg::A_SWIZZLE)
                        : encode_3d(&mapA, g.A, g.M, g.K, g.lda, a_bz ? g.batch : 1, g.stride_a, Cfg::BM, Cfg::BK,
                                    Cfg::A_SWIZZLE);
    if (e != cudaSuccess) return e;
    e = encode_3d(&mapB, g.B, g.K, g.N, g.ldb, b_bz ? g.batch : 1, g.stride_b, Cfg::BK, Cfg::BN,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    // Stream-K needs the caller's workspace; without one the schedule is whole tiles.
    Schedule s = make_schedule<Cfg>(g, g.workspace != nullptr);
    if (s.sk_ctas > 0 && g.workspace_bytes < workspace_bytes<Cfg>(s)) s = make_schedule<Cfg>(g, false);
    if (s.sk_ctas > 0 &&
        (e = schedule_attach_workspace(s, g.workspace, Cfg::CONSUMERS, !g.counters_zeroed, stream)) != cudaSuccess)
        return e;
    const bool vec = ((reinterpret_cast<uintptr_t>(g.C) & 15u) == 0) && (g.ldc % 4 == 0) &&
                     (g.batch <= 1 || g.stride_c % 4 == 0);
    Epilogue ep{g.C, g.ldc, g.batch > 1 ? g.stride_c : 0, (int)g.M, (int)g.N, g.alpha, g.beta, a_bz, b_bz};
    unsigned int *status = g.status;
    int withhold = g.withhold_it;
    void *args[] = {&mapA, &mapB, &ep, &s, &status, &withhold};
    const void *fn = vec ? reinterpret_cast<const void *>(sgemm_ffma_tma_kernel<Cfg, true, K_TAIL, DEP>)
                         : reinterpret_cast<const void *>(sgemm_ffma_tma_kernel<Cfg, false, K_TAIL, DEP>);
    // No CTA waits for another (split tiles are reduced by their last part),
    // so this is an ordinary launch; the DEP instance, behind the call's
    // layout pass, may start early (programmatic serialization), its threads
    // waiting for the pass.
    if constexpr (DEP) {
        cudaLaunchConfig_t lc = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        lc.gridDim = dim3(s.grid);
        lc.blockDim = dim3(Cfg::THREADS);
        lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
        lc.stream = stream;
        lc.attrs = attr;
        lc.numAttrs = 1;
        e = cudaLaunchKernelExC(&lc, fn, args);
    } else {
        e = cudaLaunchKernel(fn, dim3(s.grid), dim3(Cfg::THREADS), args, Cfg::SMEM_BYTES, stream);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace
}  // namespace sgemm_gb300
