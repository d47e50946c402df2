// FP32 product on the 5th-generation tensor cores by 3xTF32 splitting.
//
// Chapter 9: Optimised Matrix Multiplication, section 9.7, points past CUDA
// cores to tensor-core instructions that multiply whole tiles on a separate
// pipeline. Those take TF32 inputs (10 explicit mantissa bits), so each FP32
// operand is split as x = hi + lo with hi = tf32(x) and lo = tf32(x - hi),
// and the product keeps three of the four terms:
//     A.B ~ A_hi.B_hi + A_hi.B_lo + A_lo.B_hi      (A_lo.B_lo, ~2^-22 |A||B|, dropped)
// accumulated in FP32 in tensor memory. Integer-valued inputs with
// |x| < 2^11 have lo = 0 and stay exact; non-finite inputs do not (x - hi is
// NaN for infinite x), so this path is documented for finite inputs.
//
// Data flow of one call: two split pre-passes write A_hi, A_lo (M x Kp,
// K-major) and B_hi^T, B_lo^T (N x Kp, K-major: B is transposed on the way)
// into scratch; the product kernel then streams 128 x 16 and 256 x 16 tiles
// of all four through TMA (64-byte swizzle) into a 4-stage ring.
//
// Product kernel: persistent, one 128 x 256 output tile (or a K-slab range of
// one, under the stream-K tail of schedule.cuh) at a time per CTA.
//   warp 0      TMA producer (one thread): 4 boxes per K slab, full/empty
//               mbarriers per stage;
//   warp 1      MMA issuer (one thread) and TMEM owner: per K slab of 16,
//               2 x 3 tcgen05.mma .kind::tf32 (M 128, N 256, K 8) into a
//               TMEM accumulator; tcgen05.commit frees the stage, and at the
//               end of a tile signals the epilogue;
//   warps 4-7   epilogue: warp 4+q reads TMEM lanes 32q..32q+31 (rows of the
//               tile) with tcgen05.ld and stores them to C. For a slab range
//               of a split tile, the part that arrives last adds every part
//               in CTA order and stores the tile; the others write their
//               partial sums to their own slots and count themselves in the
//               tile's arrival counter (schedule.cuh). No CTA waits for another.
// The accumulator is double-buffered (2 x 256 of the 512 TMEM columns), so
// the epilogue of one tile overlaps the MMAs of the next. Every wait is
// bounded in time; a role that gives up sets the device error word and skips
// to the teardown (a CTA-wide barrier, then TMEM is freed); the producer
// drains its own copies before leaving.
//
// Cluster-pair variant (CM = 2): two CTAs of a cluster compute vertically
// adjacent 128 x 256 tiles that share one B tile. Each loads half of B_hi and
// B_lo and multicasts it into both CTAs' stage, so a CTA moves 32 KB per slab
// instead of 48 KB; each MMA warp multicasts its stage-release commit to both
// CTAs' empty barriers (count 2), so no stage is refilled before both have
// consumed it. Before leaving, a CTA's producer waits for the last release
// of every stage from both CTAs (no peer commit can then still be on its
// way), and the CTAs exchange a bounded "done" handshake. A launch without
// the cluster is detected (cluster size != 2) and reported, not run.
#include "common.cuh"
#include "configs.cuh"
#include "ptx.cuh"
#include "schedule.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace sgemm_gb300 {

namespace {

template <int BN_, int STAGES_, int CM_ = 1>
struct Tf32x3Cfg {
    static constexpr int BM = 128, BN = BN_, BK = 16, STAGES = STAGES_;
    static constexpr int CM = CM_;                             // CTAs per cluster, along M
    static constexpr int ROW_BYTES = BK * 4;                   // 64: 64-byte swizzle
    static constexpr int A_TILE = BM * ROW_BYTES;              // 8 KB
    static constexpr int B_TILE = BN * ROW_BYTES;              // 16 KB
    static constexpr int B_PIECE_ROWS = BN / CM;               // rows of B each CTA of a cluster loads
    static constexpr int STAGE_BYTES = 2 * A_TILE + 2 * B_TILE;
    static constexpr int NUM_BARS = 2 * STAGES + 2 + 2 + 1 + 1;  // full, empty, acc full, acc empty, drain, exit
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_BARS * 8 + 16;
    static constexpr int TMEM_COLS = 2 * BN;                   // double-buffered FP32 accumulator
    static constexpr int THREADS = 256;
    static constexpr int EPI_WARP0 = 4;
    static constexpr uint32_t IDESC = ptx::idesc_tf32_kmajor(BM, BN);
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
    static_assert(TMEM_COLS <= 512, "tensor memory columns");
    static_assert(CM == 1 || CM == 2 || CM == 4, "cluster size");
    static_assert((B_PIECE_ROWS * ROW_BYTES) % 1024 == 0, "B pieces keep the swizzle phase");
};

template <class Cfg, bool VEC_C>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
sgemm_tf32x3_kernel(const __grid_constant__ CUtensorMap mapAhi, const __grid_constant__ CUtensorMap mapAlo,
                    const __grid_constant__ CUtensorMap mapBhi, const __grid_constant__ CUtensorMap mapBlo,
                    float *__restrict__ C, int64_t ldc, int M, int N, const Schedule sched,
                    unsigned int *status, float alpha, float beta)
{
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES, CM = Cfg::CM;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bars = base + STAGES * Cfg::STAGE_BYTES;
    auto stage_a_hi = [&](int s) { return base + s * Cfg::STAGE_BYTES; };
    auto stage_a_lo = [&](int s) { return base + s * Cfg::STAGE_BYTES + Cfg::A_TILE; };
    auto stage_b_hi = [&](int s) { return base + s * Cfg::STAGE_BYTES + 2 * Cfg::A_TILE; };
    auto stage_b_lo = [&](int s) { return base + s * Cfg::STAGE_BYTES + 2 * Cfg::A_TILE + Cfg::B_TILE; };
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bars + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bars + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = bars + 8u * (2 * STAGES + 4);
    const uint32_t exit_bar = bars + 8u * (2 * STAGES + 5);
    const uint32_t tmem_slot = bars + 8u * Cfg::NUM_BARS;
    uint32_t *tmem_slot_ptr = reinterpret_cast<uint32_t *>(smem_raw + (tmem_slot - raw));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // A cluster of CM CTAs shares one schedule item: CTA `rank` computes
    // block row rank of the item's CM x 1 group of 128 x BN tiles.
    const int rank = CM > 1 ? (int)ptx::cluster_ctarank() : 0;
    const int g = (int)blockIdx.x / CM;               // schedule index (cluster)
    const int nk = sched.nk;
    constexpr uint16_t kClusterMask = (uint16_t)((1u << CM) - 1u);
    if constexpr (CM > 1) {
        // Launched without its cluster of CM CTAs, this kernel would copy to
        // and arrive at peers that do not exist: report it and do nothing.
        if (ptx::cluster_nctarank() != (uint32_t)CM) {
            if (threadIdx.x == 0) atomicOr(status, kStatusLaunchConfig);
            return;
        }
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), CM);         // one MMA commit from every CTA of the cluster
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accf_bar(b), 1);
            ptx::mbar_init(acce_bar(b), 4);
        }
        ptx::mbar_init(drain_bar, 1);
        ptx::mbar_init(exit_bar, CM);
        ptx::mbar_init_fence();
    }
    if (warp == 1) ptx::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    ptx::tc_fence_before();
    // Barriers must be initialised in every CTA before any peer copies or
    // arrives into them.
    if constexpr (CM > 1)
        ptx::cluster_sync_all();
    else
        __syncthreads();
    ptx::tc_fence_after();
    const uint32_t taddr = *tmem_slot_ptr;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        // A: this CTA's 128 rows. B: with CM > 1, this CTA loads rows
        // [rank * BN/CM, (rank + 1) * BN/CM) of the B tile and multicasts
        // them to the whole cluster, so each CTA's full barrier counts the
        // whole stage; a stage is refilled only when every CTA's MMAs have
        // released it (the empty barrier counts CM commits).
        if (lane == 0) {
            ptx::prefetch_tensormap(&mapAhi);
            ptx::prefetch_tensormap(&mapAlo);
            ptx::prefetch_tensormap(&mapBhi);
            ptx::prefetch_tensormap(&mapBlo);
            const uint64_t policy = ptx::policy_evict_last();
            int last_round[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s) last_round[s] = -1;
            uint32_t it = 0;
            bool ok = true;
            Cursor cur = cursor_init(sched, g);
            Item item;
            while (ok && next_item(sched, cur, item)) {
                int tg, tn;
                tile_coords(item.tile, sched.tiles_m, sched.tiles_n, tg, tn);
                const int tm = tg * CM + rank;
                for (int kb = item.kb0; kb < item.kb1; ++kb, ++it) {
                    const int s = (int)(it % STAGES);
                    const int round = (int)(it / STAGES);
                    if (!ptx::wait_phase(empty_bar(s), (round & 1) ^ 1)) {
                        atomicOr(status, kStatusTimeout);
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(full_bar(s), Cfg::STAGE_BYTES);
                    ptx::tma_load_2d(stage_a_hi(s), &mapAhi, full_bar(s), kb * BK, tm * BM, policy);
                    ptx::tma_load_2d(stage_a_lo(s), &mapAlo, full_bar(s), kb * BK, tm * BM, policy);
                    if constexpr (CM > 1) {
                        const uint32_t off = (uint32_t)(rank * Cfg::B_PIECE_ROWS * Cfg::ROW_BYTES);
                        const int row = tn * BN + rank * Cfg::B_PIECE_ROWS;
                        ptx::tma_load_2d_multicast(stage_b_hi(s) + off, &mapBhi, full_bar(s), kb * BK, row,
                                                   kClusterMask, policy);
                        ptx::tma_load_2d_multicast(stage_b_lo(s) + off, &mapBlo, full_bar(s), kb * BK, row,
                                                   kClusterMask, policy);
                    } else {
                        ptx::tma_load_2d(stage_b_hi(s), &mapBhi, full_bar(s), kb * BK, tn * BN, policy);
                        ptx::tma_load_2d(stage_b_lo(s), &mapBlo, full_bar(s), kb * BK, tn * BN, policy);
                    }
                    last_round[s] = round;
                }
            }
            // Every byte bound for this CTA (its own copies and the peers'
            // multicasts) must have landed before it leaves.
            for (int s = 0; s < STAGES; ++s)
                if (last_round[s] >= 0 && !ptx::wait_phase(full_bar(s), last_round[s] & 1))
                    atomicOr(status, kStatusTimeout);
            // With CM > 1, so must every commit arrival the peers' MMA warps
            // send to this CTA's empty barriers: wait for the release of each
            // stage's last round by all CM CTAs (phase r of an empty barrier
            // completes when round r of its stage has been released).
            if constexpr (CM > 1) {
                for (int s = 0; s < STAGES; ++s)
                    if (last_round[s] >= 0 && !ptx::wait_phase(empty_bar(s), last_round[s] & 1))
                        atomicOr(status, kStatusTimeout);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            uint32_t it = 0, lt = 0;
            Cursor cur = cursor_init(sched, g);
            Item item;
            for (; next_item(sched, cur, item); ++lt) {
                const int b = (int)(lt & 1);
                const uint32_t use = lt >> 1;
                if (!ptx::wait_phase(acce_bar(b), (use & 1) ^ 1)) {
                    atomicOr(status, kStatusTimeout);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = taddr + (uint32_t)(b * BN);
                bool ok = true;
                for (int kb = item.kb0; kb < item.kb1; ++kb, ++it) {
                    const int s = (int)(it % STAGES);
                    if (!ptx::wait_phase(full_bar(s), (it / STAGES) & 1)) {
                        atomicOr(status, kStatusTimeout);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < BK / 8; ++ks) {
                        const uint64_t ah = ptx::sdesc_kmajor(stage_a_hi(s) + ks * 32, Cfg::ROW_BYTES);
                        const uint64_t al = ptx::sdesc_kmajor(stage_a_lo(s) + ks * 32, Cfg::ROW_BYTES);
                        const uint64_t bh = ptx::sdesc_kmajor(stage_b_hi(s) + ks * 32, Cfg::ROW_BYTES);
                        const uint64_t bl = ptx::sdesc_kmajor(stage_b_lo(s) + ks * 32, Cfg::ROW_BYTES);
                        ptx::mma_tf32(d, ah, bh, Cfg::IDESC, (kb != item.kb0 || ks != 0) ? 1u : 0u);
                        ptx::mma_tf32(d, ah, bl, Cfg::IDESC, 1u);
                        ptx::mma_tf32(d, al, bh, Cfg::IDESC, 1u);
                    }
                    // The stage is free once these MMAs are done; with CM > 1
                    // every CTA of the cluster learns it (their producers
                    // multicast into this CTA's copy of the stage).
                    if constexpr (CM > 1)
                        ptx::mma_commit_multicast(empty_bar(s), kClusterMask);
                    else
                        ptx::mma_commit(empty_bar(s));
                }
                if (!ok) break;
                ptx::mma_commit(accf_bar(b));        // the tile's accumulator is complete
            }
            // Every MMA issued above (and so every commit arrival it sends to
            // the peers) must finish before TMEM is released.
            ptx::mma_commit(drain_bar);
            if (!ptx::wait_phase(drain_bar, 0)) atomicOr(status, kStatusTimeout);
        }
        __syncwarp();
    } else if (warp >= Cfg::EPI_WARP0) {
        // ------------------------------ epilogue ------------------------------
        const int q = warp - Cfg::EPI_WARP0;          // TMEM lane quarter (== warp % 4)
        const int et = 32 * q + lane;                 // epilogue thread: row of the tile
        uint32_t lt = 0;
        Cursor cur = cursor_init(sched, g);
        Item item;
        for (; next_item(sched, cur, item); ++lt) {
            const int b = (int)(lt & 1);
            const uint32_t use = lt >> 1;
            if (!ptx::wait_phase_warp(accf_bar(b), use & 1)) {
                if (lane == 0) atomicOr(status, kStatusTimeout);
                break;
            }
            ptx::tc_fence_after();
            int tg, tn;
            tile_coords(item.tile, sched.tiles_m, sched.tiles_n, tg, tn);
            const int tm = tg * CM + rank;
            // Partial-sum slot layout: float4 v (columns 4v..4v+3) of tile row
            // et at index v * 128 + et, so each warp's accesses are coalesced.
            // Part h of a split tile (this CTA's rank of cluster h) has the
            // slot sk_part_slot of CTA index h * CM + rank.
            const bool split = item.kb0 > 0 || item.kb1 < nk;
            int first = 0, last = 0;
            unsigned others = 0;
            unsigned *ctr = nullptr;
            bool from_tmem = false;   // reduce now, this part straight from TMEM
            if (split) {
                first = sk_first_cta(sched, item.tile);
                last = sk_last_cta(sched, item.tile);
                others = (unsigned)(last - first);
                ctr = sched.counters + ((item.tile - sched.dp_tiles) * CM + rank) * 4 + q;
                // The part holding the first slab adds the others itself when
                // they have all arrived; otherwise every part is published.
                if (g == first) {
                    unsigned seen = 0;
                    if (lane == 0) seen = ld_acquire_gpu(ctr);
                    from_tmem = __shfl_sync(0xffffffffu, seen, 0) == others;
                    if (from_tmem) (void)ld_acquire_gpu(ctr);
                }
            }
            const bool publish = split && !from_tmem;
            auto slot_ptr = [&](int h) {
                const int64_t sl = 2 * ((int64_t)h * CM + rank) + (h == first ? 1 : 0);
                return reinterpret_cast<float4 *>(sched.partials + sl * (BM * BN));
            };
            const int64_t row = (int64_t)tm * BM + et;
            float *crow = C + row * ldc;
            const int col_base = tn * BN;
            // Stores columns c0 .. c0 + 31 of this thread's row of C.
            auto store_chunk = [&](int c0, float (&f)[32]) {
                if (row >= M) return;
                const int col0 = col_base + c0;
#pragma unroll
                for (int j = 0; j < 32; ++j) f[j] *= alpha;
                if (VEC_C && (int64_t)col0 + 32 <= N) {   // 64-bit: col0 + 32 may reach 2^31
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        float4 *p = reinterpret_cast<float4 *>(crow + col0 + j);
                        float4 v = make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
                        if (beta != 0.0f) {
                            const float4 o = *p;
                            v.x = fmaf(beta, o.x, v.x);
                            v.y = fmaf(beta, o.y, v.y);
                            v.z = fmaf(beta, o.z, v.z);
                            v.w = fmaf(beta, o.w, v.w);
                        }
                        *p = v;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + j < N) crow[col0 + j] = beta != 0.0f ? fmaf(beta, crow[col0 + j], f[j]) : f[j];
                }
            };
            // Adds parts h0 .. last of columns c0 .. c0 + 31, in that order.
            auto add_parts = [&](int h0, int c0, float (&f)[32]) {
                for (int h = h0; h <= last; ++h) {
                    const float4 *src = slot_ptr(h);
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4 p4 = src[((c0 + j) / 4) * 128 + et];
                        f[j] += p4.x;
                        f[j + 1] += p4.y;
                        f[j + 2] += p4.z;
                        f[j + 3] += p4.w;
                    }
                }
            };
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t v[32];
                ptx::tmem_ld32(taddr + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * BN + c0), v);
                ptx::tmem_ld_wait();
                if (c0 == BN - 32) {
                    // Last read of this accumulator: hand it back to the MMA warp.
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(acce_bar(b));
                }
                float f[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
                if (publish) {
                    float4 *dst = slot_ptr(g);
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        dst[((c0 + j) / 4) * 128 + et] = make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
                    continue;
                }
                if (from_tmem) add_parts(first + 1, c0, f);
                store_chunk(c0, f);
            }
            if (publish) {
                __threadfence();
                __syncwarp();
                unsigned before = 0;
                if (lane == 0) before = atomic_inc_acq_rel_gpu(ctr);
                if (__shfl_sync(0xffffffffu, before, 0) == others) {
                    // The last part to arrive: every part is in its slot.
                    (void)ld_acquire_gpu(ctr);
#pragma unroll 1
                    for (int c0 = 0; c0 < BN; c0 += 32) {
                        float f[32];
                        const float4 *src = slot_ptr(first);
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            const float4 p4 = src[((c0 + j) / 4) * 128 + et];
                            f[j] = p4.x;
                            f[j + 1] = p4.y;
                            f[j + 2] = p4.z;
                            f[j + 3] = p4.w;
                        }
                        add_parts(first + 1, c0, f);
                        store_chunk(c0, f);
                    }
                }
            }
        }
        ptx::tc_fence_before();
    }

    // ------------------------------ teardown ------------------------------
    // Every role of this CTA is done: the producer has seen all bytes bound
    // for this CTA land, the MMA warp has drained its MMAs and commits.
    __syncthreads();
    if constexpr (CM > 1) {
        // No CTA leaves while a peer may still copy into its shared memory
        // or arrive on its barriers: each tells every CTA of the cluster that
        // it is done, then waits (bounded) until all have said so.
        if (threadIdx.x == 0) {
            for (int r = 0; r < CM; ++r) ptx::mbar_arrive_remote(exit_bar, (uint32_t)r);
            if (!ptx::wait_phase(exit_bar, 0)) atomicOr(status, kStatusTimeout);
        }
        __syncthreads();
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(taddr, Cfg::TMEM_COLS);
    }
}

// hi[i * ldo + k] = tf32(x), lo[i * ldo + k] = tf32(x - hi) for x = src[i * ld + k].
// One block per row at a time; VEC reads and writes float4 (source rows and
// base 16-byte aligned, cols a multiple of 4), otherwise single floats.
template <bool VEC>
__global__ void __launch_bounds__(256)
tf32_split_rows_kernel(const float *__restrict__ src, int64_t rows, int64_t cols, int64_t ld,
                       float *__restrict__ hi, float *__restrict__ lo, int64_t ldo)
{
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float *s = src + r * ld;
        float *h = hi + r * ldo;
        float *l = lo + r * ldo;
        if (VEC) {
            for (int64_t c = threadIdx.x; c < cols / 4; c += blockDim.x) {
                const float4 x = reinterpret_cast<const float4 *>(s)[c];
                float4 xh, xl;
                xh.x = ptx::to_tf32(x.x); xl.x = ptx::to_tf32(x.x - xh.x);
                xh.y = ptx::to_tf32(x.y); xl.y = ptx::to_tf32(x.y - xh.y);
                xh.z = ptx::to_tf32(x.z); xl.z = ptx::to_tf32(x.z - xh.z);
                xh.w = ptx::to_tf32(x.w); xl.w = ptx::to_tf32(x.w - xh.w);
                reinterpret_cast<float4 *>(h)[c] = xh;
                reinterpret_cast<float4 *>(l)[c] = xl;
            }
        } else {
            for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) {
                const float x = s[c];
                const float xh = ptx::to_tf32(x);
                h[c] = xh;
                l[c] = ptx::to_tf32(x - xh);
            }
        }
    }
}

// The same split of B (K x N, leading dimension ld), written transposed:
// hiT[n * ldo + k], loT[n * ldo + k]. 64 x 64 tiles through shared memory
// (padded by one column), 32 x 8 threads moving 16 elements each, so both
// the reads (along n) and the writes (along k) are 128-byte warp segments.
__global__ void __launch_bounds__(256)
tf32_split_transpose_kernel(const float *__restrict__ src, int64_t rows, int64_t cols, int64_t ld,
                            float *__restrict__ hiT, float *__restrict__ loT, int64_t ldo)
{
    __shared__ float tile[64][65];
    const int tx = threadIdx.x, ty = threadIdx.y;   // 32 x 8 threads
    const int64_t tiles_c = (cols + 63) / 64;
    const int64_t ntiles = ((rows + 63) / 64) * tiles_c;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t r0 = (t / tiles_c) * 64, c0 = (t % tiles_c) * 64;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t r = r0 + ty + 8 * i;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t c = c0 + tx + 32 * h;
                tile[ty + 8 * i][tx + 32 * h] = (r < rows && c < cols) ? src[r * ld + c] : 0.0f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t c = c0 + ty + 8 * i;   // output row c, column r
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t r = r0 + tx + 32 * h;
                if (c < cols && r < rows) {
                    const float x = tile[tx + 32 * h][ty + 8 * i];
                    const float xh = ptx::to_tf32(x);
                    hiT[c * ldo + r] = xh;
                    loT[c * ldo + r] = ptx::to_tf32(x - xh);
                }
            }
        }
        __syncthreads();
    }
}

int64_t round_up_i(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

struct Tf32x3Layout {
    int64_t kp;                  // leading dimension of the split operands
    size_t a_bytes, b_bytes;     // one split copy of A / of B^T, 256-byte rounded
    size_t total;
};

Tf32x3Layout tf32x3_layout(const GemmArgs &g)
{
    Tf32x3Layout l;
    l.kp = round_up_i(g.K, 4);
    l.a_bytes = (size_t)round_up_i(g.M * l.kp * 4, 256);
    l.b_bytes = (size_t)round_up_i(g.N * l.kp * 4, 256);
    l.total = 2 * l.a_bytes + 2 * l.b_bytes;
    return l;
}

cudaError_t encode_kmajor(CUtensorMap *map, const float *ptr, int64_t rows, int64_t k, int64_t ld, int box_rows,
                          int box_k)
{
    void *fnp = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fnp, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fnp) return cudaErrorNotSupported;
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fnp);
    const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
    const cuuint32_t box[2] = {(cuuint32_t)box_k, (cuuint32_t)box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(ptr), dims, strides,
                              box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// K-major hi/lo split of an operand with `rows` rows of K values: stored
// K-major (rows x K, leading dimension ld) when `kmajor`, else transposed
// (K x rows, leading dimension ld).
cudaError_t split_kmajor(const float *src, bool kmajor, int64_t rows, int64_t K, int64_t ld, float *hi,
                         float *lo, int64_t kp, int num_sms, cudaStream_t stream)
{
    if (kmajor) {
        // kp is a multiple of 4 and the planes are 256-byte aligned, so the
        // writes vectorise whenever the source rows do.
        const bool vec = K % 4 == 0 && ld % 4 == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0;
        const int64_t cap = (int64_t)num_sms * 8;
        const unsigned grid = (unsigned)(rows < cap ? rows : cap);
        if (vec)
            tf32_split_rows_kernel<true><<<grid, 256, 0, stream>>>(src, rows, K, ld, hi, lo, kp);
        else
            tf32_split_rows_kernel<false><<<grid, 256, 0, stream>>>(src, rows, K, ld, hi, lo, kp);
    } else {
        const int64_t tiles = ((K + 63) / 64) * ((rows + 63) / 64);
        const unsigned grid = (unsigned)(tiles < (int64_t)num_sms * 16 ? tiles : (int64_t)num_sms * 16);
        tf32_split_transpose_kernel<<<grid, dim3(32, 8), 0, stream>>>(src, K, rows, ld, hi, lo, kp);
    }
    return cudaGetLastError();
}

using Tf32x3Wide = Tf32x3Cfg<256, 4>;     // 128 x 256 tiles, 4 stages of 48 KB
using Tf32x3Square = Tf32x3Cfg<128, 6>;   // 128 x 128 tiles, 6 stages of 32 KB
using Tf32x3Pair = Tf32x3Cfg<256, 4, 2>;  // clusters of 2 CTAs sharing (multicasting) B tiles

// The schedule runs over groups of CM vertically adjacent tiles, one group
// per cluster; clusters of CM CTAs fill the SMs (every GB300 SM pair hosts
// a cluster of 2).
template <class Cfg>
Schedule tf32x3_schedule(const GemmArgs &g, bool with_sk)
{
    return plan_schedule(g.M, g.N, g.K, Cfg::BM * Cfg::CM, Cfg::BN, Cfg::BK, g.num_sms / Cfg::CM, g.sched,
                         with_sk);
}

template <class Cfg>
size_t tf32x3_workspace(const GemmArgs &g)
{
    return tf32x3_layout(g).total +
           schedule_workspace_bytes(tf32x3_schedule<Cfg>(g, true), 4 * Cfg::CM, Cfg::BM * Cfg::CM, Cfg::BN);
}

template <class Cfg>
cudaError_t prepare_cfg()
{
    cudaError_t e = cudaFuncSetAttribute(sgemm_tf32x3_kernel<Cfg, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(sgemm_tf32x3_kernel<Cfg, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg::SMEM_BYTES);
}

template <class Cfg>
cudaError_t launch_cfg(const GemmArgs &g, cudaStream_t stream)
{
    const Tf32x3Layout l = tf32x3_layout(g);
    if (!g.workspace || g.workspace_bytes < l.total) return cudaErrorInvalidValue;
    uint8_t *ws = static_cast<uint8_t *>(g.workspace);
    float *a_hi = reinterpret_cast<float *>(ws);
    float *a_lo = reinterpret_cast<float *>(ws + l.a_bytes);
    float *b_hi = reinterpret_cast<float *>(ws + 2 * l.a_bytes);
    float *b_lo = reinterpret_cast<float *>(ws + 2 * l.a_bytes + l.b_bytes);
    cudaError_t e;

    // Split pre-passes into K-major hi/lo copies: a K-major operand (A as
    // stored, or B stored transposed) is split row by row, the others go
    // through the transposing split.
    if ((e = split_kmajor(g.A, g.op_a == 0, g.M, g.K, g.lda, a_hi, a_lo, l.kp, g.num_sms, stream)) != cudaSuccess)
        return e;
    if ((e = split_kmajor(g.B, g.op_b == 1, g.N, g.K, g.ldb, b_hi, b_lo, l.kp, g.num_sms, stream)) != cudaSuccess)
        return e;

    CUtensorMap mAh, mAl, mBh, mBl;
    if ((e = encode_kmajor(&mAh, a_hi, g.M, g.K, l.kp, Cfg::BM, Cfg::BK)) != cudaSuccess) return e;
    if ((e = encode_kmajor(&mAl, a_lo, g.M, g.K, l.kp, Cfg::BM, Cfg::BK)) != cudaSuccess) return e;
    if ((e = encode_kmajor(&mBh, b_hi, g.N, g.K, l.kp, Cfg::B_PIECE_ROWS, Cfg::BK)) != cudaSuccess) return e;
    if ((e = encode_kmajor(&mBl, b_lo, g.N, g.K, l.kp, Cfg::B_PIECE_ROWS, Cfg::BK)) != cudaSuccess) return e;

    // Stream-K arrival counters (4 per CTA of a cluster per split tile) and
    // partial-sum slots (two per CTA) follow the split operands in the workspace.
    constexpr int kCounters = 4 * Cfg::CM;
    Schedule sched = tf32x3_schedule<Cfg>(g, true);
    if (sched.sk_ctas > 0 &&
        g.workspace_bytes < l.total + schedule_workspace_bytes(sched, kCounters, Cfg::BM * Cfg::CM, Cfg::BN))
        sched = tf32x3_schedule<Cfg>(g, false);
    if (sched.sk_ctas > 0 && (e = schedule_attach_workspace(sched, ws + l.total, kCounters, true, stream)) != cudaSuccess)
        return e;
    const bool vec = ((reinterpret_cast<uintptr_t>(g.C) & 15u) == 0) && (g.ldc % 4 == 0);
    float *C = g.C;
    int64_t ldc = g.ldc;
    int M = (int)g.M, N = (int)g.N;
    unsigned int *status = g.status;
    float alpha = g.alpha, beta = g.beta;
    void *args[] = {&mAh, &mAl, &mBh, &mBl, &C, &ldc, &M, &N, &sched, &status, &alpha, &beta};
    const void *fn = vec ? reinterpret_cast<const void *>(sgemm_tf32x3_kernel<Cfg, true>)
                         : reinterpret_cast<const void *>(sgemm_tf32x3_kernel<Cfg, false>);
    // Split tiles are reduced by their last part, so no CTA waits for
    // another: the only launch attribute is the cluster shape.
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attrs[1];
    int na = 0;
    if (Cfg::CM > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = Cfg::CM;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    lc.gridDim = dim3((unsigned)(sched.grid * Cfg::CM));
    lc.blockDim = dim3(Cfg::THREADS);
    lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
    lc.stream = stream;
    lc.attrs = attrs;
    lc.numAttrs = (unsigned)na;
    e = cudaLaunchKernelExC(&lc, fn, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

size_t tf32x3_workspace_bytes(int kernel, const GemmArgs &g)
{
    if (kernel == kKernTf32x3_128x128) return tf32x3_workspace<Tf32x3Square>(g);
    if (kernel == kKernTf32x3_pair) return tf32x3_workspace<Tf32x3Pair>(g);
    return tf32x3_workspace<Tf32x3Wide>(g);
}

cudaError_t prepare_tf32x3()
{
    cudaError_t e = prepare_cfg<Tf32x3Wide>();
    if (e == cudaSuccess) e = prepare_cfg<Tf32x3Square>();
    if (e == cudaSuccess) e = prepare_cfg<Tf32x3Pair>();
    return e;
}

cudaError_t launch_tf32x3(int kernel, const GemmArgs &g, cudaStream_t stream)
{
    // Batch entries run one after another, reusing the split buffers.
    for (int64_t b = 0; b < (g.batch > 1 ? g.batch : 1); ++b) {
        GemmArgs e = g;
        e.A = g.A + b * g.stride_a;
        e.B = g.B + b * g.stride_b;
        e.C = g.C + b * g.stride_c;
        e.batch = 1;
        const cudaError_t r = kernel == kKernTf32x3_128x128 ? launch_cfg<Tf32x3Square>(e, stream)
                              : kernel == kKernTf32x3_pair  ? launch_cfg<Tf32x3Pair>(e, stream)
                                                            : launch_cfg<Tf32x3Wide>(e, stream);
        if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
}

}  // namespace sgemm_gb300
