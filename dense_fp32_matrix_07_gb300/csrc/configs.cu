// Configuration table and selector (host logic only).
#include "configs.cuh"

namespace sgemm_gb300 {

const ConfigInfo kConfigTable[kNumConfigs] = {
    {"tiled16_simple", kKernTiledSimple, kSchedDataParallel, false, false, 16, 16},
    {"ffma_128x128_k32_s4", kKernFfma128x128k32s4, kSchedAuto, true, true, 128, 128},
    {"ffma2_128x128_k32_s4", kKernFfma2_128x128k32s4, kSchedAuto, true, true, 128, 128},
    {"ffma2_128x128_k16_s8", kKernFfma2_128x128k16s8, kSchedAuto, true, true, 128, 128},
    {"ffma2_128x64_k32_s4", kKernFfma2_128x64k32s4, kSchedAuto, true, true, 128, 64},
    {"ffma2_128x256_k32_s4", kKernFfma2_128x256k32s4, kSchedAuto, true, true, 128, 256},
    {"ffma2_128x128_k32_s4_dp", kKernFfma2_128x128k32s4, kSchedDataParallel, true, true, 128, 128},
    {"ffma2_128x128_k32_s4_sk", kKernFfma2_128x128k32s4, kSchedStreamK, true, true, 128, 128},
    {"ffma2_128x256_k32_s4_dp", kKernFfma2_128x256k32s4, kSchedDataParallel, true, true, 128, 256},
    {"ffma2_128x256_k32_s4_sk", kKernFfma2_128x256k32s4, kSchedStreamK, true, true, 128, 256},
    {"ladder_naive_rowmap", kKernLadderNaive, kSchedDataParallel, false, false, 16, 16},
    {"ladder_coalesced", kKernLadderCoalesced, kSchedDataParallel, false, false, 16, 16},
    {"ladder_cache_blocked_8x8", kKernLadderCacheBlocked8x8, kSchedDataParallel, false, false, 8, 8},
    {"ladder_register_tiled_2x2", kKernLadderRegisterTiled2x2, kSchedDataParallel, false, false, 16, 16},
    {"tf32x3_128x256_k16_s4", kKernTf32x3_128x256, kSchedTailSplit, true, false, 128, 256},
    {"tf32x3_128x256_k16_s4_sk", kKernTf32x3_128x256, kSchedStreamK, true, false, 128, 256},
    {"tf32x3_128x256_k16_s4_auto", kKernTf32x3_128x256, kSchedAuto, true, false, 128, 256},
    {"tf32x3_128x128_k16_s6", kKernTf32x3_128x128, kSchedDataParallel, true, false, 128, 128},
    {"tf32x3_128x256_k16_s4_dp", kKernTf32x3_128x256, kSchedDataParallel, true, false, 128, 256},
    {"tf32x3_pair_128x256_k16_s4", kKernTf32x3_pair, kSchedTailSplit, true, false, 128, 256},
    {"tf32x3_pair_128x256_k16_s4_dp", kKernTf32x3_pair, kSchedDataParallel, true, false, 128, 256},
    {"ffma2_128x256_k32_s4_ka", kKernFfma2_128x256k32s4ka, kSchedAuto, true, true, 128, 256, true},
    {"ffma2_128x128_k32_s4_ka", kKernFfma2_128x128k32s4ka, kSchedAuto, true, true, 128, 128, true},
    {"small_32x32_k256", kKernSmall32, kSchedDataParallel, false, false, 32, 32},
};

bool config_supports(int cfg, const ProblemShape &p)
{
    if (cfg < 0 || cfg >= kNumConfigs) return false;
    // One thread per output on a 2-D grid: grid.y (<= 65535 blocks of 16)
    // runs over columns (row-mapped kernel) or rows (coalesced kernel).
    if (kConfigTable[cfg].kernel == kKernLadderNaive) return p.N <= 65535 * 16;
    if (kConfigTable[cfg].kernel == kKernLadderCoalesced) return p.M <= 65535 * 16;
    if (!kConfigTable[cfg].uses_tma) return true;
    // TMA sizes are 32-bit coordinates; strides of packed operands are at
    // most (kMaxDim rounded up) * 4 bytes, within the 2^40-byte stride limit.
    return p.M <= kMaxDim && p.N <= kMaxDim && p.K <= kMaxDim &&
           p.lda < (int64_t(1) << 37) && p.ldb < (int64_t(1) << 37);
}

int select_config(const ProblemShape &p)
{
    if (!config_supports(kCfgFfma2_128x128, p)) return kCfgTiledSimple;
    // Small products (up to about 400^3, a C of at most 2^19 entries, K up to
    // 512) finish sooner in the small-product kernel: 32 x 32 tiles over many
    // SMs, each CTA's K panel loaded at once, no tensor-map set-up. Same-box
    // A/B with the L2 flushed, against the pages' register-tiled kernel that
    // had these shapes before and the TMA configuration: 256^3 10.7 us
    // (16.9, 17.9 for 128 x 64 tiles), 384^3 14.8 (23.3), 512 x 512 x 256 14.6
    // (22.1, 17.9), 64^3 8.5 (10.3 TMA); the TMA tiles lead once C grows
    // (1024 x 1024 x 64: 17.9 against 10.2 us), once K does (256 x 256 x
    // 1024: 25.2 against 22.0 us) and from 448^3 on (20.9 against 20.0 us).
    const double mn = (double)p.M * (double)p.N;
    if (mn * (double)p.K <= 67108864.0 && p.K <= 512 && mn <= 524288.0) return kCfgSmall32;
    // The widest thread tile (8x16) when there are enough 128x256 tiles to
    // give every SM one; 128x128 down to a third of that (at 1024^3, 64
    // tiles: 49.2 us against 51.2 us for 128x64), 128x64 (two CTAs per SM)
    // below. The stream-K tail evens out partial last waves in all three.
    const int64_t tiles256 = ((p.M + 127) / 128) * ((p.N + 255) / 256);
    const int64_t tiles128 = ((p.M + 127) / 128) * ((p.N + 127) / 128);
    // With A k-major in shared memory the 8x16 loop runs faster (91 % of the
    // FP32 pipe alone against 88 %); a plain A is transposed first, at about
    // 8MK bytes of traffic, which the product repays once N reaches about
    // 1300 (same-box sweep: 4096^3 86.3 % against 84.3 % of the FP32 peak,
    // 16384^3 87.8 % against 85.2 %, 2048^3 forced onto 128x256 tiles 80.0 %
    // against 79.4 %).
    // The pass also costs about 5 us whatever its size (a launch and its
    // drain), which the faster loop, about 2.5 % of the product, repays once
    // the product takes about 200 us: M*N*K >= 6e9 (same-box sweep, row-major
    // against k-major: 2048 x 2048 x 512 81.6 against 85.7 us, 1536 x 2048 x
    // 2048 212.6 against 212.7 us, 2048^3 276.1 against 274.1 us).
    const bool kmajor = p.N >= 2048 && (double)p.M * (double)p.N * (double)p.K >= 6.0e9;
    // With A k-major, the 128 x 128 tiles keep up with the 128 x 256 ones
    // and even out the last waves better while the 128 x 256 grid spans
    // under three waves (same-box A/B, 128 x 128 against 128 x 256:
    // 4097 x 3001 x 2049 789.0 against 798.1 us, 3072^3 849.7 against 854.1
    // us, 4096^3 (3.4 waves) 1975.1 against 1975.9 us, 6144^3 (7.6 waves)
    // 6586.5 against 6578.8 us).
    if (kmajor && tiles256 >= p.num_sms && tiles256 < 3 * (int64_t)p.num_sms) return kCfgFfma2_128x128_ka;
    if (tiles256 >= p.num_sms) return kmajor ? kCfgFfma2_128x256_ka : kCfgFfma2_128x256;
    // The 128x128 block's k-major twin by the same rule (8x8 loop alone 89.5 %
    // against 86.0 %; same-box sweep: 2048^3 78.3 % against 77.3 %, 2048 x
    // 2048 x 8192 84.0 % against 81.0 %, but 1024^3 50.7 % against 54.2 %).
    if (3 * tiles128 >= p.num_sms) return kmajor ? kCfgFfma2_128x128_ka : kCfgFfma2_128x128;
    return kCfgFfma2_128x64;
}

int64_t row_tail_rows(int cfg, int64_t M, int64_t N, int64_t K, int64_t batch)
{
    if (cfg < 0 || cfg >= kNumConfigs || !kConfigTable[cfg].packs || batch < 1 || batch > 65535) return 0;
    const int64_t bm = kConfigTable[cfg].bm, bn = kConfigTable[cfg].bn;
    const int64_t r = M % bm;
    if (r < 1 || r > kRowTailMax || M <= bm) return 0;
    // The padded block row costs round_up(N, bn) * bm * K FMAs of the tiled
    // product; from about 2.7e8 of them (some 7 us) the tail kernel, which
    // streams B once in a few microseconds, is the cheaper way.
    if ((double)((N + bn - 1) / bn * bn) * (double)K < 2097152.0) return 0;
    return r;
}

size_t config_workspace_bytes(int cfg, const GemmArgs &g)
{
    if (cfg < 0 || cfg >= kNumConfigs || !kConfigTable[cfg].uses_tma) return 0;
    if (kConfigTable[cfg].kernel >= kKernTf32x3_128x256) {
        GemmArgs a = g;
        a.sched = kConfigTable[cfg].sched;
        return tf32x3_workspace_bytes(kConfigTable[cfg].kernel, a);
    }
    GemmArgs a = g;
    a.sched = kConfigTable[cfg].sched;
    return ffma_tma_workspace_bytes(kConfigTable[cfg].kernel, a);
}

size_t config_counter_bytes(int cfg, const GemmArgs &g)
{
    if (cfg < 0 || cfg >= kNumConfigs || !kConfigTable[cfg].packs) return 0;
    GemmArgs a = g;
    if (a.sched != kSchedDataParallel) a.sched = kConfigTable[cfg].sched;
    return ffma_tma_counter_bytes(kConfigTable[cfg].kernel, a);
}

cudaError_t launch_config(int cfg, const GemmArgs &g, cudaStream_t stream)
{
    const int kernel = kConfigTable[cfg].kernel;
    if (kernel == kKernTiledSimple) return launch_tiled_simple(g, stream);
    if (kernel == kKernSmall32) return launch_small(g, stream);
    if (kernel >= kKernTf32x3_128x256) {
        GemmArgs a = g;
        if (a.sched != kSchedDataParallel) a.sched = kConfigTable[cfg].sched;
        return launch_tf32x3(kernel, a, stream);
    }
    if (kernel >= kKernLadderNaive) return launch_ladder(kernel, g, stream);
    GemmArgs a = g;
    if (a.sched != kSchedDataParallel) a.sched = kConfigTable[cfg].sched;
    return launch_ffma_tma(kConfigTable[cfg].kernel, a, stream);
}

cudaError_t configs_prepare_device()
{
    cudaError_t e = prepare_ffma_tma();
    if (e == cudaSuccess) e = prepare_tf32x3();
    return e != cudaSuccess ? e : prepare_small();
}

}  // namespace sgemm_gb300
