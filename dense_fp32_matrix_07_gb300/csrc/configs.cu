// Configuration table and selector (host logic only).
#include "configs.cuh"

namespace sgemm_gb300 {

const ConfigInfo kConfigTable[kNumConfigs] = {
    {"tiled16_simple", kKernTiledSimple, kSchedDataParallel, false, 16, 16},
    {"ffma_128x128_k32_s4", kKernFfma128x128k32s4, kSchedAuto, true, 128, 128},
    {"ffma2_128x128_k32_s4", kKernFfma2_128x128k32s4, kSchedAuto, true, 128, 128},
    {"ffma2_128x128_k16_s8", kKernFfma2_128x128k16s8, kSchedAuto, true, 128, 128},
    {"ffma2_128x64_k32_s4", kKernFfma2_128x64k32s4, kSchedAuto, true, 128, 64},
    {"ffma2_128x256_k32_s4", kKernFfma2_128x256k32s4, kSchedAuto, true, 128, 256},
    {"ffma2_128x128_k32_s4_dp", kKernFfma2_128x128k32s4, kSchedDataParallel, true, 128, 128},
    {"ffma2_128x128_k32_s4_sk", kKernFfma2_128x128k32s4, kSchedStreamK, true, 128, 128},
    {"ffma2_128x256_k32_s4_dp", kKernFfma2_128x256k32s4, kSchedDataParallel, true, 128, 256},
    {"ffma2_128x256_k32_s4_sk", kKernFfma2_128x256k32s4, kSchedStreamK, true, 128, 256},
};

bool config_supports(int cfg, const ProblemShape &p)
{
    if (cfg < 0 || cfg >= kNumConfigs) return false;
    if (!kConfigTable[cfg].uses_tma) return true;
    // TMA sizes are 32-bit coordinates; strides of packed operands are at
    // most (kMaxDim rounded up) * 4 bytes, within the 2^40-byte stride limit.
    return p.M <= kMaxDim && p.N <= kMaxDim && p.K <= kMaxDim &&
           p.lda < (int64_t(1) << 37) && p.ldb < (int64_t(1) << 37);
}

int select_config(const ProblemShape &p)
{
    if (!config_supports(kCfgFfma2_128x128, p)) return kCfgTiledSimple;
    // The widest thread tile (8x16) when there are enough 128x256 tiles to
    // give every SM one; below that, 128x128, and 128x64 (two CTAs per SM)
    // when even 128x128 tiles cannot fill the SMs. The stream-K tail evens
    // out partial last waves in all three.
    const int64_t tiles256 = ((p.M + 127) / 128) * ((p.N + 255) / 256);
    const int64_t tiles128 = ((p.M + 127) / 128) * ((p.N + 127) / 128);
    if (tiles256 >= p.num_sms) return kCfgFfma2_128x256;
    if (tiles128 >= p.num_sms) return kCfgFfma2_128x128;
    return kCfgFfma2_128x64;
}

size_t config_workspace_bytes(int cfg, const GemmArgs &g)
{
    if (cfg < 0 || cfg >= kNumConfigs || !kConfigTable[cfg].uses_tma) return 0;
    GemmArgs a = g;
    a.sched = kConfigTable[cfg].sched;
    return ffma_tma_workspace_bytes(kConfigTable[cfg].kernel, a);
}

cudaError_t launch_config(int cfg, const GemmArgs &g, cudaStream_t stream)
{
    if (kConfigTable[cfg].kernel == kKernTiledSimple) return launch_tiled_simple(g, stream);
    GemmArgs a = g;
    if (a.sched != kSchedDataParallel) a.sched = kConfigTable[cfg].sched;
    return launch_ffma_tma(kConfigTable[cfg].kernel, a, stream);
}

cudaError_t configs_prepare_device() { return prepare_ffma_tma(); }

}  // namespace sgemm_gb300
