// Configuration table and selector (host logic only).
#include "configs.cuh"

namespace sgemm_gb300 {

const ConfigInfo kConfigTable[kNumConfigs] = {
    {"tiled16_simple", false, 16, 16},
    {"ffma_128x128_k32_s4", true, 128, 128},
    {"ffma2_128x128_k32_s4", true, 128, 128},
    {"ffma2_128x128_k16_s8", true, 128, 128},
    {"ffma2_128x64_k32_s4", true, 128, 64},
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
    // Work per SM decides between the two block shapes: when 128x128 tiles
    // would leave SMs idle, the half-width tile doubles the CTA count.
    const int64_t tiles128 = ((p.M + 127) / 128) * ((p.N + 127) / 128);
    if (!config_supports(kCfgFfma2_128x128k32s4, p)) return kCfgTiledSimple;
    if (tiles128 < p.num_sms) return kCfgFfma2_128x64k32s4;
    return kCfgFfma2_128x128k32s4;
}

cudaError_t launch_config(int cfg, const GemmArgs &g, cudaStream_t stream)
{
    if (cfg == kCfgTiledSimple) return launch_tiled_simple(g, stream);
    return launch_ffma_tma(cfg, g, stream);
}

cudaError_t configs_prepare_device() { return prepare_ffma_tma(); }

}  // namespace sgemm_gb300
