// Kernel configurations, the selector that picks one per problem, and the
// dispatch to their launchers.
#pragma once

#include "common.cuh"

namespace sgemm_gb300 {

// Largest M, N or K: TMA coordinates are signed 32-bit.
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

// What the selector looks at (no pointers are dereferenced).
struct ProblemShape {
    int64_t M, N, K, lda, ldb, ldc;
    uint64_t a, b, c;   // operand addresses (alignment only)
    int num_sms;
};

enum ConfigId : int {
    kCfgTiledSimple = 0,       // predicated 16x16 shared-memory tiles, any layout
    kCfgFfma128x128k32s4,      // TMA ring, 128x128 block, BK 32, 4 stages, FFMA
    kCfgFfma2_128x128k32s4,    // same, paired FFMA2
    kCfgFfma2_128x128k16s8,    // 128x128 block, BK 16, 8 stages, FFMA2
    kCfgFfma2_128x64k32s4,     // 128x64 block (4 consumer warps), BK 32, 4 stages, 2 CTAs per SM
    kNumConfigs
};

struct ConfigInfo {
    const char *name;
    bool uses_tma;   // reads A and B through TMA tensor maps
    int bm, bn;      // block tile (0 for the simple kernel's 16x16)
};

extern const ConfigInfo kConfigTable[kNumConfigs];

// Host-only selection (also used by sgemm_plan(), which needs no GPU).
int select_config(const ProblemShape &p);
bool config_supports(int cfg, const ProblemShape &p);

// Runs configuration `cfg` on operands that already satisfy its alignment
// needs (the API packs misaligned operands for TMA configurations first).
cudaError_t launch_config(int cfg, const GemmArgs &g, cudaStream_t stream);

// One-time per-device set-up (shared-memory limits of the kernels, the
// tensor-map encoder); call with the device current.
cudaError_t configs_prepare_device();

// Launchers of the TMA kernels (kernels_ffma_tma.cu).
cudaError_t launch_ffma_tma(int cfg, const GemmArgs &g, cudaStream_t stream);
cudaError_t prepare_ffma_tma();

}  // namespace sgemm_gb300
