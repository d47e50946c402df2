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

// Kernel instances.
enum KernelId : int {
    kKernTiledSimple = 0,       // predicated 16x16 shared-memory tiles, any layout
    kKernFfma128x128k32s4,      // TMA ring, 128x128 block, BK 32, 4 stages, FFMA
    kKernFfma2_128x128k32s4,    // same, paired FFMA2
    kKernFfma2_128x128k16s8,    // 128x128 block, BK 16, 8 stages, FFMA2
    kKernFfma2_128x64k32s4,     // 128x64 block (4 consumer warps), 2 CTAs per SM
    kKernFfma2_128x256k32s4,    // 128x256 block, 8x16 thread tiles, FFMA2
    kKernFfma2_128x256k32s4ka,  // the same with A stored K x M (k-major slabs)
    kKernFfma2_128x128k32s4ka,  // the 128x128 FFMA2 block with A stored K x M
    // The pages' kernel ladder (kernels_ladder.cu), for measurement.
    kKernLadderNaive,           // one thread per output, threadIdx.x -> row
    kKernLadderCoalesced,       // one thread per output, threadIdx.x -> column
    kKernLadderCacheBlocked8x8, // 8x8 register micro-tiles, caches only
    kKernLadderRegisterTiled2x2, // 16x16 padded smem tiles, 2x2 per thread
    // Tensor cores (kernels_tf32x3.cu): 3xTF32 split, tcgen05.mma into TMEM.
    kKernTf32x3_128x256,
    kKernTf32x3_128x128,
    kKernTf32x3_pair,           // 128x256 per CTA, clusters of 2 along M multicasting B
    // Small products (kernels_small.cu): 32x32 tiles, the K panel loaded at once.
    kKernSmall32
};

// Configurations = kernel instance + schedule policy.
enum ConfigId : int {
    kCfgTiledSimple = 0,
    kCfgFfma128x128,
    kCfgFfma2_128x128,
    kCfgFfma2_128x128k16,
    kCfgFfma2_128x64,
    kCfgFfma2_128x256,
    kCfgFfma2_128x128_dp,
    kCfgFfma2_128x128_sk,
    kCfgFfma2_128x256_dp,
    kCfgFfma2_128x256_sk,
    kCfgLadderNaive,
    kCfgLadderCoalesced,
    kCfgLadderCacheBlocked8x8,
    kCfgLadderRegisterTiled2x2,
    kCfgTf32x3_128x256,
    kCfgTf32x3_128x256_sk,
    kCfgTf32x3_128x256_auto,
    kCfgTf32x3_128x128,
    kCfgTf32x3_128x256_dp,
    kCfgTf32x3_pair,
    kCfgTf32x3_pair_dp,
    kCfgFfma2_128x256_ka,
    kCfgFfma2_128x128_ka,
    kCfgSmall32,
    kNumConfigs
};

struct ConfigInfo {
    const char *name;
    int kernel;      // KernelId
    int sched;       // SchedPolicy
    bool uses_tma;   // TMA tensor maps (32-bit coordinates)
    bool packs;      // needs A and B with 16-byte-aligned rows (packs others)
    int bm, bn;      // block tile
    bool a_kmajor = false;   // takes A stored K x M (transposes a plain A into scratch)
};

extern const ConfigInfo kConfigTable[kNumConfigs];

// Host-only selection (also used by sgemm_plan(), which needs no GPU).
int select_config(const ProblemShape &p);
bool config_supports(int cfg, const ProblemShape &p);

// Workspace bytes configuration `cfg` wants for this product (0: none).
size_t config_workspace_bytes(int cfg, const GemmArgs &g);
// For an FFMA TMA configuration given g.workspace_bytes: the bytes at the
// start of the workspace that must be zero when the product starts (0: none).
size_t config_counter_bytes(int cfg, const GemmArgs &g);

// Runs configuration `cfg` on operands that already satisfy its alignment
// needs (the API packs misaligned operands for TMA configurations first).
// g.sched is overwritten with the configuration's policy unless it is
// kSchedDataParallel; without g.workspace the schedule is whole tiles.
cudaError_t launch_config(int cfg, const GemmArgs &g, cudaStream_t stream);

// One-time per-device set-up (shared-memory limits of the kernels, the
// tensor-map encoder); call with the device current.
cudaError_t configs_prepare_device();

// Launchers of the TMA kernels (kernels_ffma_tma.cu), by KernelId.
cudaError_t launch_ffma_tma(int kernel, const GemmArgs &g, cudaStream_t stream);
size_t ffma_tma_workspace_bytes(int kernel, const GemmArgs &g);
size_t ffma_tma_counter_bytes(int kernel, const GemmArgs &g);
cudaError_t prepare_ffma_tma();
// The same kernels trimming the last K slab, for K not a multiple of the
// slab depth (kernels_ffma_tma_ktail.cu); launch_ffma_tma() dispatches there.
cudaError_t launch_ffma_tma_ktail(int kernel, const GemmArgs &g, cudaStream_t stream);
cudaError_t prepare_ffma_tma_ktail();
// The same kernels (K a multiple of the slab depth) launched behind the
// call's layout pass with programmatic serialization
// (kernels_ffma_tma_dep.cu); launch_ffma_tma() dispatches there when
// g.behind_pack is set.
cudaError_t launch_ffma_tma_dep(int kernel, const GemmArgs &g, cudaStream_t stream);
cudaError_t prepare_ffma_tma_dep();

// The small-product kernel (kernels_small.cu), plain form only, any layout.
cudaError_t launch_small(const GemmArgs &g, cudaStream_t stream);
cudaError_t prepare_small();

// Launcher of the ladder kernels (kernels_ladder.cu), by KernelId.
cudaError_t launch_ladder(int kernel, const GemmArgs &g, cudaStream_t stream);

// The last r <= kRowTailMax rows of C of a product whose tiled part covers
// rows 0 .. m0 - 1 (kernels_row_tail.cu): C_b[m0 + i][j] = alpha * sum_k
// op(A_b)[m0 + i][k] * B_b[k][j] (+ beta * C_b[m0 + i][j] when beta != 0).
constexpr int kRowTailMax = 8;
struct RowTailArgs {
    const float *A;      // op(A_b)[m][k] at A + b * stride_a + m * a_row_stride + k * a_k_stride
    int64_t a_row_stride, a_k_stride, stride_a;
    const float *B;      // B_b: K x N row-major, ldb, rows 16-byte aligned (the TMA path's B)
    int64_t ldb, stride_b;
    float *C;
    int64_t ldc, stride_c;
    int64_t m0;          // first row of the tail
    int r;               // rows, 1 .. kRowTailMax
    int64_t N, K, batch;
    float alpha, beta;
    // With more than one K chunk per column block (row_tail_splits() > 1):
    // the arrival counters (zero at launch, row_tail_counter_bytes()) and the
    // chunk sums (row_tail_slot_bytes()).
    unsigned int *counters;
    float *slots;
};
cudaError_t launch_row_tail(const RowTailArgs &t, int num_sms, cudaStream_t stream);
// K chunks per column block of the row-tail kernel, and the bytes of its
// counters (a multiple of 256) and chunk sums; both 0 with one chunk.
int row_tail_splits(int64_t r, int64_t N, int64_t K, int64_t batch, int num_sms);
size_t row_tail_counter_bytes(int64_t r, int64_t N, int64_t K, int64_t batch, int num_sms);
size_t row_tail_slot_bytes(int64_t r, int64_t N, int64_t K, int64_t batch, int num_sms);

// Rows that a call with this configuration leaves to the row-tail kernel:
// M = 128 q + r with 1 <= r <= kRowTailMax on a TMA FFMA configuration, when
// the block row of tiles those rows would pad is worth more than the tail
// kernel's fixed cost (round_up(N, BN) * K >= 2^21); else 0.
int64_t row_tail_rows(int cfg, int64_t M, int64_t N, int64_t K, int64_t batch);

// The 3xTF32 tensor-core path (kernels_tf32x3.cu): split pre-passes into
// g.workspace, then the tcgen05 product.
cudaError_t launch_tf32x3(int kernel, const GemmArgs &g, cudaStream_t stream);
size_t tf32x3_workspace_bytes(int kernel, const GemmArgs &g);
cudaError_t prepare_tf32x3();

}  // namespace sgemm_gb300
