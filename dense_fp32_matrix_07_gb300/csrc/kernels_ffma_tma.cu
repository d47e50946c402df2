// Instantiations of the main SGEMM kernel (ffma_tma.cuh) for K a multiple
// of the slab depth, the per-device set-up of all FFMA TMA kernels, their
// workspace sizes and the dispatch by kernel id.
#include "ffma_tma.cuh"

namespace sgemm_gb300 {

cudaError_t prepare_ffma_tma()
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    cudaError_t e = get_encoder(&encode);
    if (e != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma128x128k32s4, false>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x128k32s4, false>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x128k16s8, false>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x64k32s4, false>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x256k32s4ka, false>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x128k32s4ka, false>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x256k32s4, false>()) != cudaSuccess) return e;
    if ((e = prepare_ffma_tma_ktail()) != cudaSuccess) return e;
    return prepare_ffma_tma_dep();
}

size_t ffma_tma_workspace_bytes(int kernel, const GemmArgs &g)
{
    switch (kernel) {
    case kKernFfma128x128k32s4: return workspace_bytes<CfgFfma128x128k32s4>(make_schedule<CfgFfma128x128k32s4>(g, true));
    case kKernFfma2_128x128k32s4: return workspace_bytes<CfgFfma2_128x128k32s4>(make_schedule<CfgFfma2_128x128k32s4>(g, true));
    case kKernFfma2_128x128k16s8: return workspace_bytes<CfgFfma2_128x128k16s8>(make_schedule<CfgFfma2_128x128k16s8>(g, true));
    case kKernFfma2_128x64k32s4: return workspace_bytes<CfgFfma2_128x64k32s4>(make_schedule<CfgFfma2_128x64k32s4>(g, true));
    case kKernFfma2_128x256k32s4: return workspace_bytes<CfgFfma2_128x256k32s4>(make_schedule<CfgFfma2_128x256k32s4>(g, true));
    case kKernFfma2_128x256k32s4ka: return workspace_bytes<CfgFfma2_128x256k32s4ka>(make_schedule<CfgFfma2_128x256k32s4ka>(g, true));
    case kKernFfma2_128x128k32s4ka: return workspace_bytes<CfgFfma2_128x128k32s4ka>(make_schedule<CfgFfma2_128x128k32s4ka>(g, true));
    default: return 0;
    }
}

size_t ffma_tma_counter_bytes(int kernel, const GemmArgs &g)
{
    switch (kernel) {
    case kKernFfma128x128k32s4: return counter_bytes<CfgFfma128x128k32s4>(g);
    case kKernFfma2_128x128k32s4: return counter_bytes<CfgFfma2_128x128k32s4>(g);
    case kKernFfma2_128x128k16s8: return counter_bytes<CfgFfma2_128x128k16s8>(g);
    case kKernFfma2_128x64k32s4: return counter_bytes<CfgFfma2_128x64k32s4>(g);
    case kKernFfma2_128x256k32s4: return counter_bytes<CfgFfma2_128x256k32s4>(g);
    case kKernFfma2_128x256k32s4ka: return counter_bytes<CfgFfma2_128x256k32s4ka>(g);
    case kKernFfma2_128x128k32s4ka: return counter_bytes<CfgFfma2_128x128k32s4ka>(g);
    default: return 0;
    }
}

cudaError_t launch_ffma_tma(int kernel, const GemmArgs &g, cudaStream_t stream)
{
    // B arrives K x N (transposed ones packed); A arrives M x K, except for
    // the k-major configurations, which take it K x M (op_a 1).
    const int want_op_a = (kernel == kKernFfma2_128x256k32s4ka || kernel == kKernFfma2_128x128k32s4ka) ? 1 : 0;
    if (g.op_a != want_op_a || g.op_b != 0) return cudaErrorInvalidValue;
    // A K that is not a multiple of BK runs the kernels that trim the last
    // slab (kernels_ffma_tma_ktail.cu) when that slab holds at most 3/8 of
    // BK valid k; every configuration has BK 32 or 16. The trimmed slab is
    // multiplied one k at a time, so past that point the whole zero-filled
    // slab of the main loop is the faster one (same-box sweep, trimmed
    // against whole, k_last 4 / 12 / 20 of 32: 4096 x 4096 x 2048+k_last
    // 1009.6 / 1013.7 / 1017.2 against 1013.2 us, 4096 x 3001 x 2048+k_last
    // 777.3 / 780.3 / 783.5 against 780.5 us, 4096 x 1536 x 1024+k_last on
    // the row-major 128 x 256 tiles 216.6 / 216.9 / 218.6 against 218.6 us).
    const int bk = kernel == kKernFfma2_128x128k16s8 ? 16 : 32;
    const int k_last = (int)(g.K % bk);
    if (k_last != 0 && 8 * k_last <= 3 * bk) return launch_ffma_tma_ktail(kernel, g, stream);
    // Behind the call's layout pass, the instances that may start while it
    // finishes (kernels_ffma_tma_dep.cu).
    if (g.behind_pack) return launch_ffma_tma_dep(kernel, g, stream);
    switch (kernel) {
    case kKernFfma128x128k32s4: return launch<CfgFfma128x128k32s4, false>(g, stream);
    case kKernFfma2_128x128k32s4: return launch<CfgFfma2_128x128k32s4, false>(g, stream);
    case kKernFfma2_128x128k16s8: return launch<CfgFfma2_128x128k16s8, false>(g, stream);
    case kKernFfma2_128x64k32s4: return launch<CfgFfma2_128x64k32s4, false>(g, stream);
    case kKernFfma2_128x256k32s4: return launch<CfgFfma2_128x256k32s4, false>(g, stream);
    case kKernFfma2_128x256k32s4ka: return launch<CfgFfma2_128x256k32s4ka, false>(g, stream);
    case kKernFfma2_128x128k32s4ka: return launch<CfgFfma2_128x128k32s4ka, false>(g, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace sgemm_gb300
