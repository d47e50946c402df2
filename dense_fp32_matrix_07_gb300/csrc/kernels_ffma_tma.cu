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
    // slab (kernels_ffma_tma_ktail.cu); every configuration has BK 32 or 16.
    const int bk = kernel == kKernFfma2_128x128k16s8 ? 16 : 32;
    if (g.K % bk != 0) return launch_ffma_tma_ktail(kernel, g, stream);
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
