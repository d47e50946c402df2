// Instantiations of the main SGEMM kernel (ffma_tma.cuh) that trim the last
// K slab: for a K that is not a multiple of the slab depth, the last slab of
// every tile multiplies only its k_last valid k instead of a whole slab of
// zero-filled padding. launch_ffma_tma() takes them when k_last is at most
// 3/8 of the slab depth. A separate translation unit, so these kernels
// compile in parallel with the others.
#include "ffma_tma.cuh"

namespace sgemm_gb300 {

cudaError_t prepare_ffma_tma_ktail()
{
    cudaError_t e;
    if ((e = set_smem_limit<CfgFfma128x128k32s4, true>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x128k32s4, true>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x128k16s8, true>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x64k32s4, true>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x256k32s4ka, true>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x128k32s4ka, true>()) != cudaSuccess) return e;
    return set_smem_limit<CfgFfma2_128x256k32s4, true>();
}

cudaError_t launch_ffma_tma_ktail(int kernel, const GemmArgs &g, cudaStream_t stream)
{
    switch (kernel) {
    case kKernFfma128x128k32s4: return launch<CfgFfma128x128k32s4, true>(g, stream);
    case kKernFfma2_128x128k32s4: return launch<CfgFfma2_128x128k32s4, true>(g, stream);
    case kKernFfma2_128x128k16s8: return launch<CfgFfma2_128x128k16s8, true>(g, stream);
    case kKernFfma2_128x64k32s4: return launch<CfgFfma2_128x64k32s4, true>(g, stream);
    case kKernFfma2_128x256k32s4: return launch<CfgFfma2_128x256k32s4, true>(g, stream);
    case kKernFfma2_128x256k32s4ka: return launch<CfgFfma2_128x256k32s4ka, true>(g, stream);
    case kKernFfma2_128x128k32s4ka: return launch<CfgFfma2_128x128k32s4ka, true>(g, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace sgemm_gb300
