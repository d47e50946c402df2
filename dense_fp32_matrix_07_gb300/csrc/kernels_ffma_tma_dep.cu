// Instances of the main SGEMM kernel (ffma_tma.cuh) launched right behind
// the call's layout pass (the transposed or packed operands and the zeroed
// stream-K counters) with programmatic stream serialization: their CTAs may
// take SMs and set up their barriers while the pass's last blocks run, and
// every thread waits for the pass to complete before it touches global
// memory. Kernels that trim a K tail are launched behind the pass in the
// ordinary way: with the wait compiled in, the 128 x 128 k-major one ran
// 4097 x 3001 x 2049 in 784.1 us against 780.4 us without it (same-box A/B),
// more than the early start gains. A separate translation unit, so these
// kernels compile in parallel with the others.
#include "ffma_tma.cuh"

namespace sgemm_gb300 {

cudaError_t prepare_ffma_tma_dep()
{
    cudaError_t e;
    if ((e = set_smem_limit<CfgFfma128x128k32s4, false, true>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x128k32s4, false, true>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x128k16s8, false, true>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x64k32s4, false, true>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x256k32s4ka, false, true>()) != cudaSuccess) return e;
    if ((e = set_smem_limit<CfgFfma2_128x128k32s4ka, false, true>()) != cudaSuccess) return e;
    return set_smem_limit<CfgFfma2_128x256k32s4, false, true>();
}

cudaError_t launch_ffma_tma_dep(int kernel, const GemmArgs &g, cudaStream_t stream)
{
    switch (kernel) {
    case kKernFfma128x128k32s4: return launch<CfgFfma128x128k32s4, false, true>(g, stream);
    case kKernFfma2_128x128k32s4: return launch<CfgFfma2_128x128k32s4, false, true>(g, stream);
    case kKernFfma2_128x128k16s8: return launch<CfgFfma2_128x128k16s8, false, true>(g, stream);
    case kKernFfma2_128x64k32s4: return launch<CfgFfma2_128x64k32s4, false, true>(g, stream);
    case kKernFfma2_128x256k32s4: return launch<CfgFfma2_128x256k32s4, false, true>(g, stream);
    case kKernFfma2_128x256k32s4ka: return launch<CfgFfma2_128x256k32s4ka, false, true>(g, stream);
    case kKernFfma2_128x128k32s4ka: return launch<CfgFfma2_128x128k32s4ka, false, true>(g, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace sgemm_gb300
