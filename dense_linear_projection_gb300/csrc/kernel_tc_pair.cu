// The tensor-core kernel for CTA-pair plans (cta_group::2 MMAs over a
// cluster of 2), without a fused epilogue.
#include "proj_kernel.cuh"
#include "proj_launch.h"

namespace projgb {

cudaError_t tc_configure_pair(int smem_optin) {
    return cudaFuncSetAttribute(dev::proj_tc_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_optin);
}

cudaError_t tc_launch_pair(const cudaLaunchConfig_t *cfg, const KernelParams &p, const CUtensorMap &map_w,
                           const CUtensorMap &map_x) {
    return cudaLaunchKernelEx(cfg, dev::proj_tc_kernel<false, true>, p, map_w, map_x);
}

}  // namespace projgb
