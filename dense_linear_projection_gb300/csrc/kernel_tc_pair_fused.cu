// The tensor-core kernel for CTA-pair plans with the fused epilogue
// (proj_run_fused): activation, residual, SwiGLU.
#include "proj_kernel.cuh"
#include "proj_launch.h"

namespace projgb {

cudaError_t tc_configure_pair_fused(int smem_optin) {
    return cudaFuncSetAttribute(dev::proj_tc_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_optin);
}

cudaError_t tc_launch_pair_fused(const cudaLaunchConfig_t *cfg, const KernelParams &p, const CUtensorMap &map_w,
                                 const CUtensorMap &map_x) {
    return cudaLaunchKernelEx(cfg, dev::proj_tc_kernel<true, true>, p, map_w, map_x);
}

}  // namespace projgb
