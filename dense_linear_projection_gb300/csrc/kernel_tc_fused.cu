// The tensor-core kernel with the fused epilogue (proj_run_fused): activation
// on the projection plus bias, then the residual, before the one rounding.
#include "proj_kernel.cuh"
#include "proj_launch.h"

namespace projgb {

cudaError_t tc_configure_fused(int smem_optin) {
    cudaError_t e = cudaFuncSetAttribute(dev::proj_tc_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_optin);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(dev::proj_tc_kernel<true, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

cudaError_t tc_launch_fused(const cudaLaunchConfig_t *cfg, const KernelParams &p, const CUtensorMap &map_w,
                            const CUtensorMap &map_x) {
    return cudaLaunchKernelEx(cfg, dev::proj_tc_kernel<true, false>, p, map_w, map_x);
}

}  // namespace projgb
