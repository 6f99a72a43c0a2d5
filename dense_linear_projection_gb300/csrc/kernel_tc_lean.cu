// The tensor-core kernel without a fused epilogue (every ordinary run).
#include "proj_kernel.cuh"
#include "proj_launch.h"

namespace projgb {

cudaError_t tc_configure_lean(int smem_optin) {
    cudaError_t e = cudaFuncSetAttribute(dev::proj_tc_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_optin);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(dev::proj_tc_kernel<false, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

cudaError_t tc_max_active_clusters(int *clusters, const cudaLaunchConfig_t *cfg) {
    return cudaOccupancyMaxActiveClusters(clusters, dev::proj_tc_kernel<false, false>, cfg);
}

cudaError_t tc_launch_lean(const cudaLaunchConfig_t *cfg, const KernelParams &p, const CUtensorMap &map_w,
                           const CUtensorMap &map_x) {
    return cudaLaunchKernelEx(cfg, dev::proj_tc_kernel<false, false>, p, map_w, map_x);
}

}  // namespace projgb
