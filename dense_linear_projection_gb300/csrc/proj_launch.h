// Host entry points of the tensor-core kernel.  The kernel is built four
// times, each in its own translation unit: a lean instance (no fused
// epilogue) for ordinary runs and a fused instance (activation and residual)
// for proj_run_fused, each for single CTAs and for CTA pairs (every tcgen05
// instruction of a kernel names one CTA group).  Keeping the fused code out
// of the lean instances keeps the default path's code small.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "proj_internal.h"

namespace projgb {

// Kernel attributes: the device's opt-in shared memory and cluster sizes
// above the portable 8.
cudaError_t tc_configure_lean(int smem_optin);
cudaError_t tc_configure_fused(int smem_optin);
// Clusters of the configuration's shape that can be resident at once.
cudaError_t tc_max_active_clusters(int *clusters, const cudaLaunchConfig_t *cfg);
cudaError_t tc_launch_lean(const cudaLaunchConfig_t *cfg, const KernelParams &p, const CUtensorMap &map_w,
                           const CUtensorMap &map_x);
cudaError_t tc_launch_fused(const cudaLaunchConfig_t *cfg, const KernelParams &p, const CUtensorMap &map_w,
                            const CUtensorMap &map_x);
cudaError_t tc_configure_pair(int smem_optin);
cudaError_t tc_configure_pair_fused(int smem_optin);
cudaError_t tc_launch_pair(const cudaLaunchConfig_t *cfg, const KernelParams &p, const CUtensorMap &map_w,
                           const CUtensorMap &map_x);
cudaError_t tc_launch_pair_fused(const cudaLaunchConfig_t *cfg, const KernelParams &p, const CUtensorMap &map_w,
                                 const CUtensorMap &map_x);

}  // namespace projgb
