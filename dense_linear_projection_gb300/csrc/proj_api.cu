// C ABI of the GB300 dense projection library: handle lifecycle, argument
// checks, TMA descriptor encoding and kernel launches.  See include/proj.h for
// the contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "proj.h"
#include "proj_aux.cuh"
#include "proj_internal.h"
#include "proj_launch.h"

using namespace projgb;

struct proj_plan_s {
    int device = 0;
    int64_t M = 0, N = 0, K = 0;
    int w_layout = PROJ_W_NK;
    int y_dtype = PROJ_BF16;
    int has_bias = 0;
    proj_plan_desc_t plan{};
    KernelParams params{};
    // Weights stored [K,N] load along N in 64-column boxes.  When the plan's
    // CTA pairs hold weight halves of another width, runs on weights as
    // stored (not packed) use this single-CTA plan instead.
    bool has_plan_stored = false;
    proj_plan_desc_t plan_stored{};
    KernelParams params_stored{};
    void *scratch = nullptr;
    int64_t scratch_bytes = 0;       // allocated
    int64_t scratch_clear_from = 0;  // counters and status word: [clear_from, scratch_bytes)
    // Tensor maps cached by base pointer and box rows (rebuilt when X or W
    // moves or another plan runs).
    const void *map_x_ptr = nullptr;
    const void *map_w_ptr = nullptr;
    const void *map_wp_ptr = nullptr;  // packed weights
    int32_t map_x_box = 0, map_w_box = 0;
    int32_t map_x_kpb = 0, map_x_3d = 0;  // k-blocks per stage the X map was built for; 3-D or not
    CUtensorMap map_x;  // CUtensorMap carries its own 64-byte alignment
    CUtensorMap map_w;
    CUtensorMap map_wp;
    unsigned long long *trace = nullptr;  // caller's phase-trace buffer, if any
    int overlap = PROJ_OVERLAP_PROLOGUE;    // programmatic dependent launch mode
    int prefetch_stages = kMaxStages;       // PROJ_OVERLAP_WEIGHTS: W stages before the wait
    bool prefetch_any = false;              // PROJ_PREFETCH_ANY=1: also plans that leave SMs idle
    int sm_count = 0;
    int act = 0;  // fused activation (proj_set_activation)
    // fp32 router weights: planned and run as [H | L] along K (2·kt k-blocks);
    // they exist only in packed form (the split happens in proj_pack_weights).
    int hilo = 0;
    int64_t kt = 0;  // k-blocks of K
    // Device staging for proj_run_host (allocated on first use).
    void *stage_x = nullptr;
    void *stage_y = nullptr;
};

namespace {

constexpr int64_t kDefaultWaitLimitNs = 1000000000LL;  // 1 s

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

// Host-side fault injection for tests (PROJ_FAULT, read once per process): a
// comma-separated list of "alloc" (every device allocation of the library
// fails as out of memory), "encode" (every tensor-map encoding fails) and
// "launch" (every kernel launch fails before it is queued).  The failure is
// made on the host: nothing faulty reaches the device.
constexpr int kFaultAlloc = 1, kFaultEncode = 2, kFaultLaunch = 4;

int fault_mask() {
    static const int mask = [] {
        int m = 0;
        if (const char *e = std::getenv("PROJ_FAULT")) {
            if (std::strstr(e, "alloc")) m |= kFaultAlloc;
            if (std::strstr(e, "encode")) m |= kFaultEncode;
            if (std::strstr(e, "launch")) m |= kFaultLaunch;
        }
        return m;
    }();
    return mask;
}

bool launch_faulted() { return (fault_mask() & kFaultLaunch) != 0; }

// Every device allocation of the library goes through here.
cudaError_t dev_malloc(void **p, size_t bytes) {
    if (fault_mask() & kFaultAlloc) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(p, bytes);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// 2-D bf16 tensor map: `inner` contiguous elements per row, `outer` rows,
// rows `row_bytes` apart, box [box_inner, box_outer], 128-byte swizzle,
// out-of-range elements read as zero.
bool encode_2d(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t outer, uint64_t row_bytes,
               uint32_t box_inner, uint32_t box_outer) {
    if (fault_mask() & kFaultEncode) return false;
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 tensor map: dims {64, d1, d2} with byte strides s1, s2 for the
// outer two, box {64, b1, b2}, 128-byte swizzle, zero fill outside.
bool encode_3d(CUtensorMap *map, const void *ptr, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
               uint32_t b1, uint32_t b2) {
    if (fault_mask() & kFaultEncode) return false;
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {64, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// X's tensor map for a plan: with two k-blocks a stage (K a multiple of 64),
// a 3-D view {64 K, M rows, K/64 k-blocks} whose box brings a stage's
// k-blocks in one op (*x_3d = 1); otherwise 2-D boxes of one k-block.
bool encode_x(CUtensorMap *map, const void *X, int64_t M, int64_t K, const proj_plan_desc_t &plan, int32_t *x_3d) {
    const int32_t kpb = plan_kpb(plan);
    const uint32_t rows = static_cast<uint32_t>(plan.cta_pair ? plan.block_t / 2 : plan.block_t);
    if (kpb > 1 && K % kBlockK == 0 &&
        encode_3d(map, X, static_cast<uint64_t>(M), static_cast<uint64_t>(K / kBlockK), static_cast<uint64_t>(K) * 2,
                  128, rows, static_cast<uint32_t>(kpb))) {
        *x_3d = 1;
        return true;
    }
    *x_3d = 0;
    return encode_2d(map, X, static_cast<uint64_t>(K), static_cast<uint64_t>(M), static_cast<uint64_t>(K) * 2,
                     kBlockK, rows);
}

// The packed weights' tensor map: planes of block_n rows x 64 K, one per
// (tile, k-block), tiles_n x (k_blocks x kpb) of them; box {64, the rows
// this CTA holds, kpb planes}.  With one k-block a stage, the same memory as
// a 2-D map of 64-wide rows.
bool encode_packed(CUtensorMap *map, const void *Wp, const proj_plan_desc_t &plan) {
    const uint32_t rows = static_cast<uint32_t>(plan.cta_pair ? plan.block_n / 2 : plan.block_n);
    if (plan_kpb(plan) == 1)  // one k-block a stage: a 2-D map of 64-wide rows
        return encode_2d(map, Wp, 64, static_cast<uint64_t>(plan.tiles_n * plan.k_blocks * plan.block_n), 128,
                         kBlockK, rows);
    return encode_3d(map, Wp, static_cast<uint64_t>(plan.block_n),
                     static_cast<uint64_t>(plan.tiles_n * plan_packed_kblocks(plan)), 128,
                     static_cast<uint64_t>(plan.block_n) * 128, rows, static_cast<uint32_t>(plan_kpb(plan)));
}

uint32_t make_idesc(int mma_m, int mma_n, bool a_mn_major, bool b_mn_major) {
    // tcgen05 instruction descriptor, kind::f16: fp32 accumulator (bits 4-5),
    // bf16 A (7-9) and B (10-12), A major-ness (15), B major-ness (16),
    // N >> 3 (17-22), M >> 4 (24-28).
    uint32_t d = 0;
    d |= 1u << 4;
    d |= 1u << 7;
    d |= 1u << 10;
    if (a_mn_major) d |= 1u << 15;
    if (b_mn_major) d |= 1u << 16;
    d |= static_cast<uint32_t>(mma_n >> 3) << 17;
    d |= static_cast<uint32_t>(mma_m >> 4) << 24;
    return d;
}

// Instruction descriptor of a plan: M = 128 (256 for a CTA pair), N = B rows;
// [K,N] weights are MN-major in whichever operand they occupy.
uint32_t idesc_of(const proj_plan_desc_t &plan, int w_layout) {
    const bool kn = w_layout == PROJ_W_KN;
    return make_idesc(plan.cta_pair ? 2 * kBlockA : kBlockA, plan_b_rows(plan), plan.swap_ab && kn,
                      !plan.swap_ab && kn);
}

// Rows of one TMA box of X and of W (a CTA of a pair loads half the tile's).
int32_t x_box_rows(const proj_plan_desc_t &plan) { return plan.cta_pair ? plan.block_t / 2 : plan.block_t; }
int32_t w_box_rows(const proj_plan_desc_t &plan) { return plan.cta_pair ? plan.block_n / 2 : plan.block_n; }

// Whether a plan can load weights stored [K,N]: its weight rows per CTA are
// whole 64-column boxes.
bool loads_stored_kn(const proj_plan_desc_t &plan) { return w_box_rows(plan) % 64 == 0; }

// Bytes of split-K partial tiles in the scratch (the rest is counters and
// the status word).  Cluster-split plans reduce in shared memory: none.
int64_t partial_bytes_of(const proj_plan_desc_t &plan) {
    const int64_t b_rows = plan.swap_ab ? plan.block_t : plan.block_n;
    if (plan.tiles_sk > 0 && plan.cluster_split >= 2 && plan.cluster_groups >= 2)
        return plan.tiles_sk * plan.cluster_groups * kBlockA * b_rows * 4;  // one per (tile, cluster)
    return plan.tiles_sk > 0 && plan.cluster_split < 2 ? int64_t(2) * plan.grid * kBlockA * b_rows * 4 : 0;
}

// The kernel may use up to the device's opt-in shared memory.  The attribute
// belongs to the kernel, not to a handle: every launch fits under it.
bool set_kernel_smem_limit(int smem_optin) {
    // Also allow clusters above the portable 8 CTAs (GB300 runs 16); the
    // occupancy query in plan_for_device decides whether a size fits.
    if (tc_configure_lean(smem_optin) != cudaSuccess || tc_configure_fused(smem_optin) != cudaSuccess ||
        tc_configure_pair(smem_optin) != cudaSuccess || tc_configure_pair_fused(smem_optin) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return true;
}

// Launch configuration of a tensor-core plan: the cluster shape of a
// cluster-split or CTA-pair plan and, unless off, programmatic dependent
// launch.
struct TcLaunch {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[2];
    TcLaunch(const proj_plan_desc_t &plan, cudaStream_t s, bool pdl) {
        cfg.gridDim = dim3(static_cast<unsigned>(plan.grid));
        cfg.blockDim = dim3(static_cast<unsigned>(plan.threads));
        cfg.dynamicSmemBytes = static_cast<size_t>(plan.smem_bytes);
        cfg.stream = s;
        unsigned n = 0;
        if (plan.cluster_split > 1 || plan.cta_pair) {
            attr[n].id = cudaLaunchAttributeClusterDimension;
            attr[n].val.clusterDim.x = static_cast<unsigned>(plan.cta_pair ? 2 : plan.cluster_split);
            attr[n].val.clusterDim.y = 1;
            attr[n].val.clusterDim.z = 1;
            ++n;
        }
        if (pdl) {
            attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[n].val.programmaticStreamSerializationAllowed = 1;
            ++n;
        }
        cfg.attrs = attr;
        cfg.numAttrs = n;
    }
};

// A plan whose cluster split is kept only if every tile's cluster can be
// resident at once (GPCs hold whole clusters, so not every SM count divides
// into clusters); otherwise the split size is lowered, down to the
// global-scratch split-K plans.  Needs the kernel's shared-memory limit set.
proj_status_t plan_fitted(int64_t M, int64_t N, int64_t K, proj_wlayout_t w_layout, proj_dtype_t y_dtype,
                          int has_bias, const proj_device_desc_t &dd, PlanOptions opt, proj_plan_desc_t *plan) {
    while (true) {
        proj_status_t st = plan_compute(M, N, K, w_layout, y_dtype, has_bias, &dd, opt, plan);
        if (st != PROJ_OK || plan->cluster_split < 2) return st;
        TcLaunch l(*plan, nullptr, false);
        int clusters = 0;
        const int64_t need = plan->tiles_sk * (plan->cluster_groups > 1 ? plan->cluster_groups : 1);
        if (tc_max_active_clusters(&clusters, &l.cfg) == cudaSuccess && static_cast<int64_t>(clusters) >= need)
            return PROJ_OK;
        cudaGetLastError();
        if (plan->cluster_groups > 1) {  // first one cluster per tile
            opt.cluster_groups = 1;
            continue;
        }
        opt.max_cluster = plan->cluster_split - 1;
        opt.force_cluster = 0;  // a forced size that does not fit falls back to the rule
        if (opt.max_cluster < 2) opt.max_cluster = 0;
    }
}

// Plan for this device.  With PROJ_TM_CLUSTER=1, for at most 32 tokens, a
// token-major cluster split (256 weight rows per MMA instruction) replaces a
// swapped cluster split when, both fitted to the device, it keeps at least
// 70 % as many SMs (each then streams about 1.4 times as fast).
proj_status_t plan_for_device(int64_t M, int64_t N, int64_t K, proj_wlayout_t w_layout,
                              proj_dtype_t y_dtype, int has_bias, const proj_device_desc_t &dd,
                              PlanOptions opt, proj_plan_desc_t *plan) {
    const int32_t tm = opt.tm_cluster;
    opt.tm_cluster = tm == 2 ? 2 : 0;
    const proj_status_t st = plan_fitted(M, N, K, w_layout, y_dtype, has_bias, dd, opt, plan);
    if (st != PROJ_OK || tm != 1 || opt.half_tiles == 2 || plan->kernel != PROJ_KERNEL_TC || !plan->swap_ab ||
        plan->cluster_split < 2 || M > 32)
        return st;
    PlanOptions alt_opt = opt;
    alt_opt.tm_cluster = 2;
    proj_plan_desc_t alt;
    if (plan_fitted(M, N, K, w_layout, y_dtype, has_bias, dd, alt_opt, &alt) == PROJ_OK &&
        alt.kernel == PROJ_KERNEL_TC && !alt.swap_ab && alt.cluster_split >= 2 &&
        10 * static_cast<int64_t>(alt.grid) >= 7 * static_cast<int64_t>(plan->grid))
        *plan = alt;
    return st;
}

// Y rows start on 16-byte boundaries: vector stores of 16 outputs are safe.
int y_vec_of(const void *Y, int64_t N, int y_dtype) {
    const int64_t row_bytes = N * (y_dtype == PROJ_F32 ? 4 : 2);
    return (row_bytes % 16 == 0) && (reinterpret_cast<uintptr_t>(Y) % 16 == 0);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The kernel instance a plan runs on: CTA pairs or single CTAs, with or
// without the fused epilogue.
cudaError_t launch_tc(const proj_plan_desc_t &plan, const TcLaunch &l, bool fused, const KernelParams &kp,
                      const CUtensorMap &map_w, const CUtensorMap &map_x) {
    if (launch_faulted()) return cudaErrorLaunchFailure;
    if (plan.cta_pair)
        return fused ? tc_launch_pair_fused(&l.cfg, kp, map_w, map_x) : tc_launch_pair(&l.cfg, kp, map_w, map_x);
    return fused ? tc_launch_fused(&l.cfg, kp, map_w, map_x) : tc_launch_lean(&l.cfg, kp, map_w, map_x);
}

proj_status_t check_launch() {
    return cudaGetLastError() == cudaSuccess ? PROJ_OK : PROJ_ERR_CUDA;
}

}  // namespace

extern "C" {

const char *proj_status_string(proj_status_t s) {
    switch (s) {
        case PROJ_OK: return "PROJ_OK";
        case PROJ_ERR_INVALID_ARG: return "PROJ_ERR_INVALID_ARG";
        case PROJ_ERR_UNSUPPORTED: return "PROJ_ERR_UNSUPPORTED";
        case PROJ_ERR_MISALIGNED: return "PROJ_ERR_MISALIGNED";
        case PROJ_ERR_OUT_OF_MEMORY: return "PROJ_ERR_OUT_OF_MEMORY";
        case PROJ_ERR_CUDA: return "PROJ_ERR_CUDA";
        case PROJ_ERR_DEVICE_TIMEOUT: return "PROJ_ERR_DEVICE_TIMEOUT";
    }
    return "PROJ_ERR_UNKNOWN";
}

proj_status_t proj_create(proj_handle_t *out, int64_t M, int64_t N, int64_t K,
                          proj_wlayout_t w_layout, proj_dtype_t x_dtype, proj_dtype_t w_dtype,
                          proj_dtype_t y_dtype, int has_bias, proj_dtype_t bias_dtype, void *stream) {
    if (!out) return PROJ_ERR_INVALID_ARG;
    *out = nullptr;
    if (M < 0 || N < 0 || K < 0) return PROJ_ERR_INVALID_ARG;
    if (w_layout != PROJ_W_NK && w_layout != PROJ_W_KN) return PROJ_ERR_INVALID_ARG;
    if (has_bias != 0 && has_bias != 1) return PROJ_ERR_INVALID_ARG;
    if (y_dtype != PROJ_BF16 && y_dtype != PROJ_F32) return PROJ_ERR_INVALID_ARG;
    if (x_dtype != PROJ_BF16 || (w_dtype != PROJ_BF16 && w_dtype != PROJ_F32)) return PROJ_ERR_UNSUPPORTED;
    const bool hilo = w_dtype == PROJ_F32;
    if (has_bias && bias_dtype != PROJ_BF16) return PROJ_ERR_UNSUPPORTED;
    if (K % 8 != 0) return PROJ_ERR_MISALIGNED;
    // [K,N] bf16 weights are loaded by TMA along N; fp32 weights are only read
    // by the pack kernel, element by element.
    if (w_layout == PROJ_W_KN && N % 8 != 0 && !hilo) return PROJ_ERR_MISALIGNED;

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return PROJ_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return PROJ_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return PROJ_ERR_UNSUPPORTED;  // built for sm_103a

    proj_device_desc_t dd{prop.multiProcessorCount, static_cast<int32_t>(prop.sharedMemPerBlockOptin)};
    if (!set_kernel_smem_limit(static_cast<int>(prop.sharedMemPerBlockOptin))) return PROJ_ERR_CUDA;
    proj_plan_desc_t plan;
    PlanOptions opt;  // environment overrides: tuning only
    if (const char *e = std::getenv("PROJ_FORCE_BLOCK_T")) opt.force_block_t = std::atoi(e);
    if (const char *e = std::getenv("PROJ_FORCE_BLOCK_N")) opt.force_block_n = std::atoi(e);
    if (const char *e = std::getenv("PROJ_MAX_CLUSTER")) {
        const int c = std::atoi(e);
        opt.max_cluster = c >= 2 && c <= kMaxClusterSplit ? c : 0;
    }
    if (const char *e = std::getenv("PROJ_CLUSTER_FILL_PCT")) {
        const int f = std::atoi(e);
        if (f >= 1 && f <= 100) opt.cluster_fill_pct = f;
    }
    if (const char *e = std::getenv("PROJ_CTA_PAIR")) {
        const int c = std::atoi(e);
        if (c >= 0 && c <= 2) opt.cta_pair = c;
    }
    if (const char *e = std::getenv("PROJ_HALF_TILES")) opt.half_tiles = std::atoi(e) == 2 ? 2 : 0;
    if (const char *e = std::getenv("PROJ_TM_CLUSTER")) {
        const int c = std::atoi(e);
        if (c >= 0 && c <= 2) opt.tm_cluster = c;
    }
    if (const char *e = std::getenv("PROJ_INFLIGHT_KB")) {
        const int kb = std::atoi(e);
        if (kb >= 16 && kb <= 228) opt.inflight_bytes = kb * 1024;
    }
    if (const char *e = std::getenv("PROJ_FORCE_CLUSTER")) {
        const int c = std::atoi(e);
        if (c >= 2 && c <= kMaxClusterSplit) opt.force_cluster = c;
    }
    if (const char *e = std::getenv("PROJ_PAIR_SK")) {  // tuning only
        if (std::atoi(e) == 1) opt.pair_sk = 1;
    }
    if (const char *e = std::getenv("PROJ_CLUSTER_GROUPS")) {  // tuning only
        const int g = std::atoi(e);
        if (g >= 1 && g <= 16) opt.cluster_groups = g;
    }
    // fp32 weights: the reduction runs over [H | L], twice the k-blocks of K.
    // A stage must not straddle the halves (its X k-blocks are contiguous):
    // with an odd number of k-blocks in K, one k-block a stage.
    const int64_t kt = (K + kBlockK - 1) / kBlockK;
    const int64_t k_plan = hilo ? 2 * kt * kBlockK : K;
    if (hilo && kt % 2 != 0) opt.kpb = 1;
    if (const char *e = std::getenv("PROJ_KPB")) {  // tuning only: 1 = one k-block a stage, 2 = two wherever K allows
        const int c = std::atoi(e);
        if ((c == 1 || c == 2) && !(hilo && kt % 2 != 0)) opt.kpb = c;
    }
    proj_status_t st = plan_for_device(M, N, k_plan, w_layout, y_dtype, has_bias, dd, opt, &plan);
    if (st != PROJ_OK) return st;
    if (const char *e = std::getenv("PROJ_FORCE_GRID")) {  // tuning only: fewer CTAs, all-split plans
        const int g = std::atoi(e);
        if (g >= 1 && g < plan.grid && plan.kernel == PROJ_KERNEL_TC && plan.tiles_dp == 0 &&
            plan.cluster_split < 2 && !plan.cta_pair) {
            plan.grid = g;
            const int64_t b_rows = plan.swap_ab ? plan.block_t : plan.block_n;
            const int64_t counter_bytes = ((plan.tiles_sk * 4 * 4 + 255) / 256) * 256;
            plan.scratch_bytes = int64_t(2) * g * kBlockA * b_rows * 4 + counter_bytes + 256;
        }
    }
    if (const char *e = std::getenv("PROJ_FORCE_WHOLE_TILES")) {  // tuning only
        if (std::atoi(e) == 1 && plan.kernel == PROJ_KERNEL_TC && plan.tiles_sk > 0 &&
            plan.cluster_split < 2 && !plan.cta_pair) {
            plan.tiles_dp += plan.tiles_sk;
            plan.tiles_sk = 0;
            plan.units_sk = 0;
            if (plan.tiles_dp < plan.grid) plan.grid = static_cast<int32_t>(plan.tiles_dp);  // no idle CTAs
        }
    }
    if (const char *e = std::getenv("PROJ_FORCE_STAGES")) {  // tuning only
        const int st_force = std::atoi(e);
        if (st_force >= 2 && st_force < plan.stages && plan.kernel == PROJ_KERNEL_TC) {
            plan.stages = st_force;
            plan.smem_bytes = st_force * plan_kpb(plan) * stage_bytes_for(plan_a_rows(plan), plan_cta_b_rows(plan)) +
                              plan_red_bytes(plan) + kSmemReserve;
        }
    }
    if (const char *e = std::getenv("PROJ_FORCE_RASTER_GROUP")) {  // tuning only
        const int g = std::atoi(e);
        if (g > 0 && plan.kernel == PROJ_KERNEL_TC)
            plan.raster_group = static_cast<int32_t>(g < plan.tiles_m ? g : plan.tiles_m);
    }

    proj_plan_s *h = new (std::nothrow) proj_plan_s();
    if (!h) return PROJ_ERR_OUT_OF_MEMORY;
    h->device = device;
    h->sm_count = prop.multiProcessorCount;
    h->hilo = hilo ? 1 : 0;
    h->kt = kt;
    h->M = M;
    h->N = N;
    h->K = K;
    h->w_layout = w_layout;
    h->y_dtype = y_dtype;
    h->has_bias = has_bias;
    h->plan = plan;
    if (const char *e = std::getenv("PROJ_PREFETCH_ANY")) h->prefetch_any = std::atoi(e) == 1;  // tuning only
    if (const char *e = std::getenv("PROJ_PREFETCH_STAGES")) {  // tuning only
        const int n = std::atoi(e);
        if (n >= 0 && n <= kMaxStages) h->prefetch_stages = n;
    }

    if (plan.kernel == PROJ_KERNEL_TC && w_layout == PROJ_W_KN && !hilo && !loads_stored_kn(plan)) {
        PlanOptions single = opt;
        single.cta_pair = 0;
        st = plan_for_device(M, N, k_plan, w_layout, y_dtype, has_bias, dd, single, &h->plan_stored);
        if (st != PROJ_OK) {
            delete h;
            return st;
        }
        h->has_plan_stored = true;
    }

    if (plan.kernel == PROJ_KERNEL_TC) {
        // One scratch serves both plans: partial sums first, each plan's
        // counters after its partials, the status word in the last 256 bytes.
        int64_t scratch_bytes = plan.scratch_bytes;
        if (h->has_plan_stored && h->plan_stored.scratch_bytes > scratch_bytes)
            scratch_bytes = h->plan_stored.scratch_bytes;
        if (dev_malloc(&h->scratch, static_cast<size_t>(scratch_bytes)) != cudaSuccess) {
            cudaGetLastError();
            delete h;
            return PROJ_ERR_OUT_OF_MEMORY;
        }
        uint8_t *sc = static_cast<uint8_t *>(h->scratch);
        auto init_params = [&](const proj_plan_desc_t &pl, KernelParams &kp) {
            kp.M = static_cast<int32_t>(M);
            kp.N = static_cast<int32_t>(N);
            kp.K = static_cast<int32_t>(K);
            params_from_plan(pl, kp);
            kp.idesc = idesc_of(pl, w_layout);
            kp.w_kn = w_layout == PROJ_W_KN;
            kp.y_f32 = y_dtype == PROJ_F32;
            kp.x_kb_mod = hilo ? static_cast<int32_t>(kt) : 0;
            kp.wait_limit_ns = kDefaultWaitLimitNs;
            kp.partials = reinterpret_cast<float *>(sc);
            kp.counters = reinterpret_cast<uint32_t *>(sc + partial_bytes_of(pl));
            kp.status = reinterpret_cast<int *>(sc + scratch_bytes - 256);
        };
        init_params(plan, h->params);
        int64_t partial_bytes = partial_bytes_of(plan);
        if (h->has_plan_stored) {
            init_params(h->plan_stored, h->params_stored);
            if (partial_bytes_of(h->plan_stored) < partial_bytes) partial_bytes = partial_bytes_of(h->plan_stored);
        }
        h->scratch_bytes = scratch_bytes;
        h->scratch_clear_from = partial_bytes;
        // Counters and the status word start at zero; partials need no clearing.
        if (cudaMemsetAsync(sc + partial_bytes, 0, static_cast<size_t>(scratch_bytes - partial_bytes),
                            as_stream(stream)) != cudaSuccess ||
            cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(h->scratch);
            delete h;
            return PROJ_ERR_CUDA;
        }
    }
    *out = h;
    return PROJ_OK;
}

}  // extern "C"

namespace {

// Rows of the packed weight layout (see proj_pack_weights), or -1 if they do
// not fit the 31-bit TMA coordinates.
int64_t packed_rows(const proj_plan_desc_t &plan) {
    const int64_t rows = plan.tiles_n * plan_packed_kblocks(plan) * plan.block_n;
    return rows < (int64_t(1) << 31) ? rows : -1;
}

proj_status_t run_impl(proj_handle_t h, const void *X, const void *W, bool packed, const void *bias,
                       const void *residual, void *Y, void *stream);

}  // namespace

extern "C" {

proj_status_t proj_run(proj_handle_t h, const void *X, const void *W, const void *bias, void *Y,
                       void *stream) {
    return run_impl(h, X, W, false, bias, nullptr, Y, stream);
}

proj_status_t proj_run_packed(proj_handle_t h, const void *X, const void *W_packed, const void *bias,
                              void *Y, void *stream) {
    return run_impl(h, X, W_packed, true, bias, nullptr, Y, stream);
}

proj_status_t proj_packed_weight_bytes(proj_handle_t h, size_t *bytes) {
    if (!h || !bytes) return PROJ_ERR_INVALID_ARG;
    *bytes = 0;
    if (h->plan.kernel != PROJ_KERNEL_TC) return PROJ_OK;
    const int64_t rows = packed_rows(h->plan);
    if (rows < 0) return PROJ_ERR_UNSUPPORTED;
    *bytes = static_cast<size_t>(rows) * 128;
    return PROJ_OK;
}

proj_status_t proj_pack_weights(proj_handle_t h, const void *W, void *W_packed, void *stream) {
    if (!h) return PROJ_ERR_INVALID_ARG;
    const proj_plan_desc_t &plan = h->plan;
    if (plan.kernel != PROJ_KERNEL_TC) return PROJ_OK;
    if (!W || !W_packed) return PROJ_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(W_packed)) return PROJ_ERR_MISALIGNED;
    const int64_t rows = packed_rows(plan);
    if (rows < 0) return PROJ_ERR_UNSUPPORTED;
    const int64_t chunks = rows * 8;  // 16-byte chunks
    const int64_t want = (chunks + 255) / 256;
    const int blocks = static_cast<int>(want < int64_t(h->sm_count) * 16 ? want : int64_t(h->sm_count) * 16);
    if (launch_faulted()) return PROJ_ERR_CUDA;
    if (h->hilo)
        dev::proj_pack_hilo_kernel<<<blocks, 256, 0, as_stream(stream)>>>(
            static_cast<const float *>(W), static_cast<uint16_t *>(W_packed), h->N, h->K,
            h->w_layout == PROJ_W_KN, plan.block_n, plan_packed_kblocks(plan), h->kt, chunks);
    else
        dev::proj_pack_kernel<<<blocks, 256, 0, as_stream(stream)>>>(
            static_cast<const uint16_t *>(W), static_cast<uint16_t *>(W_packed), h->N, h->K,
            h->w_layout == PROJ_W_KN, plan.block_n, plan_packed_kblocks(plan), chunks,
            h->act == PROJ_ACT_SWIGLU ? (plan.swap_ab ? 1 : 2) : 0);
    return check_launch();
}

}  // extern "C"

namespace {

proj_status_t run_impl(proj_handle_t h, const void *X, const void *W, bool packed, const void *bias,
                       const void *residual, void *Y, void *stream) {
    if (!h) return PROJ_ERR_INVALID_ARG;
    if (h->hilo && !packed && h->plan.kernel == PROJ_KERNEL_TC) return PROJ_ERR_UNSUPPORTED;
    if ((bias != nullptr) != (h->has_bias != 0)) return PROJ_ERR_INVALID_ARG;
    const bool stored = !packed && h->has_plan_stored;  // weights as stored, plan of single CTAs
    const proj_plan_desc_t &plan = stored ? h->plan_stored : h->plan;
    if (plan.kernel == PROJ_KERNEL_NONE) return PROJ_OK;
    if (!Y) return PROJ_ERR_INVALID_ARG;
    const size_t y_align = h->y_dtype == PROJ_F32 ? 4 : 2;
    if (reinterpret_cast<uintptr_t>(Y) % y_align != 0) return PROJ_ERR_MISALIGNED;
    if (residual && reinterpret_cast<uintptr_t>(residual) % y_align != 0) return PROJ_ERR_MISALIGNED;
    if (bias && reinterpret_cast<uintptr_t>(bias) % 2 != 0) return PROJ_ERR_MISALIGNED;
    cudaStream_t s = as_stream(stream);

    const bool swiglu = h->act == PROJ_ACT_SWIGLU;
    if (plan.kernel == PROJ_KERNEL_FILL) {
        // K = 0: every sum is empty.  SwiGLU of zeros is zero (no bias).
        if (launch_faulted()) return PROJ_ERR_CUDA;
        dev::proj_fill_kernel<<<plan.grid, plan.threads, 0, s>>>(
            h->M, swiglu ? h->N / 2 : h->N, static_cast<const uint16_t *>(bias), Y, h->y_dtype == PROJ_F32,
            swiglu ? 0 : h->act, residual);
        return check_launch();
    }
    // SwiGLU needs the interleaved packed weights.
    if (swiglu && !packed) return PROJ_ERR_UNSUPPORTED;

    if (!X || !W) return PROJ_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W)) return PROJ_ERR_MISALIGNED;
    if (X != h->map_x_ptr || x_box_rows(plan) != h->map_x_box || plan_kpb(plan) != h->map_x_kpb) {
        if (!encode_x(&h->map_x, X, h->M, h->K, plan, &h->map_x_3d)) {
            h->map_x_ptr = nullptr;
            return PROJ_ERR_CUDA;
        }
        h->map_x_ptr = X;
        h->map_x_box = x_box_rows(plan);
        h->map_x_kpb = plan_kpb(plan);
    }
    if (packed) {
        if (W != h->map_wp_ptr) {  // packed runs always use h->plan: one box size
            if (packed_rows(plan) < 0) return PROJ_ERR_UNSUPPORTED;
            if (!encode_packed(&h->map_wp, W, plan)) {
                h->map_wp_ptr = nullptr;
                return PROJ_ERR_CUDA;
            }
            h->map_wp_ptr = W;
        }
    } else if (W != h->map_w_ptr || w_box_rows(plan) != h->map_w_box) {
        const bool ok = h->w_layout == PROJ_W_NK
                            ? encode_2d(&h->map_w, W, h->K, h->N, h->K * 2, kBlockK, w_box_rows(plan))
                            : encode_2d(&h->map_w, W, h->N, h->K, h->N * 2, 64, kBlockK);
        if (!ok) {
            h->map_w_ptr = nullptr;
            return PROJ_ERR_CUDA;
        }
        h->map_w_ptr = W;
        h->map_w_box = w_box_rows(plan);
    }
    KernelParams kp = stored ? h->params_stored : h->params;
    kp.x_3d = h->map_x_3d;
    if (packed) {
        // Packed weights are K-major blocks whatever the stored layout.
        kp.w_packed = 1;
        kp.w_kn = 0;
        kp.idesc = idesc_of(plan, PROJ_W_NK);
    }
    kp.bias = static_cast<const uint16_t *>(bias);
    kp.Y = Y;
    kp.act = h->act;
    kp.residual = residual;
    kp.ldy = static_cast<int32_t>(swiglu ? h->N / 2 : h->N);
    // Vector stores read the residual the same way: both 16-byte aligned.
    kp.y_vec = y_vec_of(Y, kp.ldy, h->y_dtype) && (!residual || aligned16(residual));
    kp.trace = h->trace;
    // Weights stream early only when every SM has a CTA: the next kernel's
    // CTAs then start as the preceding kernel's leave, in its tail.  With SMs
    // idle they would start at once and compete with its weight stream
    // (measured slower on GB300 for the cluster-split and 128-tile plans).
    // (Not with CTA pairs, whose stages are armed by the leader for both.)
    kp.w_prefetch = h->overlap == PROJ_OVERLAP_WEIGHTS && (plan.grid >= h->sm_count || h->prefetch_any) &&
                            !plan.cta_pair
                        ? h->prefetch_stages
                        : 0;
    TcLaunch l(plan, s, h->overlap != PROJ_OVERLAP_NONE);
    // The fused instance also carries the token-major cluster reduction.
    const bool fused = kp.act != 0 || kp.residual != nullptr || (plan.cluster_split > 1 && !plan.swap_ab);
    const CUtensorMap &map_w = packed ? h->map_wp : h->map_w;
    if (launch_tc(plan, l, fused, kp, map_w, h->map_x) != cudaSuccess) {
        cudaGetLastError();
        return PROJ_ERR_CUDA;
    }
    return PROJ_OK;
}

}  // namespace

extern "C" {

namespace {
proj_status_t run_host_impl(proj_handle_t h, const void *X_host, const void *W, bool packed,
                            const void *bias, void *Y_host, void *stream);
}  // namespace

proj_status_t proj_run_host(proj_handle_t h, const void *X_host, const void *W, const void *bias,
                            void *Y_host, void *stream) {
    return run_host_impl(h, X_host, W, false, bias, Y_host, stream);
}

proj_status_t proj_run_host_packed(proj_handle_t h, const void *X_host, const void *W_packed,
                                   const void *bias, void *Y_host, void *stream) {
    return run_host_impl(h, X_host, W_packed, true, bias, Y_host, stream);
}

}  // extern "C"

namespace {

// The device address of a host buffer the device can read and write (pinned
// by cudaHostAlloc or registered by cudaHostRegister), or nullptr (pageable
// memory, or a buffer the runtime does not know).
void *host_device_pointer(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// One host <-> device copy: a copy kernel chained to its neighbours by
// programmatic dependent launch when the host buffer is device-addressable
// and both ends are 16-byte aligned, else cudaMemcpyAsync.
proj_status_t copy_host(void *dst_dev, const void *src_dev, void *dst, const void *src, size_t bytes,
                        cudaMemcpyKind kind, int sm_count, cudaStream_t s) {
    if (bytes == 0) return PROJ_OK;
    if (src_dev && dst_dev && aligned16(src_dev) && aligned16(dst_dev)) {
        const int64_t n16 = static_cast<int64_t>(bytes / 16);
        const int64_t want = (n16 + 1023) / 1024;  // four chunks a thread
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3(static_cast<unsigned>(want < 1 ? 1 : (want < 2 * sm_count ? want : 2 * sm_count)));
        cfg.blockDim = dim3(256);
        cfg.stream = s;
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (launch_faulted()) return PROJ_ERR_CUDA;
        if (cudaLaunchKernelEx(&cfg, dev::proj_copy_kernel, static_cast<const uint8_t *>(src_dev),
                               static_cast<uint8_t *>(dst_dev), static_cast<int64_t>(bytes)) != cudaSuccess) {
            cudaGetLastError();
            return PROJ_ERR_CUDA;
        }
        return PROJ_OK;
    }
    return cudaMemcpyAsync(dst, src, bytes, kind, s) == cudaSuccess ? PROJ_OK : PROJ_ERR_CUDA;
}

proj_status_t run_host_impl(proj_handle_t h, const void *X_host, const void *W, bool packed,
                            const void *bias, void *Y_host, void *stream) {
    if (!h) return PROJ_ERR_INVALID_ARG;
    if (h->plan.kernel == PROJ_KERNEL_NONE) return PROJ_OK;
    if (!Y_host || (!X_host && h->K > 0)) return PROJ_ERR_INVALID_ARG;
    const size_t xb = static_cast<size_t>(h->M) * h->K * 2;
    const size_t yb = static_cast<size_t>(h->M) * h->N * (h->y_dtype == PROJ_F32 ? 4 : 2);
    if (!h->stage_y) {
        if (xb && dev_malloc(&h->stage_x, xb) != cudaSuccess) {
            cudaGetLastError();
            return PROJ_ERR_OUT_OF_MEMORY;
        }
        if (dev_malloc(&h->stage_y, yb) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(h->stage_x);
            h->stage_x = nullptr;
            return PROJ_ERR_OUT_OF_MEMORY;
        }
    }
    cudaStream_t s = as_stream(stream);
    // Device addresses of the host buffers, looked up on every call (a buffer
    // may be freed and its address reused by memory of another kind).
    const void *x_dev = X_host ? host_device_pointer(X_host) : nullptr;
    void *y_dev = host_device_pointer(Y_host);
    proj_status_t st = copy_host(h->stage_x, x_dev, h->stage_x, X_host, xb, cudaMemcpyHostToDevice, h->sm_count, s);
    if (st != PROJ_OK) return st;
    // A device-addressable, 16-byte aligned Y is written by the projection's
    // own epilogue, through its device address (no staging, no copy kernel).
    if (y_dev && aligned16(y_dev)) return run_impl(h, h->stage_x, W, packed, bias, nullptr, y_dev, stream);
    st = run_impl(h, h->stage_x, W, packed, bias, nullptr, h->stage_y, stream);
    if (st != PROJ_OK) return st;
    return copy_host(y_dev, h->stage_y, Y_host, h->stage_y, yb, cudaMemcpyDeviceToHost, h->sm_count, s);
}
}  // namespace

extern "C" {

proj_status_t proj_device_status(proj_handle_t h, void *stream) {
    if (!h) return PROJ_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return PROJ_ERR_CUDA;
    if (h->plan.kernel != PROJ_KERNEL_TC) return PROJ_OK;
    int word = 0;
    if (cudaMemcpy(&word, h->params.status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PROJ_ERR_CUDA;
    if (word == 0) return PROJ_OK;
    const proj_status_t what = (word & (kErrSmemTooSmall | kErrLaunchShape | kErrPairTmem))
                                   ? PROJ_ERR_CUDA
                                   : PROJ_ERR_DEVICE_TIMEOUT;
    // Clear the word and the split-K counters (a run that gave up may have
    // left some mid-count) so the handle is usable again.
    if (cudaMemset(static_cast<uint8_t *>(h->scratch) + h->scratch_clear_from, 0,
                   static_cast<size_t>(h->scratch_bytes - h->scratch_clear_from)) != cudaSuccess)
        return PROJ_ERR_CUDA;
    return what;
}

proj_status_t proj_set_activation(proj_handle_t h, proj_activation_t act) {
    if (!h) return PROJ_ERR_INVALID_ARG;
    if (act != PROJ_ACT_NONE && act != PROJ_ACT_GELU && act != PROJ_ACT_SWIGLU) return PROJ_ERR_INVALID_ARG;
    // SwiGLU: stacked gate and up rows (N even), no bias, bf16 weights.
    if (act == PROJ_ACT_SWIGLU && (h->N % 2 != 0 || h->has_bias || h->hilo)) return PROJ_ERR_UNSUPPORTED;
    h->act = act;
    return PROJ_OK;
}

proj_status_t proj_run_fused(proj_handle_t h, const void *X, const void *W, int packed, const void *bias,
                             const void *residual, void *Y, void *stream) {
    if (packed != 0 && packed != 1) return PROJ_ERR_INVALID_ARG;
    return run_impl(h, X, W, packed != 0, bias, residual, Y, stream);
}

proj_status_t proj_set_overlap(proj_handle_t h, proj_overlap_t mode) {
    if (!h) return PROJ_ERR_INVALID_ARG;
    if (mode != PROJ_OVERLAP_NONE && mode != PROJ_OVERLAP_PROLOGUE && mode != PROJ_OVERLAP_WEIGHTS)
        return PROJ_ERR_INVALID_ARG;
    h->overlap = mode;
    return PROJ_OK;
}

proj_status_t proj_set_trace(proj_handle_t h, void *device_buffer, size_t bytes) {
    if (!h) return PROJ_ERR_INVALID_ARG;
    if (!device_buffer) {
        h->trace = nullptr;
        return PROJ_OK;
    }
    if (h->plan.kernel != PROJ_KERNEL_TC) return PROJ_ERR_UNSUPPORTED;
    int32_t grid = h->plan.grid;
    if (h->has_plan_stored && h->plan_stored.grid > grid) grid = h->plan_stored.grid;
    const size_t need = static_cast<size_t>(grid) * kTraceSlots * sizeof(unsigned long long);
    if (bytes < need) return PROJ_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(device_buffer) % 8 != 0) return PROJ_ERR_MISALIGNED;
    h->trace = static_cast<unsigned long long *>(device_buffer);
    return PROJ_OK;
}

proj_status_t proj_get_plan(proj_handle_t h, proj_plan_desc_t *out) {
    if (!h || !out) return PROJ_ERR_INVALID_ARG;
    *out = h->plan;
    return PROJ_OK;
}

proj_status_t proj_plan_info(proj_handle_t h, char *buf, size_t len) {
    if (!h || !buf || len == 0) return PROJ_ERR_INVALID_ARG;
    plan_to_json(h->plan, h->M, h->N, h->K, h->w_layout, h->y_dtype, h->has_bias, buf, len);
    return PROJ_OK;
}

proj_status_t proj_destroy(proj_handle_t h) {
    if (!h) return PROJ_OK;
    proj_status_t st = PROJ_OK;
    if (h->scratch && cudaFree(h->scratch) != cudaSuccess) st = PROJ_ERR_CUDA;
    if (h->stage_x && cudaFree(h->stage_x) != cudaSuccess) st = PROJ_ERR_CUDA;
    if (h->stage_y && cudaFree(h->stage_y) != cudaSuccess) st = PROJ_ERR_CUDA;
    delete h;
    return st;
}

proj_status_t proj_selftest_wait_timeout(int64_t limit_ns, void *stream) {
    if (limit_ns < 1000 || limit_ns > 1000000000LL) return PROJ_ERR_INVALID_ARG;
    int *word = nullptr;
    if (dev_malloc(reinterpret_cast<void **>(&word), sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return PROJ_ERR_OUT_OF_MEMORY;
    }
    cudaStream_t s = as_stream(stream);
    proj_status_t st = PROJ_OK;
    int host_word = 0;
    if (cudaMemsetAsync(word, 0, sizeof(int), s) != cudaSuccess) st = PROJ_ERR_CUDA;
    if (st == PROJ_OK) {
        if (launch_faulted()) {
            st = PROJ_ERR_CUDA;
        } else {
            dev::proj_selftest_wait_kernel<<<1, 32, 0, s>>>(limit_ns, word);
            st = check_launch();
        }
    }
    if (st == PROJ_OK && (cudaMemcpyAsync(&host_word, word, sizeof(int), cudaMemcpyDeviceToHost, s) !=
                              cudaSuccess ||
                          cudaStreamSynchronize(s) != cudaSuccess))
        st = PROJ_ERR_CUDA;
    cudaFree(word);
    if (st != PROJ_OK) return st;
    return host_word == kErrSelfTest ? PROJ_ERR_DEVICE_TIMEOUT : PROJ_OK;
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot call cudaMalloc: a serving loop where an allocation may
// synchronise the device and stall every other stream at an unpredictable
// moment, or a plug-in whose host application owns all device memory and
// forbids allocating behind its back.  proj_run_noalloc serves them with the
// same kernel as proj_run, taking its split-K scratch from the fixed-size
// device array below instead of a handle.  Every GPU that loads this library
// holds the array until the process exits.
//
// Layout of the array: a plan's partial sums from offset 0, its split-K
// counters after them, and one status word in the last 256 bytes.  Each call
// clears the counters it uses; the status word collects the error bits of
// every call until proj_noalloc_device_status reads and clears it.
// ----------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB: partials, counters, status
constexpr size_t kNoAllocStatusOffset = kNoAllocScratchBytes - 256;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Per-device set-up: the array's device address (the host-side name of the
// array is only a stand-in), the kernels' shared-memory limit and the
// device's SM count, redone whenever the device's current context is a
// different one (a context torn down by cudaDeviceReset takes the address
// with it).  The plan of the last shape run on the device is kept too, so a
// steady stream of calls of one shape plans once.
struct NoAllocDevice {
    bool ready = false;
    unsigned long long ctx_id = 0;
    void *scratch = nullptr;
    int sms = 0, smem = 0;
    bool has_plan = false;
    int64_t M = 0, N = 0, K = 0;
    int layout = 0, y_dtype = 0, bias = 0;
    proj_plan_desc_t plan{};
};

std::mutex g_noalloc_mutex;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// Unique id of the calling thread's current context (0 if there is none yet).
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// The set-up of `device`, which must be current (done on its first use and
// again after its context changed).  Call with g_noalloc_mutex held.
proj_status_t noalloc_setup(int device, NoAllocDevice **out) {
    if (device < 0 || device >= kNoAllocMaxDevices) return PROJ_ERR_UNSUPPORTED;
    NoAllocDevice &d = g_noalloc_dev[device];
    const unsigned long long ctx = current_context_id();
    if (d.ready && ctx != 0 && ctx == d.ctx_id) {
        *out = &d;
        return PROJ_OK;
    }
    d = NoAllocDevice{};
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return PROJ_ERR_CUDA;
    }
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess)
        return PROJ_ERR_CUDA;
    if (major != 10 || minor != 3) return PROJ_ERR_UNSUPPORTED;
    if (!set_kernel_smem_limit(d.smem)) return PROJ_ERR_CUDA;
    d.scratch = ptr;
    d.ctx_id = current_context_id();  // the symbol lookup made the context current if it was not
    d.ready = true;
    *out = &d;
    return PROJ_OK;
}

// Error bits of the device status word as a status code.
proj_status_t status_of_word(int word) {
    if (word == 0) return PROJ_OK;
    return (word & (kErrSmemTooSmall | kErrLaunchShape | kErrPairTmem)) ? PROJ_ERR_CUDA : PROJ_ERR_DEVICE_TIMEOUT;
}

}  // namespace

extern "C" proj_status_t proj_run_noalloc(int64_t M, int64_t N, int64_t K, proj_wlayout_t w_layout,
                                          proj_dtype_t y_dtype, const void *X, const void *W,
                                          const void *bias, void *Y, void *stream) {
    if (M < 0 || N < 0 || K < 0) return PROJ_ERR_INVALID_ARG;
    if (w_layout != PROJ_W_NK && w_layout != PROJ_W_KN) return PROJ_ERR_INVALID_ARG;
    if (y_dtype != PROJ_BF16 && y_dtype != PROJ_F32) return PROJ_ERR_INVALID_ARG;
    if (K % 8 != 0) return PROJ_ERR_MISALIGNED;
    if (w_layout == PROJ_W_KN && N % 8 != 0) return PROJ_ERR_MISALIGNED;
    if (M == 0 || N == 0) return PROJ_OK;
    if (!Y) return PROJ_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(Y) % (y_dtype == PROJ_F32 ? 4 : 2) != 0) return PROJ_ERR_MISALIGNED;
    if (bias && reinterpret_cast<uintptr_t>(bias) % 2 != 0) return PROJ_ERR_MISALIGNED;
    cudaStream_t s = as_stream(stream);

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return PROJ_ERR_CUDA;
    const int has_bias = bias != nullptr ? 1 : 0;
    proj_plan_desc_t plan;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        NoAllocDevice *d = nullptr;
        proj_status_t st = noalloc_setup(device, &d);
        if (st != PROJ_OK) return st;
        if (!(d->has_plan && d->M == M && d->N == N && d->K == K && d->layout == w_layout &&
              d->y_dtype == y_dtype && d->bias == has_bias)) {
            d->has_plan = false;
            proj_device_desc_t dd{d->sms, d->smem};
            st = plan_for_device(M, N, K, w_layout, y_dtype, has_bias, dd, PlanOptions{}, &d->plan);
            if (st != PROJ_OK) return st;
            if (d->plan.kernel == PROJ_KERNEL_TC && w_layout == PROJ_W_KN && !loads_stored_kn(d->plan)) {
                PlanOptions single;
                single.cta_pair = 0;
                st = plan_for_device(M, N, K, w_layout, y_dtype, has_bias, dd, single, &d->plan);
                if (st != PROJ_OK) return st;
            }
            d->M = M;
            d->N = N;
            d->K = K;
            d->layout = w_layout;
            d->y_dtype = y_dtype;
            d->bias = has_bias;
            d->has_plan = true;
        }
        plan = d->plan;
        scratch = d->scratch;
    }
    if (plan.kernel == PROJ_KERNEL_FILL) {
        if (launch_faulted()) return PROJ_ERR_CUDA;
        dev::proj_fill_kernel<<<plan.grid, plan.threads, 0, s>>>(M, N, static_cast<const uint16_t *>(bias),
                                                                 Y, y_dtype == PROJ_F32, 0, nullptr);
        return check_launch();
    }
    // The plan's scratch must fit the static array; larger problems are refused.
    if (static_cast<size_t>(plan.scratch_bytes) > kNoAllocScratchBytes) return PROJ_ERR_UNSUPPORTED;
    if (!X || !W) return PROJ_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W)) return PROJ_ERR_MISALIGNED;

    const int64_t partial_bytes = partial_bytes_of(plan);
    const int64_t counter_bytes = plan.scratch_bytes - 256 - partial_bytes;
    uint8_t *sc = static_cast<uint8_t *>(scratch);
    // The array keeps the previous call's contents: the counters must start
    // at zero (partials are fully rewritten before use; the status word is
    // left for proj_noalloc_device_status).
    if (counter_bytes > 0 &&
        cudaMemsetAsync(sc + partial_bytes, 0, static_cast<size_t>(counter_bytes), s) != cudaSuccess) {
        cudaGetLastError();
        return PROJ_ERR_CUDA;
    }

    CUtensorMap map_x, map_w;
    int32_t x_3d = 0;
    if (!encode_x(&map_x, X, M, K, plan, &x_3d)) return PROJ_ERR_CUDA;
    const bool ok = w_layout == PROJ_W_NK ? encode_2d(&map_w, W, K, N, K * 2, kBlockK, w_box_rows(plan))
                                          : encode_2d(&map_w, W, N, K, N * 2, 64, kBlockK);
    if (!ok) return PROJ_ERR_CUDA;

    KernelParams kp{};
    kp.M = static_cast<int32_t>(M);
    kp.N = static_cast<int32_t>(N);
    kp.K = static_cast<int32_t>(K);
    params_from_plan(plan, kp);
    kp.idesc = idesc_of(plan, w_layout);
    kp.w_kn = w_layout == PROJ_W_KN;
    kp.y_f32 = y_dtype == PROJ_F32;
    kp.wait_limit_ns = kDefaultWaitLimitNs;
    kp.w_prefetch = 0;
    kp.bias = static_cast<const uint16_t *>(bias);
    kp.Y = Y;
    kp.ldy = static_cast<int32_t>(N);
    kp.y_vec = y_vec_of(Y, N, y_dtype);
    kp.partials = reinterpret_cast<float *>(sc);
    kp.counters = reinterpret_cast<uint32_t *>(sc + partial_bytes);
    kp.status = reinterpret_cast<int *>(sc + kNoAllocStatusOffset);
    kp.trace = nullptr;
    kp.x_3d = x_3d;
    TcLaunch l(plan, s, false);
    if (launch_tc(plan, l, plan.cluster_split > 1 && !plan.swap_ab, kp, map_w, map_x) != cudaSuccess) {
        cudaGetLastError();
        return PROJ_ERR_CUDA;
    }
    return PROJ_OK;
}

extern "C" proj_status_t proj_noalloc_device_status(void *stream) {
    if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return PROJ_ERR_CUDA;
    int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_noalloc_scratch, sizeof word, kNoAllocStatusOffset,
                             cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return PROJ_ERR_CUDA;
    }
    if (word == 0) return PROJ_OK;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_noalloc_scratch, &zero, sizeof zero, kNoAllocStatusOffset,
                           cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return PROJ_ERR_CUDA;
    }
    return status_of_word(word);
}

extern "C" proj_status_t proj_noalloc_selftest_wait_timeout(int64_t limit_ns, void *stream) {
    if (limit_ns < 1000 || limit_ns > 1000000000LL) return PROJ_ERR_INVALID_ARG;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return PROJ_ERR_CUDA;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        NoAllocDevice *d = nullptr;
        const proj_status_t st = noalloc_setup(device, &d);
        if (st != PROJ_OK) return st;
        scratch = d->scratch;
    }
    if (launch_faulted()) return PROJ_ERR_CUDA;
    dev::proj_selftest_wait_kernel<<<1, 32, 0, as_stream(stream)>>>(
        limit_ns, reinterpret_cast<int *>(static_cast<uint8_t *>(scratch) + kNoAllocStatusOffset));
    return check_launch();
}
