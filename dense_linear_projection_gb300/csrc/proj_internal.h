// Internal definitions shared by the planner, the C ABI and the device code.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "proj.h"

#if defined(__CUDACC__)
#define PROJ_HD __host__ __device__ __forceinline__
#else
#define PROJ_HD inline
#endif

namespace projgb {

constexpr int32_t kBlockA = 128;       // rows of the MMA's A operand (tcgen05 M)
constexpr int32_t kBlockK = 64;        // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int32_t kMmaK = 16;          // K per tcgen05.mma (kind::f16)
constexpr int32_t kMaxTokenTile = 256; // tcgen05 MMA N limit for cta_group::1
constexpr int32_t kMaxStages = 16;
constexpr int32_t kInflightTarget = 160 * 1024;  // stage bytes per SM when streaming W from HBM
constexpr int32_t kMaxClusterSplit = 16;          // thread-block cluster size (16: non-portable)
constexpr int32_t kClusterFillPct = 10;           // SMs a cluster split must keep busy (%)
// CTA pairs: tensor-memory columns a pair may allocate in each of its SMs
// (both CTAs allocate together and receive the same columns).
constexpr int32_t kPairTmemMax = 512;
constexpr int32_t kThreads = 192;      // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int32_t kEpilogueThreads = 128;
constexpr int32_t kSmemReserve = 25600; // 1024-byte alignment slack + barriers + epilogue staging
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

// Phase-trace record: kTraceSlots unsigned 64-bit words per CTA, globaltimer
// nanoseconds unless noted.
constexpr int kTraceSlots = 16;
constexpr int kTraceEntry = 0;         // kernel entry (thread 0)
constexpr int kTraceSetup = 1;         // barriers initialised, tensor memory allocated
constexpr int kTraceFirstLoad = 2;     // producer issued its first TMA load
constexpr int kTraceLastLoad = 3;      // producer issued its last TMA load
constexpr int kTraceFirstData = 4;     // MMA issuer saw the first stage full
constexpr int kTraceLastMma = 5;       // MMA issuer committed its last accumulator
constexpr int kTraceFirstAcc = 6;      // epilogue warp 2 received its first accumulator
constexpr int kTraceEpilogueDone = 7;  // epilogue warp 2 finished every segment
constexpr int kTraceTeardown = 8;      // all roles joined at the final barrier
constexpr int kTraceSmid = 9;          // SM the CTA ran on (a number, not a time)
constexpr int kTraceReductions = 10;   // split tiles epilogue warp 2 reduced (a count)
constexpr int kTraceDepWait = 11;      // producer returned from the grid-dependency wait
constexpr int kTraceEpiDepWait = 12;   // epilogue warp 2 returned from the grid-dependency wait
// Epilogue warp 2, first split tile only:
constexpr int kTraceSplitPartial = 13; // its partial sums are written (shared or global memory)
constexpr int kTraceSplitReady = 14;   // it knows every partial of the tile is in (or it is not the reducer)
constexpr int kTraceSplitStored = 15;  // it stored the reduced rows (or gave them to the reducer)

// Error bits in the device status word.
constexpr int kErrWaitProducer = 1 << 0;
constexpr int kErrWaitMma = 1 << 1;
constexpr int kErrWaitEpilogue = 1 << 2;
constexpr int kErrWaitDrain = 1 << 3;
constexpr int kErrSelfTest = 1 << 4;
constexpr int kErrSmemTooSmall = 1 << 5;  // launch gave less shared memory than the ring needs
constexpr int kErrLaunchShape = 1 << 6;   // cluster shape of the launch differs from the plan's
constexpr int kErrPairTmem = 1 << 7;      // the two CTAs of a pair received different tensor memory

int32_t token_tile_for(int64_t M);
// Planner options.  force_block_t > 0 forces the swapped orientation with
// that token tile; force_block_n > 0 forces the token-rows-on-M orientation
// with that weight tile (both tuning overrides, from PROJ_FORCE_BLOCK_T /
// PROJ_FORCE_BLOCK_N in proj_create).  max_cluster bounds the cluster-split
// size (0 disables it; proj_create lowers it when the clusters would not all
// be resident at once); a cluster split must keep cluster_fill_pct percent of
// the SMs busy.
struct PlanOptions {
    int32_t force_block_t = 0;
    int32_t force_block_n = 0;
    int32_t max_cluster = kMaxClusterSplit;
    int32_t cluster_fill_pct = kClusterFillPct;
    // CTA pairs (cta_group::2 MMAs, PROJ_CTA_PAIR): 0 never; 1 where they
    // measure faster (swapped plans of 256-token tiles that keep half of the
    // SMs busy); 2 wherever the tile allows (token-major tiles too).
    int32_t cta_pair = 1;
    // Half tiles (PROJ_HALF_TILES=2): swapped tiles of 64 weight rows, for
    // any swapped plan of at most 64 tokens.  Off by default: on GB300 the
    // 2048-row decode weight ran 15.9 us on 32 half tiles in clusters of 4
    // (128 SMs) against 12.6 us on 16 full tiles in clusters of 6 (96 SMs).
    int32_t half_tiles = 0;
    // Token-major cluster split (PROJ_TM_CLUSTER) for at most 32 tokens: the
    // tokens on the MMA's M side (128 rows, the rest zero) and 256 weight rows
    // on its N side, which streams more weight bytes per MMA instruction than
    // 128 weight rows on the M side.  0 never (the default); 1 where
    // proj_create finds the swapped plan a cluster split too and this one
    // keeps at least 70 % of its SMs; 2 wherever it applies.  Off by default:
    // on GB300 the 2048-row decode weight streamed in 5.2 us instead of 7.1 us
    // per CTA, but its 8 clusters of 12 CTAs started about 5 us later after
    // the preceding call than 16 clusters of 6 (15.9 us per call vs 12.7).
    int32_t tm_cluster = 0;
    // K per pipeline stage (PROJ_KPB): 0 lets the planner choose, 1 forces
    // one 64-wide k-block a stage, 2 allows two (see the planner).
    int32_t kpb = 0;
    // Cluster split of exactly this size for swapped tiles of at most 64
    // tokens whenever the clusters fit the SMs (PROJ_FORCE_CLUSTER; 0: the
    // planner's rule).
    int32_t force_cluster = 0;
    // Stream-K over CTA pairs (PROJ_PAIR_SK=1): token-major pair tiles of
    // 256 weight columns whose K ranges are shared by all pairs (the
    // data-parallel + two-tile stream-K hybrid), instead of whole tiles of
    // the width that best fills the pairs.  Off by default.
    int32_t pair_sk = 0;
    // Clusters per tile of a swapped cluster split (PROJ_CLUSTER_GROUPS): 0
    // lets the planner choose, 1 forces one, G >= 2 forces G where the G·S
    // CTAs of every tile fit the SMs.
    int32_t cluster_groups = 0;
    // Stage bytes per SM a weight-streaming plan keeps in flight
    // (PROJ_INFLIGHT_KB).
    int32_t inflight_bytes = kInflightTarget;
};
// The planner behind proj_plan_compute (which uses the default options).
proj_status_t plan_compute(int64_t M, int64_t N, int64_t K, proj_wlayout_t w_layout,
                           proj_dtype_t y_dtype, int has_bias, const proj_device_desc_t *dev,
                           const PlanOptions &opt, proj_plan_desc_t *out);
// Shared-memory bytes of one pipeline stage: A (a_rows x 64 K: 128, or the 64
// weight rows of a half tile) plus B (b_rows x 64 K), bf16.  A CTA of a pair
// holds half of the B rows.
int32_t stage_bytes_for(int32_t a_rows, int32_t b_rows);
int plan_to_json(const proj_plan_desc_t &p, int64_t M, int64_t N, int64_t K, int w_layout,
                 int y_dtype, int has_bias, char *buf, size_t len);

// Kernel parameters (passed by value; the tensor maps travel separately as
// __grid_constant__ arguments).
struct KernelParams {
    int32_t M, N, K;
    int32_t swap;          // 1: A = weight rows, B = token rows; 0: A = token rows, B = weight rows
    int32_t block_t;       // token rows per tile
    int32_t block_n;       // weight rows per tile
    int32_t b_rows;        // rows of the B operand (MMA N): block_t if swap, else block_n
    int32_t tiles_m;       // token-row tiles
    int32_t tiles_n;       // weight-row tiles
    int32_t raster_group;  // token tiles per raster group (tile order, see tile_coords)
    int32_t k_blocks;      // pipeline stages of K per tile: ceil(K / (64 · kpb))
    int32_t kpb;           // 64-wide k-blocks per stage (1 or 2), loaded by one TMA op each for W and X
    int32_t x_3d;          // X's tensor map is 3-D (64 K, rows, k-blocks): a stage's X in one op
    int32_t tiles_dp;      // whole tiles, dealt round-robin: CTA c gets c, c+G, ...
    int32_t grid;          // work owners the tiles are dealt to: CTAs, or pairs of CTAs
    int64_t units_sk;      // split-K units after the whole tiles
    int32_t sk_pair;       // every CTA owns >= k_blocks units: a split tile has exactly 2 contributors
    int32_t sk_dense;      // units_sk >= grid: no CTA has an empty unit range
    int32_t cluster_split; // S >= 2: tile c / S split over the S CTAs of a cluster (DSMEM reduction)
    int32_t cta_pair;      // 1: each tile on a cluster of 2 CTAs, one cta_group::2 MMA of 256 rows
    int32_t acc_bufs;      // accumulator buffers in tensor memory (2: epilogue overlaps the next tile)
    int32_t stages;
    int32_t stage_bytes;   // one stage: A rows + B rows, what one CTA's loads bring into it
    int32_t a_rows;        // A rows of a tile this CTA holds: 128, or 64 (half tiles: MMA rows 64-127 unused)
    int32_t red_bytes;     // cluster split: shared memory after the ring for peers' partial sums
    int32_t tmem_cols;
    uint32_t idesc;        // tcgen05 instruction descriptor (bf16 x bf16 -> f32, M=128 or 256, N=b_rows)
    int32_t w_kn;          // W stored [K,N] (MN-major A operand)
    int32_t w_packed;      // W pre-packed: block (tile, k-block) at row (tn·k_blocks + kb)·block_n
    int32_t x_kb_mod;      // > 0: fp32 router weights as [H | L]; X k-block = kb mod x_kb_mod
    int32_t y_f32;         // store fp32 (else bf16)
    int32_t y_vec;         // Y rows start 16-byte aligned (N·size % 16 == 0, aligned base)
    int64_t wait_limit_ns; // bounded device waits give up after this long
    int32_t cluster_groups; // cluster split: clusters per tile (their sums meet in scratch), else 1
    int32_t w_prefetch;    // stages of W streamed before the preceding kernel completes (0: none)
    int32_t act;           // fused activation: 0 none, 1 GELU (on projection + bias), 2 SwiGLU
    int32_t ldy;           // Y row stride in elements: N, or N / 2 for SwiGLU (gate and up rows stacked)
    const uint16_t *bias;  // [N] bf16 or nullptr
    const void *residual;  // [M,N] in Y's dtype, added after the activation, or nullptr (may alias Y)
    void *Y;
    float *partials;       // [2*grid][128 rows][b_rows] fp32 partial tiles
    uint32_t *counters;    // [4 * (tiles - tiles_dp)]: one per (split tile, row quarter)
    int *status;           // device status word
    unsigned long long *trace;  // [grid][kTraceSlots] phase trace, or nullptr
};

// ----------------------------------------------------------------------------
// Work decomposition, shared verbatim by the kernel (every role walks the same
// sequence) and by the host introspection entry points (so the CPU tests check
// the exact code the GPU runs).
// ----------------------------------------------------------------------------
struct Segment {
    int32_t tile;   // tile index in raster order (tile_coords gives its coordinates)
    int32_t kb0;    // first k-block
    int32_t kb1;    // one past the last k-block
    int32_t slot;   // partial-sum slot (split segments), else -1
    bool split;     // the tile's K range is shared with other CTAs
};

// a / b for 0 ≤ a, 0 < b: a 32-bit division when both fit (the usual case; a
// 64-bit division is a long software sequence on the GPU).
PROJ_HD int64_t div_nonneg(int64_t a, int64_t b) {
    if (a < (int64_t(1) << 32) && b < (int64_t(1) << 32))
        return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
    return a / b;
}

// First split-K unit of CTA c: ⌊c·U/G⌋ (the integer partition that splits 128
// k-blocks over 3 CTAs as 42/43/43).
PROJ_HD int64_t unit_begin(int32_t c, int64_t U, int32_t G) {
    return div_nonneg(static_cast<int64_t>(c) * U, G);
}

// The CTA whose unit range contains unit u: the largest c with ⌊c·U/G⌋ ≤ u.
PROJ_HD int32_t cta_of_unit(int64_t u, int64_t U, int32_t G) {
    return static_cast<int32_t>(div_nonneg((u + 1) * G + U - 1, U) - 1);
}

// CTAs whose unit ranges touch split tile ts: [first, last] (some in between
// may own no units at all when there are fewer units than CTAs).
PROJ_HD void split_tile_ctas(int32_t ts, int32_t k_blocks, int64_t U, int32_t G, int32_t &first,
                             int32_t &last) {
    const int64_t x0 = static_cast<int64_t>(ts) * k_blocks;
    first = cta_of_unit(x0, U, G);
    last = cta_of_unit(x0 + k_blocks - 1, U, G);
}

PROJ_HD bool cta_has_units(int32_t c, int64_t U, int32_t G) {
    return unit_begin(c, U, G) < unit_begin(c + 1, U, G);
}

// Partial-sum slot of CTA c's segment of split tile ts: 2c for the first tile
// of c's unit range, 2c + 1 for the last (a range spans at most one partial
// tile at each end; tiles it covers whole are never split).
PROJ_HD int32_t split_slot(int32_t c, int32_t ts, int64_t U, int32_t G, int32_t k_blocks) {
    return 2 * c + (ts == static_cast<int32_t>(div_nonneg(unit_begin(c, U, G), k_blocks)) ? 0 : 1);
}

// Tile index -> (token tile, weight tile).  Tiles are ordered in groups of
// raster_group token tiles: within a group the token tile varies fastest, then
// the weight tile, so the tiles running at the same time share a few token
// panels and a band of weight panels that stay in L2 together.
PROJ_HD void tile_coords(const KernelParams &p, int32_t tile, int32_t &tm, int32_t &tn) {
    const int32_t per_group = p.raster_group * p.tiles_n;
    const int32_t g = tile / per_group;
    const int32_t idx = tile - g * per_group;
    const int32_t m_base = g * p.raster_group;
    const int32_t gm = p.tiles_m - m_base < p.raster_group ? p.tiles_m - m_base : p.raster_group;
    tm = m_base + idx % gm;
    tn = idx / gm;
}

struct WorkIter {
    int32_t cta;
    int32_t dp_next;
    int64_t u, u_end;
    int32_t first_sk_tile;

    PROJ_HD void init(const KernelParams &p, int32_t c) {
        cta = c;
        if (p.cluster_split > 1) {
            // One segment: part c % P of tile c / P, an integer share of K,
            // with P = G·S parts per tile (G clusters of S CTAs; cluster
            // c / S is group (c / S) % G of its tile, rank c % S of it).
            const int32_t P = p.cluster_split * (p.cluster_groups > 1 ? p.cluster_groups : 1);
            const int32_t part = c % P;
            const int32_t tile = c / P;
            dp_next = -1;
            u = static_cast<int64_t>(tile) * p.k_blocks + div_nonneg(static_cast<int64_t>(part) * p.k_blocks, P);
            u_end = static_cast<int64_t>(tile) * p.k_blocks + div_nonneg(static_cast<int64_t>(part + 1) * p.k_blocks, P);
            first_sk_tile = tile;
            return;
        }
        dp_next = c;
        u = unit_begin(c, p.units_sk, p.grid);
        u_end = unit_begin(c + 1, p.units_sk, p.grid);
        first_sk_tile = static_cast<int32_t>(div_nonneg(u, p.k_blocks));
    }

    // Whole tiles first (c, c+G, ... below tiles_dp), then this CTA's split-K
    // units, cut at tile boundaries.
    PROJ_HD bool next(const KernelParams &p, Segment &s) {
        if (p.cluster_split > 1) {
            if (u >= u_end) return false;
            s.tile = first_sk_tile;
            s.kb0 = static_cast<int32_t>(u - static_cast<int64_t>(first_sk_tile) * p.k_blocks);
            s.kb1 = static_cast<int32_t>(u_end - static_cast<int64_t>(first_sk_tile) * p.k_blocks);
            s.split = true;
            s.slot = -1;
            u = u_end;
            return true;
        }
        if (dp_next < p.tiles_dp) {
            s.tile = dp_next;
            s.kb0 = 0;
            s.kb1 = p.k_blocks;
            s.slot = -1;
            s.split = false;
            dp_next += p.grid;
            return true;
        }
        if (u < u_end) {
            const int32_t ts = static_cast<int32_t>(div_nonneg(u, p.k_blocks));
            const int32_t kb0 = static_cast<int32_t>(u - static_cast<int64_t>(ts) * p.k_blocks);
            const int64_t left = u_end - u;
            const int32_t kb1 = left < static_cast<int64_t>(p.k_blocks - kb0)
                                    ? kb0 + static_cast<int32_t>(left)
                                    : p.k_blocks;
            s.tile = p.tiles_dp + ts;
            s.kb0 = kb0;
            s.kb1 = kb1;
            s.split = (kb0 != 0) || (kb1 != p.k_blocks);
            s.slot = s.split ? 2 * cta + (ts == first_sk_tile ? 0 : 1) : -1;
            u += kb1 - kb0;
            return true;
        }
        return false;
    }
};

// Work-shape fields of the kernel parameters, from a plan.
// Cluster split: every CTA reserves shared memory for the partial sums its
// peers send it, S - 1 partials of 32 rows x b_rows fp32 for each row quarter
// it reduces: quarter q is reduced by rank q mod S (S <= 4, so ceil(4 / S)
// quarters per reducer) or by rank q (S > 4, one quarter each).
PROJ_HD int32_t cluster_quarters_per_reducer(int32_t S) { return S <= 4 ? (4 + S - 1) / S : 1; }
PROJ_HD int32_t cluster_red_bytes(int32_t S, int32_t b_rows) {
    return S > 1 ? cluster_quarters_per_reducer(S) * (S - 1) * 32 * b_rows * 4 : 0;
}
// Token-major cluster split (at most 32 tokens, all in row quarter 0): rank
// c mod S adds 16-column chunk c of the block_n columns, receiving S - 1
// partial chunks of 32 rows x 16 fp32 (2 KiB) for each chunk it owns.
PROJ_HD int32_t cluster_red_bytes_tm(int32_t S, int32_t block_n) {
    const int32_t chunks = block_n / 16;
    return S > 1 ? ((chunks + S - 1) / S) * (S - 1) * 2048 : 0;
}

// B rows of the MMA (its N), and the B rows one CTA holds per stage (half of
// them in a CTA pair).
PROJ_HD int32_t plan_b_rows(const proj_plan_desc_t &plan) { return plan.swap_ab ? plan.block_t : plan.block_n; }
PROJ_HD int32_t plan_cta_b_rows(const proj_plan_desc_t &plan) {
    return plan.cta_pair ? plan_b_rows(plan) / 2 : plan_b_rows(plan);
}
// A rows per CTA: the weight rows of a swapped tile (64 for half tiles, 128
// of a pair's 256), else 128 token rows.
PROJ_HD int32_t plan_a_rows(const proj_plan_desc_t &plan) {
    return plan.swap_ab ? (plan.cta_pair ? plan.block_n / 2 : plan.block_n) : kBlockA;
}
// 64-wide k-blocks per stage, and the packed layout's k-blocks per weight
// tile (whole stages: the blocks past K are zero).
PROJ_HD int32_t plan_kpb(const proj_plan_desc_t &plan) {
    return plan.block_k > kBlockK ? plan.block_k / kBlockK : 1;
}
PROJ_HD int64_t plan_packed_kblocks(const proj_plan_desc_t &plan) { return plan.k_blocks * plan_kpb(plan); }
// Shared memory after the ring for a cluster split's incoming partial sums.
PROJ_HD int32_t plan_red_bytes(const proj_plan_desc_t &plan) {
    return plan.swap_ab ? cluster_red_bytes(plan.cluster_split, plan_b_rows(plan))
                        : cluster_red_bytes_tm(plan.cluster_split, plan.block_n);
}

inline void params_from_plan(const proj_plan_desc_t &plan, KernelParams &kp) {
    kp.swap = plan.swap_ab;
    kp.block_t = plan.block_t;
    kp.block_n = plan.block_n;
    kp.b_rows = plan_b_rows(plan);
    kp.tiles_m = static_cast<int32_t>(plan.tiles_m);
    kp.tiles_n = static_cast<int32_t>(plan.tiles_n);
    kp.raster_group = plan.raster_group > 0 ? plan.raster_group : static_cast<int32_t>(plan.tiles_m);
    kp.k_blocks = static_cast<int32_t>(plan.k_blocks);
    kp.kpb = plan.block_k > kBlockK ? plan.block_k / kBlockK : 1;
    kp.tiles_dp = static_cast<int32_t>(plan.tiles_dp);
    kp.cta_pair = plan.cta_pair;
    kp.grid = plan.cta_pair ? plan.grid / 2 : plan.grid;  // pairs own tiles, not CTAs
    kp.units_sk = plan.units_sk;
    kp.sk_pair = kp.grid > 0 && plan.units_sk / kp.grid >= plan.k_blocks;
    kp.sk_dense = plan.units_sk >= kp.grid;
    kp.cluster_split = plan.cluster_split;
    kp.cluster_groups = plan.cluster_split > 1 && plan.cluster_groups > 1 ? plan.cluster_groups : 1;
    if (kp.cluster_split > 1) kp.sk_pair = kp.sk_dense = 0;
    kp.stages = plan.stages;
    kp.a_rows = plan_a_rows(plan);
    kp.stage_bytes = kp.kpb * stage_bytes_for(kp.a_rows, plan_cta_b_rows(plan));
    kp.red_bytes = plan_red_bytes(plan);
    kp.tmem_cols = plan.tmem_cols;
    kp.acc_bufs = plan.tmem_cols >= 2 * kp.b_rows ? 2 : 1;
}

}  // namespace projgb
