// Host planner: cuts one projection problem into GPU work.  Pure host code (no
// CUDA calls), so it is exercised on machines without a GPU.
//
// Design points, with the worklog sections that motivate them ("How I made
// Muse's GPU projections 1.32× faster in the Open Kernel Challenge"):
//  * Enough independent work ("Having lots of workers doesn't help if I give
//    them nothing to do", "Enough active work, with enough resources"): the
//    grid is one CTA per SM, each CTA owning a deep shared-memory pipeline;
//    when there are fewer output tiles than SMs the K reduction is split
//    ("My first useful win: split up the sum").
//  * Block count arithmetic ("How splitting changes the grid"):
//    tiles = ceil(M/BT) · ceil(N/BN).
//  * Integer partition of K blocks ("Why the later TMA/WGMMA kernel was a new
//    experiment": 128 tiles over 3 splits → 42/43/43): CTA c owns units
//    [⌊c·U/G⌋, ⌊(c+1)·U/G⌋) so every unit is covered exactly once.
//  * Tile shape: the swapped product Yᵀ = W·Xᵀ ("Prove the swapped product
//    before worrying about its speed") puts 128 weight rows on the MMA's M
//    side and the token rows (16..256) on its N side, so small M does not
//    waste a 128-row MMA dimension.
#include "proj_internal.h"

#include <cstdio>

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int32_t pow2_ceil(int32_t v) {
    int32_t p = 1;
    while (p < v) p <<= 1;
    return p;
}

}  // namespace

namespace projgb {

int32_t token_tile_for(int64_t M) {
    if (M >= kMaxTokenTile) return kMaxTokenTile;
    int64_t bt = ceil_div(M < 1 ? 1 : M, 16) * 16;
    return static_cast<int32_t>(bt < 16 ? 16 : bt);
}

int32_t stage_bytes_for(int32_t a_rows, int32_t b_rows) {
    return a_rows * kBlockK * 2 + b_rows * kBlockK * 2;
}

}  // namespace projgb

using namespace projgb;

namespace projgb {

proj_status_t plan_compute(int64_t M, int64_t N, int64_t K, proj_wlayout_t w_layout,
                           proj_dtype_t y_dtype, int has_bias, const proj_device_desc_t *dev,
                           const PlanOptions &opt, proj_plan_desc_t *out) {
    const int32_t force_block_t = opt.force_block_t;
    const int32_t force_block_n = opt.force_block_n;
    if (!dev || !out) return PROJ_ERR_INVALID_ARG;
    *out = proj_plan_desc_t{};
    if (M < 0 || N < 0 || K < 0) return PROJ_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return PROJ_ERR_UNSUPPORTED;
    if (w_layout != PROJ_W_NK && w_layout != PROJ_W_KN) return PROJ_ERR_INVALID_ARG;
    if (y_dtype != PROJ_BF16 && y_dtype != PROJ_F32) return PROJ_ERR_INVALID_ARG;
    if (has_bias != 0 && has_bias != 1) return PROJ_ERR_INVALID_ARG;
    if (dev->sm_count < 1) return PROJ_ERR_INVALID_ARG;

    out->block_n = kBlockA;
    out->block_k = kBlockK;
    out->threads = kThreads;
    if (M == 0 || N == 0) {
        out->kernel = PROJ_KERNEL_NONE;
        return PROJ_OK;
    }
    if (K == 0) {
        out->kernel = PROJ_KERNEL_FILL;
        out->grid = static_cast<int32_t>(ceil_div(M * N, 256) < dev->sm_count * 8
                                             ? ceil_div(M * N, 256)
                                             : dev->sm_count * 8);
        out->threads = 256;
        return PROJ_OK;
    }
    if (force_block_t > 0 && (force_block_t % 16 != 0 || force_block_t > kMaxTokenTile))
        return PROJ_ERR_INVALID_ARG;
    const int32_t n_step = w_layout == PROJ_W_KN ? 64 : 16;  // [K,N] weights load in 64-row boxes
    if (force_block_n > 0 && (force_block_n % n_step != 0 || force_block_n > kMaxTokenTile))
        return PROJ_ERR_INVALID_ARG;
    const int64_t sms = dev->sm_count;

    // Orientation.  The swapped product (128 weight rows on the MMA's M side,
    // up to 256 token rows on its N side) serves every shape whose swapped
    // tiles cover the SMs; it measures faster than the token-major tiles of
    // the same size for the 4096-token prefill shape.  When 256-token swapped
    // tiles would leave SMs idle and there are at least 128 token rows, the
    // tokens take the M side and the weight rows the N side, whose width (a
    // multiple of 16) is free: it is chosen so the tiles fill whole waves.
    const bool swap_fills = ceil_div(M, kMaxTokenTile) * ceil_div(N, kBlockA) >= sms;
    // Token-major cluster split (option 2, at most 32 tokens): see the
    // cluster rule below.
    const bool tm_cluster = opt.tm_cluster == 2 && M <= 32 && force_block_t <= 0 && force_block_n <= 0 &&
                            opt.max_cluster >= 2;
    const bool swap = tm_cluster ? false
                      : force_block_n > 0 ? false
                                          : (force_block_t > 0 || M < kBlockA || swap_fills);
    int32_t bt, bn;
    if (swap) {
        bn = kBlockA;
        bt = force_block_t > 0 ? force_block_t : token_tile_for(M);
        if (force_block_t <= 0) {
            // With more token rows than one tile holds but fewer tiles than
            // SMs, halve the token tile until every SM has a tile.
            const int64_t tiles_n = ceil_div(N, kBlockA);
            while (bt > 64 && ceil_div(M, bt) * tiles_n < sms) {
                const int32_t half = static_cast<int32_t>(ceil_div(bt / 2, 16) * 16);
                if (half >= bt) break;
                bt = half;
            }
        }
        // Half tiles (an option, off by default): 64 weight rows per swapped
        // tile of at most 64 tokens (the MMA keeps M = 128; its rows 64-127
        // are not used), twice the tiles of a narrow few-tile shape.
        if (opt.half_tiles == 2 && bt <= 64) bn = kBlockA / 2;
    } else {
        bt = kBlockA;
        if (tm_cluster) {
            bn = kMaxTokenTile;
        } else if (force_block_n > 0) {
            bn = force_block_n;
        } else {
            // Per-SM time ~ waves x (block_n + a fixed share for the token
            // tile's own loads); the widest block_n wins ties.
            const int64_t tiles_m = ceil_div(M, bt);
            int64_t best_cost = -1;
            bn = kMaxTokenTile;
            for (int32_t cand = kMaxTokenTile; cand >= 64; cand -= n_step) {
                const int64_t tiles = tiles_m * ceil_div(N, cand);
                const int64_t waves = ceil_div(tiles, sms);
                const int64_t cost = waves * (cand + 32);
                if (best_cost < 0 || cost < best_cost) {
                    best_cost = cost;
                    bn = cand;
                }
            }
        }
    }
    const int32_t budget = dev->smem_optin_bytes - kSmemReserve;

    // CTA pairs: a tile of 256 rows on the MMA's M side, computed by the two
    // CTAs of a cluster with one cta_group::2 MMA per K step.  Each CTA
    // stages half of the B operand (the MMA reads both halves), so a stage
    // holds 16 KiB + b_rows/2 rows instead of 16 KiB + b_rows, and each CTA
    // pulls half the weight (token-major) or token (swapped) rows from L2
    // per FLOP.  Whole tiles only, dealt to pairs; the MMA's N side (b_rows)
    // between 64 and 256, a multiple of 32 (swapped) or 16 (token-major).  Chosen for the tensor-bound
    // swapped plans of 256-token tiles that keep at least half of the SMs
    // busy (measured on GB300, 4096 x 8192 x 8192: 359 us on pairs with one
    // accumulator vs 370 us on single CTAs).  Token-major pairs (more than
    // 128 tokens) are taken with two k-blocks a stage; with one they
    // measured no faster on the 256 x 12288 x 4096 QKV shape (27.9 vs
    // 27.7 us), so then only with option 2, which takes pairs wherever the
    // tile allows them.
    {
        const bool forced = opt.cta_pair == 2;
        const int64_t pairs_max = sms / 2;
        bool pair_swapped = swap && bt % 32 == 0 && bt >= 64;
        if (!forced)
            pair_swapped = pair_swapped && bt == kMaxTokenTile && 2 * bt <= kPairTmemMax &&
                           2 * ceil_div(M, bt) * ceil_div(N, 2 * kBlockA) >= pairs_max;
        // Two k-blocks a stage (K a multiple of 64, not turned off): also
        // token-major pairs by default (see below).
        const bool kpb2_ok = K % kBlockK == 0 && opt.kpb != 1;
        const bool pair_tm = (forced || (opt.cta_pair == 1 && kpb2_ok)) && !swap && M > kBlockA &&
                             (force_block_n <= 0 || force_block_n % 16 == 0);
        if (opt.cta_pair >= 1 && sms >= 2 && (pair_swapped || pair_tm)) {
            int32_t pbt = bt, pbn = bn;
            if (swap) {
                pbn = 2 * kBlockA;
            } else {
                pbt = 2 * kBlockA;
                if (force_block_n <= 0 && opt.pair_sk) {
                    pbn = kMaxTokenTile;  // stream-K evens out the pairs' work
                } else if (force_block_n <= 0) {
                    // As for single CTAs: per-pair time ~ waves x (block_n +
                    // a fixed share); the widest block_n wins ties.  Steps of
                    // 16 (each CTA holds half, a multiple of 8 rows): the QKV
                    // shape's 12288 rows fill 70 of 76 pairs at 176.
                    const int64_t tiles_m = ceil_div(M, pbt);
                    int64_t best_cost = -1;
                    for (int32_t cand = kMaxTokenTile; cand >= 64; cand -= 16) {
                        const int64_t waves = ceil_div(tiles_m * ceil_div(N, cand), pairs_max);
                        const int64_t cost = waves * (cand + 32);
                        if (best_cost < 0 || cost < best_cost) {
                            best_cost = cost;
                            pbn = cand;
                        }
                    }
                }
            }
            const int32_t pb_rows = swap ? pbt : pbn;
            // Two k-blocks a stage whenever K allows: each CTA's operands for
            // a stage come in two TMA ops of 32 KiB instead of two of
            // 16 KiB, and the per-op pacing of the loads (see the swapped
            // streaming plans below) had held the tensor pipe back.  Measured
            // on GB300, packed: 4096 x 8192 x 8192 on swapped pairs 298.5 us
            // (1842 TFLOP/s) against 350.4 us with one k-block a stage; the
            // 256 x 12288 x 4096 QKV shape on token-major pairs 27.2 us
            // against 31.3 us on single CTAs (34.3 us single CTAs with two
            // k-blocks, whose 80 KiB stages leave room for two).
            const int32_t pkpb = kpb2_ok ? 2 : 1;
            const int32_t pstage = pkpb * stage_bytes_for(kBlockA, pb_rows / 2);
            int32_t pstages = budget / pstage;
            if (pstages > kMaxStages) pstages = kMaxStages;
            const int64_t ptiles = ceil_div(M, pbt) * ceil_div(N, pbn);
            if (pstages >= 2 && (forced || 2 * ptiles >= pairs_max)) {
                out->kernel = PROJ_KERNEL_TC;
                out->cta_pair = 1;
                out->swap_ab = swap ? 1 : 0;
                out->block_t = pbt;
                out->block_n = pbn;
                // Two accumulator buffers when they fit the pair's tensor
                // memory, else one (the epilogue then waits for the MMAs).
                out->tmem_cols = 2 * pb_rows <= kPairTmemMax ? pow2_ceil(2 * pb_rows < 32 ? 32 : 2 * pb_rows)
                                                             : pow2_ceil(pb_rows < 32 ? 32 : pb_rows);
                out->tiles_m = ceil_div(M, pbt);
                out->tiles_n = ceil_div(N, pbn);
                int64_t g = 2048 / pbt;
                if (g < 1) g = 1;
                out->raster_group = static_cast<int32_t>(out->tiles_m < g ? out->tiles_m : g);
                out->block_k = pkpb * kBlockK;
                out->k_blocks = ceil_div(K, out->block_k);
                const int64_t tiles = out->tiles_m * out->tiles_n;
                // Stream-K over pairs (option pair_sk, token-major): the last
                // partial wave and one full wave before it are shared along K
                // by all pairs, as for single CTAs.  A split tile's partial
                // slots hold the pair's 256 rows; each CTA counts its own row
                // quarters (8 counters a tile).
                int64_t sk = 0;
                if (opt.pair_sk && !swap && tiles % pairs_max != 0)
                    sk = tiles < pairs_max ? tiles : tiles % pairs_max + pairs_max;
                out->grid = static_cast<int32_t>(2 * (tiles < pairs_max && sk == 0 ? tiles : pairs_max));
                out->tiles_dp = tiles - sk;
                out->tiles_sk = sk;
                out->units_sk = sk * out->k_blocks;
                out->stages = pstages;
                out->smem_bytes = pstages * pstage + kSmemReserve;
                out->scratch_bytes = 256;  // the status word
                if (sk > 0)
                    out->scratch_bytes += int64_t(2) * out->grid * kBlockA * pb_rows * 4 + ((sk * 8 * 4 + 255) / 256) * 256;
                return PROJ_OK;
            }
        }
    }

    const int32_t b_rows = swap ? bt : bn;
    // Half tiles stage only their 64 weight rows (the MMA's rows 64-127 read
    // whatever follows them in shared memory, into accumulator rows nobody
    // reads), so their stages are small and the ring deep.
    const bool half = swap && bn < kBlockA;
    // Two k-blocks a stage for the weight-streaming swapped plans (at most 64
    // tokens): one TMA op brings both k-blocks of the weight tile and one the
    // activations'.  On GB300 a CTA's TMA loads are paced per operation, not
    // per byte: measured with the loads alone, one 16 KiB op and one 2 KiB op
    // a stage streamed 61 GB/s of weights per SM, one 32 KiB and one 4 KiB
    // op 122 GB/s, so about 64 SMs instead of 110 keep HBM busy.  The
    // activations' 3-D tensor map needs K to be a multiple of 64.
    // (PROJ_KPB=2 also allows two for the other plans, as an experiment.)
    const int32_t kpb = (((swap && bt <= 64 && opt.kpb != 1) || opt.kpb == 2) && K % kBlockK == 0) ? 2 : 1;
    out->block_k = kpb * kBlockK;
    const int32_t stage = kpb * stage_bytes_for(half ? bn : kBlockA, b_rows);
    int32_t stages = budget / stage;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return PROJ_ERR_UNSUPPORTED;

    out->kernel = PROJ_KERNEL_TC;
    out->swap_ab = swap ? 1 : 0;
    out->block_t = bt;
    out->block_n = bn;
    // Two accumulator buffers (the epilogue of one tile overlaps the MMAs of
    // the next); TMEM is allocated in powers of two, at least 32 columns.
    out->tmem_cols = pow2_ceil(2 * b_rows < 32 ? 32 : 2 * b_rows);

    out->tiles_m = ceil_div(M, bt);
    out->tiles_n = ceil_div(N, bn);
    // Raster groups of about 2048 token rows: with K = 8192 a group's token
    // panels take 32 MiB, leaving room in L2 for the weight panels its wave
    // shares.
    {
        int64_t g = 2048 / bt;
        if (g < 1) g = 1;
        out->raster_group = static_cast<int32_t>(out->tiles_m < g ? out->tiles_m : g);
    }
    out->k_blocks = ceil_div(K, out->block_k);
    const int64_t tiles = out->tiles_m * out->tiles_n;
    const int64_t units = tiles * out->k_blocks;
    const int64_t grid = units < sms ? units : sms;
    out->grid = static_cast<int32_t>(grid);
    // Whole tiles in data-parallel waves, except that the last partial wave
    // and one full wave before it are shared along K by every CTA (the
    // "data-parallel + two-tile stream-K" hybrid).  Each CTA then owns at
    // least one tile's worth of K blocks, so a split tile has exactly two
    // contributors.  With fewer tiles than CTAs everything is split.  Whole
    // tiles only when the last wave is nearly full: 95 % for the swapped
    // (weight-streaming) plans, 80 % for the tensor-bound token-major plans,
    // whose split partial tiles are large.
    //
    // Cluster split: fewer (swapped, narrow) tiles than SMs, each split along
    // K over the S CTAs of one thread-block cluster whose partial sums meet
    // in distributed shared memory (no global scratch, no atomics).
    //   * Two k-blocks a stage: whenever S = SMs / tiles >= 2.  A CTA then
    //     streams up to twice the HBM share of one SM, so the S·tiles CTAs
    //     (at least half of the SMs) keep HBM busy, and the reduction in
    //     shared memory is cheaper than stream-K's through global memory.
    //     Measured on GB300 with packed weights, 16 tokens, K = 8192: 64
    //     tiles in clusters of 2 on 128 SMs 24.8 us, stream-K on 152 SMs
    //     26.2 us (26.1-26.5 on 128-144 SMs).
    //   * One k-block a stage: only while 3·tiles < SMs, when stream-K would
    //     give a split tile more than about three contributors.  With one
    //     k-block a stage a CTA streams at most about 50 GB/s, so idle SMs
    //     cost bandwidth: 64 tiles, stream-K 25.2 us vs clusters of 2
    //     26.2 us; 16 tiles, clusters of 6 on 96 SMs 12.6 us vs stream-K
    //     13.4 us; the 2 tiles of a 256-row router weight, clusters of 8 on
    //     16 SMs 14.6 us vs 16.3 us for stream-K at its best grid.
    // S goes up to 16 (a non-portable cluster size); the clusters must keep
    // cluster_fill_pct (10) % of the SMs busy.
    //
    // Token-major cluster split (at most 32 tokens): the same split over K,
    // with the tokens as the MMA's A rows (zero beyond M) and 256 weight rows
    // as its N side.  A CTA then streams 256 weight rows per MMA instruction
    // instead of 128: measured on GB300 with 48 busy SMs, 70 GB/s per SM
    // against 51 GB/s for 128 weight rows on either side.  Its partial sums
    // are 32 token rows x 256 columns; rank c mod S adds 16-column chunk c.
    auto red_for = [&](int32_t s_) {
        return swap ? cluster_red_bytes(s_, b_rows) : cluster_red_bytes_tm(s_, bn);
    };
    int32_t S = 0;
    if (opt.force_cluster >= 2 && swap && b_rows <= 64 && int64_t(opt.force_cluster) * tiles <= sms &&
        opt.force_cluster <= out->k_blocks && budget - red_for(opt.force_cluster) >= 2 * stage) {
        S = opt.force_cluster;
    } else if ((tm_cluster || (swap && b_rows <= 64)) && opt.max_cluster >= 2 &&
               (kpb == 2 ? 2 * tiles <= sms : 3 * tiles < sms)) {
        int64_t s_try = sms / tiles;
        if (s_try > opt.max_cluster) s_try = opt.max_cluster;
        if (s_try > out->k_blocks) s_try = out->k_blocks;
        if (s_try >= 2 && 100 * tiles * s_try >= int64_t(opt.cluster_fill_pct) * sms &&
            budget - red_for(static_cast<int32_t>(s_try)) >= 2 * stage)
            S = static_cast<int32_t>(s_try);
    }
    if (tm_cluster && S < 2) {
        // Not a cluster split after all: the ordinary plan.
        PlanOptions plain = opt;
        plain.tm_cluster = 0;
        return plan_compute(M, N, K, w_layout, y_dtype, has_bias, dev, plain, out);
    }
    // Several clusters per tile (forced with option cluster_groups): the G
    // clusters of S CTAs split the tile's K range into G·S parts; their
    // sums meet in the scratch.  Swapped splits only.
    int32_t G = 1;
    if (S >= 2 && swap && !tm_cluster && opt.cluster_groups >= 2 &&
        int64_t(opt.cluster_groups) * S * tiles <= sms && int64_t(opt.cluster_groups) * S <= out->k_blocks)
        G = opt.cluster_groups;
    // The peers' partial sums get their own shared memory after the ring.
    const int32_t red_bytes = red_for(S);
    if (stages * stage + red_bytes > budget) stages = (budget - red_bytes) / stage;
    const int64_t rem = tiles % grid;
    const int64_t waves = (tiles + grid - 1) / grid;
    const int64_t fill_pct = swap ? 95 : 80;
    if (S >= 2) {
        out->cluster_split = S;
        out->cluster_groups = G;
        out->grid = static_cast<int32_t>(tiles * S * G);
        out->tiles_sk = tiles;
    } else if (rem == 0 || 100 * tiles >= fill_pct * waves * grid) {
        out->tiles_sk = 0;
    } else if (tiles < grid) {
        out->tiles_sk = tiles;
    } else {
        out->tiles_sk = rem + grid;
    }
    out->tiles_dp = tiles - out->tiles_sk;
    out->units_sk = out->tiles_sk * out->k_blocks;
    // Whole tiles only: no more CTAs than tiles (the rest would have no work).
    if (out->tiles_sk == 0 && tiles < out->grid) out->grid = static_cast<int32_t>(tiles);

    // Pipeline depth.  When the weights stream from HBM (a single token tile,
    // or any split plan), about kInflightTarget bytes of stages per SM keep
    // the memory system busy; more only lengthens its queues (measured on
    // GB300: 8 stages of 18 KiB beat 12 for the 16-token decode shapes).  A
    // CTA with few k-blocks also pays the fill of a deep ring: at most a third
    // of its k-blocks (not for half tiles, whose small stages need the depth
    // to keep as many weight bytes in flight, nor for token-major cluster
    // splits, whose 48 KiB stages allow only three).  Data-parallel plans
    // over several token tiles are tensor-bound and keep the whole ring.
    const bool streaming = out->tiles_m == 1 || out->tiles_sk > 0;
    if (streaming) {
        int32_t want = opt.inflight_bytes / stage;
        // (Counted in 64-wide k-blocks: a stage of two counts twice.)
        const int64_t units_per_cta = kpb * (out->tiles_dp * out->k_blocks + out->units_sk) / out->grid;
        if (!half && !tm_cluster && units_per_cta / 3 < want) want = static_cast<int32_t>(units_per_cta / 3);
        if (want < 2) want = 2;
        if (want < stages) stages = want;
    }
    out->stages = stages;
    out->smem_bytes = stages * stage + red_bytes + kSmemReserve;

    // Scratch: one partial tile per (CTA, first|last split segment), one
    // completion counter per (split tile, 32-row quarter), and the device
    // status word.
    // (Clusters of a split over several clusters per tile: one partial tile
    // per (tile, cluster).)
    int64_t partial_bytes = 0;
    if (out->tiles_sk > 0 && S < 2) partial_bytes = 2 * grid * int64_t(kBlockA) * b_rows * 4;
    if (S >= 2 && G >= 2) partial_bytes = out->tiles_sk * G * int64_t(kBlockA) * b_rows * 4;
    const int64_t counter_bytes = (S < 2 || G >= 2) ? ((out->tiles_sk * 4 * 4 + 255) / 256) * 256 : 0;
    out->scratch_bytes = partial_bytes + counter_bytes + 256;
    (void)has_bias;
    return PROJ_OK;
}

}  // namespace projgb

extern "C" proj_status_t proj_plan_compute(int64_t M, int64_t N, int64_t K,
                                           proj_wlayout_t w_layout, proj_dtype_t y_dtype,
                                           int has_bias, const proj_device_desc_t *dev,
                                           proj_plan_desc_t *out) {
    return plan_compute(M, N, K, w_layout, y_dtype, has_bias, dev, PlanOptions{}, out);
}

static bool plan_is_tc(const proj_plan_desc_t *plan) {
    return plan && plan->kernel == PROJ_KERNEL_TC && plan->grid > 0 && plan->k_blocks > 0 &&
           plan->tiles_m > 0;
}

extern "C" proj_status_t proj_plan_segments(const proj_plan_desc_t *plan, int32_t cta,
                                            proj_segment_t *out, int64_t cap, int64_t *count) {
    if (!count || (cap > 0 && !out) || cap < 0) return PROJ_ERR_INVALID_ARG;
    *count = 0;
    if (!plan) return PROJ_ERR_INVALID_ARG;
    if (plan->kernel != PROJ_KERNEL_TC) return PROJ_OK;
    if (!plan_is_tc(plan) || cta < 0 || cta >= plan->grid) return PROJ_ERR_INVALID_ARG;
    KernelParams kp{};
    params_from_plan(*plan, kp);
    WorkIter it;
    it.init(kp, plan->cta_pair ? cta / 2 : cta);  // both CTAs of a pair run the pair's tiles
    Segment s;
    int64_t n = 0;
    while (it.next(kp, s)) {
        if (n < cap) {
            proj_segment_t &o = out[n];
            o.tile = s.tile;
            tile_coords(kp, s.tile, o.tile_m, o.tile_n);
            o.k_block_begin = s.kb0;
            o.k_block_end = s.kb1;
            o.slot = s.slot;
            o.split = s.split ? 1 : 0;
            o.reserved = 0;
        }
        ++n;
    }
    *count = n;
    return PROJ_OK;
}

extern "C" proj_status_t proj_plan_reduction_order(const proj_plan_desc_t *plan, int64_t split_tile,
                                                   int32_t *ctas, int32_t *slots, int64_t cap,
                                                   int64_t *count) {
    if (!count || cap < 0 || (cap > 0 && (!ctas || !slots))) return PROJ_ERR_INVALID_ARG;
    *count = 0;
    if (!plan_is_tc(plan) || split_tile < 0 || split_tile >= plan->tiles_sk)
        return PROJ_ERR_INVALID_ARG;
    const int32_t ts = static_cast<int32_t>(split_tile);
    const int32_t kt = static_cast<int32_t>(plan->k_blocks);
    if (plan->cluster_split > 1) {
        // Cluster split: parts 0..P-1 of the tile (P = G·S), in K order.
        // Each cluster adds its S ranks in rank order in distributed shared
        // memory (slot -1 with one cluster per tile); with G clusters per
        // tile, cluster g's sum goes to scratch slot ts·G + g, and the G sums
        // are added in group order.
        const int32_t S = plan->cluster_split;
        const int32_t G = plan->cluster_groups > 1 ? plan->cluster_groups : 1;
        for (int32_t r = 0; r < G * S; ++r)
            if (r < cap) {
                ctas[r] = ts * G * S + r;
                slots[r] = G > 1 ? ts * G + r / S : -1;
            }
        *count = G * S;
        return PROJ_OK;
    }
    // Stream-K: CTAs (pairs, for a CTA-pair plan) in ascending order.
    const int32_t g = plan->cta_pair ? plan->grid / 2 : plan->grid;
    int32_t first, last;
    split_tile_ctas(ts, kt, plan->units_sk, g, first, last);
    int64_t n = 0;
    for (int32_t c = first; c <= last; ++c) {
        if (!cta_has_units(c, plan->units_sk, g)) continue;
        if (n < cap) {
            ctas[n] = c;
            slots[n] = split_slot(c, ts, plan->units_sk, g, kt);
        }
        ++n;
    }
    *count = n;
    return PROJ_OK;
}

namespace projgb {

int plan_to_json(const proj_plan_desc_t &p, int64_t M, int64_t N, int64_t K, int w_layout,
                 int y_dtype, int has_bias, char *buf, size_t len) {
    static const char *kernels[] = {"none", "fill", "tc_tma_tcgen05"};
    const char *kname = (p.kernel >= 0 && p.kernel <= 2) ? kernels[p.kernel] : "?";
    return std::snprintf(
        buf, len,
        "{\"kernel\": \"%s\", \"M\": %lld, \"N\": %lld, \"K\": %lld, \"w_layout\": \"%s\", "
        "\"y_dtype\": \"%s\", \"bias\": %s, \"block_n\": %d, \"block_t\": %d, \"block_k\": %d, "
        "\"stages\": %d, \"grid\": %d, \"threads\": %d, \"smem_bytes\": %d, "
        "\"tmem_cols\": %d, \"raster_group\": %d, \"swap_ab\": %d, \"cluster_split\": %d, \"cluster_groups\": %d, \"cta_pair\": %d, \"tiles_m\": %lld, \"tiles_n\": %lld, \"k_blocks\": %lld, "
        "\"tiles_dp\": %lld, \"tiles_sk\": %lld, \"units_sk\": %lld, \"scratch_bytes\": %lld}",
        kname, (long long)M, (long long)N, (long long)K, w_layout == PROJ_W_NK ? "NK" : "KN",
        y_dtype == PROJ_F32 ? "f32" : "bf16", has_bias ? "true" : "false", p.block_n,
        p.block_t, p.block_k, p.stages, p.grid, p.threads, p.smem_bytes, p.tmem_cols, p.raster_group,
        p.swap_ab, p.cluster_split, p.cluster_groups, p.cta_pair,
        (long long)p.tiles_m, (long long)p.tiles_n, (long long)p.k_blocks,
        (long long)p.tiles_dp, (long long)p.tiles_sk, (long long)p.units_sk,
        (long long)p.scratch_bytes);
}

}  // namespace projgb
