/*
 * proj.h: C ABI of the GB300 dense projection library (libproj_gb300).
 *
 * Computes the dense projection of transformer inference
 *
 *     Y[m, n] = Σ_{k=0}^{K-1} X[m, k] · W[n, k]   (+ bias[n])
 *
 * ("How I made Muse's GPU projections 1.32× faster in the Open Kernel
 * Challenge", section "The full equation, now with the letters explained";
 * the bias makes it the affine map of section "What makes it linear?").
 * X is [M, K] token activations, W holds N rows of K weights, Y is [M, N].
 * Products are bf16 × bf16 with fp32 accumulation; the output is stored as
 * fp32 or rounded once to bf16 (round-to-nearest-even), after the bias is
 * added (section "Inputs, products, accumulators, and outputs are separate
 * choices").
 *
 * Memory and ownership
 *   - Every tensor pointer passed to proj_run is a DEVICE pointer owned by the
 *     caller (e.g. allocated by PyTorch).  The library never frees or keeps
 *     them beyond the call, apart from caching the tensor-map descriptors
 *     built from them.
 *   - Streams are owned by the caller and passed as `void*` holding a
 *     cudaStream_t (NULL means the legacy default stream).
 *   - A handle owns its plan, its split-K scratch (partial sums, completion
 *     counters) and a device status word.  proj_create allocates them once;
 *     proj_run allocates nothing, never synchronises the host and may be
 *     captured into a CUDA graph.  Scratch partial sums are fully rewritten
 *     before they are read and counters return to zero inside every run, so
 *     no memset is needed between runs.
 *   - One handle must not run on two streams at the same time (its scratch is
 *     shared).  Different handles are independent.
 *
 * Layouts (section "What a matrix looks like in memory")
 *   X: [M, K] row-major, K contiguous, bf16.
 *   W: PROJ_W_NK: [N, K] row-major, element (n,k) at n·K + k.
 *      PROJ_W_KN: the copied transpose [K, N], element (n,k) at k·N + n.
 *   bias: [N] bf16 or NULL.   Y: [M, N] row-major, fp32 or bf16.
 *
 * Alignment (TMA global strides and addresses must be 16-byte multiples):
 *   X and W base addresses 16-byte aligned; K % 8 == 0 (X rows and [N,K]
 *   weight rows are whole 16-byte multiples); for PROJ_W_KN bf16 weights also
 *   N % 8 == 0 (fp32 router weights are read only by proj_pack_weights).
 *   Violations return PROJ_ERR_MISALIGNED and launch nothing.
 *
 * Errors: every call returns a proj_status_t; nothing aborts or throws across
 * the ABI.  CUDA launch failures surface as PROJ_ERR_CUDA.  Device-side waits
 * are bounded (about one second); a wait that runs out records itself in the
 * handle's status word, the kernel returns early, and proj_device_status
 * reports PROJ_ERR_DEVICE_TIMEOUT.
 *
 * Determinism: for one handle and the same inputs every run writes the same
 * bytes.  The split of K across CTAs is fixed when the handle is planned, and
 * partial sums are combined in a fixed order (no floating-point atomics).
 */
#ifndef PROJ_GB300_PROJ_H
#define PROJ_GB300_PROJ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct proj_plan_s *proj_handle_t;

typedef enum proj_status {
    PROJ_OK = 0,
    PROJ_ERR_INVALID_ARG = 1,    /* bad shape, NULL pointer, bias/has_bias mismatch */
    PROJ_ERR_UNSUPPORTED = 2,    /* dtype or device this library does not handle */
    PROJ_ERR_MISALIGNED = 3,     /* a TMA alignment rule above is violated */
    PROJ_ERR_OUT_OF_MEMORY = 4,  /* scratch allocation failed */
    PROJ_ERR_CUDA = 5,           /* a CUDA runtime/driver call failed */
    PROJ_ERR_DEVICE_TIMEOUT = 6  /* a bounded device-side wait ran out */
} proj_status_t;

typedef enum proj_dtype { PROJ_BF16 = 0, PROJ_F32 = 1 } proj_dtype_t;

typedef enum proj_wlayout { PROJ_W_NK = 0, PROJ_W_KN = 1 } proj_wlayout_t;

/* Which device code a plan runs. */
typedef enum proj_kernel {
    PROJ_KERNEL_NONE = 0,  /* M == 0 or N == 0: nothing to compute */
    PROJ_KERNEL_FILL = 1,  /* K == 0: every sum is empty, Y = bias (or 0) */
    PROJ_KERNEL_TC = 2     /* TMA + tcgen05/TMEM persistent projection kernel */
} proj_kernel_t;

/*
 * Device properties the planner needs.  Filled from cudaGetDeviceProperties by
 * proj_create; tests may pass their own (the planner is pure host code).
 */
typedef struct proj_device_desc {
    int32_t sm_count;           /* streaming multiprocessors (152 on GB300) */
    int32_t smem_optin_bytes;   /* max dynamic shared memory per block (opt-in) */
} proj_device_desc_t;

/*
 * A plan: how one problem is cut into work for the GPU.
 *
 * Tiles: block_t token rows × block_n weight rows × the whole K range, cut
 * into k_blocks blocks of block_k.  With few tokens (M < 128) the swapped
 * product Yᵀ = W·Xᵀ puts 128 weight rows on the tensor-core MMA's M side and
 * the tokens (16..112) on its N side (section "Prove the swapped product
 * before worrying about its speed"); with M ≥ 128, 128 tokens take the M side
 * and block_n weight rows (a multiple of 16, of 64 for [K,N] weights) the N
 * side, block_n chosen so the tiles fill whole waves of SMs.
 * Whole tiles are dealt out in data-parallel waves (tiles_dp); the remaining
 * tiles_sk tiles (the last partial wave plus one full wave, or every tile when
 * there are fewer tiles than CTAs; none when the last wave is nearly full) are
 * split along K
 * into units_sk k-block units shared contiguously by all CTAs ("split-K",
 * section "My first useful win: split up the sum"; CTA c takes units
 * [⌊c·U/G⌋, ⌊(c+1)·U/G⌋), the integer partition of section "Why the later
 * TMA/WGMMA kernel was a new experiment" that splits 128 tiles 42/43/43).
 * Cluster split instead (cluster_split = S ≥ 2): when there are fewer than a
 * third as many narrow swapped tiles as SMs (stream-K would give a tile more
 * than three contributors) and S CTAs per tile (S ≤ 16) keep at least 10 % of the SMs busy,
 * each tile gets its own cluster of S CTAs, grid = tiles_sk · S, and the
 * partial sums meet in distributed shared memory; no partial-sum scratch and
 * no counters.
 * CTA pairs (cta_pair = 1): the tensor-bound shapes whose tiles are computed
 * whole (several token tiles) run each tile on two CTAs of a cluster.  One
 * MMA spans both CTAs' shared memory, so each CTA holds half of the B operand
 * per stage: fewer bytes per stage, a deeper ring and half the weight (or
 * token) rows per CTA from L2.
 */
typedef struct proj_plan_desc {
    int32_t kernel;          /* proj_kernel_t */
    int32_t block_n;         /* weight rows per tile: 128 when swap_ab, else 64..256 */
    int32_t block_t;         /* token rows per tile: 16..256 when swap_ab, else 128 */
    int32_t block_k;         /* K elements per pipeline stage (64 = 128 bytes) */
    int32_t stages;          /* shared-memory pipeline depth */
    int32_t grid;            /* CTAs launched (one per SM at most) */
    int32_t threads;         /* threads per CTA */
    int32_t smem_bytes;      /* dynamic shared memory per CTA */
    int32_t tmem_cols;       /* tensor-memory columns allocated per CTA */
    int32_t raster_group;    /* token tiles per raster group: tiles are numbered group by group,
                                token tile fastest within a group, then weight tile */
    int32_t swap_ab;         /* 1: weight rows on the MMA's M side (128), tokens on its N side
                                (block_t); 0: tokens on the M side (128), weight rows on the N
                                side (block_n) */
    int32_t cluster_split;   /* 0, or S >= 2: every tile is split along K over the S CTAs of one
                                thread-block cluster (CTA c: tile c / S, rank c % S, k-blocks
                                [⌊r·k_blocks/S⌋, ⌊(r+1)·k_blocks/S⌋)), and the partial sums are
                                added through distributed shared memory in rank order */
    int32_t cta_pair;        /* 1: every tile is computed by a pair of CTAs (a cluster of 2) with
                                one 256-row tensor-core MMA (tcgen05 cta_group::2).  The pair
                                tile is 256 rows on the MMA's M side (block_n = 256 weight rows
                                when swap_ab, else block_t = 256 tokens); each CTA loads half
                                of the tile's weight rows and half of its token rows, and holds
                                128 of the M rows' accumulators.  grid counts CTAs (2 per pair);
                                tiles are dealt to pairs.  Whole tiles only (tiles_sk = 0) */
    int64_t tiles_m;         /* ceil(M / block_t) */
    int64_t tiles_n;         /* ceil(N / block_n) */
    int64_t k_blocks;        /* ceil(K / block_k) */
    int64_t tiles_dp;        /* tiles computed whole, dealt round-robin (CTA c: c, c+grid, ...);
                                a multiple of grid whenever tiles_sk > 0 */
    int64_t tiles_sk;        /* tiles split along K across CTAs */
    int64_t units_sk;        /* tiles_sk * k_blocks */
    int64_t scratch_bytes;   /* device scratch the handle owns */
    int32_t cluster_groups;  /* with cluster_split S >= 2: 0 or 1, one cluster per tile; G >= 2,
                                each tile's K range is split over G clusters of S CTAs (grid =
                                tiles_sk * G * S; CTA c: tile c / (G·S), part p = c % (G·S),
                                k-blocks [⌊p·k_blocks/(G·S)⌋, ⌊(p+1)·k_blocks/(G·S)⌋)).  Each
                                cluster adds its ranks' partial sums in rank order; the G
                                cluster sums meet in the handle's scratch and the cluster that
                                completes last adds them in group order */
} proj_plan_desc_t;

/*
 * Plan a problem without touching a GPU (pure host code).
 * Returns PROJ_ERR_INVALID_ARG for negative sizes, a bad layout, or a NULL
 * dev/out; PROJ_ERR_UNSUPPORTED if the device cannot hold two pipeline stages.
 * This is the plan proj_create uses, except that proj_create lowers
 * cluster_split (down to a plain split-K plan) when the device cannot keep
 * every tile's cluster resident at once.
 */
proj_status_t proj_plan_compute(int64_t M, int64_t N, int64_t K, proj_wlayout_t w_layout,
                                proj_dtype_t y_dtype, int has_bias,
                                const proj_device_desc_t *dev, proj_plan_desc_t *out);

/* One stretch of work a CTA executes: k-blocks [k_block_begin, k_block_end)
 * of one tile (its index in raster order and its token/weight coordinates). */
typedef struct proj_segment {
    int32_t tile;
    int32_t tile_m;          /* token-row tile */
    int32_t tile_n;          /* weight-row tile */
    int32_t k_block_begin;
    int32_t k_block_end;
    int32_t slot;            /* partial-sum slot when split, else -1 (also -1 in cluster splits) */
    int32_t split;           /* 1 if other CTAs own the rest of this tile's K range */
    int32_t reserved;
} proj_segment_t;

/*
 * Host introspection of a PROJ_KERNEL_TC plan (pure host code, the same
 * decomposition code the kernel runs): the segments CTA `cta` executes, in
 * order (in a CTA-pair plan, CTAs 2p and 2p + 1 both run pair p's tiles).  Writes min(cap, total) segments to `out` and the total to *count.
 * A plan of another kernel kind yields zero segments.  PROJ_ERR_INVALID_ARG
 * for a NULL count/plan, a negative cap, or cta outside [0, grid).
 */
proj_status_t proj_plan_segments(const proj_plan_desc_t *plan, int32_t cta, proj_segment_t *out,
                                 int64_t cap, int64_t *count);

/*
 * The order in which the partial sums of split tile `split_tile`
 * (0 ≤ split_tile < tiles_sk; tile index tiles_dp + split_tile) are added:
 * contributing CTAs (pair indices for a CTA-pair plan) in ascending order
 * with their partial-sum slots.  Writes
 * min(cap, total) pairs and the total to *count.  For a cluster split the
 * CTAs are the tile's parts, split_tile·P .. split_tile·P + P − 1 (P = G·S,
 * G = max(1, cluster_groups)), each with slot −1 when G = 1, else with its
 * cluster's scratch slot split_tile·G + (part / S): each cluster adds its
 * ranks in rank order, then the G cluster sums are added in group order.
 */
proj_status_t proj_plan_reduction_order(const proj_plan_desc_t *plan, int64_t split_tile,
                                        int32_t *ctas, int32_t *slots, int64_t cap,
                                        int64_t *count);

/*
 * Create a handle for one problem shape on the current CUDA device.
 *   M, N, K ≥ 0 (a zero M or N plans nothing; K == 0 plans Y = bias or 0).
 *   x_dtype, bias_dtype: PROJ_BF16 only (else PROJ_ERR_UNSUPPORTED).
 *   w_dtype: PROJ_BF16, or PROJ_F32 for fp32 router weights, computed as the
 *     worklog's high/low bf16 split (section "Why the high-plus-low router
 *     scheme helped"): H = roundBF16(W), L = roundBF16(W − FP32(H)),
 *     Y = X·Hᵀ + X·Lᵀ summed in one fp32 accumulator.  The split happens
 *     when the weights are packed: such a handle runs only through
 *     proj_pack_weights (fp32 W in) and proj_run_packed / proj_run_host_packed;
 *     proj_run and proj_run_host return PROJ_ERR_UNSUPPORTED.  Its plan
 *     covers [H | L] along K: k_blocks = 2·ceil(K / 64).
 *   y_dtype: PROJ_BF16 or PROJ_F32.   has_bias: 0 or 1.
 *   stream: cudaStream_t used to clear the new scratch; create synchronises it
 *   before returning, so the handle may be used on any stream afterwards.
 * Allocates scratch with cudaMalloc (PROJ_ERR_OUT_OF_MEMORY on failure).
 * The device must be compute capability 10.3 (GB300); else PROJ_ERR_UNSUPPORTED.
 * On failure *out is set to NULL.
 *
 * Tuning overrides (environment, read once here; for experiments and tests,
 * every plan they produce computes the same projection):
 *   PROJ_FORCE_BLOCK_T=t     swapped orientation with token tile t (multiple of 16)
 *   PROJ_FORCE_BLOCK_N=n     token-major orientation with weight tile n
 *   PROJ_MAX_CLUSTER=s       largest cluster split (0 or 1: none)
 *   PROJ_CLUSTER_FILL_PCT=f  SMs (%) a cluster split must keep busy
 *   PROJ_CTA_PAIR=0|2        CTA pairs off, or on wherever the tile allows them
 *   PROJ_HALF_TILES=2        swapped tiles of 64 weight rows (at most 64 tokens)
 *   PROJ_TM_CLUSTER=1|2      token-major cluster splits for at most 32 tokens (1: where they
 *                            keep 70 % of a swapped cluster split's SMs; 2: wherever they apply)
 *   PROJ_FORCE_STAGES=k      fewer pipeline stages than planned
 *   PROJ_FORCE_GRID=g        fewer CTAs for an all-split plan
 *   PROJ_FORCE_WHOLE_TILES=1 no split tiles
 *   PROJ_FORCE_RASTER_GROUP=r token tiles per raster group
 *   PROJ_PREFETCH_STAGES=k   weight stages streamed early in PROJ_OVERLAP_WEIGHTS
 *   PROJ_KPB=1|2             one 64-wide k-block a pipeline stage, or two wherever K allows
 *                            (default: two for the weight-streaming swapped plans)
 *   PROJ_INFLIGHT_KB=n       stage bytes a weight-streaming plan keeps in flight per SM
 *   PROJ_FORCE_CLUSTER=s     cluster split of s CTAs per tile where the clusters fit the SMs
 *   PROJ_CLUSTER_GROUPS=g    g clusters per tile for a swapped cluster split (1: one)
 *   PROJ_PAIR_SK=1           stream-K over CTA pairs for token-major pair tiles of 256 columns
 */
proj_status_t proj_create(proj_handle_t *out, int64_t M, int64_t N, int64_t K,
                          proj_wlayout_t w_layout, proj_dtype_t x_dtype,
                          proj_dtype_t w_dtype, proj_dtype_t y_dtype, int has_bias,
                          proj_dtype_t bias_dtype, void *stream);

/*
 * Enqueue Y = X·Wᵀ (+ bias) on `stream`.  X, W, bias, Y are device pointers
 * with the layouts above; bias must be NULL iff the handle has no bias.
 * Asynchronous: returns once the launch is queued.  No allocation, no host
 * synchronisation; safe inside CUDA-graph capture.
 */
proj_status_t proj_run(proj_handle_t h, const void *X, const void *W, const void *bias,
                       void *Y, void *stream);

/*
 * Pre-packed weights, a preparation step outside the timed call.  The
 * worklog's contract let preparation pack fixed weights (section "Preparation
 * is not secretly computing the answer"), and its C2 experiments kept each
 * output tile's weights next to each other in memory (section "Sometimes
 * moving the same numbers around was enough").
 *
 * The handle's packed layout is one block per (weight tile t, k-block b), in
 * the order t·k_blocks + b.  Each block holds block_n rows × 64 K values in
 * bf16, K contiguous (128 bytes a row).  Rows at or past N and K positions at
 * or past K are zero.  Every pipeline stage of a packed run then reads one
 * contiguous block of block_n × 128 bytes, and [K,N] weights become K-major.
 * The layout follows the plan's block_n, so packed weights are used with the
 * handle that packed them (or one with the same plan).
 *
 * proj_packed_weight_bytes: the packed size, tiles_n · k_blocks · block_n ·
 *   128 bytes (0 for plans without the tensor-core kernel).
 *   PROJ_ERR_UNSUPPORTED if the packed rows would not fit 31-bit coordinates.
 * proj_pack_weights: W (device, the handle's layout and w_dtype: bf16, or
 *   fp32 for a PROJ_F32 handle, which stores the H blocks of a tile followed
 *   by its L blocks) → W_packed (device, proj_packed_weight_bytes bytes,
 *   16-byte aligned, caller-owned), enqueued on `stream`.  W must not overlap
 *   W_packed.
 * proj_run_packed: proj_run with packed weights; same arguments otherwise.
 * PROJ_ERR_INVALID_ARG for NULL handles or pointers, PROJ_ERR_MISALIGNED for
 * unaligned pointers, PROJ_ERR_CUDA if a launch fails.
 */
proj_status_t proj_packed_weight_bytes(proj_handle_t h, size_t *bytes);
proj_status_t proj_pack_weights(proj_handle_t h, const void *W, void *W_packed, void *stream);
proj_status_t proj_run_packed(proj_handle_t h, const void *X, const void *W_packed,
                              const void *bias, void *Y, void *stream);
/*
 * Fused epilogues.  The worklog's second page writes the FFN intermediate
 * once by fusing its GELU into the projection's epilogue, and fuses the
 * residual add that follows an output projection; the first page, section
 * "Normalization and residuals also cost time", says why: the extra pass
 * over the activations costs time of its own.
 *
 *   Y = act(X·Wᵀ + bias) + residual,
 *
 * computed in fp32 and rounded once to Y's type.  act is the handle's
 * activation (proj_set_activation; PROJ_ACT_NONE by default): PROJ_ACT_GELU
 * is GELU(x) = x/2 · (1 + erf(x/√2)).  residual is an [M,N] array in Y's
 * type and layout, or NULL; it may be Y itself (each element is read before
 * it is written).  proj_run_fused: packed = 1 takes packed weights (as
 * proj_run_packed), 0 weights as stored; otherwise as proj_run.
 *
 * PROJ_ACT_SWIGLU (Shazeer, "GLU Variants Improve Transformer"; the first
 * page's expert pattern of a gate vector through a nonlinearity times an up
 * vector): W stacks the F = N / 2 gate rows, then the F up rows ([N,K], or
 * [K,N] with gate columns first), and Y[m,f] = SiLU(G[m,f]) · U[m,f]
 * (+ residual), Y and the residual [M, F], SiLU(x) = x / (1 + e^(−x)).  Set
 * it before proj_pack_weights, which interleaves each tile's gate and up rows
 * so they meet in one epilogue warp; such a handle runs only packed
 * (proj_run_packed, or proj_run_fused with packed = 1).  proj_set_activation
 * returns PROJ_ERR_UNSUPPORTED for SwiGLU on a handle with a bias, an odd N,
 * or fp32 weights; an unpacked run returns PROJ_ERR_UNSUPPORTED.
 * PROJ_ERR_INVALID_ARG for an unknown activation or packed flag;
 * PROJ_ERR_MISALIGNED for a residual not aligned to Y's element size.
 */
typedef enum proj_activation {
    PROJ_ACT_NONE = 0,
    PROJ_ACT_GELU = 1,
    PROJ_ACT_SWIGLU = 2
} proj_activation_t;

proj_status_t proj_set_activation(proj_handle_t h, proj_activation_t act);
proj_status_t proj_run_fused(proj_handle_t h, const void *X, const void *W, int packed,
                             const void *bias, const void *residual, void *Y, void *stream);

/* proj_run_host with packed weights (W_packed on the device). */
proj_status_t proj_run_host_packed(proj_handle_t h, const void *X_host, const void *W_packed,
                                   const void *bias, void *Y_host, void *stream);

/*
 * Same projection with HOST activations: copies X_host ([M,K] bf16) to a
 * device staging buffer, runs, and copies Y back to Y_host, all on `stream`.
 * W and bias stay device pointers (weights are resident, as after a
 * preparation step).  A pinned or registered X_host (16-byte aligned) is
 * copied by a small kernel chained to the projection by programmatic
 * dependent launch; a pinned or registered Y_host (16-byte aligned) is written
 * by the projection's epilogue itself, through its device address, with no
 * staging copy.  Other host memory goes through cudaMemcpyAsync and the
 * staging buffers (asynchronous only when pinned).  Y_host is valid once
 * `stream` has been synchronised.  The staging
 * buffers are allocated by the first call on a handle (so that first call is
 * not capturable) and reused afterwards.
 */
proj_status_t proj_run_host(proj_handle_t h, const void *X_host, const void *W,
                            const void *bias, void *Y_host, void *stream);

/*
 * Synchronise `stream` and read the handle's device status word.  Returns
 * PROJ_ERR_DEVICE_TIMEOUT if a bounded device wait ran out in any earlier run,
 * PROJ_ERR_CUDA if a run found its launch given less shared memory than its
 * pipeline needs or clusters of another size than its plan's (internal
 * launch errors; the kernel then did nothing) or the synchronisation failed,
 * else PROJ_OK.  A non-zero word is cleared,
 * together with the split-K counters, so the handle can be reused.
 */
proj_status_t proj_device_status(proj_handle_t h, void *stream);

/*
 * How a run may overlap the kernel launched before it on the same stream
 * (programmatic dependent launch; the worklog's section "The later version
 * really did reach 1.32×" describes the idea: start the independent part
 * early, wait where it matters).
 *   PROJ_OVERLAP_NONE      plain stream order.
 *   PROJ_OVERLAP_PROLOGUE  (default) the kernel may start while the preceding
 *                          kernel finishes, but touches no global memory (no
 *                          X, W, bias, Y or scratch) until that kernel has
 *                          completed: always safe.
 *   PROJ_OVERLAP_WEIGHTS   as above, and the first pipeline stages of W are
 *                          streamed before the preceding kernel completes,
 *                          for plans that occupy every SM.  (A plan that
 *                          leaves SMs idle would start streaming there while
 *                          the preceding kernel still streams its own data,
 *                          and delay it: such plans behave as PROLOGUE.)
 *                          The caller promises that W is not written by the
 *                          kernel launched just before the run (true for
 *                          inference weights).
 * PROJ_ERR_INVALID_ARG for a NULL handle or an unknown mode.
 */
typedef enum proj_overlap {
    PROJ_OVERLAP_NONE = 0,
    PROJ_OVERLAP_PROLOGUE = 1,
    PROJ_OVERLAP_WEIGHTS = 2
} proj_overlap_t;

proj_status_t proj_set_overlap(proj_handle_t h, proj_overlap_t mode);

/*
 * Phase trace (diagnostics).  With a device buffer of at least
 * grid × 16 × 8 bytes (grid from the plan) every later proj_run writes, per
 * CTA, 16 unsigned 64-bit words: [0] kernel entry, [1] set-up done,
 * [2] first TMA load issued, [3] last TMA load issued, [4] first stage seen
 * by the MMA issuer, [5] last accumulator committed, [6] first accumulator
 * received by the epilogue, [7] epilogue finished, [8] final barrier
 * (globaltimer nanoseconds), [9] the SM id, [10] split tiles reduced by the
 * CTA's first epilogue warp, [11] producer past the grid-dependency wait,
 * [12] epilogue past it; for the first split tile of that warp: [13] its
 * partial sums written, [14] all partials of the tile known to be in (or,
 * for a warp that does not reduce, the same as [13]), [15] the reduced rows
 * stored (or handed over).  The caller owns the buffer; a
 * NULL buffer turns tracing off.  PROJ_ERR_INVALID_ARG if the buffer is too
 * small, PROJ_ERR_MISALIGNED if not 8-byte aligned, PROJ_ERR_UNSUPPORTED for
 * plans without the tensor-core kernel.
 */
proj_status_t proj_set_trace(proj_handle_t h, void *device_buffer, size_t bytes);

/* Copy the handle's plan. */
proj_status_t proj_get_plan(proj_handle_t h, proj_plan_desc_t *out);

/*
 * Write a one-line JSON description of the plan into buf (NUL-terminated,
 * truncated to len).  PROJ_ERR_INVALID_ARG for a NULL handle or buffer.
 */
proj_status_t proj_plan_info(proj_handle_t h, char *buf, size_t len);

/*
 * Allocation-free variant of proj_run, for callers that cannot call
 * cudaMalloc: a serving loop where an allocation may synchronise the device
 * and stall every other stream, or a plug-in whose host application owns all
 * device memory.  The worklog has no counterpart of this call; it is an
 * interface addition of this library.
 *
 * Same computation, layouts and argument rules as proj_create + proj_run
 * (bf16 X, W, bias; y_dtype PROJ_BF16 or PROJ_F32; bias NULL for none), with
 * no handle.  The caller passes inputs and outputs; the split-K scratch comes
 * from one fixed device array of 8 MiB inside the library, which every GPU
 * that loads the library holds until the process exits.  Nothing is allocated
 * and no allocating library routine is called.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Problems whose plan needs more scratch than 8 MiB (for example 64
 *     token rows against 20,000 weight rows, where K is split) return
 *     PROJ_ERR_UNSUPPORTED.
 *   - Every call shares the array: calls that overlap on the GPU (other
 *     streams, other threads) race and give wrong results.  Each call clears
 *     the split-K counters it uses on `stream` before its kernel.
 *   - The first call on a device (and the first after the device's context
 *     changed) also sets the kernels' shared-memory limit; the plan of the
 *     last shape run on each device is kept, so repeated calls of one shape
 *     plan once.
 * Returns the argument and launch status codes of proj_create/proj_run.  A
 * bounded device wait that gave up inside the kernel is not known when the
 * call returns: the kernel records it in the array's status word, which
 * collects the error bits of every call until proj_noalloc_device_status
 * reads and clears it.
 */
proj_status_t proj_run_noalloc(int64_t M, int64_t N, int64_t K, proj_wlayout_t w_layout,
                               proj_dtype_t y_dtype, const void *X, const void *W,
                               const void *bias, void *Y, void *stream);

/*
 * Device status of proj_run_noalloc, the allocation-free counterpart of
 * proj_device_status: synchronises `stream`, reads the fixed array's status
 * word and clears it.  PROJ_OK if no call since the last read recorded an
 * error; PROJ_ERR_DEVICE_TIMEOUT if a bounded wait gave up (the output of
 * that call is incomplete); PROJ_ERR_CUDA for a launch whose shared memory
 * or cluster shape did not match its plan, or if the read itself failed.
 * Allocates nothing.  The worklog has no counterpart of this call.
 */
proj_status_t proj_noalloc_device_status(void *stream);

/*
 * proj_selftest_wait_timeout for the allocation-free path: one CTA waits on a
 * barrier nothing arrives on, gives up after `limit_ns` (1 µs .. 1 s) and
 * records the timeout in the fixed array's status word, where
 * proj_noalloc_device_status then reports PROJ_ERR_DEVICE_TIMEOUT.
 * Asynchronous on `stream`; allocates nothing; PROJ_ERR_INVALID_ARG for a
 * limit out of range.  No fault, trap or hang is involved.
 */
proj_status_t proj_noalloc_selftest_wait_timeout(int64_t limit_ns, void *stream);

/* Free the handle and its scratch (synchronises the device).  NULL is a no-op. */
proj_status_t proj_destroy(proj_handle_t h);

/* Static human-readable name of a status code (never NULL). */
const char *proj_status_string(proj_status_t s);

/*
 * Self-test of the bounded device wait: launch one CTA that waits on a
 * shared-memory barrier nothing ever arrives on, with a limit of
 * `limit_ns` nanoseconds (1 µs .. 1 s).  The wait gives up, the kernel writes
 * its status and returns; the call synchronises `stream` and returns
 * PROJ_ERR_DEVICE_TIMEOUT when the timeout path worked (PROJ_OK would mean
 * the wait did not give up).  No fault, trap or hang is involved.
 */
proj_status_t proj_selftest_wait_timeout(int64_t limit_ns, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* PROJ_GB300_PROJ_H */
