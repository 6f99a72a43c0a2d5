// Device code of the GB300 dense projection Y = X·Wᵀ (+ bias).
//
// One persistent kernel, one CTA per SM, warp-specialised:
//   warp 0      TMA producer: streams W tiles [128 rows × 64 K] and X tiles
//               [block_t rows × 64 K] (128-byte swizzle) into a ring of
//               shared-memory stages ("How I made Muse's GPU projections 1.32×
//               faster in the Open Kernel Challenge", section "How a pipeline
//               hides waiting": load the next tile while computing this one).
//   warp 1      allocates tensor memory and issues tcgen05.mma (bf16 × bf16 →
//               fp32) for the swapped product Yᵀ = W·Xᵀ (section "Prove the
//               swapped product before worrying about its speed"): weight rows
//               are the MMA's M = 128 side, token rows its N = block_t side, so
//               a handful of tokens still fills the tensor core's long side.
//   warps 2..5  epilogue: tensor memory → registers → (+ bias) → fp32/bf16 Y,
//               or → fp32 partial sums for a tile whose K range is split.
//
// Stage hand-off uses "full" and "empty" mbarriers with phase parity (section
// "A transfer being issued does not mean the data is ready": ready-to-read and
// safe-to-reuse are separate signals).  Accumulators are double-buffered in
// tensor memory so one tile's epilogue overlaps the next tile's MMAs.
//
// Split-K (section "My first useful win: split up the sum"): CTAs that share a
// tile write fp32 partials to scratch and bump a per-(tile, 32-row quarter)
// counter; the warp that arrives last adds the partials in ascending CTA order
// (= ascending K), adds the bias and stores Y.  The fixed order makes every
// run bit-identical; no floating-point atomics are used (section "Could I avoid
// reading all those router partials back?" shows why those are not).  The
// counter returns to zero inside the run (section "Why a last-block scheme was
// more complicated than it sounded": every replay needs a fresh counter).
//
// Cluster split (decode shapes with fewer narrow tiles than SMs): each tile's
// K range is shared by the S CTAs of one thread-block cluster.  The partial
// sums are sent through distributed shared memory to one rank per 32-row
// quarter, which adds them in rank (= K) order; no scratch, no counters.
//
// Every mbarrier wait is bounded in time; a wait that runs out records a bit in
// the device status word, raises a CTA-wide abort flag, drains in-flight copies
// and MMAs (again bounded), frees tensor memory and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include "proj_internal.h"

namespace projgb {
namespace dev {

// ----------------------------------------------------------------------------
// PTX wrappers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// The same test with acquire at cluster scope: the arrivals came from other
// CTAs of the cluster, whose shared-memory writes must then be visible.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait for the phase of `bar` with the given parity to complete.
// Returns false (and raises the CTA abort flag, recording `code` in the status
// word) if `limit_ns` passes, or false at once if another role aborted.
template <bool kClusterScope = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           int *status, int code, int64_t limit_ns) {
    auto test = [&]() {
        return kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (test()) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (test()) return true;
        if (*abort_flag) return false;
        if (static_cast<int64_t>(globaltimer_ns() - t0) > limit_ns) {
            *abort_flag = 1;
            atomicOr(status, code);
            return false;
        }
    }
}

// Thread-block clusters (cluster split): this CTA's rank, the address of the
// same shared-memory location in another CTA of the cluster, arrivals and
// loads through that window, and the cluster-wide barrier.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t c;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(c));
    return c;
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
    return d;
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

__device__ __forceinline__ void st_cluster_f4(uint32_t cluster_addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t cluster_addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t saddr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(saddr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_prefetch_map(const void *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled TMA load into shared memory, completing on `bar` (transaction bytes).
// x is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *map, uint32_t bar, int32_t x,
                                            int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// 3-D tiled TMA load (x innermost): the box's z planes land one after another.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *map, uint32_t bar, int32_t x, int32_t y,
                                            int32_t z, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void *map, uint32_t bar, int32_t x,
                                                 int32_t y, int32_t z, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// CTA pairs: the same load, completing on an mbarrier that may sit in the
// other CTA of the pair (`bar` is then a shared::cluster address from mapa).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void *map, uint32_t bar, int32_t x,
                                                 int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// Tensor-memory allocation.  Every tcgen05 instruction of a kernel names the
// same CTA group: cta_group::2 in the CTA-pair instance, where one warp of
// each CTA of the pair takes part in the allocation and the release.
template <bool kPair>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    if constexpr (kPair)
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(ncols)
                     : "memory");
}

template <bool kPair>
__device__ __forceinline__ void tmem_relinquish() {
    if constexpr (kPair)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <bool kPair>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    if constexpr (kPair)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                     : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] · B[smem]ᵀ, kind::f16 (bf16 operands, fp32 accumulate).
// cta_group::2 (issued by the even CTA of a pair): M = 256, the A rows and
// the accumulator rows split 128/128 between the two CTAs, B's rows split in
// halves (the even CTA holds the first), each CTA's operands at the same
// shared-memory offsets, so the descriptors of the issuing CTA serve both.
template <bool kPair>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    if constexpr (kPair)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Arrive once on `bar` when every tcgen05 op this thread issued so far completes.
template <bool kPair>
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    if constexpr (kPair)
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         bar)
                     : "memory");
    else
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         bar)
                     : "memory");
}

// CTA pairs: the same arrival on the mbarrier at this shared-memory offset in
// both CTAs of the pair (cluster ranks 0 and 1).
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(static_cast<uint16_t>(3))
        : "memory");
}

// Load 16 consecutive fp32 columns of this thread's tensor-memory lane and wait
// for them (the wait sits in the same asm block so no use can move above it).
__device__ __forceinline__ void tmem_load16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 columns of this thread's tensor-memory lane in one load
// and one wait (four 16-column chunks: one round trip instead of four).
__device__ __forceinline__ void tmem_load64(uint32_t taddr, float (&v)[64]) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor (tcgen05 format), 128-byte swizzle.
// lbo/sbo in bytes: for K-major tiles sbo is the 8-row group stride (1024);
// for MN-major tiles lbo is the stride between 64-element MN blocks and sbo
// the stride between 8-row K groups.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;  // swizzle mode: 128-byte
    return d;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Programmatic dependent launch: let the next kernel on the stream start its
// set-up now / wait until the preceding kernel has completed and its memory
// is visible.  Both are no-ops for a launch without the PDL attribute.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint32_t sm_id() {
    uint32_t id;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(id));
    return id;
}

// Phase trace (off unless the handle has a trace buffer): one globaltimer
// stamp per phase per CTA, see proj_set_trace in proj.h for the layout.
__device__ __forceinline__ void trace_stamp(const KernelParams &p, int slot) {
    if (p.trace) p.trace[static_cast<size_t>(blockIdx.x) * kTraceSlots + slot] = globaltimer_ns();
}

// Fused epilogue (the FFN activation written once; a residual added back):
// y = act(projection + bias) + residual, in fp32, then one rounding to the
// output type.  GELU is x/2 · (1 + erf(x/√2)).  The tensor-core kernel is
// built twice: kFused = false leaves all of this out of the default path.
__device__ __forceinline__ float gelu_f32(float v) {
    return 0.5f * v * (1.0f + erff(v * 0.7071067811865476f));
}

// Out of line, four values a call (passed in registers): one copy of the code
// instead of one per unrolled store site (the epilogue runs once per tile,
// from a cold instruction cache), one call per four values.
static __device__ __noinline__ float4 gelu4(float4 v) {
    return make_float4(gelu_f32(v.x), gelu_f32(v.y), gelu_f32(v.z), gelu_f32(v.w));
}

// SwiGLU's gate: SiLU(g)·u for four (gate, up) pairs a call, out of line.
static __device__ __noinline__ float4 swiglu4(float4 g, float4 u) {
    return make_float4(g.x / (1.0f + expf(-g.x)) * u.x, g.y / (1.0f + expf(-g.y)) * u.y,
                       g.z / (1.0f + expf(-g.z)) * u.z, g.w / (1.0f + expf(-g.w)) * u.w);
}

// The activation over n values (n a multiple of 4), four per call.
template <bool kFused, int n>
__device__ __forceinline__ void apply_act_n(const KernelParams &p, float *v) {
    if constexpr (kFused) {
        if (p.act == 1) {
#pragma unroll
            for (int i = 0; i < n; i += 4) {
                const float4 g = gelu4(make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
                v[i] = g.x;
                v[i + 1] = g.y;
                v[i + 2] = g.z;
                v[i + 3] = g.w;
            }
        }
    }
}

__device__ __forceinline__ float residual_at(const KernelParams &p, size_t off) {
    return p.y_f32 ? static_cast<const float *>(p.residual)[off]
                   : __bfloat162float(static_cast<const __nv_bfloat16 *>(p.residual)[off]);
}

// 4 consecutive residual values (16-byte aligned fp32, or 8-byte aligned bf16).
__device__ __forceinline__ float4 residual4(const KernelParams &p, size_t off) {
    if (p.y_f32) return *reinterpret_cast<const float4 *>(static_cast<const float *>(p.residual) + off);
    const uint2 u = *reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p.residual) + off);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// One output value (+ residual), rounded to Y's type.
template <bool kFused>
__device__ __forceinline__ void store_y(const KernelParams &p, size_t off, float y) {
    if constexpr (kFused)
        if (p.residual) y += residual_at(p, off);
    if (p.y_f32)
        static_cast<float *>(p.Y)[off] = y;
    else
        static_cast<__nv_bfloat16 *>(p.Y)[off] = __float2bfloat16_rn(y);
}

// 8 consecutive outputs at a 16-byte aligned offset (+ residual): one fp32
// pair of float4 stores or one bf16 16-byte store.
template <bool kFused>
__device__ __forceinline__ void store_y8(const KernelParams &p, size_t off, float4 a, float4 b) {
    if constexpr (kFused)
        if (p.residual) {
            a = add4(a, residual4(p, off));
            b = add4(b, residual4(p, off + 4));
        }
    if (p.y_f32) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.Y) + off);
        dst[0] = a;
        dst[1] = b;
    } else {
        *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.Y) + off) =
            make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
    }
}

// 4 consecutive fp32 outputs at a 16-byte aligned offset (+ residual).
template <bool kFused>
__device__ __forceinline__ void store_y4_f32(const KernelParams &p, size_t off, float4 v) {
    if constexpr (kFused)
        if (p.residual) v = add4(v, residual4(p, off));
    *reinterpret_cast<float4 *>(static_cast<float *>(p.Y) + off) = v;
}

// Acquire-release add at GPU scope: one lane publishes the partial sums its
// whole warp wrote (ordered before it by __syncwarp) and observes the other
// contributors' partials.
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t *ptr, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(ptr), "r"(v)
                 : "memory");
    return old;
}

__device__ __forceinline__ void store_relaxed_gpu(uint32_t *ptr, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

// Partial sums in scratch are chunk-major: a slot of 128 rows x b_rows fp32
// holds, for each 16-column chunk, the 128 rows' 16 values one after another
// (64 bytes a row).  A warp's 32 rows of one chunk are then 2 KiB contiguous
// however wide the tile; for a 16-column tile this is plain row order.
constexpr int32_t kPartialChunkStride = kBlockA * 16;  // floats from one chunk to the next

// Chunk ch of one partial-sum row (`row` points at the row's first chunk):
// four 16-byte loads through L2 (partials are written by other SMs).
__device__ __forceinline__ void load_partial16(const float *row, int32_t ch, float4 (&o)[4]) {
    const float4 *src = reinterpret_cast<const float4 *>(row + ch * kPartialChunkStride);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = __ldcg(src + i);
}

// ----------------------------------------------------------------------------
// Shared-memory layout
// ----------------------------------------------------------------------------
constexpr int kYTileStride = 36;  // floats per token row of y_tile (32 + 4: 16-byte rows, fewer conflicts)

struct SmemCtl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint64_t ready[4];  // cluster split: the other ranks' partials of a quarter are in place
    uint32_t tmem_base;
    int abort_flag;
    float bias_tile[4][kMaxTokenTile];  // token-major: each epilogue warp's copy of the tile's bias
    // Output staging, one area per epilogue warp: swapped tiles, 16 tokens x
    // 32 weight rows (fp32, stride kYTileStride); token-major tiles, 32 token
    // rows x 32 columns (fp32 stride kYTileStride, or bf16 stride 40).
    float y_tile[4][32 * kYTileStride];
};
static_assert(offsetof(SmemCtl, y_tile) % 16 == 0, "y_tile rows are read as 16-byte vectors");
static_assert(sizeof(SmemCtl) + 1023 <= kSmemReserve, "the reserve holds SmemCtl and the alignment slack");

// ----------------------------------------------------------------------------
// The kernel
// ----------------------------------------------------------------------------
template <bool kFused, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    proj_tc_kernel(const __grid_constant__ KernelParams p, const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_x) {
    extern __shared__ uint8_t smem_raw[];
    // Stage buffers need 1024-byte alignment (128-byte swizzle atoms).
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    {
        // The ring, its barriers and the alignment slack must fit the dynamic
        // shared memory this launch received; otherwise record the error and
        // leave before touching any of it.
        uint32_t dyn_bytes;
        asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_bytes));
        const uint64_t need = static_cast<uint64_t>(base_addr - raw_addr) +
                              static_cast<uint64_t>(p.stages) * static_cast<uint32_t>(p.stage_bytes) +
                              static_cast<uint32_t>(p.red_bytes) + sizeof(SmemCtl);
        if (p.stages > kMaxStages || need > dyn_bytes) {
            if (threadIdx.x == 0) atomicOr(p.status, kErrSmemTooSmall);
            return;
        }
        // A cluster-split plan needs clusters of exactly its size (every CTA
        // of the launch sees the same cluster size, so all leave together,
        // before any cluster barrier).
        if (p.cluster_split > 1 && cluster_nctarank() != static_cast<uint32_t>(p.cluster_split)) {
            if (threadIdx.x == 0) atomicOr(p.status, kErrLaunchShape);
            return;
        }
        // A CTA-pair plan runs on the pair instance, in clusters of 2.
        if ((p.cta_pair != 0) != kPair || (kPair && cluster_nctarank() != 2u)) {
            if (threadIdx.x == 0) atomicOr(p.status, kErrLaunchShape);
            return;
        }
    }
    // The CTA's index in the plan: in a cluster split, cluster c's rank r is
    // CTA c·S + r (tile c, K range r), taken from the hardware's own numbering.
    // A CTA pair owns tiles as one: its index is the cluster's.
    const int32_t cta = kPair ? static_cast<int32_t>(cluster_id_x())
                        : p.cluster_split > 1
                            ? static_cast<int32_t>(cluster_id_x() * static_cast<uint32_t>(p.cluster_split) +
                                                   cluster_ctarank())
                            : static_cast<int32_t>(blockIdx.x);
    // CTA pairs: rank 0 (the leader) issues the MMAs and owns the barriers
    // they wait on; rank 1 loads its halves of the operands and runs the
    // epilogue of its 128 accumulator rows.
    const uint32_t pair_rank = kPair ? cluster_ctarank() : 0u;
    const bool leader = pair_rank == 0u;
    uint8_t *smem = smem_raw + (base_addr - raw_addr);
    // [ring: stages x stage_bytes][peers' partial sums: red_bytes][SmemCtl]
    const uint32_t red_addr = base_addr + static_cast<uint32_t>(p.stages * p.stage_bytes);
    SmemCtl *ctl = reinterpret_cast<SmemCtl *>(smem + p.stages * p.stage_bytes + p.red_bytes);
    volatile int *abort_flag = &ctl->abort_flag;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int32_t stages = p.stages;
    // A region of a stage: 128 rows (16 KiB), or the 64 weight rows of a
    // half tile (8 KiB: the MMA's A rows 64-127 are then the bytes after
    // them, shared memory the kernel owns, read into accumulator rows that
    // are never used).
    const uint32_t a_bytes = static_cast<uint32_t>(p.a_rows) * kBlockK * 2;
    // B region of one k-block (the B rows this CTA holds).
    const uint32_t b_bytes = static_cast<uint32_t>(p.stage_bytes / p.kpb) - a_bytes;
    // A stage holds kpb k-blocks: [A of each k-block][B of each k-block].
    // Where W and X land in a stage: W is the A operand when swapped, else B.
    const uint32_t w_off = p.swap ? 0u : a_bytes * static_cast<uint32_t>(p.kpb);
    const uint32_t x_off = p.swap ? a_bytes * static_cast<uint32_t>(p.kpb) : 0u;
    const uint32_t w_blk = p.swap ? a_bytes : b_bytes;  // one k-block's W bytes

    if (threadIdx.x == 0) trace_stamp(p, kTraceEntry);
    if (warp == 2) {
        // Barrier set-up, a few barriers per lane of an epilogue warp (idle
        // until the first accumulator), while the producer lane works out its
        // first segment below.
        for (int st = lane; st < stages; st += 32) {
            mbar_init(smem_u32(&ctl->full[st]), 1);
            mbar_init(smem_u32(&ctl->empty[st]), 1);
        }
        if (lane < 2) {
            mbar_init(smem_u32(&ctl->acc_full[lane]), 1);
            // Pairs: the leader's accumulator is free once both CTAs' epilogue
            // warps have read their halves.
            mbar_init(smem_u32(&ctl->acc_empty[lane]), (kPair ? 2 : 1) * kEpilogueThreads / 32);
        } else if (lane == 2) {
            mbar_init(smem_u32(&ctl->drain), 1);
            ctl->abort_flag = 0;
        } else if (lane >= 4 && lane < 8 && p.cluster_split > 1) {
            mbar_init(smem_u32(&ctl->ready[lane - 4]), static_cast<uint32_t>(32 * (p.cluster_split - 1)));
        }
        fence_barrier_init();
    }
    // The producer's cache policies and first segment.  This single-lane
    // integer work (the work iterator alone takes about 0.5 µs) runs during
    // set-up instead of between set-up and the first load, where it had
    // delayed the CTAs that start only as the preceding kernel's leave.
    uint64_t pol_w = 0, pol_x = 0;
    WorkIter prod_it;
    Segment prod_s;
    bool prod_more = false;
    int32_t prod_tm = 0, prod_tn = 0;
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmap_w);
        tma_prefetch_map(&tmap_x);
        // W is evict-first even where several token tiles reuse a weight
        // panel: the raster order runs those tiles in the same wave, in step
        // along K, so a panel's k-block is shared while it is in L2 anyway,
        // and evicting it first leaves more of the L2 to the raster group's
        // token panels.  (4096 x 8192 x 8192 on GB300: the same time as
        // evict-normal; DRAM traffic varied more between GPUs than between
        // the two hints.)
        pol_w = l2_policy_evict_first();
        pol_x = l2_policy_evict_last();  // X is reread by every CTA
        prod_it.init(p, cta);
        prod_more = prod_it.next(p, prod_s);
        if (prod_more) tile_coords(p, prod_s.tile, prod_tm, prod_tn);
    }
    if (warp == 1) {
        tmem_alloc<kPair>(smem_u32(&ctl->tmem_base), static_cast<uint32_t>(p.tmem_cols));
        // A single CTA gives up its right to allocate at once (the next
        // kernel's CTA on this SM may then allocate while this one runs).  A
        // pair keeps it until its teardown, after both CTAs have allocated.
        if constexpr (!kPair) tmem_relinquish<false>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // Cluster split: announce that this CTA's barriers exist.  A thread waits
    // for the whole cluster's announcement (cluster_waited) before its first
    // access to another CTA's shared memory, and at the latest at teardown.
    const bool clustered = kPair || p.cluster_split > 1;
    bool cluster_waited = false;
    if (clustered) cluster_arrive();
    // CTA pairs: both CTAs' barriers and tensor memory exist before any role
    // starts (the producer's first load completes on the leader's barrier,
    // the leader's first commit arrives on the peer's).  Every thread waits
    // here, each warp whole: a cluster-barrier wait from one lane while the
    // rest of its warp is elsewhere did not return on GB300.
    if constexpr (kPair) {
        cluster_wait();
        cluster_waited = true;
    }
    const uint32_t tmem_base = ctl->tmem_base;
    const uint32_t half_cols = static_cast<uint32_t>(p.tmem_cols / 2);
    // Accumulator buffer of the n-th tile and the parity of its use.
    auto acc_buf = [&](int32_t n) { return p.acc_bufs == 2 ? n & 1 : 0; };
    auto acc_use = [&](int32_t n) { return static_cast<uint32_t>(p.acc_bufs == 2 ? n >> 1 : n) & 1u; };
    if (threadIdx.x == 0) {
        // Only on-chip state has been touched so far; the next kernel may begin
        // its own set-up.  Global memory is touched only after griddep_wait().
        griddep_launch_dependents();
        if (p.trace) {
            trace_stamp(p, kTraceSetup);
            p.trace[static_cast<size_t>(blockIdx.x) * kTraceSlots + kTraceSmid] = sm_id();
        }
    }

    int64_t issued = 0;   // producer: stage loads issued (for the abort drain)
    int32_t reductions = 0;  // epilogue warp 2: split tiles this warp finished

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint32_t stage_bytes = static_cast<uint32_t>(p.stage_bytes);
            // CTA pairs: this CTA's halves of the tile's weight and token rows.
            const int32_t w_row_off = static_cast<int32_t>(pair_rank) * (p.block_n / 2);
            const int32_t x_row_off = static_cast<int32_t>(pair_rank) * (p.block_t / 2);
            const int32_t w_rows = kPair ? p.block_n / 2 : p.block_n;
            // Loads complete on the leader's "full" barrier (the MMA issuer's).
            auto full_bar = [&](int32_t st) {
                const uint32_t a = smem_u32(&ctl->full[st]);
                return (kPair && !leader) ? map_to_rank(a, 0u) : a;
            };
            auto load = [&](uint32_t dst, const CUtensorMap *map, uint32_t bar, int32_t x, int32_t y,
                            uint64_t pol) {
                if constexpr (kPair)
                    tma_load_2d_pair(dst, map, bar, x, y, pol);
                else
                    tma_load_2d(dst, map, bar, x, y, pol);
            };
            auto load3 = [&](uint32_t dst, const CUtensorMap *map, uint32_t bar, int32_t x, int32_t y, int32_t z,
                             uint64_t pol) {
                if constexpr (kPair)
                    tma_load_3d_pair(dst, map, bar, x, y, z, pol);
                else
                    tma_load_3d(dst, map, bar, x, y, z, pol);
            };
            // Stage kb of a weight tile: its kpb k-blocks of [block_n rows x
            // 64 K]; for [K,N] weights, each k-block is block_n/64 boxes of
            // 64 N-rows x 64 K, 8 KiB apart (the MN-major operand layout).
            auto load_w = [&](uint32_t dst, uint32_t full, int32_t tn, int32_t kb) {
                const int32_t kb64 = kb * p.kpb;  // first 64-wide k-block of the stage
                if (p.w_packed) {
                    // Pre-packed: every (tile, k-block) is one contiguous block
                    // of block_n rows x 128 bytes.  Two k-blocks a stage: planes
                    // of a 3-D map, consecutive, one op; one: rows of a 2-D map
                    // (a 2-D op is the quicker of the two for the TMA unit).
                    if (p.kpb > 1)
                        load3(dst, &tmap_w, full, 0, w_row_off, tn * p.k_blocks * p.kpb + kb64, pol_w);
                    else
                        load(dst, &tmap_w, full, 0, (tn * p.k_blocks + kb) * p.block_n + w_row_off, pol_w);
                } else if (!p.w_kn) {
                    for (int32_t j = 0; j < p.kpb; ++j)
                        load(dst + static_cast<uint32_t>(j) * w_blk, &tmap_w, full, (kb64 + j) * kBlockK,
                             tn * p.block_n + w_row_off, pol_w);
                } else {
                    for (int32_t j = 0; j < p.kpb; ++j)
                        for (int32_t i = 0; i < w_rows / 64; ++i)
                            load(dst + static_cast<uint32_t>(j) * w_blk + static_cast<uint32_t>(i) * 8192u, &tmap_w,
                                 full, tn * p.block_n + w_row_off + 64 * i, (kb64 + j) * kBlockK, pol_w);
                }
            };
            // Optional weight prefetch: fill the ring with W before the
            // preceding kernel has finished (W must not be written by it).
            int64_t pre = 0;
            if (!kPair && p.w_prefetch > 0) {
                const int32_t pre_max = min(p.w_prefetch, stages);
                WorkIter it = prod_it;  // from the first segment onwards
                Segment s = prod_s;
                int32_t tn = prod_tn;
                bool more = prod_more;
                while (pre < pre_max && more) {
                    for (int32_t kb = s.kb0; kb < s.kb1 && pre < pre_max; ++kb) {
                        const uint32_t full = smem_u32(&ctl->full[pre]);
                        mbar_arrive_expect_tx(full, stage_bytes);  // W + X bytes of the stage
                        load_w(base_addr + static_cast<uint32_t>(pre) * stage_bytes + w_off, full, tn, kb);
                        ++pre;
                    }
                    if (pre < pre_max) {
                        more = it.next(p, s);
                        int32_t tm_unused;
                        if (more) tile_coords(p, s.tile, tm_unused, tn);
                    }
                }
                if (pre > 0) trace_stamp(p, kTraceFirstLoad);
            }
            // X (and everything else) may come from the preceding kernel: the
            // grid-dependency wait comes right before the first load of this
            // loop, after the work decomposition and the first stage's barrier
            // are ready (that code's first run, instruction fetch included,
            // then overlaps the preceding kernel instead of following it).
            bool dep_done = false;
            auto dep_wait = [&]() {
                if (!dep_done) {
                    griddep_wait();
                    trace_stamp(p, kTraceDepWait);
                    dep_done = true;
                }
            };
            int32_t stage = 0;
            uint32_t phase = 0;
            WorkIter &it = prod_it;
            Segment &s = prod_s;
            int32_t tm = prod_tm, tn = prod_tn;
            bool more = prod_more;
            bool ok = true;
            while (ok && more) {
                for (int32_t kb = s.kb0; kb < s.kb1; ++kb) {
                    const uint32_t full = full_bar(stage);
                    const uint32_t st_base = base_addr + stage * stage_bytes;
                    if (issued >= pre) {
                        if (!wait_phase<kPair>(smem_u32(&ctl->empty[stage]), phase ^ 1u, abort_flag, p.status,
                                               kErrWaitProducer, p.wait_limit_ns)) {
                            ok = false;
                            break;
                        }
                        // The leader expects both CTAs' bytes of the stage.
                        if (leader) mbar_arrive_expect_tx(full, (kPair ? 2u : 1u) * stage_bytes);
                        dep_wait();
                        load_w(st_base + w_off, full, tn, kb);
                    }
                    dep_wait();
                    // fp32 router weights run as [H | L] along K: the second
                    // half multiplies the same X k-blocks again (a stage never
                    // straddles the halves: kpb divides their k-blocks).
                    const int32_t kb64 = kb * p.kpb;
                    const int32_t xkb = (p.x_kb_mod > 0 && kb64 >= p.x_kb_mod) ? kb64 - p.x_kb_mod : kb64;
                    if (p.x_3d) {
                        // The stage's k-blocks of X: planes of a 3-D map, one op.
                        load3(st_base + x_off, &tmap_x, full, 0, tm * p.block_t + x_row_off, xkb, pol_x);
                    } else {
                        const uint32_t x_blk = p.swap ? b_bytes : a_bytes;  // one k-block's X bytes
                        for (int32_t j = 0; j < p.kpb; ++j)
                            load(st_base + x_off + static_cast<uint32_t>(j) * x_blk, &tmap_x, full,
                                 (xkb + j) * kBlockK, tm * p.block_t + x_row_off, pol_x);
                    }
                    if (issued == 0 && pre == 0) trace_stamp(p, kTraceFirstLoad);
                    ++issued;
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                more = it.next(p, s);
                if (more) tile_coords(p, s.tile, tm, tn);
            }
            if (issued < pre) issued = pre;  // stages armed by the prefetch (abort drain)
            trace_stamp(p, kTraceLastLoad);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // (CTA pairs: the leader's, for both CTAs.)  Per MMA the issuing
        // thread only adds a constant to the stage's descriptors, whose
        // address field (bits 0-13, 16-byte units) holds every shared-memory
        // offset without a carry: with fewer instructions between MMAs the
        // tensor core gets them faster (one lane issuing 128 x 16 x 16 MMAs
        // with precomputed descriptors: about 120 cycles each on GB300).
        if (lane == 0 && leader) {
            const bool a_mn = p.swap && p.w_kn;   // weights [K,N] as the A operand
            const bool b_mn = !p.swap && p.w_kn;  // weights [K,N] as the B operand
            // K-major: the next 16 K values start 32 bytes further along the
            // 128-byte swizzled row.  MN-major (W stored [K,N]): 16 more K
            // rows, 16 × 128 bytes further; its 64-wide MN blocks are 8 KiB
            // apart.
            const uint64_t a_desc0 = a_mn ? smem_desc_sw128(base_addr, 8192, 1024) : smem_desc_sw128(base_addr, 16, 1024);
            const uint32_t b0 = base_addr + a_bytes * static_cast<uint32_t>(p.kpb);
            const uint64_t b_desc0 = b_mn ? smem_desc_sw128(b0, 8192, 1024) : smem_desc_sw128(b0, 16, 1024);
            const uint64_t a_kstep = a_mn ? (kMmaK * 128) >> 4 : (kMmaK * 2) >> 4;
            const uint64_t b_kstep = b_mn ? (kMmaK * 128) >> 4 : (kMmaK * 2) >> 4;
            const uint64_t a_jstep = a_bytes >> 4, b_jstep = b_bytes >> 4;
            const uint64_t stage_step = static_cast<uint64_t>(p.stage_bytes) >> 4;
            auto waited = [&](uint32_t bar, uint32_t parity) {
                return wait_phase<kPair>(bar, parity, abort_flag, p.status, kErrWaitMma, p.wait_limit_ns);
            };
            int32_t stage = 0;
            uint32_t phase = 0;
            int32_t seg_idx = 0;
            WorkIter it;
            it.init(p, cta);
            Segment s;
            bool ok = true;
            while (ok && it.next(p, s)) {
                const int32_t buf = acc_buf(seg_idx);
                const uint32_t use = acc_use(seg_idx);
                if (!waited(smem_u32(&ctl->acc_empty[buf]), use ^ 1u)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf) * half_cols;
                for (int32_t kb = s.kb0; kb < s.kb1; ++kb) {
                    if (!waited(smem_u32(&ctl->full[stage]), phase)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    if (seg_idx == 0 && kb == s.kb0) trace_stamp(p, kTraceFirstData);
                    const uint64_t st = static_cast<uint64_t>(stage) * stage_step;
                    for (int32_t j = 0; j < p.kpb; ++j) {
                        const uint64_t ad = a_desc0 + st + static_cast<uint64_t>(j) * a_jstep;
                        const uint64_t bd = b_desc0 + st + static_cast<uint64_t>(j) * b_jstep;
                        const uint32_t first = (kb > s.kb0 || j > 0) ? 1u : 0u;
#pragma unroll
                        for (int kk = 0; kk < kBlockK / kMmaK; ++kk)
                            tc_mma<kPair>(d_tmem, ad + kk * a_kstep, bd + kk * b_kstep, p.idesc,
                                          kk > 0 ? 1u : first);
                    }
                    // The stage is free (in both CTAs of a pair) once these MMAs finish.
                    if constexpr (kPair)
                        tc_commit_pair(smem_u32(&ctl->empty[stage]));
                    else
                        tc_commit<false>(smem_u32(&ctl->empty[stage]));
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                // The accumulator is ready (both CTAs' halves of it, for a pair).
                if constexpr (kPair)
                    tc_commit_pair(smem_u32(&ctl->acc_full[buf]));
                else
                    tc_commit<false>(smem_u32(&ctl->acc_full[buf]));
                ++seg_idx;
            }
            trace_stamp(p, kTraceLastMma);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;              // tensor-memory lane quarter of this warp
        const int r = q * 32 + lane;         // row within the 128-row weight tile
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const int64_t U = p.units_sk;
        griddep_wait();  // partials, counters and Y may be in use by the preceding kernel
        if (warp == 2 && lane == 0) trace_stamp(p, kTraceEpiDepWait);
        if (clustered && !cluster_waited) {
            cluster_wait();  // every CTA of the cluster has initialised its barriers (whole warps)
            cluster_waited = true;
        }
        // CTA pairs: the MMAs write the accumulator at the leader's address in
        // both CTAs' tensor memory.  Both CTAs allocate together and receive
        // the same columns; a difference is recorded (and the leader's used).
        uint32_t acc_base = tmem_base;
        if (kPair && !leader) {
            acc_base = ld_cluster_u32(map_to_rank(smem_u32(&ctl->tmem_base), 0u));
            if (acc_base != tmem_base && warp == 2 && lane == 0) atomicOr(p.status, kErrPairTmem);
        }
        // Where this CTA's epilogue warps report an accumulator read.
        const uint32_t acc_empty_bar0 =
            kPair ? map_to_rank(smem_u32(&ctl->acc_empty[0]), 0u) : smem_u32(&ctl->acc_empty[0]);
        int32_t seg_idx = 0;
        bool split_traced = false;  // the split-epilogue stamps cover the first split tile
        float *bias_s = ctl->bias_tile[q];
        WorkIter it;
        it.init(p, cta);
        Segment s;
        while (it.next(p, s)) {
            const int32_t buf = acc_buf(seg_idx);
            const uint32_t use = acc_use(seg_idx);
            int32_t tm, tn;
            tile_coords(p, s.tile, tm, tn);
            // Tensor-memory lane r holds one A row, columns hold B rows.
            // Swapped: lane = weight row n, columns = token rows m.
            // Otherwise: lane = token row m, columns = weight rows n.
            // A CTA of a pair holds A rows 128·rank .. 128·rank + 127 of the
            // pair's 256 and every B row (column).
            int32_t m0 = tm * p.block_t;
            int32_t n0 = tn * p.block_n;
            if (kPair) {
                if (p.swap)
                    n0 += kBlockA * static_cast<int32_t>(pair_rank);
                else
                    m0 += kBlockA * static_cast<int32_t>(pair_rank);
            }
            const int32_t lane_row = (p.swap ? n0 : m0) + r;
            const bool lane_ok = r < p.a_rows && lane_row < (p.swap ? p.N : p.M);
            const int32_t ccount = p.swap ? min(p.block_t, p.M - m0) : min(p.block_n, p.N - n0);
            const int32_t nchunks = (ccount + 15) / 16;
            const uint32_t tbase = acc_base + lane_off + static_cast<uint32_t>(buf) * half_cols;
            // The bias is fetched before the accumulator wait, so that a DRAM
            // round trip under the weight stream's load overlaps the MMAs:
            // swapped, one value per lane (its weight row); token-major, the
            // tile's block_n values into this warp's shared-memory slice.
            const float bias_lane =
                (p.swap && p.bias != nullptr && lane_ok) ? bf16_bits_to_float(p.bias[lane_row]) : 0.f;
            if (!p.swap && p.bias != nullptr) {
                for (int32_t j = lane; j < p.block_n; j += 32)
                    bias_s[j] = n0 + j < p.N ? bf16_bits_to_float(p.bias[n0 + j]) : 0.f;
                __syncwarp();
            }
            if (!wait_phase<kPair>(smem_u32(&ctl->acc_full[buf]), use, abort_flag, p.status,
                                   kErrWaitEpilogue, p.wait_limit_ns))
                break;
            tc_fence_after_sync();
            if (warp == 2 && lane == 0 && seg_idx == 0) trace_stamp(p, kTraceFirstAcc);
            if (q * 32 >= p.a_rows) {
                // Half tiles: this warp's accumulator rows come from the
                // unused half of the A region.  Nothing to store or reduce.
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t bar = acc_empty_bar0 + static_cast<uint32_t>(buf) * 8u;
                    if constexpr (kPair)
                        mbar_arrive_remote(bar);
                    else
                        mbar_arrive(bar);
                }
                ++seg_idx;
                continue;
            }
            const bool stamp_split = s.split && !split_traced && warp == 2 && lane == 0;
            if (s.split) split_traced = true;
            // Store one chunk of 16 columns of this lane's row (+ bias, the
            // activation and the residual).  Every
            // lane of the warp calls it (the swapped path shuffles through
            // shared memory).
            auto store_chunk = [&](int32_t ch, const float (&y)[16]) {
                if constexpr (kFused) {
                    if (p.act == 2) {
                        // SwiGLU.  Packing interleaved the stacked gate and up
                        // rows: swapped tiles hold, in each 32-row quarter,
                        // 16 gate rows (lanes 0-15) and the same 16 features'
                        // up rows (lanes 16-31); token-major chunks hold 8
                        // gate columns then the same 8 features' up columns.
                        // Output feature f of this tile: n0 / 2 + ...; Y rows
                        // are ldy = F apart.  There is no bias.
                        const int32_t F = p.ldy;
                        if (p.swap) {
                            float up[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) up[i] = __shfl_xor_sync(0xFFFFFFFFu, y[i], 16);
                            const int32_t f = n0 / 2 + q * 16 + lane;
                            const int32_t fb = n0 / 2 + q * 16;  // the warp's first feature
                            const int32_t mb = m0 + ch * 16;
                            if (p.y_vec && fb + 16 <= F && mb + 16 <= p.M) {
                                // 16 features (lanes 0-15) x 16 tokens through shared
                                // memory, stored as 16-byte row segments.
                                float *t = ctl->y_tile[q];
                                if (lane < 16) {
#pragma unroll
                                    for (int i = 0; i < 16; i += 4) {
                                        const float4 o = swiglu4(make_float4(y[i], y[i + 1], y[i + 2], y[i + 3]),
                                                                 make_float4(up[i], up[i + 1], up[i + 2], up[i + 3]));
                                        t[(i + 0) * kYTileStride + lane] = o.x;
                                        t[(i + 1) * kYTileStride + lane] = o.y;
                                        t[(i + 2) * kYTileStride + lane] = o.z;
                                        t[(i + 3) * kYTileStride + lane] = o.w;
                                    }
                                }
                                __syncwarp();
                                if (p.y_f32) {
#pragma unroll
                                    for (int pass = 0; pass < 2; ++pass) {
                                        const int32_t mi = pass * 8 + lane / 4, c = (lane % 4) * 4;
                                        store_y4_f32<kFused>(p, static_cast<size_t>(mb + mi) * F + fb + c,
                                                             *reinterpret_cast<const float4 *>(t + mi * kYTileStride + c));
                                    }
                                } else {
                                    const int32_t mi = lane / 2, c = (lane % 2) * 8;
                                    store_y8<kFused>(p, static_cast<size_t>(mb + mi) * F + fb + c,
                                                     *reinterpret_cast<const float4 *>(t + mi * kYTileStride + c),
                                                     *reinterpret_cast<const float4 *>(t + mi * kYTileStride + c + 4));
                                }
                                __syncwarp();  // the tile is reused by the next chunk
                                return;
                            }
                            if (lane < 16 && f < F) {
#pragma unroll
                                for (int i = 0; i < 16; i += 4) {
                                    const float4 o = swiglu4(make_float4(y[i], y[i + 1], y[i + 2], y[i + 3]),
                                                             make_float4(up[i], up[i + 1], up[i + 2], up[i + 3]));
                                    const float ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                                    for (int j = 0; j < 4; ++j) {
                                        const int32_t m = m0 + ch * 16 + i + j;
                                        if (m < p.M) store_y<kFused>(p, static_cast<size_t>(m) * F + f, ov[j]);
                                    }
                                }
                            }
                        } else {
                            if (!lane_ok) return;
                            const int32_t m = lane_row;
                            const int32_t f0 = n0 / 2 + ch * 8;
                            const float4 a = swiglu4(make_float4(y[0], y[1], y[2], y[3]), make_float4(y[8], y[9], y[10], y[11]));
                            const float4 b = swiglu4(make_float4(y[4], y[5], y[6], y[7]), make_float4(y[12], y[13], y[14], y[15]));
                            const size_t off = static_cast<size_t>(m) * F + f0;
                            if (p.y_vec && f0 + 8 <= F) {
                                store_y8<kFused>(p, off, a, b);
                            } else {
                                const float ov[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    if (f0 + j < F) store_y<kFused>(p, off + j, ov[j]);
                            }
                        }
                        return;
                    }
                }
                if (p.swap) {
                    // The warp holds 32 consecutive weight rows (lanes) x 16
                    // tokens (registers), but Y rows run along the weight rows:
                    // transpose through shared memory and store 16-byte vectors
                    // (2 stores a lane for bf16, 4 for fp32, instead of 16).
                    const int32_t mb = m0 + ch * 16;   // first token of the chunk
                    const int32_t nw = n0 + q * 32;    // first weight row of the warp
                    if (p.y_vec && nw + 32 <= p.N && mb + 16 <= p.M) {
                        float *t = ctl->y_tile[q];
                        float a16[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) a16[i] = y[i] + bias_lane;
                        apply_act_n<kFused, 16>(p, a16);
#pragma unroll
                        for (int i = 0; i < 16; ++i) t[i * kYTileStride + lane] = a16[i];
                        __syncwarp();
                        if (p.y_f32) {
#pragma unroll
                            for (int pass = 0; pass < 4; ++pass) {
                                const int32_t mi = pass * 4 + lane / 8, nc = (lane % 8) * 4;
                                store_y4_f32<kFused>(p, static_cast<size_t>(mb + mi) * p.N + nw + nc,
                                             *reinterpret_cast<const float4 *>(t + mi * kYTileStride + nc));
                            }
                        } else {
#pragma unroll
                            for (int pass = 0; pass < 2; ++pass) {
                                const int32_t mi = pass * 8 + lane / 4, nc = (lane % 4) * 8;
                                store_y8<kFused>(p, static_cast<size_t>(mb + mi) * p.N + nw + nc,
                                         *reinterpret_cast<const float4 *>(t + mi * kYTileStride + nc),
                                         *reinterpret_cast<const float4 *>(t + mi * kYTileStride + nc + 4));
                            }
                        }
                        __syncwarp();  // the tile is reused by the next chunk
                        return;
                    }
                    if (!lane_ok) return;
                    const int32_t n = lane_row;
                    float a16[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) a16[i] = y[i] + bias_lane;
                    apply_act_n<kFused, 16>(p, a16);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int32_t m = mb + i;
                        if (m < p.M) store_y<kFused>(p, static_cast<size_t>(m) * p.N + n, a16[i]);
                    }
                } else {
                    if (!lane_ok) return;
                    const int32_t m = lane_row;
                    const int32_t nb = n0 + ch * 16;
                    float v[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = y[i] + (p.bias != nullptr ? bias_s[ch * 16 + i] : 0.f);
                    apply_act_n<kFused, 16>(p, v);
                    const size_t off = static_cast<size_t>(m) * p.N + nb;
                    if (p.y_vec && nb + 16 <= p.N) {
                        // 16 consecutive outputs of one row: vector stores.
#pragma unroll
                        for (int i = 0; i < 2; ++i)
                            store_y8<kFused>(p, off + 8 * i, make_float4(v[8 * i], v[8 * i + 1], v[8 * i + 2], v[8 * i + 3]),
                                     make_float4(v[8 * i + 4], v[8 * i + 5], v[8 * i + 6], v[8 * i + 7]));
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (nb + i < p.N) store_y<kFused>(p, off + i, v[i]);
                    }
                }
            };
            // Token-major: store 32 columns [n0 + 16·ch, +32) of the warp's 32
            // token rows (+ bias, activation, residual).  Each lane holds one
            // row, so the block goes through shared memory and leaves as whole
            // row segments (bf16: 8 rows of 64 bytes per store instruction,
            // fp32: 4 rows of 128),
            // not 32 rows touched by every instruction.  Every lane calls it.
            auto store_cols32 = [&](int32_t ch, const float *y) {
                const int32_t nb = n0 + ch * 16;
                const int32_t mw = m0 + q * 32;
                float *t = ctl->y_tile[q];
                float b[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) b[i] = y[i] + (p.bias != nullptr ? bias_s[ch * 16 + i] : 0.f);
                apply_act_n<kFused, 32>(p, b);
                bool with_residual = false;
                if constexpr (kFused) with_residual = p.residual != nullptr;
                if (!p.y_f32 && !with_residual) {
                    // bf16 without a residual: stage the rounded values (64-byte
                    // rows, stride 80 bytes: conflict-free 16-byte accesses).
                    uint8_t *tb = reinterpret_cast<uint8_t *>(t);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<uint4 *>(tb + lane * 80 + 16 * j) =
                            make_uint4(pack_bf16x2(b[8 * j], b[8 * j + 1]), pack_bf16x2(b[8 * j + 2], b[8 * j + 3]),
                                       pack_bf16x2(b[8 * j + 4], b[8 * j + 5]), pack_bf16x2(b[8 * j + 6], b[8 * j + 7]));
                    __syncwarp();
#pragma unroll
                    for (int pass = 0; pass < 4; ++pass) {
                        const int32_t r = pass * 8 + lane / 4, c = (lane % 4) * 8;
                        if (mw + r < p.M)
                            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.Y) +
                                                       static_cast<size_t>(mw + r) * p.N + nb + c) =
                                *reinterpret_cast<const uint4 *>(tb + r * 80 + c * 2);
                    }
                    __syncwarp();  // the staging area is reused by the next block
                    return;
                }
                // fp32 staging otherwise: a residual is added before the one
                // rounding.  The block's residual values are all loaded before
                // they are used (one memory round trip per block, not one per
                // store).
                if (p.y_f32) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<float4 *>(t + lane * kYTileStride + 4 * j) =
                            make_float4(b[4 * j], b[4 * j + 1], b[4 * j + 2], b[4 * j + 3]);
                    float4 res[8];
                    if constexpr (kFused) {
#pragma unroll
                        for (int pass = 0; pass < 8; ++pass) {
                            const int32_t r = pass * 4 + lane / 8, c = (lane % 8) * 4;
                            res[pass] = (with_residual && mw + r < p.M)
                                            ? residual4(p, static_cast<size_t>(mw + r) * p.N + nb + c)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    }
                    __syncwarp();
#pragma unroll
                    for (int pass = 0; pass < 8; ++pass) {
                        const int32_t r = pass * 4 + lane / 8, c = (lane % 8) * 4;
                        float4 v = *reinterpret_cast<const float4 *>(t + r * kYTileStride + c);
                        if constexpr (kFused) v = add4(v, res[pass]);
                        if (mw + r < p.M)
                            *reinterpret_cast<float4 *>(static_cast<float *>(p.Y) +
                                                        static_cast<size_t>(mw + r) * p.N + nb + c) = v;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<float4 *>(t + lane * kYTileStride + 4 * j) =
                            make_float4(b[4 * j], b[4 * j + 1], b[4 * j + 2], b[4 * j + 3]);
                    uint4 res[4];
                    if constexpr (kFused) {
#pragma unroll
                        for (int pass = 0; pass < 4; ++pass) {
                            const int32_t r = pass * 8 + lane / 4, c = (lane % 4) * 8;
                            res[pass] = (with_residual && mw + r < p.M)
                                            ? *reinterpret_cast<const uint4 *>(
                                                  static_cast<const __nv_bfloat16 *>(p.residual) +
                                                  static_cast<size_t>(mw + r) * p.N + nb + c)
                                            : make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    __syncwarp();
#pragma unroll
                    for (int pass = 0; pass < 4; ++pass) {
                        const int32_t r = pass * 8 + lane / 4, c = (lane % 4) * 8;
                        float4 a = *reinterpret_cast<const float4 *>(t + r * kYTileStride + c);
                        float4 bb = *reinterpret_cast<const float4 *>(t + r * kYTileStride + c + 4);
                        if constexpr (kFused) {
                            const uint4 u = res[pass];
                            a = add4(a, make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                                                    __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u)));
                            bb = add4(bb, make_float4(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xFFFF0000u),
                                                      __uint_as_float(u.w << 16), __uint_as_float(u.w & 0xFFFF0000u)));
                        }
                        if (mw + r < p.M)
                            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.Y) +
                                                       static_cast<size_t>(mw + r) * p.N + nb + c) =
                                make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(bb.x, bb.y),
                                           pack_bf16x2(bb.z, bb.w));
                    }
                }
                __syncwarp();  // the staging area is reused by the next block
            };
            auto release_accumulator = [&]() {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t bar = acc_empty_bar0 + static_cast<uint32_t>(buf) * 8u;
                    if constexpr (kPair)
                        mbar_arrive_remote(bar);  // the leader's barrier (release at cluster scope)
                    else
                        mbar_arrive(bar);
                }
            };

            if (!s.split) {
                // Whole tile: tensor memory -> (+ bias) -> Y, four chunks per
                // tensor-memory round trip while whole groups of four remain.
                int32_t ch = 0;
                for (; ch + 4 <= nchunks; ch += 4) {
                    float v[64];
                    tmem_load64(tbase + ch * 16, v);
                    bool cols32 = !p.swap && p.y_vec && n0 + (ch + 4) * 16 <= p.N;
                    if constexpr (kFused) cols32 = cols32 && p.act != 2;  // SwiGLU stores per chunk
                    if (cols32) {
                        store_cols32(ch, v);
                        store_cols32(ch + 2, v + 32);
                    } else {
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            store_chunk(ch + u, *reinterpret_cast<const float(*)[16]>(v + 16 * u));
                    }
                }
                for (; ch < nchunks; ++ch) {
                    float v[16];
                    tmem_load16(tbase + ch * 16, v);
                    store_chunk(ch, v);
                }
                release_accumulator();
            } else if (kFused && p.cluster_split > 1 && !p.swap) {
                // Token-major cluster split (at most 32 tokens, so only row
                // quarter 0 holds results; built into the fused instance
                // only, which every such plan runs on, to keep the lean
                // instance's epilogue code small).  The S ranks hold the tile's
                // partial sums over consecutive K ranges.  Rank c mod S adds
                // 16-column chunk c: every other rank stores its partial
                // chunk (32 rows x 16 fp32, [float4][lane]) into the owner's
                // shared memory, then every lane arrives on each other
                // rank's barrier (releasing its stores).  The owner adds all
                // ranks in rank (= K) order, so every run gives the same bits.
                if (q == 0) {
                    const uint32_t S = static_cast<uint32_t>(p.cluster_split);
                    const uint32_t rank = static_cast<uint32_t>(cta) % S;  // = %cluster_ctarank
                    const int32_t nch = p.block_n / 16;
                    const uint32_t lane_off16 = static_cast<uint32_t>(lane) * 16u;
                    // Slot (o, j): the owner's o-th chunk from contributor j.
                    auto slot_addr = [&](uint32_t o, uint32_t j) {
                        return red_addr + (o * (S - 1u) + j) * 2048u + lane_off16;
                    };
                    if (stamp_split) trace_stamp(p, kTraceSplitPartial);
                    for (int32_t c = 0; c < nch; ++c) {
                        const uint32_t owner = static_cast<uint32_t>(c) % S;
                        if (owner == rank) continue;
                        const uint32_t dst =
                            map_to_rank(slot_addr(static_cast<uint32_t>(c) / S, rank < owner ? rank : rank - 1u), owner);
                        float v[16];
                        tmem_load16(tbase + c * 16, v);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            st_cluster_f4(dst + static_cast<uint32_t>(i) * 512u,
                                          make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
                    }
                    for (uint32_t r2 = 0; r2 < S; ++r2)
                        if (r2 != rank) mbar_arrive_remote(map_to_rank(smem_u32(&ctl->ready[0]), r2));
                    if (wait_phase<true>(smem_u32(&ctl->ready[0]), 0u, abort_flag, p.status, kErrWaitEpilogue,
                                         p.wait_limit_ns)) {
                        if (stamp_split) trace_stamp(p, kTraceSplitReady);
                        for (int32_t c = static_cast<int32_t>(rank); c < nch; c += static_cast<int32_t>(S)) {
                            if (c * 16 >= ccount) break;  // past N: nothing to store
                            const uint32_t o = static_cast<uint32_t>(c) / S;
                            float own[16], acc[16];
                            tmem_load16(tbase + c * 16, own);
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc[i] = 0.f;
                            for (uint32_t rk = 0; rk < S; ++rk) {
                                if (rk == rank) {
#pragma unroll
                                    for (int i = 0; i < 16; ++i) acc[i] += own[i];
                                    continue;
                                }
                                const uint32_t src = slot_addr(o, rk < rank ? rk : rk - 1u);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const float4 w4 = ld_shared_f4(src + static_cast<uint32_t>(i) * 512u);
                                    acc[4 * i] += w4.x;
                                    acc[4 * i + 1] += w4.y;
                                    acc[4 * i + 2] += w4.z;
                                    acc[4 * i + 3] += w4.w;
                                }
                            }
                            store_chunk(c, acc);
                        }
                        if (stamp_split) trace_stamp(p, kTraceSplitStored);
                    }
                }
                release_accumulator();
            } else if (p.cluster_split > 1) {
                // (Not `clustered`: a CTA pair is a cluster too, but its split
                // tiles go through the scratch below.)
                // Cluster split: the S CTAs of this cluster hold the tile's
                // partial sums over consecutive K ranges (rank order = K
                // order).  Quarter q is reduced by rank q mod S (S <= 4) or q
                // (S > 4).  Every other rank stores its 32 rows straight into
                // the reducer's shared memory and arrives there (every lane,
                // releasing its own stores); the reducer then reads them
                // locally and adds all ranks in ascending order, so every run
                // gives the same bits.
                const uint32_t S = static_cast<uint32_t>(p.cluster_split);
                const uint32_t rank = static_cast<uint32_t>(cta) % S;  // = %cluster_ctarank
                const uint32_t reducer = S <= 4 ? static_cast<uint32_t>(q) % S : static_cast<uint32_t>(q);
                const uint32_t slot_q = S <= 4 ? static_cast<uint32_t>(q) / S : 0u;
                const uint32_t part_bytes = 32u * static_cast<uint32_t>(p.b_rows) * 4u;
                // A partial is [16-column chunk][float4 of the chunk][lane]:
                // 16 consecutive bytes per lane, a warp's accesses contiguous.
                const uint32_t lane_off16 = static_cast<uint32_t>(lane) * 16u;
                const uint32_t quarter_base = red_addr + slot_q * (S - 1u) * part_bytes + lane_off16;
                if (rank != reducer) {
                    const uint32_t j = rank < reducer ? rank : rank - 1u;  // contributor index
                    const uint32_t dst = map_to_rank(quarter_base + j * part_bytes, reducer);
                    for (int32_t ch = 0; ch < nchunks; ++ch) {
                        float v[16];
                        tmem_load16(tbase + ch * 16, v);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            st_cluster_f4(dst + static_cast<uint32_t>(ch * 4 + i) * 512u,
                                          make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
                    }
                    release_accumulator();
                    if (stamp_split) trace_stamp(p, kTraceSplitPartial);
                    mbar_arrive_remote(map_to_rank(smem_u32(&ctl->ready[q]), reducer));
                    if (stamp_split) {
                        trace_stamp(p, kTraceSplitReady);
                        trace_stamp(p, kTraceSplitStored);
                    }
                } else {
                    if (stamp_split) trace_stamp(p, kTraceSplitPartial);
                    if (wait_phase<true>(smem_u32(&ctl->ready[q]), 0u, abort_flag, p.status,
                                         kErrWaitEpilogue, p.wait_limit_ns)) {
                        if (stamp_split) trace_stamp(p, kTraceSplitReady);
                        if (warp == 2 && lane == 0) ++reductions;
                        // Several clusters per tile: this cluster's sum of the
                        // quarter goes to its scratch slot [tile·G + group]
                        // (laid out like a split tile's partial) instead of Y.
                        const int32_t G = p.cluster_groups;
                        const int32_t grp = (cta / static_cast<int32_t>(S)) % G;
                        float *mine = G > 1 ? p.partials + static_cast<size_t>(s.tile * G + grp) * kBlockA * p.b_rows + r * 16
                                            : nullptr;
                        for (int32_t ch = 0; ch < nchunks; ++ch) {
                            float own[16], acc[16];
                            tmem_load16(tbase + ch * 16, own);
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc[i] = 0.f;
                            for (uint32_t rk = 0; rk < S; ++rk) {
                                if (rk == rank) {
#pragma unroll
                                    for (int i = 0; i < 16; ++i) acc[i] += own[i];
                                    continue;
                                }
                                const uint32_t src = quarter_base + (rk < rank ? rk : rk - 1u) * part_bytes +
                                                     static_cast<uint32_t>(ch * 4) * 512u;
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const float4 o = ld_shared_f4(src + static_cast<uint32_t>(i) * 512u);
                                    acc[4 * i] += o.x;
                                    acc[4 * i + 1] += o.y;
                                    acc[4 * i + 2] += o.z;
                                    acc[4 * i + 3] += o.w;
                                }
                            }
                            if (G > 1) {
                                float4 *dst = reinterpret_cast<float4 *>(mine + ch * kPartialChunkStride);
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    dst[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
                            } else {
                                store_chunk(ch, acc);
                            }
                        }
                        if (G > 1) {
                            // One acquire-release add per (tile, quarter) and
                            // cluster: it releases this warp's sums (ordered
                            // before it by the __syncwarp) and, for the cluster
                            // that completes last, acquires the others'.  That
                            // one adds the G sums in group order, starting
                            // from group 0's, so the bits do not depend on
                            // which cluster completes last.
                            __syncwarp();
                            int last = 0;
                            uint32_t *ctr = p.counters + static_cast<size_t>(s.tile) * 4 + q;
                            if (lane == 0) {
                                const uint32_t old = atom_add_acq_rel_gpu(ctr, 1u);
                                last = (old == static_cast<uint32_t>(G - 1)) ? 1 : 0;
                                if (last) store_relaxed_gpu(ctr, 0u);  // fresh for the next run
                            }
                            last = __shfl_sync(0xFFFFFFFFu, last, 0);
                            __syncwarp();
                            if (last) {
                                const float *g0 = p.partials + static_cast<size_t>(s.tile * G) * kBlockA * p.b_rows + r * 16;
                                const size_t gstride = static_cast<size_t>(kBlockA) * p.b_rows;
                                for (int32_t ch = 0; ch < nchunks; ++ch) {
                                    float sum[16];
                                    float4 o[4];
                                    load_partial16(g0, ch, o);
#pragma unroll
                                    for (int i = 0; i < 4; ++i) {
                                        sum[4 * i] = o[i].x;
                                        sum[4 * i + 1] = o[i].y;
                                        sum[4 * i + 2] = o[i].z;
                                        sum[4 * i + 3] = o[i].w;
                                    }
                                    for (int32_t gg = 1; gg < G; ++gg) {
                                        load_partial16(g0 + static_cast<size_t>(gg) * gstride, ch, o);
#pragma unroll
                                        for (int i = 0; i < 4; ++i) {
                                            sum[4 * i] += o[i].x;
                                            sum[4 * i + 1] += o[i].y;
                                            sum[4 * i + 2] += o[i].z;
                                            sum[4 * i + 3] += o[i].w;
                                        }
                                    }
                                    store_chunk(ch, sum);
                                }
                            }
                        }
                        if (stamp_split) trace_stamp(p, kTraceSplitStored);
                    }
                    release_accumulator();
                }
            } else {
                // Split tile.  This lane's row of fp32 partial sums goes to
                // scratch: slot [128 rows x b_rows], chunk-major (see
                // kPartialChunkStride).  A CTA pair's slot holds its 256 rows
                // as two such halves, each CTA writing and reading its own;
                // each CTA counts its own row quarters.
                auto partial_row = [&](int32_t slot) {
                    return p.partials +
                           (static_cast<size_t>(slot) * (kPair ? 2 : 1) + (kPair ? pair_rank : 0u)) * kBlockA * p.b_rows +
                           r * 16;
                };
                float *own = partial_row(s.slot);
                for (int32_t ch = 0; ch < nchunks; ++ch) {
                    float v[16];
                    tmem_load16(tbase + ch * 16, v);
                    float4 *dst = reinterpret_cast<float4 *>(own + ch * kPartialChunkStride);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                }
                // Contributors of this tile, in K order.
                const int32_t ts = s.tile - p.tiles_dp;
                int32_t c_first = 0, c_last = 0, nseg = 2, first_slot = 0;
                if (!p.sk_pair) {
                    split_tile_ctas(ts, p.k_blocks, U, p.grid, c_first, c_last);
                    if (p.sk_dense) {
                        // Every CTA owns units: c_first may have started in an
                        // earlier tile; every later contributor starts inside
                        // this one (slot 2c).
                        nseg = c_last - c_first + 1;
                        first_slot = 2 * c_first +
                                     (unit_begin(c_first, U, p.grid) < static_cast<int64_t>(ts) * p.k_blocks ? 1 : 0);
                    } else {
                        nseg = 0;
                        for (int32_t c = c_first; c <= c_last; ++c) nseg += cta_has_units(c, U, p.grid) ? 1 : 0;
                    }
                }
                if (stamp_split) trace_stamp(p, kTraceSplitPartial);
                // Publish (release) and count arrivals per 32-row quarter.
                __syncwarp();
                int last = 0;
                uint32_t *ctr = p.counters + static_cast<size_t>(ts) * (kPair ? 8 : 4) + (kPair ? pair_rank * 4u : 0u) + q;
                if (lane == 0) {
                    // One acquire-release add: releases this warp's partials
                    // (ordered before it by the __syncwarp above) and, for the
                    // last contributor, acquires everyone else's.
                    const uint32_t old = atom_add_acq_rel_gpu(ctr, 1u);
                    last = (old == static_cast<uint32_t>(nseg - 1)) ? 1 : 0;
                    if (last) store_relaxed_gpu(ctr, 0u);  // fresh for the next run
                }
                last = __shfl_sync(0xFFFFFFFFu, last, 0);
                __syncwarp();
                if (stamp_split) trace_stamp(p, kTraceSplitReady);
                if (last && warp == 2 && lane == 0) ++reductions;

                if (last && p.sk_pair) {
                    // Two contributors: own accumulator (still in tensor
                    // memory) + the other's partial.  Two-operand addition is
                    // commutative, so the bits do not depend on who is last.
                    const int32_t other_slot =
                        s.kb0 == 0 ? 2 * (cta + 1) : 2 * (cta - 1) + 1;
                    const float *other = partial_row(other_slot);
                    for (int32_t ch0 = 0; ch0 < nchunks; ch0 += 4) {
                        float4 o[4][4];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            if (ch0 + u < nchunks) load_partial16(other, ch0 + u, o[u]);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if (ch0 + u >= nchunks) break;
                            float v[16];
                            tmem_load16(tbase + (ch0 + u) * 16, v);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                v[4 * i] += o[u][i].x;
                                v[4 * i + 1] += o[u][i].y;
                                v[4 * i + 2] += o[u][i].z;
                                v[4 * i + 3] += o[u][i].w;
                            }
                            store_chunk(ch0 + u, v);
                        }
                    }
                    release_accumulator();
                } else {
                    release_accumulator();
                    if (last) {
                        // Several contributors: add every partial (own
                        // included) in ascending CTA order, i.e. ascending K,
                        // four contributors' loads in flight at a time.
                        for (int32_t ch = 0; ch < nchunks; ++ch) {
                            float acc[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc[i] = 0.f;
                            for (int32_t c = c_first; c <= c_last; c += 4) {
                                float4 o[4][4];
                                bool valid[4];
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    const int32_t cc = c + k;
                                    valid[k] = cc <= c_last && (p.sk_dense || cta_has_units(cc, U, p.grid));
                                    if (valid[k]) {
                                        const int32_t slot =
                                            p.sk_dense ? (cc == c_first ? first_slot : 2 * cc)
                                                       : split_slot(cc, ts, U, p.grid, p.k_blocks);
                                        load_partial16(partial_row(slot),
                                                       ch, o[k]);
                                    }
                                }
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    if (valid[k]) {
#pragma unroll
                                        for (int i = 0; i < 4; ++i) {
                                            acc[4 * i] += o[k][i].x;
                                            acc[4 * i + 1] += o[k][i].y;
                                            acc[4 * i + 2] += o[k][i].z;
                                            acc[4 * i + 3] += o[k][i].w;
                                        }
                                    }
                            }
                            store_chunk(ch, acc);
                        }
                    }
                }
                if (stamp_split) trace_stamp(p, kTraceSplitStored);
            }
            ++seg_idx;
        }
        if (warp == 2 && lane == 0) trace_stamp(p, kTraceEpilogueDone);
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    if (p.trace && warp == 2 && lane == 0) {
        trace_stamp(p, kTraceTeardown);
        p.trace[static_cast<size_t>(blockIdx.x) * kTraceSlots + kTraceReductions] =
            static_cast<unsigned long long>(reductions);
    }
    if (*abort_flag) {
        // Let every copy and MMA already in flight land before the CTA leaves.
        if (kPair && !leader && warp == 0 && lane == 0 && issued > 0) {
            // The peer's loads complete on the leader's barriers: give them a
            // fixed 100 µs (an in-bounds TMA copy lands in a few).
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 100000ull) {
            }
        } else if (warp == 0 && lane == 0) {
            for (int32_t st = 0; st < stages; ++st) {
                const int64_t times = issued > st ? (issued - 1 - st) / stages + 1 : 0;
                if (times > 0) {
                    volatile int never = 0;
                    wait_phase(smem_u32(&ctl->full[st]), static_cast<uint32_t>((times - 1) & 1),
                               &never, p.status, kErrWaitDrain, p.wait_limit_ns);
                }
            }
        }
        if (warp == 1 && lane == 0 && leader) {
            tc_commit<kPair>(smem_u32(&ctl->drain));
            volatile int never = 0;
            wait_phase(smem_u32(&ctl->drain), 0, &never, p.status, kErrWaitDrain, p.wait_limit_ns);
        }
        __syncthreads();
    }
    if (clustered) {
        // No CTA leaves while another may still read its shared memory or
        // arrive on its barriers.  Every role reaches this point: all of its
        // waits are bounded.
        if (!cluster_waited) cluster_wait();
        cluster_arrive();
        cluster_wait();
    }
    if (warp == 1) {
        tc_fence_after_sync();
        if constexpr (kPair) tmem_relinquish<true>();
        tmem_dealloc<kPair>(tmem_base, static_cast<uint32_t>(p.tmem_cols));
    }
}

}  // namespace dev
}  // namespace projgb
