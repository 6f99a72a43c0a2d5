// Device code besides the tensor-core kernel: weight packing (preparation),
// the K = 0 fill, and the bounded-wait self-test.  Only the C-ABI translation
// unit includes this file.
#pragma once

#include "proj_kernel.cuh"

namespace projgb {
namespace dev {

// Weight packing (preparation, not part of a run): packed block (tn, kb) holds
// rows tn·block_n + r, r < block_n, and K positions kb·64 + c, c < 64, K
// contiguous; positions past N or K are zero.  One thread writes 16 bytes (8
// values).  [N,K] weights: consecutive threads take consecutive K chunks of a
// row (contiguous reads); [K,N] weights: consecutive threads take consecutive
// rows of one K chunk (contiguous reads along N).
//
// SwiGLU weights (interleave 1 or 2): W stacks F = N / 2 gate rows then F up
// rows.  Packed row r of tile tn takes feature f, its gate row (f) or its up
// row (F + f): interleave 1 (swapped tiles), r = 32·q + l with f = tn·(block_n
// / 2) + 16·q + l mod 16, gate for l < 16; interleave 2 (token-major tiles),
// r = 16·c + j with f = tn·(block_n / 2) + 8·c + j mod 8, gate for j < 8.  So a
// warp quarter, or a 16-column chunk, holds both halves of its features.
__device__ __forceinline__ int64_t packed_source_row(int64_t tn, int64_t r, int32_t block_n, int64_t N,
                                                     int interleave) {
    if (interleave == 0) return tn * block_n + r;
    const int64_t F = N / 2;
    int64_t f;
    bool up;
    if (interleave == 1) {
        f = tn * (block_n / 2) + (r / 32) * 16 + (r % 16);
        up = (r % 32) >= 16;
    } else {
        f = tn * (block_n / 2) + (r / 16) * 8 + (r % 8);
        up = (r % 16) >= 8;
    }
    if (f >= F) return N;  // past the weights: zero
    return up ? F + f : f;
}

__global__ void proj_pack_kernel(const uint16_t *W, uint16_t *P, int64_t N, int64_t K, int w_kn,
                                 int32_t block_n, int64_t k_blocks, int64_t chunks, int interleave) {
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < chunks;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int64_t blk, r, c8;
        if (!w_kn) {
            c8 = e & 7;
            const int64_t row = e >> 3;
            blk = row / block_n;
            r = row - blk * block_n;
        } else {
            const int64_t per_blk = static_cast<int64_t>(block_n) * 8;
            blk = e / per_blk;
            const int64_t rem = e - blk * per_blk;
            c8 = rem / block_n;
            r = rem - c8 * block_n;
        }
        const int64_t tn = blk / k_blocks;
        const int64_t kb = blk - tn * k_blocks;
        const int64_t n = packed_source_row(tn, r, block_n, N, interleave);
        const int64_t k0 = kb * 64 + c8 * 8;
        uint4 out = make_uint4(0u, 0u, 0u, 0u);
        if (n < N && k0 < K) {  // K % 8 == 0: the 8 values are all in range
            if (!w_kn) {
                out = *reinterpret_cast<const uint4 *>(W + n * K + k0);
            } else {
                uint32_t w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    w[j] = static_cast<uint32_t>(W[(k0 + 2 * j) * N + n]) |
                           (static_cast<uint32_t>(W[(k0 + 2 * j + 1) * N + n]) << 16);
                out = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        *reinterpret_cast<uint4 *>(P + ((blk * block_n + r) * 64 + c8 * 8)) = out;
    }
}

// fp32 router weights ("How I made Muse's GPU projections 1.32× faster in the
// Open Kernel Challenge", section "Why the high-plus-low router scheme
// helped"): H = roundBF16(W), R = W − FP32(H) (an fp32 subtraction), L =
// roundBF16(R), packed as [H | L] along K: packed k-block kb' < kt holds H's
// k-block kb', kb' >= kt holds L's k-block kb' − kt (kt = k-blocks of K), in
// the block layout of proj_pack_kernel.  One thread writes 16 bytes.
__global__ void proj_pack_hilo_kernel(const float *W, uint16_t *P, int64_t N, int64_t K, int w_kn,
                                      int32_t block_n, int64_t k_blocks, int64_t kt, int64_t chunks) {
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < chunks;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int64_t blk, r, c8;
        if (!w_kn) {
            c8 = e & 7;
            const int64_t row = e >> 3;
            blk = row / block_n;
            r = row - blk * block_n;
        } else {
            const int64_t per_blk = static_cast<int64_t>(block_n) * 8;
            blk = e / per_blk;
            const int64_t rem = e - blk * per_blk;
            c8 = rem / block_n;
            r = rem - c8 * block_n;
        }
        const int64_t tn = blk / k_blocks;
        const int64_t kbp = blk - tn * k_blocks;
        const bool low = kbp >= kt;
        const int64_t n = tn * block_n + r;
        const int64_t k0 = (low ? kbp - kt : kbp) * 64 + c8 * 8;
        uint32_t w4[4] = {0u, 0u, 0u, 0u};
        if (n < N && k0 < K) {  // K % 8 == 0: the 8 values are all in range
            float v[8];
            if (!w_kn) {
                const float4 a = *reinterpret_cast<const float4 *>(W + n * K + k0);
                const float4 b = *reinterpret_cast<const float4 *>(W + n * K + k0 + 4);
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
                v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = W[(k0 + j) * N + n];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint16_t h2[2];
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const float w = v[2 * j + t];
                    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
                    const __nv_bfloat16 part = low ? __float2bfloat16_rn(__fsub_rn(w, __bfloat162float(hi))) : hi;
                    h2[t] = *reinterpret_cast<const uint16_t *>(&part);
                }
                w4[j] = static_cast<uint32_t>(h2[0]) | (static_cast<uint32_t>(h2[1]) << 16);
            }
        }
        *reinterpret_cast<uint4 *>(P + ((blk * block_n + r) * 64 + c8 * 8)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
}

// Host <-> device copy of proj_run_host through memory the device can address
// (pinned or registered host buffers): `bytes` from src to dst, 16 bytes a
// thread while whole 16-byte chunks remain (both pointers 16-byte aligned),
// then the tail byte by byte.  Launched with programmatic dependent launch
// around the projection: it waits for the preceding kernel first (so it never
// writes a buffer that kernel still reads) and only then lets the next one
// start its set-up.
__global__ void proj_copy_kernel(const uint8_t *src, uint8_t *dst, int64_t bytes) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t n16 = bytes / 16;
    const uint4 *s16 = reinterpret_cast<const uint4 *>(src);
    uint4 *d16 = reinterpret_cast<uint4 *>(dst);
    // Four loads in flight per thread before their stores (the far side of
    // the host link has a long round trip); each access stays coalesced.
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (i + u * stride < n16) v[u] = s16[i + u * stride];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (i + u * stride < n16) d16[i + u * stride] = v[u];
    }
    const int64_t tail = bytes - n16 * 16;
    if (blockIdx.x == 0 && threadIdx.x < tail) dst[n16 * 16 + threadIdx.x] = src[n16 * 16 + threadIdx.x];
}

// K == 0: every sum is empty, so Y = act(bias or 0) + residual.
__global__ void proj_fill_kernel(int64_t M, int64_t N, const uint16_t *bias, void *Y, int y_f32, int act,
                                 const void *residual) {
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = i % N;
        float y = bias ? bf16_bits_to_float(bias[n]) : 0.f;
        if (act == 1) y = gelu_f32(y);
        if (residual)
            y += y_f32 ? static_cast<const float *>(residual)[i]
                       : __bfloat162float(static_cast<const __nv_bfloat16 *>(residual)[i]);
        if (y_f32)
            static_cast<float *>(Y)[i] = y;
        else
            static_cast<__nv_bfloat16 *>(Y)[i] = __float2bfloat16_rn(y);
    }
}

// Self-test of the bounded wait: a barrier nothing arrives on.
__global__ void proj_selftest_wait_kernel(int64_t limit_ns, int *status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool ok = wait_phase(smem_u32(&bar), 0, &abort_flag, status, kErrSelfTest, limit_ns);
        if (ok) atomicOr(status, 1 << 30);  // would mean the wait completed: it must not
    }
}

}  // namespace dev
}  // namespace projgb
