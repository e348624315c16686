// shard_combine.cuh -- the standalone on-device combines of the sharded
// linear layers, both bound by HBM bandwidth:
//
//   shard_reduce  Y[r, c] = sum_i P[i, r, c]   (all-reduce -> on-device sum)
//   shard_concat  Y[:, cols of shard i] = Ys[i] (all-gather -> on-device concat)
//
// Both stream 16-byte vectors with fully coalesced loads and stores; the grid
// is a whole number of waves over the SMs and each thread walks a grid
// stride.  Partials are read with the streaming (evict-first) hint since
// every byte is touched exactly once.
#pragma once

#include "tp_device.cuh"

namespace tpk {

__device__ __forceinline__ float4 ld_stream_f4(const float4 *p) { return __ldcs(p); }

__device__ __forceinline__ void add4(float4 &a, const float4 &b) {
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
}

// Each thread owns 8 consecutive output elements per step: it loads the 8
// fp32 values of every shard (2 x 16 bytes per shard, all loads issued before
// the first add when NS is a compile-time constant), adds them in ascending
// shard order and stores 16 bytes (bf16) or 32 bytes (fp32).  Lanes never
// need each other's data, so no cross-lane combine is required.
template <int NS, bool OUT_BF16>
__global__ void __launch_bounds__(256) shard_reduce_kernel(const float *__restrict__ P,
                                                           void *__restrict__ Y, int64_t n_vec8,
                                                           int64_t shard_stride, int n_shards) {
    const int ns = NS > 0 ? NS : n_shards;
    const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const float4 *P4 = reinterpret_cast<const float4 *>(P);
    const int64_t s4 = shard_stride / 4;
    for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < n_vec8;
         v += step) {
        float4 a0, a1;
        if constexpr (NS > 0) {
            float4 t[NS][2];
#pragma unroll
            for (int s = 0; s < NS; ++s) {
                t[s][0] = ld_stream_f4(P4 + s * s4 + 2 * v);
                t[s][1] = ld_stream_f4(P4 + s * s4 + 2 * v + 1);
            }
            a0 = t[0][0];
            a1 = t[0][1];
#pragma unroll
            for (int s = 1; s < NS; ++s) {
                add4(a0, t[s][0]);
                add4(a1, t[s][1]);
            }
        } else {
            a0 = ld_stream_f4(P4 + 2 * v);
            a1 = ld_stream_f4(P4 + 2 * v + 1);
            for (int s = 1; s < ns; ++s) {
                add4(a0, ld_stream_f4(P4 + s * s4 + 2 * v));
                add4(a1, ld_stream_f4(P4 + s * s4 + 2 * v + 1));
            }
        }
        if constexpr (OUT_BF16) {
            uint4 u = make_uint4(pack_bf16x2(a0.x, a0.y), pack_bf16x2(a0.z, a0.w),
                                 pack_bf16x2(a1.x, a1.y), pack_bf16x2(a1.z, a1.w));
            reinterpret_cast<uint4 *>(Y)[v] = u;
        } else {
            float4 *y4 = reinterpret_cast<float4 *>(Y);
            y4[2 * v] = a0;
            y4[2 * v + 1] = a1;
        }
    }
}

// Element-wise fallback for sizes that are not a multiple of 8 elements:
// same ascending-order fp32 sum, one element per thread.
template <bool OUT_BF16>
__global__ void shard_reduce_scalar_kernel(const float *__restrict__ P, void *__restrict__ Y,
                                           int64_t total, int n_shards) {
    const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += step) {
        float acc = P[t];
        for (int s = 1; s < n_shards; ++s) acc += P[static_cast<int64_t>(s) * total + t];
        if constexpr (OUT_BF16)
            static_cast<__nv_bfloat16 *>(Y)[t] = __float2bfloat16_rn(acc);
        else
            static_cast<float *>(Y)[t] = acc;
    }
}

// Concat: grid.y walks output rows, grid.x x threads walk the 16-byte vectors
// of a row.  Output vector cv of a row decomposes into (column group b,
// shard i, offset j) with two multiply-high divisions; the source is vector
// b*swv + j of row `row` of shard i.  Stores are row-contiguous, loads are
// contiguous within each shard's run.
__global__ void __launch_bounds__(256) shard_concat_kernel(const uint4 *__restrict__ Ys,
                                                           uint4 *__restrict__ Y, int64_t rows,
                                                           uint32_t ncv, FastDiv gwv, FastDiv swv,
                                                           uint32_t nlv) {
    const uint32_t cv = blockIdx.x * blockDim.x + threadIdx.x;
    if (cv >= ncv) return;
    const uint32_t b = fastdiv(cv, gwv);
    const uint32_t rem = cv - b * gwv.d;
    const uint32_t i = fastdiv(rem, swv);
    const uint32_t j = rem - i * swv.d;
    for (int64_t row = blockIdx.y; row < rows; row += gridDim.y) {
        const uint4 v = __ldcs(Ys + (static_cast<int64_t>(i) * rows + row) * nlv + b * swv.d + j);
        __stcs(Y + row * ncv + cv, v);
    }
}

}  // namespace tpk
