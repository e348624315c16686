// simt_linear.cuh -- fp32 sharded linear on the CUDA cores.
//
// Serves fp32 inputs (where tensor cores would round to tf32) and any shape
// or alignment.  One thread per output element; the contraction runs in
// ascending k with fused multiply-adds in fp32, shard by shard:
//   p_i = sum_{k in K_i} x[k] * w[k]      (fp32 FMA chain)
//   y   = ((p_0 + p_1) + p_2) + ...       (ascending shard order)
// With k_shards = 1 this is the plain column-parallel product.  Products and
// sums of integer values below 2^24 are exact, so integer-valued inputs give
// bit-exact results for either split.
#pragma once

#include "tp_device.cuh"

namespace tpk {

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ void from_f32(float v, float *dst) { *dst = v; }
__device__ __forceinline__ void from_f32(float v, __nv_bfloat16 *dst) { *dst = __float2bfloat16_rn(v); }

struct SimtArgs {
    int64_t M, K, N;
    int64_t k_shards;   // contraction shards (row split); 1 for the column split
    int act_gelu;
    float *partials;    // optional [k_shards, M, N] fp32 partial outputs
    const void *bias;   // optional [N] (input dtype), added after the shard sum
    int64_t shard_sw, shard_gw, shard_nl;  // shard-major copy layout (column split)
};

template <typename Tin, typename Tout>
__global__ void simt_linear_kernel(const Tin *__restrict__ X, const Tin *__restrict__ W,
                                   Tout *__restrict__ Y, Tout *__restrict__ Ys, const SimtArgs a) {
    const int64_t col = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (col >= a.N) return;
    const int64_t ks = a.K / a.k_shards;
    for (int64_t row = static_cast<int64_t>(blockIdx.y) * blockDim.y + threadIdx.y; row < a.M;
         row += static_cast<int64_t>(gridDim.y) * blockDim.y) {
        const Tin *x = X + row * a.K;
        float y = 0.0f;
        for (int64_t s = 0; s < a.k_shards; ++s) {
            float p = 0.0f;
            for (int64_t k = s * ks; k < (s + 1) * ks; ++k)
                p = fmaf(to_f32(x[k]), to_f32(W[k * a.N + col]), p);
            if (a.partials) a.partials[(s * a.M + row) * a.N + col] = p;
            y = (s == 0) ? p : y + p;
        }
        if (a.bias) y += to_f32(static_cast<const Tin *>(a.bias)[col]);
        if (a.act_gelu) y = gelu_f32(y);
        if (Y) from_f32(y, Y + row * a.N + col);
        if (Ys) {
            const int64_t b = col / a.shard_gw;
            const int64_t cc = col - b * a.shard_gw;
            const int64_t i = cc / a.shard_sw;
            const int64_t j = cc - i * a.shard_sw;
            from_f32(y, Ys + (i * a.M + row) * a.shard_nl + b * a.shard_sw + j);
        }
    }
}

}  // namespace tpk
