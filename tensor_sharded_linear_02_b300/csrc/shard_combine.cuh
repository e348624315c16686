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

// Streaming reduce through shared memory: a persistent kernel, one CTA per
// SM.  The output is cut into chunks of `chunk` elements (a multiple of 8);
// CTA b takes chunks b, b + grid, ...  For each chunk one thread issues one
// bulk copy per shard (chunk * 4 contiguous bytes of P_i) into a stage of a
// RED_STAGES-deep ring in shared memory, all counted on the stage's `full`
// barrier; the 256 consumer threads add the shards of 8 consecutive
// elements in ascending shard order in fp32 from shared memory and store 16
// bytes of bf16 (or 32 of fp32), and each consumer warp releases the stage.
// Large contiguous copies keep every DRAM page open for long runs, and the
// copies are issued by one thread, so no register file holds data in flight.
constexpr int RED_STAGES = 3;
constexpr int RED_STAGE_BYTES = 64 * 1024;
constexpr int RED_CONSUMERS = 256;
constexpr int RED_THREADS = 32 + RED_CONSUMERS;
constexpr int RED_SMEM_BYTES = RED_STAGES * RED_STAGE_BYTES + 128;

template <bool OUT_BF16>
__global__ void __launch_bounds__(RED_THREADS, 1)
    shard_reduce_bulk_kernel(const float *__restrict__ P, void *__restrict__ Y, int64_t total,
                             int n_shards, int chunk, uint64_t limit_ns) {
    extern __shared__ __align__(128) uint8_t red_smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(red_smem + RED_STAGES * RED_STAGE_BYTES);
    uint64_t *empty = full + RED_STAGES;
    uint32_t *abort = reinterpret_cast<uint32_t *>(empty + RED_STAGES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < RED_STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), RED_CONSUMERS / 32);
        }
        *abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) grid_dep_trigger();
    grid_dep_wait();

    const int64_t n_chunks = (total + chunk - 1) / chunk;
    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool issued = false, ok = true;
            for (int64_t c = blockIdx.x; c < n_chunks && ok; c += gridDim.x) {
                if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, limit_ns, abort,
                                       SITE_PRODUCER_EMPTY)) {
                    ok = false;
                    break;
                }
                const int64_t e0 = c * chunk;
                const int64_t n = total - e0 < chunk ? total - e0 : chunk;
                const uint32_t bytes = static_cast<uint32_t>(n * 4);
                const uint32_t fb = smem_u32(&full[stage]);
                mbar_arrive_expect_tx(fb, bytes * static_cast<uint32_t>(n_shards));
                const uint32_t dst = smem_u32(red_smem + stage * RED_STAGE_BYTES);
                for (int i = 0; i < n_shards; ++i)
                    bulk_load(dst + static_cast<uint32_t>(i) * static_cast<uint32_t>(chunk) * 4u,
                              P + static_cast<int64_t>(i) * total + e0, bytes, fb);
                issued = true;
                if (++stage == RED_STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // every stage released before exit (a copy still landing after
            // an abort is waited for the same way, with the drain limit)
            for (int s = 0; s < RED_STAGES && issued; ++s) {
                if (ok) {
                    ok = mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, limit_ns, abort,
                                           SITE_PRODUCER_EMPTY);
                } else {
                    mbar_wait_drain(smem_u32(&full[stage]), phase ^ 1u, limit_ns);
                }
                if (++stage == RED_STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        __syncwarp();
    } else {
        const int t = threadIdx.x - 32;
        int stage = 0;
        uint32_t phase = 0;
        for (int64_t c = blockIdx.x; c < n_chunks; c += gridDim.x) {
            if (!mbar_wait_warp(smem_u32(&full[stage]), phase, limit_ns, abort, SITE_MMA_FULL))
                break;
            const int64_t e0 = c * chunk;
            const int n = static_cast<int>(total - e0 < chunk ? total - e0 : chunk);
            const float *src = reinterpret_cast<const float *>(red_smem + stage * RED_STAGE_BYTES);
            for (int e = t * 8; e < n; e += RED_CONSUMERS * 8) {
                float4 a0 = *reinterpret_cast<const float4 *>(src + e);
                float4 a1 = *reinterpret_cast<const float4 *>(src + e + 4);
                for (int i = 1; i < n_shards; ++i) {
                    const float *q = src + static_cast<int64_t>(i) * chunk + e;
                    add4(a0, *reinterpret_cast<const float4 *>(q));
                    add4(a1, *reinterpret_cast<const float4 *>(q + 4));
                }
                if constexpr (OUT_BF16) {
                    const uint4 u = make_uint4(pack_bf16x2(a0.x, a0.y), pack_bf16x2(a0.z, a0.w),
                                               pack_bf16x2(a1.x, a1.y), pack_bf16x2(a1.z, a1.w));
                    __stcs(reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(Y) + e0 + e), u);
                } else {
                    float4 *y = reinterpret_cast<float4 *>(static_cast<float *>(Y) + e0 + e);
                    __stcs(y, a0);
                    __stcs(y + 1, a1);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
            if (++stage == RED_STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    __syncthreads();
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
