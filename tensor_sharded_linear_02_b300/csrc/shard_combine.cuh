// shard_combine.cuh -- the standalone on-device combines of the sharded
// linear layers, both bound by HBM bandwidth:
//
//   shard_reduce  Y[r, c] = sum_i P[i, r, c]   (all-reduce -> on-device sum)
//   shard_concat  Y[:, cols of shard i] = Ys[i] (all-gather -> on-device concat)
//
// Both stream through a shared-memory ring filled by bulk/TMA copies issued
// by one thread per SM: the reduce copies large contiguous chunks of every
// partial and adds them in registers, the concat moves tiles from the shards
// to their place in the output without touching registers.
#pragma once

#include "tp_device.cuh"

namespace tpk {

__device__ __forceinline__ void add4(float4 &a, const float4 &b) {
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
}

// Streaming reduce through shared memory: a persistent kernel, one CTA per
// SM.  The output is cut into chunks of `chunk` elements (a multiple of 8);
// CTA b takes chunks b, b + grid, ...  For each chunk one thread issues one
// bulk copy per shard (chunk * 4 contiguous bytes of P_i) into a stage of a
// RED_STAGES-deep ring in shared memory, all counted on the stage's `full`
// barrier (cutting the copies into 4-32 KiB pieces measured the same); the 256 consumer threads add the shards of 8 consecutive
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
                             int n_shards, int chunk, uint64_t limit_ns,
                             const __nv_bfloat16 *__restrict__ bias, int64_t cols) {
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
                if (bias) {  // once, after the sum; cols % 8 == 0 keeps the 8 in one row
                    const uint4 bv = __ldg(reinterpret_cast<const uint4 *>(
                        bias + (e0 + e) % cols));
                    a0.x += __uint_as_float(bv.x << 16); a0.y += __uint_as_float(bv.x & 0xffff0000u);
                    a0.z += __uint_as_float(bv.y << 16); a0.w += __uint_as_float(bv.y & 0xffff0000u);
                    a1.x += __uint_as_float(bv.z << 16); a1.y += __uint_as_float(bv.z & 0xffff0000u);
                    a1.z += __uint_as_float(bv.w << 16); a1.w += __uint_as_float(bv.w & 0xffff0000u);
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
                                           int64_t total, int n_shards,
                                           const __nv_bfloat16 *__restrict__ bias, int64_t cols) {
    const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += step) {
        float acc = P[t];
        for (int s = 1; s < n_shards; ++s) acc += P[static_cast<int64_t>(s) * total + t];
        if (bias) acc += __bfloat162float(bias[t % cols]);
        if constexpr (OUT_BF16)
            static_cast<__nv_bfloat16 *>(Y)[t] = __float2bfloat16_rn(acc);
        else
            static_cast<float *>(Y)[t] = acc;
    }
}

// Concat through shared memory with tiled TMA copies: a persistent kernel,
// one CTA (one working thread) per SM.  A unit is a box of `box_rows` rows x
// `box_cols` columns of one column group b of one shard i: loaded from Ys
// (viewed as [n][rows][shard_cols]) at (b*sw + j0, r0, i) and stored to Y
// (viewed as [rows][n*shard_cols]) at (b*gw + i*sw + j0, r0); the bytes never
// pass through registers.  Loads run CAT_LAG units ahead of stores in a
// CAT_STAGES-deep ring; a stage is reused once the store that read it has
// left shared memory.  Rows past the end are zero-filled by the load and
// clipped by the store.  Measured on the 8 x [8192, 1536] bf16 concat (L2
// flushed clean): boxes of 32 KiB in a 6-deep ring, loads 4 ahead, 63.5 us
// (0.98 of copy bandwidth); 16 KiB boxes in a 12-deep ring, loads 8 ahead,
// 72 us; the same bytes in flight split over 2 or 4 CTAs per SM, 63.5 us.
constexpr int CAT_STAGES = 6;
constexpr int CAT_LAG = 4;
constexpr int CAT_BOX_BYTES = 32 * 1024;
constexpr int CAT_SMEM_BYTES = CAT_STAGES * CAT_BOX_BYTES + 128;

struct CatArgs {
    int n, groups;         // shards, column groups
    int sw, gw;            // columns a shard owns per group, output columns per group (n*sw)
    int box_cols, box_rows;
    int col_boxes;         // sw / box_cols
    int64_t units;         // row blocks * n * groups * col_boxes
    uint32_t box_bytes;
    uint64_t wait_limit_ns;
};

__global__ void __launch_bounds__(32, 1)
    shard_concat_tma_kernel(const __grid_constant__ CUtensorMap tmSrc,
                            const __grid_constant__ CUtensorMap tmDst, const CatArgs a) {
    extern __shared__ __align__(128) uint8_t cat_smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(cat_smem + CAT_STAGES * CAT_BOX_BYTES);
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        for (int st = 0; st < CAT_STAGES; ++st) mbar_init(smem_u32(&full[st]), 1);
        abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmSrc);
        tma_prefetch_desc(&tmDst);
    }
    __syncwarp();
    if (threadIdx.x == 0) grid_dep_trigger();
    grid_dep_wait();
    if (threadIdx.x != 0) return;

    // this CTA's units: blockIdx.x, blockIdx.x + gridDim.x, ...
    const int64_t mine = a.units > blockIdx.x ? (a.units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    bool ok = true;
    int64_t issued = 0, stored = 0;  // units loaded / stored so far
    for (int64_t step = 0; step < mine + CAT_LAG && ok; ++step) {
        if (step < mine) {
            const int st = static_cast<int>(step % CAT_STAGES);
            // the store of unit step - CAT_STAGES (issued CAT_LAG steps after
            // its load) has left this stage: at most CAT_STAGES - 1 - CAT_LAG
            // younger stores may still be reading
            bulk_wait_read_n<CAT_STAGES - 1 - CAT_LAG>();
            const int64_t u = blockIdx.x + step * gridDim.x;
            int64_t t = u;
            const int jb = static_cast<int>(t % a.col_boxes); t /= a.col_boxes;
            const int b = static_cast<int>(t % a.groups); t /= a.groups;
            const int i = static_cast<int>(t % a.n); t /= a.n;
            const int r0 = static_cast<int>(t) * a.box_rows;
            const uint32_t fb = smem_u32(&full[st]);
            mbar_arrive_expect_tx(fb, a.box_bytes);
            tma_load_3d(smem_u32(cat_smem + st * CAT_BOX_BYTES), &tmSrc, fb,
                        b * a.sw + jb * a.box_cols, r0, i);
            issued = step + 1;
        }
        const int64_t j = step - CAT_LAG;
        if (j >= 0 && j < mine) {
            const int st = static_cast<int>(j % CAT_STAGES);
            const uint32_t par = static_cast<uint32_t>((j / CAT_STAGES) & 1);
            if (!mbar_wait_bounded(smem_u32(&full[st]), par, a.wait_limit_ns, &abort_flag,
                                   SITE_MMA_FULL)) {
                ok = false;
                break;
            }
            const int64_t u = blockIdx.x + j * gridDim.x;
            int64_t t = u;
            const int jb = static_cast<int>(t % a.col_boxes); t /= a.col_boxes;
            const int b = static_cast<int>(t % a.groups); t /= a.groups;
            const int i = static_cast<int>(t % a.n); t /= a.n;
            const int r0 = static_cast<int>(t) * a.box_rows;
            tma_store_3d(&tmDst, smem_u32(cat_smem + st * CAT_BOX_BYTES),
                         b * a.gw + i * a.sw + jb * a.box_cols, r0, 0);
            bulk_commit_group();
            stored = j + 1;
        }
    }
    // after an abort, loads issued but not stored must land before the CTA
    // exits (at most CAT_LAG of them, each in its own stage)
    for (int64_t j = stored; j < issued; ++j)
        mbar_wait_drain(smem_u32(&full[j % CAT_STAGES]),
                        static_cast<uint32_t>((j / CAT_STAGES) & 1), a.wait_limit_ns);
    bulk_wait_read0();  // the stores have left shared memory
}

// Column-segment copy with TMA boxes: the same ring as the concat, driven
// by a table of segments.  Segment k copies columns [src_col, src_col +
// width) of slot src_slot of the source (viewed as [slots][rows][cols]) to
// columns [dst_col, dst_col + width) of slot dst_slot of the destination.
// A source segment may be copied to several destinations (replication).
// Used for the shard-local outputs of the grouped-query QKV projection.
constexpr int SEG_MAX = 192;

struct SegTable {
    int n_seg;
    int box_cols, box_rows;
    int col_boxes;          // sum over segments of width / box_cols
    int64_t units;          // row blocks * col_boxes
    uint32_t box_bytes;
    uint64_t wait_limit_ns;
    int prefix[SEG_MAX + 1];  // col-box index where segment k starts
    int src_slot[SEG_MAX], src_col[SEG_MAX], dst_slot[SEG_MAX], dst_col[SEG_MAX];
};

__device__ __forceinline__ void seg_decode(const SegTable &t, int64_t u, int &k, int &cb, int &r0) {
    const int64_t rb = u / t.col_boxes;
    const int c = static_cast<int>(u - rb * t.col_boxes);
    k = 0;
    while (t.prefix[k + 1] <= c) ++k;
    cb = c - t.prefix[k];
    r0 = static_cast<int>(rb) * t.box_rows;
}

__global__ void __launch_bounds__(32, 1)
    segment_copy_tma_kernel(const __grid_constant__ CUtensorMap tmSrc,
                            const __grid_constant__ CUtensorMap tmDst,
                            const __grid_constant__ SegTable t) {
    extern __shared__ __align__(128) uint8_t seg_smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(seg_smem + CAT_STAGES * CAT_BOX_BYTES);
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        for (int st = 0; st < CAT_STAGES; ++st) mbar_init(smem_u32(&full[st]), 1);
        abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmSrc);
        tma_prefetch_desc(&tmDst);
    }
    __syncwarp();
    if (threadIdx.x == 0) grid_dep_trigger();
    grid_dep_wait();
    if (threadIdx.x != 0) return;

    const int64_t mine = t.units > blockIdx.x ? (t.units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    bool ok = true;
    int64_t issued = 0, stored = 0;
    for (int64_t step = 0; step < mine + CAT_LAG && ok; ++step) {
        if (step < mine) {
            const int st = static_cast<int>(step % CAT_STAGES);
            bulk_wait_read_n<CAT_STAGES - 1 - CAT_LAG>();
            int k, cb, r0;
            seg_decode(t, blockIdx.x + step * gridDim.x, k, cb, r0);
            const uint32_t fb = smem_u32(&full[st]);
            mbar_arrive_expect_tx(fb, t.box_bytes);
            tma_load_3d(smem_u32(seg_smem + st * CAT_BOX_BYTES), &tmSrc, fb,
                        t.src_col[k] + cb * t.box_cols, r0, t.src_slot[k]);
            issued = step + 1;
        }
        const int64_t j = step - CAT_LAG;
        if (j >= 0 && j < mine) {
            const int st = static_cast<int>(j % CAT_STAGES);
            if (!mbar_wait_bounded(smem_u32(&full[st]), static_cast<uint32_t>((j / CAT_STAGES) & 1),
                                   t.wait_limit_ns, &abort_flag, SITE_MMA_FULL)) {
                ok = false;
                break;
            }
            int k, cb, r0;
            seg_decode(t, blockIdx.x + j * gridDim.x, k, cb, r0);
            tma_store_3d(&tmDst, smem_u32(seg_smem + st * CAT_BOX_BYTES),
                         t.dst_col[k] + cb * t.box_cols, r0, t.dst_slot[k]);
            bulk_commit_group();
            stored = j + 1;
        }
    }
    for (int64_t j = stored; j < issued; ++j)
        mbar_wait_drain(smem_u32(&full[j % CAT_STAGES]),
                        static_cast<uint32_t>((j / CAT_STAGES) & 1), t.wait_limit_ns);
    bulk_wait_read0();  // the stores have left shared memory
}

}  // namespace tpk
