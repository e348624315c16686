// gemm_tcgen05.cuh -- bf16 GEMM on the sm_103a tensor cores for the sharded
// linear layers:  out[M, N] = act( sum over the k-range of A[M, K] . B[K, N] ).
//
//   A  row-major [M, K]   (X, or the hidden activation H)  -> K-major operand
//   B  row-major [K, N]   (the weight W as stored)          -> MN-major operand
//
// Data path: TMA (128-byte swizzle) -> 4-stage shared-memory ring (mbarrier
// full/empty pairs) -> tcgen05.mma.kind::f16, 128 x 256 x 16 per instruction,
// issued by one thread -> fp32 accumulator in tensor memory -> tcgen05.ld by
// the epilogue warps -> optional GeLU -> bf16 (RNE) or fp32 -> global store.
//
// Warp roles (320 threads): warp 0 = TMA producer, warp 1 = TMEM owner and
// MMA issuer, warps 2..9 = epilogue (warp w reads TMEM lanes 32*(w%4)..+31,
// warps 2..5 the first 128 accumulator columns, warps 6..9 the last 128).
//
// Two kernels:
//   gemm_persistent_kernel  one CTA per SM walks work units (tile, k-group);
//       the accumulator is double-buffered in TMEM (2 x 256 columns) so the
//       epilogue of one tile overlaps the main loop of the next.  k-group g
//       selects shard g's K range through the 3-D tensor maps and its output
//       goes to out + g * out_group_stride (per-shard partials); with one
//       k-group the K loop walks shard 0's rows, then shard 1's, ..., so the
//       row-parallel partial sums are added inside the accumulator.
//   gemm_cluster_sum_kernel  for outputs with too few tiles to fill the GPU:
//       the S CTAs of a cluster share one output tile, CTA r accumulates the
//       r-th contiguous slice of the K blocks (with K/n a multiple of the
//       block depth and S dividing n, slice r is exactly shard group r).  CTA
//       r owns rows [r*128/S, (r+1)*128/S) of the tile.  Once every CTA of the
//       cluster has finished its main loop (a cluster barrier: from then on no
//       ring is in use), every CTA stores the fp32 partial rows it holds into
//       slot `its rank` of the owner's shared memory (distributed shared
//       memory stores), and after a second barrier each owner adds its S
//       slots in ascending slice order.
#pragma once

#include "tp_device.cuh"

namespace tpk {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK * 2;      // 16 KiB
constexpr int B_CHUNK_N = 64;                   // N columns per TMA box (128 bytes)
constexpr int B_CHUNK_BYTES = BK * B_CHUNK_N * 2;  // 8 KiB
constexpr int B_STAGE_BYTES = BK * BN * 2;      // 32 KiB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
#ifndef TP_EPI_WARPS
#define TP_EPI_WARPS 8
#endif
// Epilogue warps: a multiple of 4 (each TMEM lane quadrant is read by
// EPI_WARPS/4 warps, each taking an equal share of the columns).
constexpr int EPI_WARPS = TP_EPI_WARPS;
constexpr int EPI_COL_CHUNKS = BN / 32 / (EPI_WARPS / 4);  // 32-column chunks per epilogue warp
constexpr int GEMM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int RED_LD = BN + 4;  // fp32 row pitch of the parked partial tile (bank spread)

constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, true);

// A descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
// B descriptor: MN-major, 128-byte swizzle; a 64-column chunk holds all BK
// k-rows (BK * 128 bytes), 8-k-row groups 1024 bytes apart.
constexpr uint32_t A_SBO = 1024;
constexpr uint32_t B_LBO = B_CHUNK_BYTES;
constexpr uint32_t B_SBO = 1024;

struct SmemBarriers {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    uint32_t abort;
};

constexpr int GEMM_SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;

struct GemmArgs {
    int M, N;
    int k_blocks;        // BK-deep blocks per k-group (ceil)
    int k_groups;        // 1, or the shard count for per-shard partial outputs
    int m_tiles, n_tiles;
    int num_units;       // m_tiles * n_tiles * k_groups (persistent kernel)
    int split;           // cluster size S (cluster kernel)
    void *out;           // [M, N] row-major
    int64_t out_group_stride;  // elements between k-group outputs
    int out_f32;         // 1: fp32 output, 0: bf16
    int act_gelu;
    void *out_shards;    // optional shard-major copy (column split)
    int shard_sw;        // columns a shard owns in each column group
    int shard_gw;        // columns per column group
    int shard_nl;        // local columns per shard
    uint64_t wait_limit_ns;
};

// ---------------------------------------------------------------------------
// Epilogue: activation, rounding and store of 8 consecutive columns of one
// output row (row < M, col < N, col a multiple of 8).  Writes the plain
// output (k-group g) and, if requested, the shard-major copy.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store_vec8(const GemmArgs &a, int g, int row, int col,
                                           float (&f)[8]) {
    if (a.act_gelu) {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = gelu_f32(f[i]);
    }
    uint4 u;
    if (!a.out_f32)
        u = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                       pack_bf16x2(f[6], f[7]));
    if (a.out) {
        const int64_t off = static_cast<int64_t>(g) * a.out_group_stride +
                            static_cast<int64_t>(row) * a.N + col;
        if (a.out_f32) {
            float4 *p = reinterpret_cast<float4 *>(static_cast<float *>(a.out) + off);
            p[0] = make_float4(f[0], f[1], f[2], f[3]);
            p[1] = make_float4(f[4], f[5], f[6], f[7]);
        } else {
            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + off) = u;
        }
    }
    if (a.out_shards) {
        // column -> (group b, shard i, offset j); the shard width per group is
        // a multiple of 8, so the vector stays inside one shard.
        const int b = col / a.shard_gw;
        const int cc = col - b * a.shard_gw;
        const int i = cc / a.shard_sw;
        const int j = cc - i * a.shard_sw;
        const int64_t off = (static_cast<int64_t>(i) * a.M + row) * a.shard_nl +
                            static_cast<int64_t>(b) * a.shard_sw + j;
        if (a.out_f32) {
            float4 *p = reinterpret_cast<float4 *>(static_cast<float *>(a.out_shards) + off);
            p[0] = make_float4(f[0], f[1], f[2], f[3]);
            p[1] = make_float4(f[4], f[5], f[6], f[7]);
        } else {
            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out_shards) + off) = u;
        }
    }
}

// 32 consecutive accumulator columns of one row, as read from TMEM.
__device__ __forceinline__ void store_row_chunk32(const GemmArgs &a, int g, int row, int col0,
                                                  const uint32_t (&r)[32]) {
    if (row >= a.M) return;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int col = col0 + v * 8;
        if (col >= a.N) break;  // N is a multiple of 8
        float f[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(r[v * 8 + i]);
        store_vec8(a, g, row, col, f);
    }
}

__device__ __forceinline__ void decode_unit(const GemmArgs &a, int u, int &m_tile, int &n_tile,
                                            int &g) {
    const int tiles = a.m_tiles * a.n_tiles;
    g = u / tiles;
    const int t = u - g * tiles;
    m_tile = t % a.m_tiles;
    n_tile = t / a.m_tiles;
}

// ---------------------------------------------------------------------------
// Producer: one thread issues the TMA loads of k-blocks [kb0, kb1) of one
// unit into the ring.  Returns false on abort.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool produce_kblocks(const CUtensorMap *tmA, const CUtensorMap *tmB,
                                                uint8_t *ring, SmemBarriers *bars, int &stage,
                                                uint32_t &phase, uint32_t &issued_mask,
                                                uint32_t &issued_parity, int m_tile, int n_tile,
                                                int g, int kb0, int kb1, uint64_t limit) {
    for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&bars->empty[stage]), phase ^ 1u, limit, &bars->abort,
                               SITE_PRODUCER_EMPTY))
            return false;
        const uint32_t fb = smem_u32(&bars->full[stage]);
        mbar_arrive_expect_tx(fb, STAGE_BYTES);
        uint8_t *sa = ring + stage * STAGE_BYTES;
        uint8_t *sb = sa + A_STAGE_BYTES;
        tma_load_3d(smem_u32(sa), tmA, fb, kb * BK, g, m_tile * BM);
#pragma unroll
        for (int j = 0; j < BN / B_CHUNK_N; ++j)
            tma_load_3d(smem_u32(sb + j * B_CHUNK_BYTES), tmB, fb, n_tile * BN + j * B_CHUNK_N,
                        kb * BK, g);
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
        }
    }
    return true;
}

// After an abort, wait (bounded) for every load the producer issued, so no
// copy is still landing in shared memory when the CTA exits.
__device__ __forceinline__ void producer_drain(SmemBarriers *bars, uint32_t issued_mask,
                                               uint32_t issued_parity, uint64_t limit) {
    for (int s = 0; s < STAGES; ++s)
        if (issued_mask & (1u << s))
            mbar_wait_drain(smem_u32(&bars->full[s]), (issued_parity >> s) & 1u, limit);
}

// MMA issuer: accumulate k-blocks [kb0, kb1) into TMEM columns at d_tmem.
__device__ __forceinline__ bool mma_kblocks(uint8_t *ring, SmemBarriers *bars, int &stage,
                                            uint32_t &phase, uint32_t d_tmem, int kb0, int kb1,
                                            uint64_t limit) {
    for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&bars->full[stage]), phase, limit, &bars->abort,
                               SITE_MMA_FULL))
            return false;
        tc_fence_after();
        const uint32_t sa = smem_u32(ring + stage * STAGE_BYTES);
        const uint32_t sb = sa + A_STAGE_BYTES;
#pragma unroll
        for (int k = 0; k < BK / UMMA_K; ++k) {
            // A: advance 16 bf16 (32 bytes) along K inside the swizzle row.
            // B: advance 16 k-rows = two 8-row groups of 1024 bytes.
            const uint64_t da = smem_desc_sw128(sa + k * (UMMA_K * 2), 16, A_SBO);
            const uint64_t db = smem_desc_sw128(sb + k * (UMMA_K / 8) * B_SBO, B_LBO, B_SBO);
            umma_f16(d_tmem, da, db, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
        }
        umma_commit(smem_u32(&bars->empty[stage]));
        if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
        }
    }
    return true;
}

__device__ __forceinline__ void mma_drain(SmemBarriers *bars, uint64_t limit) {
    umma_commit(smem_u32(&bars->drain));
    mbar_wait_drain(smem_u32(&bars->drain), 0, limit);
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void gemm_setup(SmemBarriers *bars, uint32_t tmem_cols, int epi_arrivals,
                                           const CUtensorMap *tmA, const CUtensorMap *tmB) {
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&bars->full[s]), 1);
            mbar_init(smem_u32(&bars->empty[s]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bars->acc_full[i]), 1);
            mbar_init(smem_u32(&bars->acc_empty[i]), epi_arrivals);
        }
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && (threadIdx.x & 31) == 0) {
        tma_prefetch_desc(tmA);
        tma_prefetch_desc(tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// ---------------------------------------------------------------------------
// Persistent kernel.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_persistent_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB, const GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = align1024(smem_raw);
    SmemBarriers *bars = reinterpret_cast<SmemBarriers *>(ring + STAGES * STAGE_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr uint32_t TMEM_COLS = 2 * BN;

    gemm_setup(bars, TMEM_COLS, EPI_WARPS, &tmA, &tmB);
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(&bars->tmem_base);
    const uint64_t limit = a.wait_limit_ns;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued_mask = 0, issued_parity = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < a.num_units && ok; u += gridDim.x) {
                int mt, nt, g;
                decode_unit(a, u, mt, nt, g);
                ok = produce_kblocks(&tmA, &tmB, ring, bars, stage, phase, issued_mask,
                                     issued_parity, mt, nt, g, 0, a.k_blocks, limit);
            }
            if (!ok) producer_drain(bars, issued_mask, issued_parity, limit);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, local = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < a.num_units && ok; u += gridDim.x, ++local) {
                const int acc = local & 1;
                const uint32_t acc_par = (local >> 1) & 1;
                ok = mbar_wait_bounded(smem_u32(&bars->acc_empty[acc]), acc_par ^ 1u, limit,
                                       &bars->abort, SITE_MMA_ACC_EMPTY);
                if (!ok) break;
                tc_fence_after();
                ok = mma_kblocks(ring, bars, stage, phase, tmem_base + acc * BN, 0, a.k_blocks,
                                 limit);
                if (!ok) break;
                umma_commit(smem_u32(&bars->acc_full[acc]));
            }
            if (!ok) mma_drain(bars, limit);
        }
        __syncwarp();
    } else {
        const int q = warp & 3;                             // TMEM lane quadrant
        const int c0 = ((warp - 2) >> 2) * EPI_COL_CHUNKS;  // first 32-column chunk
        int local = 0;
        for (int u = blockIdx.x; u < a.num_units; u += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t acc_par = (local >> 1) & 1;
            if (!mbar_wait_warp(smem_u32(&bars->acc_full[acc]), acc_par, limit, &bars->abort,
                                SITE_EPI_ACC_FULL))
                break;
            tc_fence_after();
            int mt, nt, g;
            decode_unit(a, u, mt, nt, g);
            const int row = mt * BM + q * 32 + lane;
            const uint32_t taddr = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
            for (int c = c0; c < c0 + EPI_COL_CHUNKS; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + c * 32, r);
                tmem_ld_wait();
                store_row_chunk32(a, g, row, nt * BN + c * 32, r);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[acc]));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Cluster split kernel: grid = S * tiles CTAs, cluster = S CTAs along x.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_cluster_sum_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB, const GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = align1024(smem_raw);
    SmemBarriers *bars = reinterpret_cast<SmemBarriers *>(ring + STAGES * STAGE_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr uint32_t TMEM_COLS = BN;

    const int S = a.split;
    const int rank = static_cast<int>(cluster_ctarank());
    const int tile = blockIdx.x / S;
    const int mt = tile % a.m_tiles;
    const int nt = tile / a.m_tiles;
    const int kb0 = static_cast<int>((static_cast<int64_t>(a.k_blocks) * rank) / S);
    const int kb1 = static_cast<int>((static_cast<int64_t>(a.k_blocks) * (rank + 1)) / S);

    gemm_setup(bars, TMEM_COLS, EPI_WARPS, &tmA, &tmB);
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(&bars->tmem_base);
    const uint64_t limit = a.wait_limit_ns;
    float *red = reinterpret_cast<float *>(ring);  // parks the fp32 partial tile

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued_mask = 0, issued_parity = 0;
            if (!produce_kblocks(&tmA, &tmB, ring, bars, stage, phase, issued_mask, issued_parity,
                                 mt, nt, 0, kb0, kb1, limit))
                producer_drain(bars, issued_mask, issued_parity, limit);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            if (mma_kblocks(ring, bars, stage, phase, tmem_base, kb0, kb1, limit))
                umma_commit(smem_u32(&bars->acc_full[0]));
            else
                mma_drain(bars, limit);
        }
        __syncwarp();
    } else {
        if (mbar_wait_warp(smem_u32(&bars->acc_full[0]), 0, limit, &bars->abort,
                           SITE_EPI_ACC_FULL))
            tc_fence_after();
    }

    // Every CTA of the cluster has finished its main loop: from here on no
    // ring is in use by TMA or MMA, so each can take parked partial rows.
    cluster_sync_all();

    if (warp >= 2 && !bars->abort) {
        // Push: row `rit` of this CTA's fp32 partial goes to slot `rank` of
        // its owner's parking area [S][BM/S][RED_LD] (local or remote).
        fence_proxy_async_smem();
        const int q = warp & 3;
        const int c0 = ((warp - 2) >> 2) * EPI_COL_CHUNKS;
        const int rows_per = BM / S;
        const int rit = q * 32 + lane;  // row in tile
        const int owner = rit / rows_per;
        const int slot_row = rank * rows_per + (rit - owner * rows_per);
        float *dst = red + slot_row * RED_LD;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
        for (int c = c0; c < c0 + EPI_COL_CHUNKS; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + c * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const float4 val =
                    make_float4(__uint_as_float(r[v * 4 + 0]), __uint_as_float(r[v * 4 + 1]),
                                __uint_as_float(r[v * 4 + 2]), __uint_as_float(r[v * 4 + 3]));
                float *p = dst + c * 32 + v * 4;
                if (owner == rank)
                    *reinterpret_cast<float4 *>(p) = val;
                else
                    dsmem_st_f4(dsmem_map(smem_u32(p), static_cast<uint32_t>(owner)), val);
            }
        }
    }

    // Every CTA of the cluster has delivered its partial rows.
    cluster_sync_all();

    if (warp >= 2) {
        // Owner: rows [rank*BM/S, (rank+1)*BM/S) of the tile, S slots each,
        // added in ascending slice order from local shared memory.
        const int rows_per = BM / S;
        const int cl = lane * 8;  // 8 consecutive columns per lane, BN = 32 * 8
        for (int rr = warp - 2; rr < rows_per; rr += EPI_WARPS) {
            const int row = mt * BM + rank * rows_per + rr;
            const float *src = red + rr * RED_LD + cl;
            float4 s0 = *reinterpret_cast<const float4 *>(src);
            float4 s1 = *reinterpret_cast<const float4 *>(src + 4);
            for (int p = 1; p < S; ++p) {
                const float *sp = src + p * rows_per * RED_LD;
                const float4 t0 = *reinterpret_cast<const float4 *>(sp);
                const float4 t1 = *reinterpret_cast<const float4 *>(sp + 4);
                s0.x += t0.x; s0.y += t0.y; s0.z += t0.z; s0.w += t0.w;
                s1.x += t1.x; s1.y += t1.y; s1.z += t1.z; s1.w += t1.w;
            }
            const int col = nt * BN + cl;
            if (row < a.M && col < a.N) {
                float f[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                store_vec8(a, 0, row, col, f);
            }
        }
    }

    // No CTA leaves while a peer could still be writing into its shared memory.
    cluster_sync_all();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

}  // namespace tpk
