// gemm_tcgen05.cuh -- bf16 GEMM on the sm_103a tensor cores for the sharded
// linear layers:  out[M, N] = act( sum over the k-range of A[M, K] . B[K, N] ).
//
//   A  row-major [M, K]   (X, or the hidden activation H)  -> K-major operand
//   B  row-major [K, N]   (the weight W as stored)          -> MN-major operand
//
// Every kernel runs on CTA pairs (clusters of 2, or of 4 for the split
// kernel) and issues tcgen05.mma.cta_group::2: one 256 x bn output tile per
// pair (bn = 256 or 128), 256 x bn x 16 per instruction.  The even CTA of a
// pair stages A rows 0..127 and B columns 0..bn/2-1 of the tile, the odd CTA
// rows 128..255 and columns bn/2..bn-1; the tensor cores of both SMs read B
// from both shared memories, so each SM stages half of B and only its own
// rows of A.  The fp32 accumulator rows 0..127 live in the even CTA's tensor
// memory (TMEM), rows 128..255 in the odd CTA's.
//
// Data path per CTA: TMA (128-byte swizzle) -> shared-memory ring of 128-deep
// K stages (3 of 64 KiB for 256-wide tiles, 4 of 48 KiB for 128-wide: deep
// stages, because issuing an MMA, a commit or a TMA copy costs a thread
// 60-100 cycles, and a 64-deep stage of 4 MMAs holds only 512 tensor
// cycles of work per SM); the TMA bytes of
// both CTAs are counted on the even CTA's `full` barrier; one thread of the
// even CTA issues the MMAs and releases a stage in both CTAs with a multicast
// commit; the epilogue warps of each CTA read its own TMEM (tcgen05.ld),
// add the optional bias, apply the optional GeLU, round to bf16 (RNE) or
// keep fp32, and write through swizzled shared-memory boxes and TMA stores.
//
// Warp roles (320 threads): warp 0 = TMA producer, warp 1 = TMEM owner (and
// MMA issuer in the even CTA), warps 2..9 = epilogue (warp w reads TMEM lanes
// 32*(w%4)..+31; warps 2..5 take the first half of the accumulator columns,
// warps 6..9 the second half).
//
// The tile width of a launch (256 or 128) is a run-time value no larger than
// the ring's template width.
//
// Kernels:
//   gemm_persistent_kernel<MAXBN>  one pair per two SMs walks work units
//       (tile, k-group); the accumulator is double-buffered in TMEM (2 x 256
//       columns) so the epilogue of one tile overlaps the main loop of the
//       next.  k-group g selects shard g's K range through the 3-D tensor
//       maps and its output goes to group g of the output (per-shard
//       partials); with one k-group the K loop walks shard 0's rows, then
//       shard 1's, ..., so the row-parallel partial sums are added inside the
//       accumulator.
//   gemm_cluster_sum_kernel  256-wide tiles for outputs with too few tiles to
//       fill the GPU: the two pairs of a cluster of 4 share one output tile,
//       pair p accumulating the p-th half of the K blocks (with K/n a
//       multiple of 256 and n even, half p is exactly shard group p).  Each
//       CTA sends the 64 accumulator rows its partner owns, in 4 KiB bulk
//       copies between shared memories, and adds the partner's chunks to
//       its own rows as they land; the sum never touches HBM.
#pragma once

#include "tp_device.cuh"

namespace tpk {

constexpr int BM = 128;              // accumulator rows held by one CTA
constexpr int PAIR_M = 2 * BM;       // rows of a pair tile
constexpr int MAX_BN = 256;          // widest tile (accumulator columns)
constexpr int BK = 128;              // K depth of one ring stage
constexpr int BK_BOX = 64;           // K depth of one A box: one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;
constexpr int A_BOX_BYTES = BM * BK_BOX * 2;        // 16 KiB
constexpr int A_STAGE_BYTES = (BK / BK_BOX) * A_BOX_BYTES;  // 32 KiB
constexpr int B_CHUNK_N = 64;                       // N columns per TMA box (128 bytes)
constexpr int B_CHUNK_BYTES = BK * B_CHUNK_N * 2;   // 16 KiB: 64 columns x 128 k-rows
constexpr int EPI_WARPS = 8;  // two per TMEM lane quadrant, each half of the columns
constexpr int GEMM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int STG_BYTES = 32 * 128;  // one epilogue warp's store box: 32 rows x 128 bytes
constexpr int ACC_STRIDE = MAX_BN;   // TMEM columns between the two accumulators
constexpr uint32_t TMEM_COLS_PERSISTENT = 2 * ACC_STRIDE;
#ifndef TP_RING_KB
#define TP_RING_KB 192
#endif
constexpr int RING_BUDGET = TP_RING_KB * 1024;  // shared memory for the operand ring
constexpr int MAX_STAGES = 8;

// Shared-memory ring for tiles up to MAXBN columns: ring | EPI_WARPS store
// boxes (1024-byte aligned, for the 128-byte swizzle) | barriers.
template <int MAXBN>
struct Ring {
    static constexpr int B_STAGE_BYTES = BK * (MAXBN / 2) * 2;
    static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
    static constexpr int STAGES = RING_BUDGET / STAGE_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int SMEM_BYTES = RING_BYTES + EPI_WARPS * STG_BYTES + 1024 + 512;
    static_assert(STAGES <= MAX_STAGES, "barrier array");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

// A descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart;
// a stage holds two such boxes (K 0..63 and 64..127), 16 KiB apart.
// B descriptor: MN-major, 128-byte swizzle; a 64-column chunk holds all BK
// k-rows (BK * 128 bytes), 8-k-row groups 1024 bytes apart.
constexpr uint32_t A_SBO = 1024;
constexpr uint32_t B_LBO = B_CHUNK_BYTES;
constexpr uint32_t B_SBO = 1024;

struct SmemBarriers {
    uint64_t full[MAX_STAGES];   // even CTA: TMA bytes of both CTAs of the pair
    uint64_t empty[MAX_STAGES];  // both CTAs: stage consumed (multicast commit)
    uint64_t acc_full[2];        // both CTAs: accumulator ready (multicast commit)
    uint64_t acc_empty[2];       // even CTA: epilogue warps of both CTAs done
    uint64_t drain;
    uint64_t ready;              // split kernel: the partner's ring is free
    uint64_t xfer[16];           // split kernel: one partial-row chunk landed
    uint32_t tmem_base;
    uint32_t abort;
};
static_assert(sizeof(SmemBarriers) <= 512, "barrier block");

// Epilogue modes of the TMA-store path (bf16 outputs):
//   EPI_PLAIN      out = act(acc)                      -> tmC
//   EPI_DUAL       out = acc -> tmC, and GeLU(acc)      -> tmAux
//   EPI_GELU_GRAD  out = acc * GeLU'(z), z (bf16 [M, N]) read from global memory
enum EpiMode : int { EPI_PLAIN = 0, EPI_DUAL = 1, EPI_GELU_GRAD = 2 };

// Bytes both CTAs of a pair land per k-block of a bn-wide tile.
__host__ __device__ constexpr uint32_t pair_stage_tx(int bn) {
    return 2u * static_cast<uint32_t>(A_STAGE_BYTES + BK * (bn / 2) * 2);
}

struct GemmArgs {
    int M, N;
    int bn;              // tile width: 256 or 128
    int k_blocks;        // BK-deep blocks per k-group (ceil)
    int k_groups;        // 1, or the shard count for per-shard partial outputs
    int m_tiles, n_tiles;  // pair tiles (PAIR_M x bn)
    int group_m;         // persistent order: tiles walk groups of group_m tile rows,
                         // row fastest within a group (L2 reuse, see decode_unit)
    int num_units;       // work units of the persistent kernel
    int full_units;      // units 0 .. full_units-1 are whole bn-wide tiles; each later
                         // unit is one half (bn/2 columns) of the remaining tiles, so
                         // that a last, partly filled round of tiles runs as half-width
                         // tiles on up to twice as many pairs
    int split;           // pairs per cluster S (cluster kernel)
    void *out;           // [M, N] row-major
    int64_t out_group_stride;  // elements between k-group outputs
    int out_f32;         // 1: fp32 output, 0: bf16
    int act_gelu;
    int tma_store;       // 1: the plain output goes through shared memory and TMA
                         //    stores (tensor map tmC); 0: per-thread vector stores
    int epi;             // EPI_PLAIN, EPI_DUAL or EPI_GELU_GRAD (TMA-store path, bf16)
    const __nv_bfloat16 *bias;  // optional [N]: added to the accumulator before the
                                // activation (after the whole K range: once per output)
    const __nv_bfloat16 *aux;   // EPI_GELU_GRAD: z, bf16 [M, N]
    void *out_shards;    // optional shard-major copy (column split)
    int shard_sw;        // columns a shard owns in each column group
    int shard_gw;        // columns per column group
    int shard_nl;        // local columns per shard
    uint64_t wait_limit_ns;
};

// ---------------------------------------------------------------------------
// Direct stores: activation, rounding and store of 8 consecutive columns of
// one output row (row < M, col < N, col a multiple of 8).  Writes the plain
// output (k-group g) and, if requested, the shard-major copy.
// ---------------------------------------------------------------------------
// Adds bias[col .. col+7] (bf16; col a multiple of 8, col < N) to f.
__device__ __forceinline__ void add_bias8(const __nv_bfloat16 *bias, int col, float *f) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(bias + col));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        f[2 * h] += __uint_as_float(w[h] << 16);
        f[2 * h + 1] += __uint_as_float(w[h] & 0xffff0000u);
    }
}

__device__ __forceinline__ void store_vec8(const GemmArgs &a, int g, int row, int col,
                                           float (&f)[8]) {
    if (a.bias) add_bias8(a.bias, col, f);
    if (a.act_gelu) {
#pragma unroll
        for (int i = 0; i < 8; i += 2) gelu2_f32(f[i], f[i + 1]);
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

// Hands the accumulator back to the MMA issuer once this warp's tensor
// memory reads are complete.
__device__ __forceinline__ void release_accumulator(uint32_t acc_empty_addr) {
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive_cluster(acc_empty_addr);
}

// Direct epilogue (per-thread 16-byte stores, one row per lane): used when a
// shard-major copy is requested.  `ncols` accumulator columns starting at
// column `cofs` of the accumulator at taddr, output columns col_base + cofs...
__device__ __forceinline__ void epilogue_direct(const GemmArgs &a, uint32_t taddr, int row,
                                                int col_base, int cofs, int ncols, int g,
                                                uint32_t acc_empty_addr) {
#pragma unroll 1
    for (int c = 0; c < ncols; c += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + cofs + c, r);
        tmem_ld_wait();
        store_row_chunk32(a, g, row, col_base + cofs + c, r);
    }
    release_accumulator(acc_empty_addr);
}

// Stages one 32-row x 128-byte box (8 16-byte chunks per row, held by lane =
// row) in this warp's store buffer with the 128-byte swizzle (chunk c of row
// r at position c ^ (r mod 8): conflict-free, 4 wavefronts per chunk column)
// and sends it to global memory with one TMA store.
__device__ __forceinline__ void stage_and_store_box(const CUtensorMap *tmC, uint32_t stg,
                                                    const uint32_t (&pk)[32], int col, int row,
                                                    int g) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) bulk_wait_read0();  // the previous box has left the buffer
    __syncwarp();
    const uint32_t row_addr = stg + lane * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        st_shared_v4(row_addr + ((c ^ (lane & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                     pk[4 * c + 3]);
    fence_proxy_async_smem();  // generic-proxy writes -> visible to the TMA engine
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(tmC, stg, col, row, g);
        bulk_commit_group();
    }
}

// TMA-store epilogue: the warp's 32 rows (starting at `row0`) and `ncols`
// accumulator columns (starting at `cofs` within the tile at `col_base`).
// bf16 output: 64-column boxes; fp32 output: 32-column boxes.  The
// accumulator is released as soon as its last tensor-memory load is done.
// Rows >= M and columns >= N of a box are clipped by the TMA unit.
// With a bias (bf16 [N]), bias[col] is added to every row's accumulator
// before the activation; every lane reads the same bias vectors (broadcast
// loads), columns >= N are skipped (the TMA store clips them anyway).
__device__ __forceinline__ void bias_chunk32(const __nv_bfloat16 *bias, int N, int col0,
                                             uint32_t (&r)[32]) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        if (col0 + 8 * v < N) {
            float f[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(r[8 * v + i]);
            add_bias8(bias, col0 + 8 * v, f);
#pragma unroll
            for (int i = 0; i < 8; ++i) r[8 * v + i] = __float_as_uint(f[i]);
        }
    }
}

__device__ __forceinline__ void epilogue_tma_store(const CUtensorMap *tmC, bool out_f32, bool gelu,
                                                   uint32_t taddr, uint32_t stg, int row0,
                                                   int col_base, int cofs, int ncols, int g,
                                                   uint32_t acc_empty_addr,
                                                   const __nv_bfloat16 *bias = nullptr,
                                                   int N = 0) {
    if (!out_f32) {
#pragma unroll 1
        for (int c = 0; c < ncols; c += 64) {
            uint32_t r0[32], r1[32];
            tmem_ld_32x32b_x32(taddr + cofs + c, r0);
            tmem_ld_32x32b_x32(taddr + cofs + c + 32, r1);
            tmem_ld_wait();
            if (c + 64 >= ncols) release_accumulator(acc_empty_addr);
            if (bias) {
                bias_chunk32(bias, N, col_base + cofs + c, r0);
                bias_chunk32(bias, N, col_base + cofs + c + 32, r1);
            }
            if (gelu) {
                gelu_chunk32(r0);
                gelu_chunk32(r1);
            }
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                pk[i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
                pk[16 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
            }
            stage_and_store_box(tmC, stg, pk, col_base + cofs + c, row0, g);
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < ncols; c += 32) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + cofs + c, r);
            tmem_ld_wait();
            if (c + 32 >= ncols) release_accumulator(acc_empty_addr);
            if (bias) bias_chunk32(bias, N, col_base + cofs + c, r);
            if (gelu) gelu_chunk32(r);
            stage_and_store_box(tmC, stg, r, col_base + cofs + c, row0, g);
        }
    }
}

// Dual epilogue (bf16): the raw accumulator to tmC and its GeLU to tmAux,
// 64 columns at a time.
__device__ __forceinline__ void epilogue_dual(const CUtensorMap *tmC, const CUtensorMap *tmAux,
                                              uint32_t taddr, uint32_t stg, int row0, int col_base,
                                              int cofs, int ncols, uint32_t acc_empty_addr) {
#pragma unroll 1
    for (int c = 0; c < ncols; c += 64) {
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(taddr + cofs + c, r0);
        tmem_ld_32x32b_x32(taddr + cofs + c + 32, r1);
        tmem_ld_wait();
        if (c + 64 >= ncols) release_accumulator(acc_empty_addr);
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            pk[i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
            pk[16 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
        }
        stage_and_store_box(tmC, stg, pk, col_base + cofs + c, row0, 0);
        gelu_chunk32(r0);
        gelu_chunk32(r1);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            pk[i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
            pk[16 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
        }
        stage_and_store_box(tmAux, stg, pk, col_base + cofs + c, row0, 0);
    }
}

// GeLU-gradient epilogue (bf16): out = acc * GeLU'(z), z (bf16 [M, N]) read
// from global memory by each lane for its own row (8 read-only 16-byte
// loads per 64-column box, issued before the tensor-memory loads so that
// their latency overlaps them; rows >= M and columns >= N read as 0).
__device__ __forceinline__ void epilogue_gelu_grad(const CUtensorMap *tmC,
                                                   const __nv_bfloat16 *z, int M, int N,
                                                   uint32_t taddr, uint32_t stg, int row0,
                                                   int col_base, int cofs, int ncols,
                                                   uint32_t acc_empty_addr) {
    const int lane = threadIdx.x & 31;
    const int row = row0 + lane;
#pragma unroll 1
    for (int c = 0; c < ncols; c += 64) {
        const int col = col_base + cofs + c;
        uint4 zv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            zv[q] = make_uint4(0u, 0u, 0u, 0u);
            if (row < M && col + 8 * q < N)
                zv[q] = __ldg(reinterpret_cast<const uint4 *>(z + static_cast<int64_t>(row) * N +
                                                              col + 8 * q));
        }
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(taddr + cofs + c, r0);
        tmem_ld_32x32b_x32(taddr + cofs + c + 32, r1);
        tmem_ld_wait();
        if (c + 64 >= ncols) release_accumulator(acc_empty_addr);
        uint32_t pk[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {  // columns 8q .. 8q+7 of the box
            const uint32_t zw[4] = {zv[q].x, zv[q].y, zv[q].z, zv[q].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int i = 8 * q + 2 * h;
                const float z0 = __uint_as_float(zw[h] << 16);
                const float z1 = __uint_as_float(zw[h] & 0xffff0000u);
                const float a0 = __uint_as_float(i < 32 ? r0[i] : r1[i - 32]);
                const float a1 = __uint_as_float(i + 1 < 32 ? r0[i + 1] : r1[i - 31]);
                pk[i / 2] = pack_bf16x2(a0 * gelu_grad_f32(z0), a1 * gelu_grad_f32(z1));
            }
        }
        stage_and_store_box(tmC, stg, pk, col, row0, 0);
    }
}

// Unit u of the persistent kernel -> k-group g, pair-tile row m_tile, first
// output column col0 and width bn of its tile.  Tiles are numbered group by
// group: a group is group_m consecutive tile rows (fewer in the last one)
// and walks its tile columns one after the other, the rows of a column
// fastest; then the next group, then the next k-group.  The pairs run
// consecutive units at the same time, so a round of P units touches about
// group_m rows of A and P / group_m columns of B: with group_m ~ sqrt(P)
// that is the fewest operand bytes a round can touch, and the round's
// successor shares the group's rows of A (L2 reuse).  Units below
// full_units are whole tiles, the rest are the two column halves of the
// last tiles.  Neither the order nor halving changes any element's
// accumulation order, so results do not depend on them.
__device__ __forceinline__ void decode_unit(const GemmArgs &a, int u, int &m_tile, int &col0,
                                            int &g, int &bn) {
    int t = u, half = 0;
    bn = a.bn;
    if (u >= a.full_units) {
        const int v = u - a.full_units;
        t = a.full_units + (v >> 1);
        half = v & 1;
        bn = a.bn >> 1;
    }
    const int tiles = a.m_tiles * a.n_tiles;
    g = t / tiles;
    const int r = t - g * tiles;
    const int per_group = a.group_m * a.n_tiles;
    const int grp = r / per_group;
    const int in = r - grp * per_group;
    const int rows = min(a.group_m, a.m_tiles - grp * a.group_m);
    m_tile = grp * a.group_m + in % rows;
    col0 = (in / rows) * a.bn + half * bn;
}

// ---------------------------------------------------------------------------
// Producer (one thread in each CTA of the pair): TMA loads of this CTA's
// half of k-blocks [kb0, kb1) of one pair tile into its ring, counted on the
// even CTA's full barrier (`full_remote` = its shared::cluster address for
// stage 0; stages are 8 bytes apart).  The even CTA also announces the pair's
// transaction bytes.  Returns false on abort.
// ---------------------------------------------------------------------------
struct ProducerState {
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0;  // 1 once any load was issued
};

// A_MN: A is stored [K][M] (M contiguous; e.g. X^T of a weight gradient),
// loaded as two 64-row x 128-k boxes.  B_KM: B is stored [N][K] (K
// contiguous; e.g. W^T of an input gradient), loaded as two 64-k x bn/2-row
// boxes.  Otherwise A is [M][K] and B is [K][N].
template <int MAXBN, bool A_MN = false, bool B_KM = false>
__device__ __forceinline__ bool produce_kblocks(const CUtensorMap *tmA, const CUtensorMap *tmB,
                                                uint8_t *ring, SmemBarriers *bars,
                                                uint32_t full_remote, bool leader, int half,
                                                ProducerState &ps, int m_tile, int tile_col0,
                                                int bn, int g, int kb0, int kb1, uint64_t limit) {
    using R = Ring<MAXBN>;
    const int row0 = m_tile * PAIR_M + half * BM;
    const int col0 = tile_col0 + half * (bn / 2);
    const int chunks = bn / 2 / B_CHUNK_N;
    const uint32_t tx = pair_stage_tx(bn);
    for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&bars->empty[ps.stage]), ps.phase ^ 1u, limit,
                               &bars->abort, SITE_PRODUCER_EMPTY))
            return false;
        if (leader) mbar_arrive_expect_tx(smem_u32(&bars->full[ps.stage]), tx);
        const uint32_t fb = full_remote + ps.stage * 8;
        uint8_t *sa = ring + ps.stage * R::STAGE_BYTES;
        uint8_t *sb = sa + A_STAGE_BYTES;
#pragma unroll
        for (int j = 0; j < BK / BK_BOX; ++j) {
            if (A_MN)
                tma_load_3d_pair(smem_u32(sa + j * A_BOX_BYTES), tmA, fb, row0 + j * 64, kb * BK,
                                 0);
            else
                tma_load_3d_pair(smem_u32(sa + j * A_BOX_BYTES), tmA, fb, kb * BK + j * BK_BOX, g,
                                 row0);
        }
        if (B_KM) {
#pragma unroll
            for (int j = 0; j < BK / BK_BOX; ++j)
                tma_load_3d_pair(smem_u32(sb + j * (bn / 2) * BK_BOX * 2), tmB, fb,
                                 kb * BK + j * BK_BOX, col0, 0);
        } else {
            for (int j = 0; j < chunks; ++j)
                tma_load_3d_pair(smem_u32(sb + j * B_CHUNK_BYTES), tmB, fb, col0 + j * B_CHUNK_N,
                                 kb * BK, g);
        }
        ps.issued = 1;
        if (++ps.stage == R::STAGES) {
            ps.stage = 0;
            ps.phase ^= 1u;
        }
    }
    return true;
}

// After the last load: wait until every stage of this CTA's ring has been
// released by the MMA issuer.  The releases are multicast commits from the
// even CTA; none may still be on its way when the CTA exits.
template <int MAXBN>
__device__ __forceinline__ bool producer_tail(SmemBarriers *bars, ProducerState &ps,
                                              uint64_t limit) {
    for (int i = 0; i < Ring<MAXBN>::STAGES; ++i) {
        if (!mbar_wait_bounded(smem_u32(&bars->empty[ps.stage]), ps.phase ^ 1u, limit,
                               &bars->abort, SITE_PRODUCER_EMPTY))
            return false;
        if (++ps.stage == Ring<MAXBN>::STAGES) {
            ps.stage = 0;
            ps.phase ^= 1u;
        }
    }
    return true;
}

// After an abort the loads this CTA issued are counted on the even CTA's
// barrier, which this CTA cannot wait on; give them a fixed time to land
// (far above any load latency) before the CTA may leave.
__device__ __forceinline__ void producer_drain(const ProducerState &ps) {
    if (!ps.issued) return;
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) {
    }
}

// MMA issuer (even CTA): accumulate k-blocks [kb0, kb1) of a bn-wide tile
// into TMEM columns at d_tmem of both CTAs; each consumed stage is released
// in both CTAs.  The shared-memory descriptors are formed once: the start
// address field (bits 0-13, address >> 4) of a stage's descriptor is the
// ring's plus stage * STAGE_BYTES / 16; a 16-deep K step adds 32 bytes (2)
// inside A's swizzle row (the second A box starts 16 KiB, 1024, further) or
// two 8-row groups (2048 bytes, 128) of B.  Shared addresses stay below
// 2^18, so no add carries out of the field.
// The operands arrive through the async proxy (TMA) and are read through it
// (tcgen05.mma), so the full-barrier wait alone orders them; no tcgen05
// fence is needed per k-block.
// With A_MN the A stage is two 64-row chunks (LBO 16 KiB) of 128 k-rows and
// a K step adds two 8-row groups (128); with B_KM the B stage is two 64-k
// boxes of bn/2 rows, like A's K-major layout.
template <int MAXBN, bool A_MN = false, bool B_KM = false>
__device__ __forceinline__ bool mma_kblocks(uint8_t *ring, SmemBarriers *bars, int &stage,
                                            uint32_t &phase, uint32_t d_tmem, uint32_t idesc,
                                            uint16_t pair_mask, int kb0, int kb1, int bn,
                                            uint64_t limit) {
    using R = Ring<MAXBN>;
    const uint64_t a_ring = A_MN ? smem_desc_sw128(smem_u32(ring), A_BOX_BYTES, A_SBO)
                                 : smem_desc_sw128(smem_u32(ring), 16, A_SBO);
    const uint64_t b_ring = B_KM ? smem_desc_sw128(smem_u32(ring) + A_STAGE_BYTES, 16, B_SBO)
                                 : smem_desc_sw128(smem_u32(ring) + A_STAGE_BYTES, B_LBO, B_SBO);
    const uint64_t b_box = static_cast<uint64_t>(((bn / 2) * BK_BOX * 2) >> 4);
    for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&bars->full[stage]), phase, limit, &bars->abort,
                               SITE_MMA_FULL))
            return false;
        const uint64_t so = static_cast<uint64_t>(stage * (R::STAGE_BYTES >> 4));
        const uint64_t da = a_ring + so, db = b_ring + so;
        constexpr int KPB = BK_BOX / UMMA_K;  // K steps per 64-deep box
        umma_f16_pair(d_tmem, da, db, idesc, kb > kb0 ? 1u : 0u);
#pragma unroll
        for (int k = 1; k < BK / UMMA_K; ++k) {
            const uint64_t ak = A_MN ? da + 128 * k
                                     : da + (A_BOX_BYTES >> 4) * (k / KPB) + 2 * (k % KPB);
            const uint64_t bk = B_KM ? db + b_box * (k / KPB) + 2 * (k % KPB) : db + 128 * k;
            umma_f16_pair(d_tmem, ak, bk, idesc, 1u);
        }
        umma_commit_pair_mc(smem_u32(&bars->empty[stage]), pair_mask);
        if (++stage == R::STAGES) {
            stage = 0;
            phase ^= 1u;
        }
    }
    return true;
}

__device__ __forceinline__ void mma_drain(SmemBarriers *bars, uint64_t limit) {
    umma_commit_pair(smem_u32(&bars->drain));
    mbar_wait_drain(smem_u32(&bars->drain), 0, limit);
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Barrier init and TMEM allocation in both CTAs of every pair, then a
// cluster barrier: no CTA sends bytes or arrivals to a peer barrier before
// the peer has initialised it.  Then the programmatic-launch hand-off: the
// next kernel of the stream may start launching, and this one waits for the
// previous kernel to complete.
__device__ __forceinline__ void gemm_setup(SmemBarriers *bars, int stages, uint32_t tmem_cols,
                                           const CUtensorMap *const *maps, int nmaps,
                                           bool split_barriers = false) {
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_u32(&bars->full[s]), 1);
            mbar_init(smem_u32(&bars->empty[s]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bars->acc_full[i]), 1);
            mbar_init(smem_u32(&bars->acc_empty[i]), 2 * EPI_WARPS);
        }
        mbar_init(smem_u32(&bars->drain), 1);
        if (split_barriers) {
            mbar_init(smem_u32(&bars->ready), 1);
            for (int i = 0; i < 16; ++i) mbar_init(smem_u32(&bars->xfer[i]), 1);
        }
        bars->abort = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && (threadIdx.x & 31) == 0) {
        for (int i = 0; i < nmaps; ++i) tma_prefetch_desc(maps[i]);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&bars->tmem_base), tmem_cols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    // Everything above is private to this CTA pair, so it overlaps the tail
    // of the previous kernel; the inputs (possibly that kernel's output) and
    // the outputs are touched only after it has completed.
    if (threadIdx.x == 0) grid_dep_trigger();
    grid_dep_wait();
}

__device__ __forceinline__ void gemm_teardown(uint32_t tmem_base, uint32_t tmem_cols) {
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no peer still reads this CTA's ring or signals its barriers
    tc_fence_after();
    if ((threadIdx.x >> 5) == 1) tmem_dealloc_pair(tmem_base, tmem_cols);
}

// ---------------------------------------------------------------------------
// Persistent kernel: cluster = one pair, grid = 2 x (pairs launched).
// ---------------------------------------------------------------------------
template <int MAXBN, bool A_MN = false, bool B_KM = false, int EPI = EPI_PLAIN>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_persistent_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmC,
                           const __grid_constant__ CUtensorMap tmAux, const GemmArgs a) {
    using R = Ring<MAXBN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = align1024(smem_raw);
    uint8_t *staging = ring + R::RING_BYTES;
    SmemBarriers *bars = reinterpret_cast<SmemBarriers *>(staging + EPI_WARPS * STG_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int half = static_cast<int>(cluster_ctarank());  // 0 = even (leader), 1 = odd
    const bool leader = half == 0;
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;

    const CUtensorMap *maps[4] = {&tmA, &tmB, &tmC, &tmAux};
    gemm_setup(bars, R::STAGES, TMEM_COLS_PERSISTENT, maps,
               (EPI == EPI_DUAL || (B_KM && a.full_units < a.num_units)) ? 4
                                                                         : (a.tma_store ? 3 : 2));
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(&bars->tmem_base);
    const uint64_t limit = a.wait_limit_ns;

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t full_remote = dsmem_map(smem_u32(&bars->full[0]), 0);
            ProducerState ps;
            bool ok = true;
            for (int u = pair; u < a.num_units && ok; u += num_pairs) {
                int mt, c0, g, bn;
                decode_unit(a, u, mt, c0, g, bn);
                // [N][K] B: the half-width units read boxes of half as many
                // rows, through the second map (tmAux is otherwise unused there)
                const CUtensorMap *mb = (B_KM && bn != a.bn) ? &tmAux : &tmB;
                ok = produce_kblocks<MAXBN, A_MN, B_KM>(&tmA, mb, ring, bars, full_remote,
                                                        leader, half, ps, mt, c0, bn, g, 0,
                                                        a.k_blocks, limit);
            }
            if (ok) ok = producer_tail<MAXBN>(bars, ps, limit);
            if (!ok) producer_drain(ps);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (leader && lane == 0) {
            int stage = 0, local = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = pair; u < a.num_units && ok; u += num_pairs, ++local) {
                int mt, c0, g, bn;
                decode_unit(a, u, mt, c0, g, bn);
                const uint32_t idesc = idesc_bf16_f32(PAIR_M, bn, !B_KM, A_MN);
                const int acc = local & 1;
                const uint32_t acc_par = (local >> 1) & 1;
                ok = mbar_wait_bounded(smem_u32(&bars->acc_empty[acc]), acc_par ^ 1u, limit,
                                       &bars->abort, SITE_MMA_ACC_EMPTY);
                if (!ok) break;
                tc_fence_after();
                ok = mma_kblocks<MAXBN, A_MN, B_KM>(ring, bars, stage, phase,
                                                    tmem_base + acc * ACC_STRIDE, idesc, 0x3, 0,
                                                    a.k_blocks, bn, limit);
                if (!ok) break;
                umma_commit_pair_mc(smem_u32(&bars->acc_full[acc]), 0x3);
            }
            if (!ok) mma_drain(bars, limit);
        }
        __syncwarp();
    } else {
        const int q = warp & 3;                         // TMEM lane quadrant
        const int chalf = (warp - 2) >> 2;              // this warp's half of the columns
        const uint32_t acc_empty_remote = dsmem_map(smem_u32(&bars->acc_empty[0]), 0);
        const uint32_t stg = smem_u32(staging + (warp - 2) * STG_BYTES);
        int local = 0;
        for (int u = pair; u < a.num_units; u += num_pairs, ++local) {
            const int acc = local & 1;
            const uint32_t acc_par = (local >> 1) & 1;
            if (!mbar_wait_warp(smem_u32(&bars->acc_full[acc]), acc_par, limit, &bars->abort,
                                SITE_EPI_ACC_FULL))
                break;
            tc_fence_after();
            int mt, c0, g, bn;
            decode_unit(a, u, mt, c0, g, bn);
            const int cofs = chalf * (bn / 2);
            const uint32_t taddr =
                tmem_base + acc * ACC_STRIDE + (static_cast<uint32_t>(q * 32) << 16);
            const uint32_t release = acc_empty_remote + acc * 8;
            const int row0 = mt * PAIR_M + half * BM + q * 32;
            if constexpr (EPI == EPI_GELU_GRAD) {
                epilogue_gelu_grad(&tmC, a.aux, a.M, a.N, taddr, stg, row0, c0, cofs, bn / 2,
                                   release);
            } else if constexpr (EPI == EPI_DUAL) {
                epilogue_dual(&tmC, &tmAux, taddr, stg, row0, c0, cofs, bn / 2, release);
            } else if (a.tma_store) {
                epilogue_tma_store(&tmC, a.out_f32 != 0, a.act_gelu != 0, taddr, stg, row0,
                                   c0, cofs, bn / 2, g, release, a.bias, a.N);
            } else {
                epilogue_direct(a, taddr, row0 + lane, c0, cofs, bn / 2, g, release);
            }
        }
        if (lane == 0) bulk_wait_read0();  // every store box has left shared memory
        __syncwarp();
    }

    gemm_teardown(tmem_base, TMEM_COLS_PERSISTENT);
}

// ---------------------------------------------------------------------------
// Cluster split kernel (256-wide tiles, two pairs per tile): grid = 4 * tiles
// CTAs, cluster = 4 CTAs along x (cluster rank 2p + h is half h of pair p).
// Pair p accumulates K slice p.  The two CTAs that hold the same 128 rows
// (ranks h and 2 + h, partners) split them: pair p owns rows [64p, 64p + 64)
// of the half.  Each epilogue warp covers 32 rows (its tensor-memory lane
// quadrant) and 128 columns; a warp whose rows the partner owns is a sender,
// the partner's warp with the same rows and columns its receiver (one of
// four links).  The sender moves its 32 x 128 fp32 partial in four chunks of
// 32 columns: tensor memory -> its own shared memory (16-byte chunk v of row
// r at v ^ (r mod 8): conflict-free) -> one bulk copy into the receiver's
// shared memory, counted on the receiver's barrier for that chunk.  The
// receiver adds each chunk to its own partial as it lands (two fp32
// operands: the sum does not depend on their order) and stores the result,
// so the transfer overlaps the epilogue.  Chunks land in the receiver's
// operand ring, so a sender first waits until the partner's main loop is
// done (`ready`, arrived on by the partner).  The sum never touches HBM.
// ---------------------------------------------------------------------------
constexpr int XFER_COLS = 32;                            // columns per chunk
constexpr int XFER_BYTES = 32 * XFER_COLS * 4;           // 32 rows x 32 fp32
constexpr int XFER_CHUNKS = (MAX_BN / 2) / XFER_COLS;    // chunks per link
constexpr int XFER_LINKS = 4;                            // (row block, column half)
static_assert(XFER_LINKS * XFER_CHUNKS <= 16, "transfer barriers");
static_assert(2 * XFER_LINKS * XFER_CHUNKS * XFER_BYTES <= Ring<256>::RING_BYTES,
              "send and receive areas fit in the ring");

__device__ __forceinline__ uint32_t xfer_slot(uint32_t buf, int lane, int v) {
    return buf + lane * (XFER_COLS * 4) + ((v ^ (lane & 7)) << 4);
}

__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_cluster_sum_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmC, const GemmArgs a) {
    using R = Ring<256>;
    constexpr int BN = 256;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = align1024(smem_raw);
    uint8_t *staging = ring + R::RING_BYTES;
    SmemBarriers *bars = reinterpret_cast<SmemBarriers *>(staging + EPI_WARPS * STG_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr uint32_t TMEM_COLS = BN;

    const int rank = static_cast<int>(cluster_ctarank());
    const int p = rank >> 1;      // pair = K slice
    const int half = rank & 1;    // which 128 rows of the tile
    const bool leader = half == 0;
    const uint32_t partner = static_cast<uint32_t>(rank ^ 2);
    const int tile = blockIdx.x / 4;
    const int mt = tile % a.m_tiles;
    const int nt = tile / a.m_tiles;
    const int kb0 = p == 0 ? 0 : a.k_blocks / 2;
    const int kb1 = p == 0 ? a.k_blocks / 2 : a.k_blocks;

    const CUtensorMap *maps[3] = {&tmA, &tmB, &tmC};
    gemm_setup(bars, R::STAGES, TMEM_COLS, maps, a.tma_store ? 3 : 2, true);
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(&bars->tmem_base);
    const uint64_t limit = a.wait_limit_ns;
    const uint16_t pair_mask = static_cast<uint16_t>(0x3u << (2 * p));

    if (warp == 0) {
        if (lane == 0) {
            // every chunk this CTA receives: 4 KiB each
            for (int i = 0; i < XFER_LINKS * XFER_CHUNKS; ++i)
                mbar_arrive_expect_tx(smem_u32(&bars->xfer[i]), XFER_BYTES);
            const uint32_t full_remote =
                dsmem_map(smem_u32(&bars->full[0]), static_cast<uint32_t>(2 * p));
            ProducerState ps;
            if (!produce_kblocks<256>(&tmA, &tmB, ring, bars, full_remote, leader, half, ps, mt,
                                      nt * BN, BN, 0, kb0, kb1, limit) ||
                !producer_tail<256>(bars, ps, limit))
                producer_drain(ps);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            if (mma_kblocks<256>(ring, bars, stage, phase, tmem_base,
                                 idesc_bf16_f32(PAIR_M, BN, true), pair_mask, kb0, kb1, BN,
                                 limit))
                umma_commit_pair_mc(smem_u32(&bars->acc_full[0]), pair_mask);
            else
                mma_drain(bars, limit);
        }
        __syncwarp();
    } else {
        // The transfer runs whether or not a wait gave up before (then the
        // rows are meaningless), so that every chunk lands before the CTAs
        // exit.
        const bool acc_ok = mbar_wait_warp(smem_u32(&bars->acc_full[0]), 0, limit, &bars->abort,
                                           SITE_EPI_ACC_FULL);
        if (acc_ok) tc_fence_after();
        // This CTA's main loop is done, its ring free: the partner may send.
        if (warp == 2 && lane == 0) mbar_arrive_cluster(dsmem_map(smem_u32(&bars->ready), partner));
        const int q = warp & 3;              // tensor-memory lane quadrant
        const int chalf = (warp - 2) >> 2;   // column half
        const int cofs = chalf * (BN / 2);
        const int link = (q & 1) + 2 * chalf;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + cofs;
        const uint32_t send = smem_u32(ring) + link * XFER_CHUNKS * XFER_BYTES;
        const uint32_t recv = send + XFER_LINKS * XFER_CHUNKS * XFER_BYTES;
        if ((q >> 1) != p) {
            // sender: the partner owns these rows
#pragma unroll 1
            for (int c = 0; c < XFER_CHUNKS; ++c) {
                const uint32_t buf = send + c * XFER_BYTES;
                if (acc_ok) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + c * XFER_COLS, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        st_shared_v4(xfer_slot(buf, lane, v), r[4 * v], r[4 * v + 1],
                                     r[4 * v + 2], r[4 * v + 3]);
                }
                fence_proxy_async_smem();  // generic-proxy writes -> the bulk copy
                __syncwarp();
                if (lane == 0) {
                    if (c == 0) mbar_wait_drain(smem_u32(&bars->ready), 0, limit);
                    bulk_copy_to_peer(
                        dsmem_map(recv + c * XFER_BYTES, partner), buf, XFER_BYTES,
                        dsmem_map(smem_u32(&bars->xfer[link * XFER_CHUNKS + c]), partner));
                }
            }
        } else if (acc_ok) {
            // receiver: own rows, 64 columns (two chunks) at a time
            const uint32_t stg = smem_u32(staging + (warp - 2) * STG_BYTES);
            const int row0 = mt * PAIR_M + half * BM + q * 32;
            const int col0 = nt * BN + cofs;
#pragma unroll 1
            for (int c = 0; c < XFER_CHUNKS; c += 2) {
                uint32_t r0[32], r1[32];
                tmem_ld_32x32b_x32(taddr + c * XFER_COLS, r0);
                tmem_ld_32x32b_x32(taddr + (c + 1) * XFER_COLS, r1);
                const bool ok0 = mbar_wait_warp(smem_u32(&bars->xfer[link * XFER_CHUNKS + c]), 0,
                                                limit, &bars->abort, SITE_EPI_SPLIT);
                const bool ok1 =
                    ok0 && mbar_wait_warp(smem_u32(&bars->xfer[link * XFER_CHUNKS + c + 1]), 0,
                                          limit, &bars->abort, SITE_EPI_SPLIT);
                tmem_ld_wait();
                if (!ok1) break;
                const uint32_t b0 = recv + c * XFER_BYTES, b1 = b0 + XFER_BYTES;
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const uint4 u0 = ld_shared_v4(xfer_slot(b0, lane, v));
                    const uint4 u1 = ld_shared_v4(xfer_slot(b1, lane, v));
                    const uint32_t w0[4] = {u0.x, u0.y, u0.z, u0.w};
                    const uint32_t w1[4] = {u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        r0[4 * v + i] = __float_as_uint(__uint_as_float(r0[4 * v + i]) +
                                                        __uint_as_float(w0[i]));
                        r1[4 * v + i] = __float_as_uint(__uint_as_float(r1[4 * v + i]) +
                                                        __uint_as_float(w1[i]));
                    }
                }
                const int col = col0 + c * XFER_COLS;
                if (!a.tma_store) {  // shard-major copy requested: direct stores
                    store_row_chunk32(a, 0, row0 + lane, col, r0);
                    store_row_chunk32(a, 0, row0 + lane, col + XFER_COLS, r1);
                    continue;
                }
                if (a.bias) {
                    bias_chunk32(a.bias, a.N, col, r0);
                    bias_chunk32(a.bias, a.N, col + XFER_COLS, r1);
                }
                if (a.act_gelu) {
                    gelu_chunk32(r0);
                    gelu_chunk32(r1);
                }
                if (a.out_f32) {  // boxes of 32 fp32 columns
                    stage_and_store_box(&tmC, stg, r0, col, row0, 0);
                    stage_and_store_box(&tmC, stg, r1, col + XFER_COLS, row0, 0);
                } else {  // boxes of 64 bf16 columns
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        pk[i] = pack_bf16x2(__uint_as_float(r0[2 * i]),
                                            __uint_as_float(r0[2 * i + 1]));
                        pk[16 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]),
                                                 __uint_as_float(r1[2 * i + 1]));
                    }
                    stage_and_store_box(&tmC, stg, pk, col, row0, 0);
                }
            }
            if (lane == 0) bulk_wait_read0();  // every store box has left shared memory
            __syncwarp();
        }
    }
    // Every chunk the partner sends has landed before this CTA may exit.
    if (threadIdx.x == 0) {
        for (int i = 0; i < XFER_LINKS * XFER_CHUNKS; ++i)
            mbar_wait_drain(smem_u32(&bars->xfer[i]), 0, limit);
    }
    gemm_teardown(tmem_base, TMEM_COLS);  // cluster barrier: no copy reads a CTA that left
}

}  // namespace tpk
