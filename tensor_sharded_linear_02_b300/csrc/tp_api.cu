// tp_api.cu -- host side of the C ABI declared in include/tp.h: argument
// validation, tensor-map encoding, kernel selection and launch.  This is the
// library's only translation unit; the kernels come in through the headers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/tp.h"
#include "gemm_tcgen05.cuh"
#include "shard_combine.cuh"
#include "simt_linear.cuh"

namespace {

using namespace tpk;

constexpr int kMaxDevices = 64;
constexpr int64_t kInt32Max = 0x7FFFFFFF;
// Largest element count of one matrix (2^40: 2 TiB of bf16, far above any
// device's memory).  With it every byte count below (elements x at most 4
// bytes x at most TP_MAX_SHARDS) stays far inside int64 / size_t.
constexpr int64_t kMaxElems = int64_t(1) << 40;

// a * b <= kMaxElems for non-negative a, b, without forming the product.
bool elems_ok(int64_t a, int64_t b) { return a == 0 || b <= kMaxElems / a; }

// ----------------------------------------------------------------- devices --

struct DeviceInfo {
    int sm_count = 0;
    int max_pairs = 0;          // clusters of 2 GEMM CTAs that fit at once
    int max_split_clusters = 0;  // clusters of 4 CTAs (two pairs) of the split kernel at once
    bool ready = false;
};

// How many clusters of `size` GEMM CTAs can be resident at once (0 if the
// size cannot be launched).
int active_clusters(const void *kernel, int size, int smem_bytes) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(size), 1, 1);
    cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(size);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];

tp_status device_info(DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TP_ERR_CUDA;
        if (cudaFuncSetAttribute(gemm_persistent_kernel<256>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Ring<256>::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(gemm_persistent_kernel<128>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Ring<128>::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(gemm_persistent_kernel<256, true, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Ring<256>::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(gemm_persistent_kernel<256, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Ring<256>::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(gemm_persistent_kernel<128, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Ring<128>::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(gemm_persistent_kernel<256, false, true, EPI_GELU_GRAD>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Ring<256>::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(gemm_persistent_kernel<256, false, false, EPI_DUAL>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Ring<256>::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(gemm_cluster_sum_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Ring<256>::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(shard_reduce_bulk_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 RED_SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(shard_reduce_bulk_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 RED_SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(shard_concat_tma_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 CAT_SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(segment_copy_tma_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 CAT_SMEM_BYTES) != cudaSuccess)
            return TP_ERR_CUDA;
        d.max_pairs = active_clusters(reinterpret_cast<const void *>(gemm_persistent_kernel<256>),
                                      2, Ring<256>::SMEM_BYTES);
        const int p128 = active_clusters(
            reinterpret_cast<const void *>(gemm_persistent_kernel<128>), 2, Ring<128>::SMEM_BYTES);
        if (p128 < d.max_pairs) d.max_pairs = p128;
        if (d.max_pairs < 1) return TP_ERR_CUDA;
        d.max_split_clusters = active_clusters(
            reinterpret_cast<const void *>(gemm_cluster_sum_kernel), 4, Ring<256>::SMEM_BYTES);
        d.ready = true;
    }
    *out = &d;
    return TP_OK;
}

uint64_t wait_limit_ns() {
    static uint64_t limit = [] {
        const char *e = std::getenv("TP_WAIT_LIMIT_MS");
        uint64_t ms = e ? std::strtoull(e, nullptr, 10) : 4000ull;
        if (ms < 1) ms = 1;
        return ms * 1000000ull;
    }();
    return limit;
}

// ------------------------------------------------------------ tensor maps --

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 3-D tensor map (bf16 unless f32), 128-byte swizzle, zero fill out of bounds.
bool encode_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1,
               uint32_t b2, bool f32 = false,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
              const_cast<void *>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A tensor map depends only on its arguments, so encoded maps are kept in a
// small least-recently-used cache: a call with the buffers and sizes of an
// earlier one (every step of a model) skips the driver's encoder.  A buffer
// freed and reallocated at the same address with the same sizes gets the
// same map, which is the correct one.
struct MapKey {
    const void *base;
    uint64_t dims[3], strides[2];
    uint32_t box[3];
    uint32_t f32, swizzle;
};

struct MapEntry {
    MapKey key;
    CUtensorMap map;
    uint64_t stamp;
};

constexpr int kMapCache = 32;
std::mutex g_map_mutex;
MapEntry g_maps[kMapCache];
uint64_t g_map_clock = 0;

bool encode_3d_cached(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1,
                      uint32_t b2, bool f32 = false,
                      CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    MapKey k;
    std::memset(&k, 0, sizeof(k));
    k.base = base;
    k.dims[0] = d0; k.dims[1] = d1; k.dims[2] = d2;
    k.strides[0] = stride1_bytes; k.strides[1] = stride2_bytes;
    k.box[0] = b0; k.box[1] = b1; k.box[2] = b2;
    k.f32 = f32 ? 1u : 0u;
    k.swizzle = static_cast<uint32_t>(swizzle);
    {
        std::lock_guard<std::mutex> lock(g_map_mutex);
        for (MapEntry &e : g_maps) {
            if (e.stamp != 0 && std::memcmp(&e.key, &k, sizeof(k)) == 0) {
                *m = e.map;
                e.stamp = ++g_map_clock;
                return true;
            }
        }
    }
    if (!encode_3d(m, base, d0, d1, d2, stride1_bytes, stride2_bytes, b0, b1, b2, f32, swizzle))
        return false;
    std::lock_guard<std::mutex> lock(g_map_mutex);
    MapEntry *victim = &g_maps[0];
    for (MapEntry &e : g_maps)
        if (e.stamp < victim->stamp) victim = &e;
    victim->key = k;
    victim->map = *m;
    victim->stamp = ++g_map_clock;
    return true;
}

// ------------------------------------------------------------- validation --

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A pointer is required unless the buffer it names holds no bytes.
bool present(const void *p, size_t bytes) { return p != nullptr || bytes == 0; }

size_t dtype_size(tp_dtype t) { return t == TP_BF16 ? 2 : 4; }

bool valid_dtype(tp_dtype t) { return t == TP_F32 || t == TP_BF16; }

bool overlaps(const void *a, size_t abytes, const void *b, size_t bbytes) {
    if (!a || !b || abytes == 0 || bbytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

tp_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

// -------------------------------------------------------------- launchers --

struct GemmCall {
    const void *A;  // [M, K] bf16 row-major, or [K, M] when a_mn
    const void *B;  // [K, N] bf16 row-major, or [N, K] when b_km
    int64_t M, N, K;
    int k_groups;   // 1: one accumulator over all of K; n: one output per shard
    void *out;
    int64_t out_group_stride;
    bool out_f32;
    bool gelu;
    void *out_shards;
    int n_shards, col_groups;
    bool allow_split;
    bool a_mn = false;         // A stored transposed (M contiguous)
    bool b_km = false;         // B stored transposed (K contiguous)
    int epi = EPI_PLAIN;       // EPI_DUAL / EPI_GELU_GRAD use aux (bf16 [M, N])
    void *aux = nullptr;
    const void *bias = nullptr;  // bf16 [N], added before the activation
};

// Tile rows per group of the persistent kernel's tile order (about the
// square root of the 74 pairs that run at once; see decode_unit), and the
// share of the 126 MB L2 that one operand may claim to stay resident.
// Measured (4096 x 4096 x 16384 products): the column GEMM (A = 32 MB) is
// fastest with all 16 tile rows in one group (A read once), the weight-
// gradient product with A = 128 MB (64 tile rows) 23 % faster with groups
// of 8 than with one group.
constexpr int kGroupM = 8;
constexpr int64_t kL2Budget = int64_t(48) << 20;

// Launch plan of one GEMM: tile width, and split = 2 for the cluster split
// kernel (two pairs per tile), 1 for the persistent kernel.
struct GemmPlan {
    int bn = 256;
    int split = 1;
};

// Optional override of the automatic plan, for measurements:
// TP_GEMM_PLAN = "256" | "128" | "split2".
// Read at every launch, so that a process can compare plans.
int plan_override() {
    const char *e = std::getenv("TP_GEMM_PLAN");
    if (!e) return 0;
    if (!std::strcmp(e, "256")) return 1;
    if (!std::strcmp(e, "128")) return 2;
    if (!std::strcmp(e, "split2")) return 3;
    return 0;
}

// Picks the plan with the smallest estimated time, in units of one k-block
// of a 256-wide pair tile (128 deep, about 1024 tensor-core cycles):
//   persistent, width bn: waves * k_blocks * (bn / 256) * overhead(bn) plus
//       the exposed epilogue of the last tile (larger with GeLU); for the
//       256-wide plan a last round that fills at most half of the pairs
//       runs as 128-wide half tiles (`half_tail`) and counts 0.75;
//   split over two pairs (256-wide, one wave of clusters): k_blocks / 2
//       plus the exchange of the partial rows between the two pairs (64 KiB
//       of fp32 per CTA through distributed shared memory) and the tail.
// A 128-wide k-block carries half the tensor work of a 256-wide one but the
// same issue work (MMA and TMA instructions per stage) and 3/4 of its
// operand bytes; measured, it takes about 0.75 of the 256-wide time.
GemmPlan plan_gemm(int64_t M, int64_t N, int k_blocks, int k_groups, bool allow_split, bool gelu,
                   bool half_tail, const DeviceInfo &dev) {
    const int64_t m_tiles = (M + PAIR_M - 1) / PAIR_M;
    const int64_t u256 = m_tiles * ((N + 255) / 256) * k_groups;
    const int64_t u128 = m_tiles * ((N + 127) / 128) * k_groups;
    const int64_t P = dev.max_pairs;
    const double tail = gelu ? 6.0 : 2.0;
    const int64_t rem256 = u256 % P;
    const double rounds256 = static_cast<double>(u256 / P) +
                             (rem256 == 0 ? 0.0
                                          : (half_tail && u256 > P && 2 * rem256 <= P ? 0.75 : 1.0));
    const double c256 = rounds256 * k_blocks + tail;
    const double c128 = static_cast<double>((u128 + P - 1) / P) * k_blocks * 0.5 * 1.5 + tail / 2;
    GemmPlan best;
    double cbest = c256;
    if (c128 < cbest) {
        best.bn = 128;
        cbest = c128;
    }
    const bool can_split = allow_split && k_groups == 1;
    const bool split_fits = can_split && u256 <= dev.max_split_clusters && k_blocks >= 2;
    if (split_fits) {
        const double cs = static_cast<double>((k_blocks + 1) / 2) + 4.0 + tail;
        if (cs < cbest) {
            best.bn = 256;
            best.split = 2;
            cbest = cs;
        }
    }
    switch (plan_override()) {
        case 1: return GemmPlan{256, 1};
        case 2: return GemmPlan{128, 1};
        case 3: if (split_fits) return GemmPlan{256, 2}; break;
        default: break;
    }
    return best;
}

tp_status launch_gemm(const GemmCall &c, cudaStream_t s) {
    DeviceInfo *dev = nullptr;
    tp_status st = device_info(&dev);
    if (st != TP_OK) return st;

    const int64_t Kg = c.K / c.k_groups;
    // plans: the K-major-B product (input gradients) may also be 128 wide;
    // transposed A and the dual / GeLU' epilogues use 256-wide tiles
    const bool plain = !c.a_mn && c.epi == EPI_PLAIN;
    const GemmPlan plan = plain ? plan_gemm(c.M, c.N, static_cast<int>((Kg + BK - 1) / BK),
                                            c.k_groups, c.allow_split && !c.b_km, c.gelu,
                                            true, *dev)
                                : GemmPlan{256, 1};
    CUtensorMap tmA, tmB, tmAux;
    if (c.a_mn) {
        // A^T stored [K][M]: viewed as [1][K][M]; box = 128 k-rows x 64 columns.
        if (!encode_3d_cached(&tmA, c.A, c.M, c.K, 1, c.M * 2, c.K * c.M * 2, 64, BK, 1))
            return TP_ERR_CUDA;
    } else {
        // A viewed as [M][k_groups][Kg]; box = 128 rows x 64 k of one group.
        if (!encode_3d_cached(&tmA, c.A, Kg, c.k_groups, c.M, Kg * 2, c.K * 2, BK_BOX, 1, BM))
            return TP_ERR_CUDA;
    }
    if (c.b_km) {
        // B^T stored [N][K]: viewed as [1][N][K]; box = bn/2 rows x 64 k.
        if (!encode_3d_cached(&tmB, c.B, c.K, c.N, 1, c.K * 2, c.N * c.K * 2, BK_BOX,
                              static_cast<uint32_t>(plan.bn / 2), 1))
            return TP_ERR_CUDA;
    } else {
        // B viewed as [k_groups][Kg][N]; box = 128 k-rows x 64 columns of one group.
        if (!encode_3d_cached(&tmB, c.B, c.N, Kg, c.k_groups, c.N * 2, Kg * c.N * 2, B_CHUNK_N,
                              BK, 1))
            return TP_ERR_CUDA;
    }
    std::memset(&tmAux, 0, sizeof(tmAux));
    if (c.epi == EPI_DUAL) {
        // second bf16 output [M, N], same boxes as the first
        if (!encode_3d_cached(&tmAux, c.aux, c.N, c.M, 1, c.N * 2, c.M * c.N * 2, 64, 32, 1))
            return TP_ERR_CUDA;
    }

    // Output viewed as [k_groups][M][N]; box = 32 rows x 128 bytes of one group.
    CUtensorMap tmC;
    const bool tma_store = c.out != nullptr && c.out_shards == nullptr;
    std::memset(&tmC, 0, sizeof(tmC));
    if (tma_store) {
        const uint64_t es = c.out_f32 ? 4 : 2;
        if (!encode_3d_cached(&tmC, c.out, c.N, c.M, c.k_groups, c.N * es,
                       (c.k_groups > 1 ? c.out_group_stride : c.M * c.N) * es,
                       static_cast<uint32_t>(128 / es), 32, 1, c.out_f32))
            return TP_ERR_CUDA;
    }

    GemmArgs a{};
    a.tma_store = tma_store ? 1 : 0;
    a.epi = c.epi;
    a.bias = static_cast<const __nv_bfloat16 *>(c.bias);
    a.aux = static_cast<const __nv_bfloat16 *>(c.aux);
    a.M = static_cast<int>(c.M);
    a.N = static_cast<int>(c.N);
    a.k_blocks = static_cast<int>((Kg + BK - 1) / BK);
    a.k_groups = c.k_groups;
    a.bn = plan.bn;
    a.m_tiles = static_cast<int>((c.M + PAIR_M - 1) / PAIR_M);
    a.n_tiles = static_cast<int>((c.N + a.bn - 1) / a.bn);
    const int64_t units = static_cast<int64_t>(a.m_tiles) * a.n_tiles * c.k_groups;
    if (units > kInt32Max / 2) return TP_ERR_SHAPE;
    a.num_units = static_cast<int>(units);
    a.full_units = a.num_units;
    // tile order: when all of A (the k-group's rows x K) fits the L2 budget
    // it stays resident while B streams past once, so the rows of a group
    // are all of them; otherwise groups of kGroupM rows keep each round's
    // operand footprint near its minimum
    const int64_t a_bytes = static_cast<int64_t>(a.m_tiles) * PAIR_M * Kg * 2;
    a.group_m = (a_bytes <= kL2Budget || a.m_tiles < kGroupM) ? a.m_tiles : kGroupM;
    // A last round of 256-wide tiles that fills at most half of the pairs
    // runs as twice as many 128-wide half tiles (each about 3/4 of a tile's
    // time).  The [N][K] (transposed) B operand's tensor-map box is as tall
    // as half a tile, so the half tiles read it through a second map, in the
    // kernel's auxiliary map slot (unused by those kernels otherwise).
    if (plan.split == 1 && a.bn == 256 && !(c.b_km && c.epi == EPI_DUAL) &&
        a.num_units > dev->max_pairs) {
        const int rem = a.num_units % dev->max_pairs;
        if (rem > 0 && 2 * rem <= dev->max_pairs) {
            a.full_units = a.num_units - rem;
            a.num_units += rem;
            if (c.b_km && !encode_3d_cached(&tmAux, c.B, c.K, c.N, 1, c.K * 2, c.N * c.K * 2,
                                            BK_BOX, static_cast<uint32_t>(a.bn / 4), 1))
                return TP_ERR_CUDA;
        }
    }
    a.out = c.out;
    a.out_group_stride = c.out_group_stride;
    a.out_f32 = c.out_f32 ? 1 : 0;
    a.act_gelu = c.gelu ? 1 : 0;
    a.out_shards = c.out_shards;
    if (c.out_shards) {
        a.shard_gw = static_cast<int>(c.N / c.col_groups);
        a.shard_sw = a.shard_gw / c.n_shards;
        a.shard_nl = a.shard_sw * c.col_groups;
    }
    a.wait_limit_ns = wait_limit_ns();

    const int tiles = a.m_tiles * a.n_tiles;
    const int S = plan.split;
    a.split = S;
    const int pairs = S > 1 ? tiles * S : (a.num_units < dev->max_pairs ? a.num_units
                                                                         : dev->max_pairs);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(a.bn == 128 ? Ring<128>::SMEM_BYTES
                                                           : Ring<256>::SMEM_BYTES);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(2 * S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // Programmatic dependent launch: the kernel's set-up (barriers, tensor
    // memory, descriptor prefetch) overlaps the previous kernel's tail; it
    // waits on the device (griddepcontrol.wait) before touching memory.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e;
    if (S > 1)
        e = cudaLaunchKernelEx(&cfg, gemm_cluster_sum_kernel, tmA, tmB, tmC, a);
    else if (c.a_mn)
        e = cudaLaunchKernelEx(&cfg, gemm_persistent_kernel<256, true, false>, tmA, tmB, tmC,
                               tmAux, a);
    else if (c.b_km && c.epi == EPI_GELU_GRAD)
        e = cudaLaunchKernelEx(&cfg, gemm_persistent_kernel<256, false, true, EPI_GELU_GRAD>,
                               tmA, tmB, tmC, tmAux, a);
    else if (c.b_km && a.bn == 128)
        e = cudaLaunchKernelEx(&cfg, gemm_persistent_kernel<128, false, true>, tmA, tmB, tmC,
                               tmAux, a);
    else if (c.b_km)
        e = cudaLaunchKernelEx(&cfg, gemm_persistent_kernel<256, false, true>, tmA, tmB, tmC,
                               tmAux, a);
    else if (c.epi == EPI_DUAL)
        e = cudaLaunchKernelEx(&cfg, gemm_persistent_kernel<256, false, false, EPI_DUAL>, tmA,
                               tmB, tmC, tmAux, a);
    else if (a.bn == 128)
        e = cudaLaunchKernelEx(&cfg, gemm_persistent_kernel<128>, tmA, tmB, tmC, tmAux, a);
    else
        e = cudaLaunchKernelEx(&cfg, gemm_persistent_kernel<256>, tmA, tmB, tmC, tmAux, a);
    if (e != cudaSuccess) return TP_ERR_CUDA;
    return launch_status();
}

template <typename Tin, typename Tout>
tp_status launch_simt_t(const void *X, const void *W, void *Y, void *Ys, const SimtArgs &a,
                        cudaStream_t s) {
    dim3 block(32, 8);
    const int64_t gx = (a.N + 31) / 32;
    int64_t gy = (a.M + 7) / 8;
    if (gy > 65535) gy = 65535;
    if (gx > 0x7FFFFFFF) return TP_ERR_SHAPE;
    simt_linear_kernel<Tin, Tout><<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)),
                                    block, 0, s>>>(
        static_cast<const Tin *>(X), static_cast<const Tin *>(W), static_cast<Tout *>(Y),
        static_cast<Tout *>(Ys), a);
    return launch_status();
}

tp_status launch_simt(const void *X, const void *W, void *Y, void *Ys, const SimtArgs &a,
                      tp_dtype in_t, tp_dtype out_t, cudaStream_t s) {
    if (in_t == TP_F32 && out_t == TP_F32) return launch_simt_t<float, float>(X, W, Y, Ys, a, s);
    if (in_t == TP_F32 && out_t == TP_BF16)
        return launch_simt_t<float, __nv_bfloat16>(X, W, Y, Ys, a, s);
    if (in_t == TP_BF16 && out_t == TP_F32)
        return launch_simt_t<__nv_bfloat16, float>(X, W, Y, Ys, a, s);
    return launch_simt_t<__nv_bfloat16, __nv_bfloat16>(X, W, Y, Ys, a, s);
}

int reduce_grid(int64_t work_items, int sm_count) {
    // whole waves of 256-thread blocks, 8 resident per SM, no more than needed
    int64_t blocks = (work_items + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

template <bool BF16>
tp_status launch_reduce_t(const float *P, void *Y, int64_t total, int n, int sm_count,
                          const void *bias, int64_t cols, cudaStream_t s) {
    const __nv_bfloat16 *b = static_cast<const __nv_bfloat16 *>(bias);
    if (total % 8 == 0 && (!bias || cols % 8 == 0)) {
        // bulk-copy pipeline: each stage holds `chunk` elements of every shard
        const int chunk = (RED_STAGE_BYTES / (4 * n)) & ~7;
        const int64_t n_chunks = (total + chunk - 1) / chunk;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(n_chunks < sm_count ? n_chunks : sm_count), 1, 1);
        cfg.blockDim = dim3(RED_THREADS, 1, 1);
        cfg.dynamicSmemBytes = RED_SMEM_BYTES;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, shard_reduce_bulk_kernel<BF16>, P, Y, total, n, chunk,
                               wait_limit_ns(), b, cols) != cudaSuccess)
            return TP_ERR_CUDA;
        return launch_status();
    }
    shard_reduce_scalar_kernel<BF16><<<reduce_grid(total, sm_count), 256, 0, s>>>(P, Y, total, n,
                                                                                  b, cols);
    return launch_status();
}

// Y = sum_i P_i (+ bias [cols], bf16, once after the sum).
tp_status launch_reduce(const float *P, void *Y, int64_t total, int n, tp_dtype out_t,
                        cudaStream_t s, const void *bias = nullptr, int64_t cols = 1) {
    DeviceInfo *dev = nullptr;
    tp_status st = device_info(&dev);
    if (st != TP_OK) return st;
    return out_t == TP_BF16
               ? launch_reduce_t<true>(P, Y, total, n, dev->sm_count, bias, cols, s)
               : launch_reduce_t<false>(P, Y, total, n, dev->sm_count, bias, cols, s);
}

// ------------------------------------------------------- shared validation --

tp_status check_shards(int n_shards) {
    return (n_shards >= 1 && n_shards <= TP_MAX_SHARDS) ? TP_OK : TP_ERR_DIVISIBILITY;
}

tp_status check_sizes(int64_t M, int64_t K, int64_t N) {
    if (M < 0 || K < 0 || N < 0) return TP_ERR_SHAPE;
    if (M > kInt32Max || K > kInt32Max || N > kInt32Max) return TP_ERR_SHAPE;
    if (!elems_ok(M, K) || !elems_ok(K, N) || !elems_ok(M, N)) return TP_ERR_SHAPE;
    return TP_OK;
}

tp_status column_impl(const void *X, const void *W, const void *bias, void *Y, void *Ys,
                      int64_t M, int64_t K, int64_t N, int n, int G, tp_dtype in_t,
                      tp_dtype out_t, tp_act act, cudaStream_t s) {
    tp_status st = check_sizes(M, K, N);
    if (st != TP_OK) return st;
    if (!valid_dtype(in_t) || !valid_dtype(out_t) || (act != TP_ACT_NONE && act != TP_ACT_GELU))
        return TP_ERR_DTYPE;
    const size_t it = dtype_size(in_t), ot = dtype_size(out_t);
    const size_t xb = M * K * it, wb = K * N * it, yb = M * N * ot;
    if (!present(X, xb) || !present(W, wb) || (!Y && !Ys && yb > 0)) return TP_ERR_NULL;
    if ((st = check_shards(n)) != TP_OK) return st;
    if (G < 1 || N % G != 0 || (N / G) % n != 0) return TP_ERR_DIVISIBILITY;
    const size_t bb = N * it;
    if (overlaps(Y, yb, X, xb) || overlaps(Y, yb, W, wb) || overlaps(Ys, yb, X, xb) ||
        overlaps(Ys, yb, W, wb) || overlaps(Y, yb, Ys, yb) || overlaps(Y, yb, bias, bb) ||
        overlaps(Ys, yb, bias, bb))
        return TP_ERR_ALIAS;
    const int64_t sw = N / G / n;
    if (in_t == TP_BF16) {
        if (!aligned(X, 16) || !aligned(W, 16) || !aligned(Y, 16) || !aligned(Ys, 16) ||
            !aligned(bias, 16))
            return TP_ERR_ALIGNMENT;
        if (K % 8 != 0 || N % 8 != 0 || (Ys && sw % 8 != 0)) return TP_ERR_ALIGNMENT;
    } else {
        if (!aligned(X, 4) || !aligned(W, 4) || !aligned(Y, ot) || !aligned(Ys, ot) ||
            !aligned(bias, 4))
            return TP_ERR_ALIGNMENT;
    }
    if (M == 0 || N == 0) return TP_OK;
    if (K == 0 && bias) {  // empty contraction: every output is act(bias)
        SimtArgs a{};
        a.M = M; a.K = 0; a.N = N; a.k_shards = 1; a.act_gelu = (act == TP_ACT_GELU);
        a.partials = nullptr; a.bias = bias;
        a.shard_gw = N / G; a.shard_sw = sw; a.shard_nl = sw * G;
        return launch_simt(X, W, Y, Ys, a, in_t, out_t, s);
    }
    if (K == 0) {  // empty contraction: every output is act(0) = 0
        if (Y && cudaMemsetAsync(Y, 0, yb, s) != cudaSuccess) return TP_ERR_CUDA;
        if (Ys && cudaMemsetAsync(Ys, 0, yb, s) != cudaSuccess) return TP_ERR_CUDA;
        return TP_OK;
    }
    if (in_t == TP_BF16) {
        GemmCall c{};
        c.A = X; c.B = W; c.M = M; c.N = N; c.K = K;
        c.k_groups = 1;
        c.out = Y; c.out_group_stride = 0; c.out_f32 = (out_t == TP_F32);
        c.gelu = (act == TP_ACT_GELU);
        c.out_shards = Ys; c.n_shards = n; c.col_groups = G;
        c.allow_split = true;
        c.bias = bias;
        return launch_gemm(c, s);
    }
    SimtArgs a{};
    a.M = M; a.K = K; a.N = N; a.k_shards = 1; a.act_gelu = (act == TP_ACT_GELU);
    a.partials = nullptr; a.bias = bias;
    a.shard_gw = N / G; a.shard_sw = sw; a.shard_nl = sw * G;
    return launch_simt(X, W, Y, Ys, a, in_t, out_t, s);
}

// ------------------------------------------------------------ row split --

tp_status row_impl(const void *X, const void *W, const void *bias, void *Y, float *P_out,
                   int64_t M, int64_t K, int64_t Nout, int n_shards, tp_dtype in_t,
                   tp_dtype out_t, cudaStream_t s) {
    tp_status st = check_sizes(M, K, Nout);
    if (st != TP_OK) return st;
    if (!valid_dtype(in_t) || !valid_dtype(out_t)) return TP_ERR_DTYPE;
    if ((st = check_shards(n_shards)) != TP_OK) return st;
    const size_t it = dtype_size(in_t), ot = dtype_size(out_t);
    const size_t xb = M * K * it, wb = K * Nout * it, yb = M * Nout * ot;
    const size_t pb = static_cast<size_t>(n_shards) * M * Nout * 4;
    if (!present(X, xb) || !present(W, wb) || (!Y && !P_out && yb > 0)) return TP_ERR_NULL;
    if (K % n_shards != 0) return TP_ERR_DIVISIBILITY;
    const size_t bb = Nout * it;
    if (overlaps(Y, yb, X, xb) || overlaps(Y, yb, W, wb) || overlaps(P_out, pb, X, xb) ||
        overlaps(P_out, pb, W, wb) || overlaps(Y, yb, P_out, pb) || overlaps(Y, yb, bias, bb) ||
        overlaps(P_out, pb, bias, bb))
        return TP_ERR_ALIAS;
    const int64_t Kg = K / n_shards;
    if (in_t == TP_BF16) {
        if (!aligned(X, 16) || !aligned(W, 16) || !aligned(Y, 16) || !aligned(P_out, 16) ||
            !aligned(bias, 16))
            return TP_ERR_ALIGNMENT;
        if (K % 8 != 0 || Nout % 8 != 0 || (P_out && Kg % 8 != 0)) return TP_ERR_ALIGNMENT;
    } else {
        if (!aligned(X, 4) || !aligned(W, 4) || !aligned(Y, ot) || !aligned(P_out, 4) ||
            !aligned(bias, 4))
            return TP_ERR_ALIGNMENT;
    }
    if (P_out && Y && (!aligned(P_out, 16) || !aligned(Y, 16))) return TP_ERR_ALIGNMENT;
    if (M == 0 || Nout == 0) return TP_OK;
    if (K == 0 && bias) {  // empty contraction: Y = bias on every row, partials 0
        SimtArgs a{};
        a.M = M; a.K = 0; a.N = Nout; a.k_shards = n_shards; a.act_gelu = 0;
        a.partials = P_out; a.bias = bias;
        a.shard_gw = Nout; a.shard_sw = Nout; a.shard_nl = Nout;
        return launch_simt(X, W, Y, nullptr, a, in_t, out_t, s);
    }
    if (K == 0) {
        if (Y && cudaMemsetAsync(Y, 0, yb, s) != cudaSuccess) return TP_ERR_CUDA;
        if (P_out && cudaMemsetAsync(P_out, 0, pb, s) != cudaSuccess) return TP_ERR_CUDA;
        return TP_OK;
    }
    if (in_t == TP_BF16) {
        GemmCall c{};
        c.A = X; c.B = W; c.M = M; c.N = Nout; c.K = K;
        c.out_f32 = false; c.gelu = false; c.out_shards = nullptr; c.n_shards = n_shards;
        c.col_groups = 1;
        if (P_out) {
            // one fp32 partial per shard: k-group g = shard g's rows of W
            c.k_groups = n_shards;
            c.out = P_out;
            c.out_group_stride = M * Nout;
            c.out_f32 = true;
            c.allow_split = false;
            if ((st = launch_gemm(c, s)) != TP_OK) return st;
            // the bias, if any, is added once by the reduce, after the sum
            return Y ? launch_reduce(P_out, Y, M * Nout, n_shards, out_t, s, bias, Nout) : TP_OK;
        }
        // fused: the K loop walks the shards in ascending order into one
        // fp32 accumulator (or shard groups summed through the cluster)
        c.k_groups = 1;
        c.out = Y;
        c.out_group_stride = 0;
        c.out_f32 = (out_t == TP_F32);
        c.allow_split = true;
        c.bias = bias;  // in the epilogue: after the whole K range, i.e. once
        return launch_gemm(c, s);
    }
    SimtArgs a{};
    a.M = M; a.K = K; a.N = Nout; a.k_shards = n_shards; a.act_gelu = 0;
    a.partials = P_out; a.bias = bias;
    a.shard_gw = Nout; a.shard_sw = Nout; a.shard_nl = Nout;
    return launch_simt(X, W, Y, nullptr, a, in_t, out_t, s);
}

// ------------------------------------------------------- segment copies --

// Copies the segments of table t (all other fields filled by the caller)
// from src [src_slots][rows][src_cols] to dst [dst_slots][rows][dst_cols].
tp_status launch_segment_copy(const void *src, int64_t src_slots, int64_t src_cols, void *dst,
                              int64_t dst_slots, int64_t dst_cols, int64_t rows, bool f32,
                              SegTable &t, cudaStream_t s) {
    DeviceInfo *dev = nullptr;
    tp_status st = device_info(&dev);
    if (st != TP_OK) return st;
    const int64_t es = f32 ? 4 : 2;
    t.box_rows = static_cast<int>(CAT_BOX_BYTES / (t.box_cols * es));
    if (t.box_rows > 256) t.box_rows = 256;
    t.units = (rows + t.box_rows - 1) / t.box_rows * t.col_boxes;
    t.box_bytes = static_cast<uint32_t>(t.box_cols * t.box_rows * es);
    t.wait_limit_ns = wait_limit_ns();
    CUtensorMap tmSrc, tmDst;
    if (!encode_3d_cached(&tmSrc, src, src_cols, rows, src_slots, src_cols * es,
                          rows * src_cols * es, static_cast<uint32_t>(t.box_cols),
                          static_cast<uint32_t>(t.box_rows), 1, f32, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_3d_cached(&tmDst, dst, dst_cols, rows, dst_slots, dst_cols * es,
                          rows * dst_cols * es, static_cast<uint32_t>(t.box_cols),
                          static_cast<uint32_t>(t.box_rows), 1, f32, CU_TENSOR_MAP_SWIZZLE_NONE))
        return TP_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    const int64_t grid = t.units < dev->sm_count ? t.units : dev->sm_count;
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(32, 1, 1);
    cfg.dynamicSmemBytes = CAT_SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, segment_copy_tma_kernel, tmSrc, tmDst, t) != cudaSuccess)
        return TP_ERR_CUDA;
    return launch_status();
}

// ------------------------------------------------------------ MLP block --

tp_status mlp_impl(const void *X, const void *W1, const void *b1, const void *W2,
                   const void *b2, void *Y, void *ws, size_t ws_bytes, int64_t M, int64_t d,
                   int64_t f, int n_shards, tp_dtype in_t, tp_dtype out_t, cudaStream_t s) {
    tp_status st = check_sizes(M, d, f);
    if (st != TP_OK) return st;
    if (!valid_dtype(in_t) || !valid_dtype(out_t)) return TP_ERR_DTYPE;
    const size_t it = dtype_size(in_t), ot = dtype_size(out_t);
    const size_t xb = M * d * it, w1b = d * f * it, w2b = f * d * it, yb = M * d * ot;
    const size_t hb = M * f * it;
    if (!present(X, xb) || !present(W1, w1b) || !present(W2, w2b) || !present(Y, yb))
        return TP_ERR_NULL;
    if ((st = check_shards(n_shards)) != TP_OK) return st;
    if (f % n_shards != 0) return TP_ERR_DIVISIBILITY;
    const size_t need = tp_mlp_block_workspace_size(M, f, in_t);
    if (need > 0 && (!ws || ws_bytes < need)) return TP_ERR_WORKSPACE;
    const size_t b1b = f * it, b2b = d * it;
    if (overlaps(Y, yb, X, xb) || overlaps(Y, yb, W1, w1b) || overlaps(Y, yb, W2, w2b) ||
        overlaps(Y, yb, ws, hb) || overlaps(ws, hb, X, xb) || overlaps(ws, hb, W1, w1b) ||
        overlaps(ws, hb, W2, w2b) || overlaps(Y, yb, b1, b1b) || overlaps(Y, yb, b2, b2b) ||
        overlaps(ws, hb, b1, b1b) || overlaps(ws, hb, b2, b2b))
        return TP_ERR_ALIAS;
    if (in_t == TP_BF16) {
        if (!aligned(X, 16) || !aligned(W1, 16) || !aligned(W2, 16) || !aligned(Y, 16) ||
            !aligned(ws, 16) || !aligned(b1, 16) || !aligned(b2, 16))
            return TP_ERR_ALIGNMENT;
        if (d % 8 != 0 || f % 8 != 0) return TP_ERR_ALIGNMENT;
    } else {
        if (!aligned(X, 4) || !aligned(W1, 4) || !aligned(W2, 4) || !aligned(Y, ot) ||
            !aligned(ws, 4) || !aligned(b1, 4) || !aligned(b2, 4))
            return TP_ERR_ALIGNMENT;
    }
    if (M == 0 || d == 0) return TP_OK;
    if (f == 0)  // empty hidden layer: Y = b2 on every row (or 0)
        return row_impl(nullptr, nullptr, b2, Y, nullptr, M, 0, d, 1, in_t, out_t, s);

    if (in_t == TP_BF16) {
        // step 1: H = GeLU(X . W1), column-parallel, H_i = column block i of H
        GemmCall c1{};
        c1.A = X; c1.B = W1; c1.M = M; c1.N = f; c1.K = d;
        c1.k_groups = 1; c1.out = ws; c1.out_group_stride = 0; c1.out_f32 = false;
        c1.gelu = true; c1.out_shards = nullptr; c1.n_shards = n_shards; c1.col_groups = 1;
        c1.allow_split = true;
        c1.bias = b1;  // each shard's slice of b1, before the GeLU
        if ((st = launch_gemm(c1, s)) != TP_OK) return st;
        // step 2: Y = sum_i H_i . W2_i, shard partials added in the accumulator
        GemmCall c2{};
        c2.A = ws; c2.B = W2; c2.M = M; c2.N = d; c2.K = f;
        c2.k_groups = 1; c2.out = Y; c2.out_group_stride = 0; c2.out_f32 = (out_t == TP_F32);
        c2.gelu = false; c2.out_shards = nullptr; c2.n_shards = n_shards; c2.col_groups = 1;
        c2.allow_split = true;
        c2.bias = b2;  // once, after the sum over all shards
        return launch_gemm(c2, s);
    }
    SimtArgs a1{};
    a1.M = M; a1.K = d; a1.N = f; a1.k_shards = 1; a1.act_gelu = 1; a1.partials = nullptr;
    a1.bias = b1;
    a1.shard_gw = f; a1.shard_sw = f; a1.shard_nl = f;
    if ((st = launch_simt(X, W1, ws, nullptr, a1, TP_F32, TP_F32, s)) != TP_OK) return st;
    SimtArgs a2{};
    a2.M = M; a2.K = f; a2.N = d; a2.k_shards = n_shards; a2.act_gelu = 0; a2.partials = nullptr;
    a2.bias = b2;
    a2.shard_gw = d; a2.shard_sw = d; a2.shard_nl = d;
    return launch_simt(ws, W2, Y, nullptr, a2, TP_F32, out_t, s);
}

// ------------------------------------------------------------- backward --

// dW = X^T . dY  [K, N]  and  dX = dY . W^T  [M, K], bf16 inputs.  The two
// products are the same for the column and the row split; only what a shard
// owns differs (see include/tp.h).  Either output may be NULL.
tp_status linear_backward_impl(const void *X, const void *W, const void *dY, void *dX, void *dW,
                               int64_t M, int64_t K, int64_t N, tp_dtype in_t, tp_dtype out_t,
                               cudaStream_t s) {
    const size_t ot = dtype_size(out_t);
    const size_t xb = M * K * 2, wb = K * N * 2, yb = M * N * 2;
    const size_t dxb = M * K * ot, dwb = K * N * ot;
    if (!present(X, xb) || !present(W, wb) || !present(dY, yb)) return TP_ERR_NULL;
    if (in_t != TP_BF16 || !valid_dtype(out_t)) return TP_ERR_DTYPE;
    if (!aligned(X, 16) || !aligned(W, 16) || !aligned(dY, 16) || !aligned(dX, 16) ||
        !aligned(dW, 16) || K % 8 != 0 || N % 8 != 0)
        return TP_ERR_ALIGNMENT;
    const void *ins[3] = {X, W, dY};
    const size_t inb[3] = {xb, wb, yb};
    for (int i = 0; i < 3; ++i)
        if (overlaps(dX, dxb, ins[i], inb[i]) || overlaps(dW, dwb, ins[i], inb[i]))
            return TP_ERR_ALIAS;
    if (overlaps(dX, dxb, dW, dwb)) return TP_ERR_ALIAS;
    tp_status st;
    if (dW && K > 0 && N > 0) {
        if (M == 0) {
            if (cudaMemsetAsync(dW, 0, dwb, s) != cudaSuccess) return TP_ERR_CUDA;
        } else {
            GemmCall c{};
            c.A = X; c.a_mn = true;  // X^T: X is [M][K] = [K'][M'] with M' = K
            c.B = dY;                // [M][N] = [K'][N']
            c.M = K; c.N = N; c.K = M;
            c.k_groups = 1; c.out = dW; c.out_f32 = (out_t == TP_F32);
            c.n_shards = 1; c.col_groups = 1;
            if ((st = launch_gemm(c, s)) != TP_OK) return st;
        }
    }
    if (dX && M > 0 && K > 0) {
        if (N == 0) {
            if (cudaMemsetAsync(dX, 0, dxb, s) != cudaSuccess) return TP_ERR_CUDA;
        } else {
            GemmCall c{};
            c.A = dY;                // [M][N]: K' = N walks the output columns (shards) in order
            c.B = W; c.b_km = true;  // W^T: W is [K][N] = [N'][K'] with N' = K
            c.M = M; c.N = K; c.K = N;
            c.k_groups = 1; c.out = dX; c.out_f32 = (out_t == TP_F32);
            c.n_shards = 1; c.col_groups = 1;
            if ((st = launch_gemm(c, s)) != TP_OK) return st;
        }
    }
    return TP_OK;
}

}  // namespace

// =================================================================== C ABI ==

extern "C" {

const char *tp_status_string(tp_status st) {
    switch (st) {
        case TP_OK: return "TP_OK";
        case TP_ERR_NULL: return "TP_ERR_NULL: a required pointer is NULL";
        case TP_ERR_SHAPE: return "TP_ERR_SHAPE: invalid or inconsistent sizes";
        case TP_ERR_DIVISIBILITY: return "TP_ERR_DIVISIBILITY: split axis not divisible, or shard count out of range";
        case TP_ERR_ALIGNMENT: return "TP_ERR_ALIGNMENT: pointer or row pitch misaligned";
        case TP_ERR_DTYPE: return "TP_ERR_DTYPE: unsupported dtype or activation";
        case TP_ERR_WORKSPACE: return "TP_ERR_WORKSPACE: workspace missing or too small";
        case TP_ERR_CUDA: return "TP_ERR_CUDA: a CUDA call failed";
        case TP_ERR_DEVICE_TIMEOUT: return "TP_ERR_DEVICE_TIMEOUT: a bounded device wait ran out";
        case TP_ERR_ALIAS: return "TP_ERR_ALIAS: an output overlaps an input";
    }
    return "TP_ERR_UNKNOWN";
}

tp_status tp_column_linear(const void *X, const void *W, void *Y, void *Y_shards, int64_t M,
                           int64_t K, int64_t Nout, int n_shards, tp_dtype in_t, tp_dtype out_t,
                           tp_act act, cudaStream_t s) {
    return column_impl(X, W, nullptr, Y, Y_shards, M, K, Nout, n_shards, 1, in_t, out_t, act, s);
}

tp_status tp_column_linear_bias(const void *X, const void *W, const void *bias, void *Y,
                                void *Y_shards, int64_t M, int64_t K, int64_t Nout, int n_shards,
                                tp_dtype in_t, tp_dtype out_t, tp_act act, cudaStream_t s) {
    return column_impl(X, W, bias, Y, Y_shards, M, K, Nout, n_shards, 1, in_t, out_t, act, s);
}

tp_status tp_column_linear_grouped(const void *X, const void *W, void *Y, void *Y_shards,
                                   int64_t M, int64_t K, int64_t Nout, int n_shards,
                                   int col_groups, tp_dtype in_t, tp_dtype out_t, tp_act act,
                                   cudaStream_t s) {
    return column_impl(X, W, nullptr, Y, Y_shards, M, K, Nout, n_shards, col_groups, in_t, out_t,
                       act, s);
}

tp_status tp_row_linear(const void *X, const void *W, void *Y, float *P_out, int64_t M, int64_t K,
                        int64_t Nout, int n_shards, tp_dtype in_t, tp_dtype out_t,
                        cudaStream_t s) {
    return row_impl(X, W, nullptr, Y, P_out, M, K, Nout, n_shards, in_t, out_t, s);
}

tp_status tp_row_linear_bias(const void *X, const void *W, const void *bias, void *Y,
                             float *P_out, int64_t M, int64_t K, int64_t Nout, int n_shards,
                             tp_dtype in_t, tp_dtype out_t, cudaStream_t s) {
    return row_impl(X, W, bias, Y, P_out, M, K, Nout, n_shards, in_t, out_t, s);
}

tp_status tp_sharded_linear(const void *X, const void *W, void *Y, int64_t M, int64_t K,
                            int64_t Nout, int n_shards, tp_split split, tp_dtype in_t,
                            tp_dtype out_t, tp_act act, cudaStream_t s) {
    if (split == TP_SPLIT_COLS)
        return tp_column_linear(X, W, Y, nullptr, M, K, Nout, n_shards, in_t, out_t, act, s);
    if (split == TP_SPLIT_ROWS) {
        if (act != TP_ACT_NONE) return TP_ERR_DTYPE;
        return tp_row_linear(X, W, Y, nullptr, M, K, Nout, n_shards, in_t, out_t, s);
    }
    return TP_ERR_SHAPE;
}

tp_status tp_shard_reduce(const float *P, void *Y, int64_t rows, int64_t cols, int n_shards,
                          tp_dtype out_t, cudaStream_t s) {
    if (rows < 0 || cols < 0 || !elems_ok(rows, cols)) return TP_ERR_SHAPE;
    if (!valid_dtype(out_t)) return TP_ERR_DTYPE;
    const int64_t total = rows * cols;
    if (!present(P, total) || !present(Y, total)) return TP_ERR_NULL;
    tp_status st = check_shards(n_shards);
    if (st != TP_OK) return st;
    if (!aligned(P, 16) || !aligned(Y, 16)) return TP_ERR_ALIGNMENT;
    if (overlaps(Y, total * dtype_size(out_t), P, static_cast<size_t>(n_shards) * total * 4))
        return TP_ERR_ALIAS;
    if (total == 0) return TP_OK;
    return launch_reduce(P, Y, total, n_shards, out_t, s);
}

tp_status tp_shard_concat_grouped(const void *Ys, void *Y, int64_t rows, int64_t shard_cols,
                                  int n_shards, int col_groups, tp_dtype t, cudaStream_t s) {
    if (rows < 0 || shard_cols < 0 || !elems_ok(rows, shard_cols)) return TP_ERR_SHAPE;
    if (!present(Ys, rows * shard_cols) || !present(Y, rows * shard_cols)) return TP_ERR_NULL;
    if (!valid_dtype(t)) return TP_ERR_DTYPE;
    tp_status st = check_shards(n_shards);
    if (st != TP_OK) return st;
    if (col_groups < 1 || shard_cols % col_groups != 0) return TP_ERR_DIVISIBILITY;
    const int64_t es = static_cast<int64_t>(dtype_size(t));
    const int64_t vec = 16 / es;
    const int64_t sw = shard_cols / col_groups;
    if (!aligned(Ys, 16) || !aligned(Y, 16) || sw % vec != 0) return TP_ERR_ALIGNMENT;
    const int64_t bytes = rows * shard_cols * n_shards * es;
    if (overlaps(Y, bytes, Ys, bytes)) return TP_ERR_ALIAS;
    const int64_t ncv = shard_cols * n_shards / vec;  // output vectors per row
    if (ncv > kInt32Max || rows > kInt32Max) return TP_ERR_SHAPE;
    if (rows == 0 || ncv == 0) return TP_OK;
    // boxes: the widest of 256, 128, ... columns dividing sw, rows to fill
    // CAT_BOX_BYTES (at most 256)
    int box_cols = 256;
    while (box_cols > vec && sw % box_cols != 0) box_cols /= 2;
    int box_rows = static_cast<int>(CAT_BOX_BYTES / (box_cols * es));
    if (box_rows > 256) box_rows = 256;
    DeviceInfo *dev = nullptr;
    if ((st = device_info(&dev)) != TP_OK) return st;
    const bool f32 = (t == TP_F32);
    const int64_t sc = shard_cols, N = sc * n_shards;
    CUtensorMap tmSrc, tmDst;
    if (!encode_3d_cached(&tmSrc, Ys, sc, rows, n_shards, sc * es, rows * sc * es,
                          static_cast<uint32_t>(box_cols), static_cast<uint32_t>(box_rows), 1, f32,
                          CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_3d_cached(&tmDst, Y, N, rows, 1, N * es, rows * N * es,
                          static_cast<uint32_t>(box_cols), static_cast<uint32_t>(box_rows), 1, f32,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
        return TP_ERR_CUDA;
    CatArgs a{};
    a.n = n_shards;
    a.groups = col_groups;
    a.sw = static_cast<int>(sw);
    a.gw = static_cast<int>(sw * n_shards);
    a.box_cols = box_cols;
    a.box_rows = box_rows;
    a.col_boxes = static_cast<int>(sw / box_cols);
    a.units = (rows + box_rows - 1) / box_rows * n_shards * col_groups * a.col_boxes;
    a.box_bytes = static_cast<uint32_t>(box_cols * box_rows * es);
    a.wait_limit_ns = wait_limit_ns();
    cudaLaunchConfig_t cfg{};
    const int64_t grid = a.units < dev->sm_count ? a.units : dev->sm_count;
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(32, 1, 1);
    cfg.dynamicSmemBytes = CAT_SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, shard_concat_tma_kernel, tmSrc, tmDst, a) != cudaSuccess)
        return TP_ERR_CUDA;
    return launch_status();
}

tp_status tp_qkv_linear(const void *X, const void *W, void *Y, void *Y_shards, int64_t M,
                        int64_t K, int64_t n_q_heads, int64_t n_kv_heads, int64_t head_dim,
                        int n_shards, tp_dtype in_t, tp_dtype out_t, cudaStream_t s) {
    if (n_q_heads < 1 || n_kv_heads < 1 || head_dim < 1) return TP_ERR_SHAPE;
    if (n_q_heads > kInt32Max || n_kv_heads > kInt32Max ||
        n_q_heads + 2 * n_kv_heads > kInt32Max / head_dim)
        return TP_ERR_SHAPE;  // the projection's width must fit the GEMM's int sizes
    if (n_q_heads % n_kv_heads != 0) return TP_ERR_SHAPE;
    tp_status st = check_shards(n_shards);
    if (st != TP_OK) return st;
    if (n_q_heads % n_shards != 0 ||
        (n_kv_heads % n_shards != 0 && n_shards % n_kv_heads != 0))
        return TP_ERR_DIVISIBILITY;
    if (!Y) return TP_ERR_NULL;
    const int64_t N = (n_q_heads + 2 * n_kv_heads) * head_dim;
    const int64_t qs = n_q_heads / n_shards;
    const int64_t kvs = n_kv_heads >= n_shards ? n_kv_heads / n_shards : 1;
    const int64_t nl = (qs + 2 * kvs) * head_dim;
    const int64_t es = static_cast<int64_t>(dtype_size(out_t));
    if (!valid_dtype(out_t)) return TP_ERR_DTYPE;
    if (Y_shards && (head_dim * es) % 16 != 0) return TP_ERR_ALIGNMENT;
    if (overlaps(Y_shards, static_cast<size_t>(n_shards) * M * nl * es, Y, M * N * es))
        return TP_ERR_ALIAS;
    if (3 * n_shards > SEG_MAX) return TP_ERR_SHAPE;
    // the full projection in Wqkv's column order (KV heads computed once)
    if ((st = column_impl(X, W, nullptr, Y, nullptr, M, K, N, 1, 1, in_t, out_t, TP_ACT_NONE,
                          s)) != TP_OK)
        return st;
    if (!Y_shards || M == 0) return TP_OK;
    if (overlaps(Y_shards, static_cast<size_t>(n_shards) * M * nl * es, X, M * K * dtype_size(in_t)) ||
        overlaps(Y_shards, static_cast<size_t>(n_shards) * M * nl * es, W, K * N * dtype_size(in_t)))
        return TP_ERR_ALIAS;
    if (!aligned(Y_shards, 16)) return TP_ERR_ALIGNMENT;
    // each shard's Q heads, then the K and V heads its Q heads read
    SegTable t;
    std::memset(&t, 0, sizeof(t));
    int box = 256;
    while (box > 16 / es && head_dim % box != 0) box /= 2;
    t.box_cols = box;
    int nseg = 0, boxes = 0;
    auto add = [&](int64_t src_col, int64_t dst_slot, int64_t dst_col, int64_t width) {
        t.prefix[nseg] = boxes;
        t.src_slot[nseg] = 0;
        t.src_col[nseg] = static_cast<int>(src_col);
        t.dst_slot[nseg] = static_cast<int>(dst_slot);
        t.dst_col[nseg] = static_cast<int>(dst_col);
        boxes += static_cast<int>(width / box);
        ++nseg;
    };
    for (int64_t i = 0; i < n_shards; ++i) {
        const int64_t kv0 = n_kv_heads >= n_shards ? i * kvs : (i * n_kv_heads) / n_shards;
        add(i * qs * head_dim, i, 0, qs * head_dim);
        add((n_q_heads + kv0) * head_dim, i, qs * head_dim, kvs * head_dim);
        add((n_q_heads + n_kv_heads + kv0) * head_dim, i, (qs + kvs) * head_dim, kvs * head_dim);
    }
    t.prefix[nseg] = boxes;
    t.n_seg = nseg;
    t.col_boxes = boxes;
    return launch_segment_copy(Y, 1, N, Y_shards, n_shards, nl, M, out_t == TP_F32, t, s);
}

tp_status tp_shard_concat(const void *Ys, void *Y, int64_t rows, int64_t shard_cols,
                          int n_shards, tp_dtype t, cudaStream_t s) {
    return tp_shard_concat_grouped(Ys, Y, rows, shard_cols, n_shards, 1, t, s);
}

size_t tp_mlp_block_workspace_size(int64_t M, int64_t f, tp_dtype t) {
    if (M < 0 || f < 0 || M > kInt32Max || f > kInt32Max || !elems_ok(M, f) || !valid_dtype(t))
        return 0;
    const size_t b = static_cast<size_t>(M) * static_cast<size_t>(f) * dtype_size(t);
    return (b + 255) & ~static_cast<size_t>(255);
}

tp_status tp_mlp_block(const void *X, const void *W1, const void *W2, void *Y, void *ws,
                       size_t ws_bytes, int64_t M, int64_t d, int64_t f, int n_shards,
                       tp_dtype in_t, tp_dtype out_t, cudaStream_t s) {
    return mlp_impl(X, W1, nullptr, W2, nullptr, Y, ws, ws_bytes, M, d, f, n_shards, in_t, out_t,
                    s);
}

tp_status tp_mlp_block_bias(const void *X, const void *W1, const void *b1, const void *W2,
                            const void *b2, void *Y, void *ws, size_t ws_bytes, int64_t M,
                            int64_t d, int64_t f, int n_shards, tp_dtype in_t, tp_dtype out_t,
                            cudaStream_t s) {
    return mlp_impl(X, W1, b1, W2, b2, Y, ws, ws_bytes, M, d, f, n_shards, in_t, out_t, s);
}

// ----------------------------------------------------------- backward ----

tp_status tp_column_linear_backward(const void *X, const void *W, const void *dY, void *dX,
                                    void *dW, int64_t M, int64_t K, int64_t Nout, int n_shards,
                                    tp_dtype in_t, tp_dtype out_t, cudaStream_t s) {
    tp_status st = check_sizes(M, K, Nout);
    if (st != TP_OK) return st;
    if ((st = check_shards(n_shards)) != TP_OK) return st;
    if (Nout % n_shards != 0) return TP_ERR_DIVISIBILITY;
    return linear_backward_impl(X, W, dY, dX, dW, M, K, Nout, in_t, out_t, s);
}

tp_status tp_row_linear_backward(const void *X, const void *W, const void *dY, void *dX,
                                 void *dW, int64_t M, int64_t K, int64_t Nout, int n_shards,
                                 tp_dtype in_t, tp_dtype out_t, cudaStream_t s) {
    tp_status st = check_sizes(M, K, Nout);
    if (st != TP_OK) return st;
    if ((st = check_shards(n_shards)) != TP_OK) return st;
    if (K % n_shards != 0) return TP_ERR_DIVISIBILITY;
    return linear_backward_impl(X, W, dY, dX, dW, M, K, Nout, in_t, out_t, s);
}

size_t tp_mlp_block_backward_workspace_size(int64_t M, int64_t f, tp_dtype t) {
    if (M < 0 || f < 0 || M > kInt32Max || f > kInt32Max || !elems_ok(M, f) || t != TP_BF16)
        return 0;
    return 3 * ((static_cast<size_t>(M) * static_cast<size_t>(f) * 2 + 255) &
                ~static_cast<size_t>(255));
}

tp_status tp_mlp_block_backward(const void *X, const void *W1, const void *W2, const void *dY,
                                void *dX, void *dW1, void *dW2, void *ws, size_t ws_bytes,
                                int64_t M, int64_t d, int64_t f, int n_shards, tp_dtype in_t,
                                tp_dtype out_t, cudaStream_t s) {
    tp_status st = check_sizes(M, d, f);
    if (st != TP_OK) return st;
    if (in_t != TP_BF16 || !valid_dtype(out_t)) return TP_ERR_DTYPE;
    if ((st = check_shards(n_shards)) != TP_OK) return st;
    if (f % n_shards != 0) return TP_ERR_DIVISIBILITY;
    const size_t ot = dtype_size(out_t);
    const size_t xb = M * d * 2, w1b = d * f * 2, w2b = f * d * 2, yb = M * d * 2;
    const size_t dxb = M * d * ot, dw1b = d * f * ot, dw2b = f * d * ot;
    if (!present(X, xb) || !present(W1, w1b) || !present(W2, w2b) || !present(dY, yb))
        return TP_ERR_NULL;
    const size_t part = (static_cast<size_t>(M) * f * 2 + 255) & ~static_cast<size_t>(255);
    const size_t need = tp_mlp_block_backward_workspace_size(M, f, in_t);
    if (need > 0 && (!ws || ws_bytes < need)) return TP_ERR_WORKSPACE;
    if (!aligned(X, 16) || !aligned(W1, 16) || !aligned(W2, 16) || !aligned(dY, 16) ||
        !aligned(dX, 16) || !aligned(dW1, 16) || !aligned(dW2, 16) || !aligned(ws, 16) ||
        d % 8 != 0 || f % 8 != 0)
        return TP_ERR_ALIGNMENT;
    const void *ins[5] = {X, W1, W2, dY, ws};
    const size_t inb[5] = {xb, w1b, w2b, yb, need};
    void *outs[3] = {dX, dW1, dW2};
    const size_t outb[3] = {dxb, dw1b, dw2b};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 5; ++i)
            if (overlaps(outs[o], outb[o], ins[i], inb[i])) return TP_ERR_ALIAS;
        for (int p = o + 1; p < 3; ++p)
            if (overlaps(outs[o], outb[o], outs[p], outb[p])) return TP_ERR_ALIAS;
    }
    for (int i = 0; i < 4; ++i)
        if (overlaps(ws, need, ins[i], inb[i])) return TP_ERR_ALIAS;
    if (M == 0 || d == 0 || f == 0) {
        // empty contractions give zero gradients
        if (dW1 && d > 0 && f > 0 && cudaMemsetAsync(dW1, 0, dw1b, s) != cudaSuccess)
            return TP_ERR_CUDA;
        if (dW2 && d > 0 && f > 0 && cudaMemsetAsync(dW2, 0, dw2b, s) != cudaSuccess)
            return TP_ERR_CUDA;
        if (dX && M > 0 && d > 0 && cudaMemsetAsync(dX, 0, dxb, s) != cudaSuccess)
            return TP_ERR_CUDA;
        return TP_OK;
    }
    uint8_t *Z = static_cast<uint8_t *>(ws), *H = Z + part, *dZ = H + part;
    const bool f32 = (out_t == TP_F32);
    // 1. recompute Z = X . W1 and H = GeLU(Z) (bf16, one launch)
    {
        GemmCall c{};
        c.A = X; c.B = W1; c.M = M; c.N = f; c.K = d;
        c.k_groups = 1; c.out = Z; c.epi = EPI_DUAL; c.aux = H;
        c.n_shards = 1; c.col_groups = 1;
        if ((st = launch_gemm(c, s)) != TP_OK) return st;
    }
    // 2. dZ = (dY . W2^T) * GeLU'(Z): every shard's block of columns of dZ
    if (dW1 || dX) {
        GemmCall c{};
        c.A = dY; c.B = W2; c.b_km = true;  // W2 is [f][d] = [N'][K']
        c.M = M; c.N = f; c.K = d;
        c.k_groups = 1; c.out = dZ; c.epi = EPI_GELU_GRAD; c.aux = Z;
        c.n_shards = 1; c.col_groups = 1;
        if ((st = launch_gemm(c, s)) != TP_OK) return st;
    }
    // 3. dW2 = H^T . dY (rows block i = shard i)
    if (dW2) {
        GemmCall c{};
        c.A = H; c.a_mn = true; c.B = dY; c.M = f; c.N = d; c.K = M;
        c.k_groups = 1; c.out = dW2; c.out_f32 = f32; c.n_shards = 1; c.col_groups = 1;
        if ((st = launch_gemm(c, s)) != TP_OK) return st;
    }
    // 4. dW1 = X^T . dZ (columns block i = shard i)
    if (dW1) {
        GemmCall c{};
        c.A = X; c.a_mn = true; c.B = dZ; c.M = d; c.N = f; c.K = M;
        c.k_groups = 1; c.out = dW1; c.out_f32 = f32; c.n_shards = 1; c.col_groups = 1;
        if ((st = launch_gemm(c, s)) != TP_OK) return st;
    }
    // 5. dX = dZ . W1^T: the K loop walks the hidden columns, shard 0's first,
    //    so the shards' contributions are added in ascending order
    if (dX) {
        GemmCall c{};
        c.A = dZ; c.B = W1; c.b_km = true;  // W1 is [d][f] = [N'][K']
        c.M = M; c.N = d; c.K = f;
        c.k_groups = 1; c.out = dX; c.out_f32 = f32; c.n_shards = 1; c.col_groups = 1;
        if ((st = launch_gemm(c, s)) != TP_OK) return st;
    }
    return TP_OK;
}

tp_status tp_get_device_status(cudaStream_t s) {
    if (cudaStreamSynchronize(s) != cudaSuccess) return TP_ERR_CUDA;
    unsigned int word = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)) != cudaSuccess) return TP_ERR_CUDA;
    if (word != 0) {
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return TP_ERR_CUDA;
        if (cudaMemcpyToSymbol(g_timeout_site, &zero, sizeof(zero)) != cudaSuccess) return TP_ERR_CUDA;
        return TP_ERR_DEVICE_TIMEOUT;
    }
    return TP_OK;
}

}  // extern "C"

// ------------------------------------------------------- bounded-wait test --

namespace tpk {
// One CTA waits on a barrier that expects one arrival nobody makes.
__global__ void selftest_wait_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_wait_bounded(smem_u32(&bar), 0, limit_ns, &abort_flag, SITE_SELFTEST);
    }
    __syncthreads();
}
}  // namespace tpk

extern "C" tp_status tp_selftest_bounded_wait(uint64_t limit_ns, cudaStream_t s) {
    if (limit_ns < 1000ull) limit_ns = 1000ull;
    if (limit_ns > 5000000000ull) limit_ns = 5000000000ull;
    tpk::selftest_wait_kernel<<<1, 32, 0, s>>>(limit_ns);
    return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}
