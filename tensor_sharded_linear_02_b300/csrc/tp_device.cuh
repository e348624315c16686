// tp_device.cuh -- device-side building blocks for sm_103a: the library's
// status word, bounded mbarrier waits, TMA tensor loads and the tcgen05
// (5th-generation tensor core) instructions, all as inline PTX.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tpk {

// ---------------------------------------------------------------------------
// Status word.  Bit 0: a bounded wait ran out.  The site word records which
// wait gave up first (for diagnostics only).
// ---------------------------------------------------------------------------
__device__ unsigned int g_status_word = 0;
__device__ unsigned int g_timeout_site = 0;

enum WaitSite : uint32_t {
    SITE_PRODUCER_EMPTY = 1,
    SITE_MMA_FULL = 2,
    SITE_MMA_ACC_EMPTY = 3,
    SITE_EPI_ACC_FULL = 4,
    SITE_DRAIN = 5,
    SITE_EPI_SPLIT = 6,
    SITE_SELFTEST = 9,
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start while the previous kernel of the stream is still
// running; `grid_dep_wait` blocks until that kernel has completed and its
// memory operations are visible, so everything before it must touch no
// global data the previous kernel could read or write.  `grid_dep_trigger`
// lets the next kernel of the stream start launching (it still waits for
// this one to complete before touching memory).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void grid_dep_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive on a barrier that may belong to another CTA of the cluster (address
// in the shared::cluster window, from mapa).  Used by the epilogue to hand a
// drained accumulator back: the data it guards is tensor memory whose reads
// were completed (tcgen05.wait::ld) and fenced before the arrive, so the
// default release at CTA scope is enough and no global store has to drain.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void record_timeout(uint32_t site) {
    atomicOr(&g_status_word, 1u);
    atomicCAS(&g_timeout_site, 0u, site);
}

// Wait until the phase with the given parity of barrier `bar` has completed,
// for at most limit_ns.  Returns false (and raises *abort and the status
// word) if the limit runs out, or returns false at once if *abort is already
// raised by another role.  `abort` lives in shared memory.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                  volatile uint32_t *abort, uint32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    uint32_t spins = 0;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((++spins & 15u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                *abort = 1;
                record_timeout(site);
                return false;
            }
        }
    }
}

// Same, ignoring the abort flag: used while draining work already in flight
// after an abort.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            record_timeout(SITE_DRAIN);
            return false;
        }
    }
    return true;
}

// Warp-uniform variant: lane 0 waits, the verdict is broadcast, so that every
// lane of the warp takes the same branch (the tcgen05.ld that follows is a
// warp-collective instruction).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                               volatile uint32_t *abort, uint32_t site) {
    uint32_t ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, limit_ns, abort, site) ? 1u : 0u;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) -- tiled 3-D load into this CTA's shared memory,
// completion signalled on an mbarrier with transaction bytes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Untiled bulk copy global -> this CTA's shared memory (both addresses 16-byte
// aligned, bytes a multiple of 16), completion counted on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// Bulk copy from this CTA's shared memory to shared memory of another CTA of
// the cluster (dst and the barrier in the shared::cluster window, from mapa;
// 16-byte aligned, bytes a multiple of 16), completion counted on the
// destination CTA's barrier.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src,
                                                  uint32_t bytes, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst_cluster),
        "r"(src), "r"(bytes), "r"(bar_cluster)
        : "memory");
}

// Same load for a CTA pair that issues one tcgen05.mma.cta_group::2: the data
// lands in this CTA's shared memory, the completed bytes are counted on the
// barrier at `cluster_bar`, which may belong to the peer CTA of the pair.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t cluster_bar, int32_t c0, int32_t c1,
                                                 int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// TMA tiled store of a box from this CTA's shared memory, tracked as a bulk
// async group of the issuing thread.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int32_t c0,
                                             int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until no committed bulk store of this thread still reads shared memory.
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until at most N of this thread's committed bulk stores still read
// shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read_n() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait0() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 for a CTA pair (cta_group::2): one thread of the even CTA issues
// M = 256 MMAs whose A rows 0..127 and B columns 0..N/2-1 come from its own
// shared memory and A rows 128..255 and B columns N/2..N-1 from the peer's
// (same offsets); accumulator rows 0..127 land in the even CTA's tensor
// memory and rows 128..255 in the odd CTA's.  Allocation is collective over
// one warp of each CTA of the pair.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void umma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the barrier at offset `bar` in every CTA of `cta_mask` when
// all pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void umma_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
}

// Arrive on this CTA's barrier at `bar` when the pair MMAs issued so far by
// this thread have completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory (TMEM) allocation, MMA, commit, loads and fences.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], bf16/fp16 inputs, one instruction of shape
// M x N x 16 as encoded in idesc.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives
// row (lane base + t), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// ---------------------------------------------------------------------------
// Shared-memory matrix descriptors for tcgen05.mma (64-bit).
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-47  descriptor version (1 on this architecture)
//   bits 49-51  base offset (0: swizzle atoms are 1024-byte aligned)
//   bit  52     leading-dimension offset mode (0: relative)
//   bits 61-63  swizzle mode (2 = 128-byte swizzle)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor for kind::f16 with bf16 A and B, fp32 D.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   bit 15 A major (0 = K-major), bit 16 B major (1 = MN-major),
//   bits 17-22 N >> 3, bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n, bool b_mn_major,
                                                      bool a_mn_major = false) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// ---------------------------------------------------------------------------
// Thread-block cluster helpers (distributed shared memory).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t dsmem_map(uint32_t local_addr, uint32_t cta_rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(cta_rank));
    return r;
}

// ---------------------------------------------------------------------------
// Numerics shared by the epilogues.
// ---------------------------------------------------------------------------
// Exact (erf-form) GeLU, x * Phi(x) with Phi(x) = (1 + erf(x / sqrt 2)) / 2,
// in fp32, written as
//     GeLU(x) = max(x, 0) - |x| h,   h = Phi(-|x|) = erfc(|x| / sqrt 2) / 2,
// with h accurate RELATIVE to its value over the whole range: for x < 0,
// GeLU(x) = x h shrinks like exp(-x^2 / 2), so an error bound that is only
// absolute (as for the rational approximations of erf) says nothing there.
//
// h uses the functional form of the Chebyshev-fitted complementary error
// function of Press, Teukolsky, Vetterling & Flannery, "Numerical Recipes
// in C" (2nd ed.), section 6.2: erfc(z) = t exp(-z^2 + P(t)) with
// t = 1 / (1 + z / 2), P a polynomial.  As z runs over [0, inf), t runs
// over (0, 1] and ln(erfc(z) exp(z^2) / t) is smooth, so a polynomial of
// degree 7 fits it; the coefficients below come from a least-squares
// Chebyshev fit over t in [0.09, 1] (|x| up to 28; fit_gelu.py in the
// package), folded for the base-2 exponential and the factor 1/2:
//     t = 1 / (1 + |x| / (2 sqrt 2)),
//     h = t * 2^(G(t) - x^2 log2(e) / 2),   G(t) = log2(e) (P(t) - ln 2).
// Relative error of h in double: 7.4e-7.  In fp32 (one hardware reciprocal,
// 8 fused multiply-adds, one hardware base-2 exponential, a multiply, a max
// and a fused multiply-add, two elements per packed fma.rn.f32x2 /
// mul.rn.f32x2 instruction where the operation allows) an emulation over
// every bf16 input in [-12, 12] gives a GeLU relative error of at most
// 6.5e-6 (the rounding of the exponent's argument, largest in the far
// tail), and the bf16 rounding of every value equal to the round-to-
// nearest-even of the exact GeLU.  Straight-line code: no branch, so no
// code is replicated per element in the unrolled epilogues.  For |x| past
// ~13 the exponential underflows to 0 (ftz) and GeLU(x) = max(x, 0), the
// correct limit to fp32 precision.
constexpr float GELU_T_SCALE = 3.535533906e-01f;  // 1 / (2 sqrt 2)
constexpr float GELU_G0 = -2.825663090e+00f;
constexpr float GELU_G1 = 1.440122604e+00f;
constexpr float GELU_G2 = 5.716950893e-01f;
constexpr float GELU_G3 = -6.818283349e-02f;
constexpr float GELU_G4 = 5.251461267e-01f;
constexpr float GELU_G5 = -1.465897799e+00f;
constexpr float GELU_G6 = 1.096563697e+00f;
constexpr float GELU_G7 = -2.737848759e-01f;
constexpr float GELU_HALF_LOG2E = 7.213475204e-01f;  // log2(e) / 2
constexpr float INV_SQRT_2PI = 3.989422804e-01f;

__device__ __forceinline__ float rcp_approx(float a) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

__device__ __forceinline__ float ex2_approx(float a) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

// h = Phi(-|x|), relative error ~1e-6 (see above).
__device__ __forceinline__ float normal_tail_f32(float x) {
    const float u = fabsf(x);
    const float t = rcp_approx(fmaf(u, GELU_T_SCALE, 1.0f));
    float g = fmaf(GELU_G7, t, GELU_G6);
    g = fmaf(g, t, GELU_G5);
    g = fmaf(g, t, GELU_G4);
    g = fmaf(g, t, GELU_G3);
    g = fmaf(g, t, GELU_G2);
    g = fmaf(g, t, GELU_G1);
    g = fmaf(g, t, GELU_G0);
    return t * ex2_approx(fmaf(x * -GELU_HALF_LOG2E, x, g));
}

__device__ __forceinline__ float gelu_f32(float x) {
    return fmaf(-fabsf(x), normal_tail_f32(x), fmaxf(x, 0.0f));
}

// Two fp32 values in one 64-bit register (lo in bits 0-31) and the packed
// fp32x2 arithmetic of sm_100-class GPUs (each lane rounded exactly like the
// scalar instruction, so packed and scalar evaluations agree bit for bit).
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t splat2(float c) { return f32x2_pack(c, c); }

// gelu_f32 of two values at once (same operations, same results).
__device__ __forceinline__ void gelu2_f32(float &x0, float &x1) {
    const uint64_t u = f32x2_pack(fabsf(x0), fabsf(x1));
    const uint64_t den = fma_f32x2(u, splat2(GELU_T_SCALE), splat2(1.0f));
    float d0, d1;
    f32x2_unpack(den, d0, d1);
    const uint64_t t = f32x2_pack(rcp_approx(d0), rcp_approx(d1));
    uint64_t g = fma_f32x2(splat2(GELU_G7), t, splat2(GELU_G6));
    g = fma_f32x2(g, t, splat2(GELU_G5));
    g = fma_f32x2(g, t, splat2(GELU_G4));
    g = fma_f32x2(g, t, splat2(GELU_G3));
    g = fma_f32x2(g, t, splat2(GELU_G2));
    g = fma_f32x2(g, t, splat2(GELU_G1));
    g = fma_f32x2(g, t, splat2(GELU_G0));
    const uint64_t xx = f32x2_pack(x0, x1);
    const uint64_t a = fma_f32x2(mul_f32x2(xx, splat2(-GELU_HALF_LOG2E)), xx, g);
    float a0, a1;
    f32x2_unpack(a, a0, a1);
    const uint64_t h = mul_f32x2(t, f32x2_pack(ex2_approx(a0), ex2_approx(a1)));
    const uint64_t nu = f32x2_pack(-fabsf(x0), -fabsf(x1));
    const uint64_t y = fma_f32x2(nu, h, f32x2_pack(fmaxf(x0, 0.0f), fmaxf(x1, 0.0f)));
    f32x2_unpack(y, x0, x1);
}

// GeLU of 32 values held as fp32 bit patterns (one tensor-memory load).
__device__ __forceinline__ void gelu_chunk32(uint32_t (&r)[32]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float a = __uint_as_float(r[2 * i]), b = __uint_as_float(r[2 * i + 1]);
        gelu2_f32(a, b);
        r[2 * i] = __float_as_uint(a);
        r[2 * i + 1] = __float_as_uint(b);
    }
}

// GeLU'(x) = Phi(x) + x phi(x), phi(x) = exp(-x^2/2) / sqrt(2 pi), in fp32:
// Phi from the same normal tail as gelu_f32 (Phi = 1 - h for x >= 0, h for
// x < 0, so relative accuracy holds in the negative tail too), the density
// from the hardware base-2 exponential (exp(-x^2/2) = 2^(-x^2 log2(e) / 2)).
__device__ __forceinline__ float gelu_grad_f32(float x) {
    const float h = normal_tail_f32(x);
    const float phi_cdf = x >= 0.0f ? 1.0f - h : h;
    const float e = ex2_approx(x * -GELU_HALF_LOG2E * x);
    return fmaf(x * INV_SQRT_2PI, e, phi_cdf);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace tpk
