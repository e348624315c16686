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
// in fp32, in two parts.
//
// Main part (x >= -3, and every x of a 32-value chunk with none below -3):
// erf from the rational approximation of Abramowitz and Stegun, "Handbook of
// Mathematical Functions" (1964), formula 7.1.28: for z >= 0,
//     erfc(z) = 1 - erf(z) ~ (1 + a1 z + a2 z^2 + ... + a6 z^6)^-16,
// absolute error at most 3e-7.  With z = |x| / sqrt 2 and h = erfc(z) / 2,
// Phi(x) = 1 - h for x >= 0 and h for x < 0, so
//     GeLU(x) = max(x, 0) - |x| h.
// The constants are folded into the polynomial: with u = -|x| and
// k = 2^(1/16), P(u) = sum_i d_i u^i, d_i = k a_i (-1/sqrt 2)^i (d_0 = k),
// equals k (1 + a1 z + ... + a6 z^6), so P^16 = 2 / erfc(z) and
// h = 1 / P^16.  Cost per element: 6 fused multiply-adds, 4 squarings, one
// hardware reciprocal, a max and a fused multiply-add; the packed variant
// does two elements per fp32x2 instruction (fma.rn.f32x2 / mul.rn.f32x2,
// each lane rounded exactly like the scalar fmaf / multiply).
// The bound 3e-7 is absolute: relative to GeLU(x) = x h for x < 0 it grows
// as h shrinks.  Evaluated in double, the relative error of this form is at
// most 6.4e-5 over x >= -3 (largest near x = -2.97; below 1e-6 for x > 0),
// 3.7e-3 at x = -4 and 4.7e-2 at x = -5.
//
// Tail (x < -3): GeLU(x) = x * Phi(x) with CUDA's normcdff, whose error is a
// few ulp relative over its whole range, so the tail is as accurate
// relatively as the rest.  It is a branch taken only for chunks that hold
// such a value (for N(0, 1) pre-activations 1.35e-3 of the values).
//
// For |x| above ~28 the 16th power overflows to +inf and h = 0, the correct
// limit on the positive side.
constexpr float GELU_D0 = 1.04427373409271240e+00f;
constexpr float GELU_D1 = -5.20751625299453735e-02f;
constexpr float GELU_D2 = 2.20769979059696198e-02f;
constexpr float GELU_D3 = -3.42273921705782413e-03f;
constexpr float GELU_D4 = 3.96861360059119761e-05f;
constexpr float GELU_D5 = -5.10552090418059379e-05f;
constexpr float GELU_D6 = 5.62129980608006008e-06f;
constexpr float GELU_TAIL_X = -3.0f;
// x < -3 (or a negative NaN) exactly when the fp32 bit pattern, read as an
// unsigned integer, exceeds that of -3.0f (0xC0400000): positive values
// have the sign bit clear, and among negative values a larger magnitude has
// a larger pattern.
constexpr uint32_t GELU_TAIL_BITS = 0xC0400000u;

// Inlined at every use: an out-of-line call would make the epilogues save
// their live accumulator registers around it (measured: stack spills in the
// cluster kernel), and the branch that reaches it is rarely taken.
__device__ __forceinline__ float normcdf_tail_f32(float x) { return normcdff(x); }
__device__ __forceinline__ float gelu_tail_f32(float x) { return x * normcdf_tail_f32(x); }

__device__ __forceinline__ float gelu_main_f32(float x) {
    const float u = -fabsf(x);
    float p = fmaf(GELU_D6, u, GELU_D5);
    p = fmaf(p, u, GELU_D4);
    p = fmaf(p, u, GELU_D3);
    p = fmaf(p, u, GELU_D2);
    p = fmaf(p, u, GELU_D1);
    p = fmaf(p, u, GELU_D0);
    p = __fmul_rn(p, p);  // ^2
    p = __fmul_rn(p, p);  // ^4
    p = __fmul_rn(p, p);  // ^8
    p = __fmul_rn(p, p);  // ^16
    float h;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(h) : "f"(p));
    return fmaf(u, h, fmaxf(x, 0.0f));
}

__device__ __forceinline__ float gelu_f32(float x) {
    return x < GELU_TAIL_X ? gelu_tail_f32(x) : gelu_main_f32(x);
}

// Two fp32 values in one 64-bit register (lo in bits 0-31) and the packed
// fp32x2 arithmetic of sm_100-class GPUs.
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

// gelu_main_f32 of two values at once (same operations, same results).
__device__ __forceinline__ void gelu2_main_f32(float &x0, float &x1) {
    const uint64_t u = f32x2_pack(-fabsf(x0), -fabsf(x1));
    uint64_t p = fma_f32x2(f32x2_pack(GELU_D6, GELU_D6), u, f32x2_pack(GELU_D5, GELU_D5));
    p = fma_f32x2(p, u, f32x2_pack(GELU_D4, GELU_D4));
    p = fma_f32x2(p, u, f32x2_pack(GELU_D3, GELU_D3));
    p = fma_f32x2(p, u, f32x2_pack(GELU_D2, GELU_D2));
    p = fma_f32x2(p, u, f32x2_pack(GELU_D1, GELU_D1));
    p = fma_f32x2(p, u, f32x2_pack(GELU_D0, GELU_D0));
    p = mul_f32x2(p, p);
    p = mul_f32x2(p, p);
    p = mul_f32x2(p, p);
    p = mul_f32x2(p, p);
    float q0, q1, h0, h1;
    f32x2_unpack(p, q0, q1);
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(h0) : "f"(q0));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(h1) : "f"(q1));
    const uint64_t y =
        fma_f32x2(u, f32x2_pack(h0, h1), f32x2_pack(fmaxf(x0, 0.0f), fmaxf(x1, 0.0f)));
    f32x2_unpack(y, x0, x1);
}

// gelu_f32 of two values at once.
__device__ __forceinline__ void gelu2_f32(float &x0, float &x1) {
    const float a = x0, b = x1;
    gelu2_main_f32(x0, x1);
    if (fminf(a, b) < GELU_TAIL_X) {
        if (a < GELU_TAIL_X) x0 = gelu_tail_f32(a);
        if (b < GELU_TAIL_X) x1 = gelu_tail_f32(b);
    }
}

// GeLU of 32 values held as fp32 bit patterns (one tensor-memory load).  The
// common case (no value below -3: one unsigned maximum over the patterns)
// runs the packed main part only; otherwise the values are taken pair by
// pair with the tail check.
__device__ __forceinline__ void gelu_chunk32(uint32_t (&r)[32]) {
    uint32_t mx = r[0];
#pragma unroll
    for (int i = 1; i < 32; ++i) mx = max(mx, r[i]);
    if (mx <= GELU_TAIL_BITS) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float a = __uint_as_float(r[2 * i]), b = __uint_as_float(r[2 * i + 1]);
            gelu2_main_f32(a, b);
            r[2 * i] = __float_as_uint(a);
            r[2 * i + 1] = __float_as_uint(b);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float a = __uint_as_float(r[2 * i]), b = __uint_as_float(r[2 * i + 1]);
            gelu2_f32(a, b);
            r[2 * i] = __float_as_uint(a);
            r[2 * i + 1] = __float_as_uint(b);
        }
    }
}

// GeLU'(x) = Phi(x) + x * phi(x), phi(x) = exp(-x^2/2) / sqrt(2 pi), in fp32:
// Phi from the same folded Abramowitz & Stegun 7.1.28 polynomial as
// gelu_main_f32 (Phi = 1 - h for x >= 0, h for x < 0) and, for x < -3, from
// CUDA's normcdff (relative accuracy in the tail, as for the GeLU itself);
// the density from the hardware base-2 exponential
// (exp(-x^2/2) = 2^(-x^2/2 * log2 e)).
__device__ __forceinline__ float gelu_grad_f32(float x) {
    const float u = -fabsf(x);
    float p = fmaf(GELU_D6, u, GELU_D5);
    p = fmaf(p, u, GELU_D4);
    p = fmaf(p, u, GELU_D3);
    p = fmaf(p, u, GELU_D2);
    p = fmaf(p, u, GELU_D1);
    p = fmaf(p, u, GELU_D0);
    p = __fmul_rn(p, p);
    p = __fmul_rn(p, p);
    p = __fmul_rn(p, p);
    p = __fmul_rn(p, p);
    float h;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(h) : "f"(p));
    float phi_cdf = x >= 0.0f ? 1.0f - h : h;
    if (x < GELU_TAIL_X) phi_cdf = normcdf_tail_f32(x);
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * x * -0.72134752044448170368f));
    return fmaf(x * 0.39894228040143267794f, e, phi_cdf);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace tpk
