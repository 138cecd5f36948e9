// ptx.cuh -- inline-PTX wrappers for sm_103a: mbarrier (with bounded waits),
// TMA tensor loads, tcgen05 (TMEM allocation, MMA, commit, loads) and fences.
//
// Every wait here is bounded by a wall-clock budget read from %globaltimer;
// when the budget runs out the wait returns false and the caller records an
// error status and winds down instead of spinning forever.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace fp8ll {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

// The same arrive issued by lane 0 of a converged warp as one predicated
// instruction: no branch, so the warp does not split and reconverge around it.
__device__ __forceinline__ void mbar_arrive_lane0(uint32_t bar, int lane) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.eq.s32 p, %1, 0;\n\t@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar),
                 "r"(lane)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
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

// One poll of two barriers in one statement (the two latencies overlap).
__device__ __forceinline__ void mbar_try_wait2(uint32_t b1, uint32_t p1, uint32_t b2, uint32_t p2, bool& ok1,
                                               bool& ok2) {
    uint32_t r1, r2;
    asm volatile(
        "{\n\t.reg .pred q1, q2;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q1, [%2], %3;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q2, [%4], %5;\n\t"
        "selp.u32 %0, 1, 0, q1;\n\t"
        "selp.u32 %1, 1, 0, q2;\n\t}"
        : "=r"(r1), "=r"(r2)
        : "r"(b1), "r"(p1), "r"(b2), "r"(p2)
        : "memory");
    ok1 = r1 != 0;
    ok2 = r2 != 0;
}

// Wait until the phase with the given parity has completed, for at most
// budget_ns of wall-clock time.  Returns false on time-out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t budget_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > budget_ns) return false;
    }
}

// Wait for two phases (each bounded as mbar_wait); both polled at once first.
__device__ __forceinline__ bool mbar_wait2(uint32_t b1, uint32_t p1, uint32_t b2, uint32_t p2, uint64_t budget_ns) {
    bool ok1, ok2;
    mbar_try_wait2(b1, p1, b2, p2, ok1, ok2);
    if (!ok1) ok1 = mbar_wait(b1, p1, budget_ns);
    if (ok1 && !ok2) ok2 = mbar_wait(b2, p2, budget_ns);
    return ok1 && ok2;
}

// Warp-wide forms of the two waits above, for a converged warp: every lane
// polls and the warp leaves together as soon as any lane has seen the phase
// complete (a completed phase stays complete until the thread that owns the
// barrier's next phase, which waits on this warp, moves it on), so the lanes
// never split and need no vote afterwards.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, uint64_t budget_ns) {
    if (__any_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (__any_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if (__any_sync(0xffffffffu, global_timer_ns() - t0 > budget_ns)) return false;
    }
}

__device__ __forceinline__ bool mbar_wait2_warp(uint32_t b1, uint32_t p1, uint32_t b2, uint32_t p2,
                                                uint64_t budget_ns) {
    bool ok1, ok2;
    mbar_try_wait2(b1, p1, b2, p2, ok1, ok2);
    if (__any_sync(0xffffffffu, ok1 && ok2)) return true;
    return mbar_wait_warp(b1, p1, budget_ns) && mbar_wait_warp(b2, p2, budget_ns);
}

// Orders this thread's earlier generic-proxy accesses to shared memory before
// later async-proxy (TMA) accesses.  A consumer that read a TMA-filled stage
// with ordinary loads issues it before releasing the stage, so the next TMA
// fill of that stage cannot overtake the reads.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of the box at (x, y) (x innermost) into shared memory,
// completing transaction bytes on the mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                            int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// ------------------------------------------------------------------ clusters
//
// A CTA pair (a cluster of two CTAs on two SMs) shares one tcgen05 MMA: rank 0
// (the leader) issues it, both CTAs supply half of each operand and each
// receives its half of the accumulator.  Addresses in the peer's shared memory
// are formed with mapa.

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// the shared::cluster address of this CTA's shared-memory offset `addr` in CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
    return d;
}

// every thread of both CTAs: earlier memory operations of the cluster are
// visible to later ones on both sides
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Lane 0 of a converged warp arrives on an mbarrier of either CTA of the
// cluster (a mapa address), one predicated instruction.  Relaxed: it orders
// nothing by itself, and is used only where what it announces has already
// completed (tensor-memory loads finished by tcgen05.wait::ld).  A
// cluster-scope release here measured ~1000 cycles per arrive.
__device__ __forceinline__ void mbar_arrive_remote_lane0(uint32_t cluster_addr, int lane) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.eq.s32 p, %1, 0;\n\t"
        "@p mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];\n\t}" ::"r"(cluster_addr),
        "r"(lane)
        : "memory");
}

// tma_load_2d into this CTA's shared memory, counting the bytes on an
// mbarrier of either CTA of the pair (a mapa address)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}

// -------------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// CTA-pair forms: one warp of each CTA of the pair executes alloc, relinquish
// and dealloc together; both get the same columns of their own tensor memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, fp8 operands (kind::f8f6f4), fp32 accumulator.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The pair's MMA (issued by one thread of the leader): M = 256 rows, rows
// 0..127 from the leader's A tile and 128..255 from the peer's at the same
// shared-memory offset; N columns, the first N/2 from the leader's B tile and
// the rest from the peer's; each CTA's tensor memory at d_tmem receives its
// own 128 rows.
__device__ __forceinline__ void mma_f8f6f4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier at offset `bar` of every CTA in cta_mask when
// all pair MMAs this thread issued before have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(cta_mask)
        : "memory");
}

// Arrive once on the mbarrier when all previously issued tcgen05 async ops of
// this thread have completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Two 16-lane TMEM loads of 32 columns each (shape 16x256b, 4 repetitions),
// one at lane offset +0 and one at +16 of the warp's quadrant, completed by one
// wait inside the same statement.  Fragment of thread t for repetition i
// (columns 8i..8i+7 from the address): lo[2i] = row t/4, columns
// 8i + 2(t%4) + {0,1}; lo[2i+1] = row t/4 + 8, same columns; hi[] the same for
// rows +16.  Each 64-bit value packs the even column in its low half.
__device__ __forceinline__ void tmem_ld_16x256b_x4_pairs2(uint32_t a, uint32_t b, uint64_t (&lo)[8], uint64_t (&hi)[8]) {
    asm volatile(
        "{\n\t.reg .b32 t<32>;\n\t"
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31}, [%17];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\tmov.b64 %1, {t2, t3};\n\tmov.b64 %2, {t4, t5};\n\tmov.b64 %3, {t6, t7};\n\tmov.b64 %4, {t8, t9};\n\tmov.b64 %5, {t10, t11};\n\tmov.b64 %6, {t12, t13};\n\tmov.b64 %7, {t14, t15};\n\tmov.b64 %8, {t16, t17};\n\tmov.b64 %9, {t18, t19};\n\tmov.b64 %10, {t20, t21};\n\tmov.b64 %11, {t22, t23};\n\tmov.b64 %12, {t24, t25};\n\tmov.b64 %13, {t26, t27};\n\tmov.b64 %14, {t28, t29};\n\tmov.b64 %15, {t30, t31};\n\t}"
        : "=l"(lo[0]), "=l"(lo[1]), "=l"(lo[2]), "=l"(lo[3]), "=l"(lo[4]), "=l"(lo[5]), "=l"(lo[6]), "=l"(lo[7]), "=l"(hi[0]), "=l"(hi[1]), "=l"(hi[2]), "=l"(hi[3]), "=l"(hi[4]), "=l"(hi[5]), "=l"(hi[6]), "=l"(hi[7])
        : "r"(a), "r"(b)
        : "memory");
}

// packed fp32x2 arithmetic on 64-bit register pairs (low half = first element);
// each lane rounds to nearest exactly as the scalar mul / fma would
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}

__device__ __forceinline__ float2 unpack_f32x2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row groups 1024 bytes apart.
//   bits  0-13 start address >> 4
//   bits 16-29 leading-dimension byte offset >> 4 (unused for swizzled K-major)
//   bits 32-45 stride-dimension byte offset >> 4 (1024 B between 8-row groups)
//   bits 46-47 descriptor version (1 on this architecture)
//   bits 61-63 swizzle mode (2 = 128-byte swizzle)
__device__ __forceinline__ uint64_t smem_desc_k_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// ------------------------------------------------------------ conversions

// two fp32 -> two fp8 codes (round to nearest even, saturating to +-max);
// `lo` lands in the low byte.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint16_t cvt_e5m2x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace fp8ll
