// Inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk / .tensor), tcgen05
// (TMEM alloc, MMA, commit, ld/st, fences), cluster DSMEM, and a bounded mbarrier wait.
#pragma once
#include <cstdint>
#include <cuda.h>

#ifndef W4A16_SPIN_MODE
#define W4A16_SPIN_MODE 0  // MMA issuers: 0 = try_wait, 2 = test_wait polling
#endif

namespace w4g {

// ---- status word -----------------------------------------------------------------
// Status codes mirror w4a16_status in include/w4a16.h.
constexpr int kStatusFormat = -5;
constexpr int kStatusTimeout = -4;

__device__ __forceinline__ void record_status(int* status, int code) {
    if (status != nullptr) atomicCAS(status, 0, code);  // the first error sticks
}

// ---- addresses / timers ----------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t lane_id() {
    uint32_t l;
    asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
    return l;
}

// ---- explicit shared-memory loads (32-bit shared addresses) -------------------------
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// ---- mbarrier ----------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test: returns at once (no hardware suspension window).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Same, but the thread may sleep in hardware (up to kSuspendNs) until the phase
// completes, instead of re-issuing the test: waiting warps then take no issue slots.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "n"(kSuspendNs)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Gives up when the
// CTA-wide abort flag is raised or after `limit_ns` of wall time; the first waiter to
// time out raises the abort flag and records kStatusTimeout.  Returns true on success.
template <int kMode>  // 0: try_wait, 1: try_wait with sleep hint, 2: test_wait polling
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                            volatile int* abort_flag, int* status,
                                            uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        const bool done = kMode == 1 ? mbar_try_wait_sleep(bar, parity)
                        : kMode == 2 ? mbar_test_wait(bar, parity)
                                     : mbar_try_wait(bar, parity);
        if (done) return true;
        if ((it & (kMode == 2 ? 255u : 3u)) == 0u) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                record_status(status, kStatusTimeout);
                return false;
            }
        }
    }
}

#ifndef W4A16_WAIT_MODE
#define W4A16_WAIT_MODE 1  // other waiters: 1 = try_wait with a sleep hint, 2 = test_wait polling
#endif
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag, int* status,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow<W4A16_WAIT_MODE>(bar, parity, abort_flag, status, limit_ns);
}

// Same bound, but never sleeps: for the latency-critical MMA-issuing threads.
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, int* status,
                                               uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow<W4A16_SPIN_MODE>(bar, parity, abort_flag, status, limit_ns);
}

// Warp-uniform form: every lane waits, and the warp proceeds only if all lanes succeeded,
// so that the .sync.aligned tcgen05 instructions that follow see a converged warp.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, int* status,
                                               uint64_t limit_ns) {
    const bool ok = mbar_wait_bounded(bar, parity, abort_flag, status, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

// Warp-uniform form of mbar_wait_spin.
__device__ __forceinline__ bool mbar_wait_spin_warp(uint32_t bar, uint32_t parity,
                                                    volatile int* abort_flag, int* status,
                                                    uint64_t limit_ns) {
    const bool ok = mbar_wait_spin(bar, parity, abort_flag, status, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

// ---- L2 cache policies -------------------------------------------------------------
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---- TMA -----------------------------------------------------------------------------
// Contiguous bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void tma_bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                             uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// 2-D tiled tensor copy global -> shared; coordinates {c0 (innermost), c1}.
__device__ __forceinline__ void tma_tensor_2d_g2s(uint32_t dst, const CUtensorMap* map,
                                                  int c0, int c1, uint32_t bar,
                                                  uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar),
          "l"(policy)
        : "memory");
}

// 3-D tiled tensor copy global -> shared; coordinates {c0 (innermost), c1, c2}.
__device__ __forceinline__ void tma_tensor_3d_g2s(uint32_t dst, const CUtensorMap* map,
                                                  int c0, int c1, int c2, uint32_t bar,
                                                  uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2),
          "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- tcgen05: tensor memory --------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] . B[smem]^T, kind::f16 (fp16 or bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The eight K = 16 MMAs of one 128-K block and the commits that track them, issued by
// lane 0 while the whole warp executes the statement (no branch around it, so the operands,
// computed by every lane, stay warp-uniform): D[d] (+)= A[a_j] . B[b_j]^T for j = 0..7, the
// first accumulating only if `accumulate`; then an arrive on bar0 and, unless bar1 is 0,
// on bar1 once they are done.  Lane 0 is the issuing thread of every block, so its later
// commits track all of them.
__device__ __forceinline__ void tc_mma_block_lane0(uint32_t d_tmem, const uint32_t (&a)[8],
                                                   const uint64_t (&b)[8], uint32_t idesc,
                                                   uint32_t accumulate, uint32_t bar0,
                                                   uint32_t bar1) {
    asm volatile(
        "{\n\t.reg .pred p, q, e, c;\n\t.reg .b32 l;\n\t"
        "mov.u32 l, %%laneid;\n\t"
        "setp.eq.u32 e, l, 0;\n\t"
        "setp.ne.b32 p, %18, 0;\n\t"
        "setp.ne.b32 q, %17, 0;\n\t"  // idesc is never 0: a true predicate
        "setp.ne.b32 c, %20, 0;\n\t"
        "and.pred c, c, e;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %9, %17, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %10, %17, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %11, %17, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %12, %17, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %13, %17, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %14, %17, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %15, %17, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], %16, %17, q;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%19];\n\t"
        "@c tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%20];\n\t}"
        ::"r"(d_tmem), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]),
          "r"(a[6]), "r"(a[7]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]),
          "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(idesc), "r"(accumulate), "r"(bar0), "r"(bar1)
        : "memory");
}

// Arrive (once) on an mbarrier when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
        ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
          "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
          "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
          "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
          "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte-swizzle
// canonical layout: 8-row x 128-byte atoms, atoms 1024 bytes apart along the
// M/N dimension (stride byte offset), start address 16-byte granular.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(1u) << 16;                  // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;          // stride byte offset
    d |= static_cast<uint64_t>(1u) << 46;                  // descriptor version (sm_100+)
    d |= static_cast<uint64_t>(2u) << 61;                  // swizzle: 128 B
    return d;
}

// Instruction descriptor, kind::f16, fp32 accumulator, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int dtype, int M, int N) {
    return (1u << 4)                                   // D format: F32
           | (static_cast<uint32_t>(dtype) << 7)      // A format: 0 F16, 1 BF16
           | (static_cast<uint32_t>(dtype) << 10)     // B format
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// ---- cluster ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t caddr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(caddr) : "memory");
    return v;
}

// Cluster barrier in two halves, so that the arrive can be issued early and the wait
// late (all threads of every CTA of the cluster take part in both).
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// Arrive without ordering this thread's memory operations: for barrier phases that only
// signal progress (the memory they protect is ordered by other means, e.g. an mbarrier
// initialisation fenced with fence.mbarrier_init.release.cluster, or a completed
// complete_tx).  A release arrive waits for the thread's prior accesses to be performed at
// cluster scope, which is measurably slower on the critical path.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Generic-proxy shared-memory writes -> visible to the async proxy (TMA / bulk copies).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bulk copy from this CTA's shared memory into a peer CTA's shared memory; completes
// `bytes` of transaction count on the peer's mbarrier (both cluster addresses).
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst_cluster, uint32_t src_cta,
                                               uint32_t bytes, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes"
        " [%0], [%1], %2, [%3];"
        ::"r"(dst_cluster), "r"(src_cta), "r"(bytes), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until the source side of every committed bulk copy has been read.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ---- programmatic dependent launch ---------------------------------------------------
__device__ __forceinline__ void grid_dep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace w4g
