// Inline-PTX wrappers for the sm_103a features the kernels use: mbarriers,
// bulk async copies (TMA, non-tensor form), L2 cache policies, and the 5th
// generation tensor core (tcgen05: TMEM allocation, MMA, commit, loads).
#pragma once

#include <cstdint>

namespace fp8bs {
namespace ptx {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes the initialised barriers visible to the async proxy (bulk copies, MMA).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// mbar_arrive where pred holds (the predicate inside the instruction)
__device__ __forceinline__ void mbar_arrive_if(uint64_t* bar, bool pred) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\t@q mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(
                     smem_addr(bar)),
                 "r"(static_cast<uint32_t>(pred))
                 : "memory");
}

// One non-blocking probe of the barrier phase: true once the phase with the
// given parity has completed.  test_wait never suspends the thread, so a spin
// on it sees a completion (of a bulk copy or an MMA commit) at once; the
// potentially blocking try_wait was measured waking only at its internal time
// limit, ~0.8 us after the phase had completed.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Four probes in one go: bit j of the result is set once barrier j's phase
// with parity pj has completed.  A probe takes about 180 cycles to answer;
// issued together the four answer in about the time of one.
__device__ __forceinline__ uint32_t mbar_test4(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1, uint64_t* b2,
                                               uint32_t p2, uint64_t* b3, uint32_t p3) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred q0, q1, q2, q3;\n\t.reg .b32 t0, t1, t2, t3;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q0, [%1], %2;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q2, [%5], %6;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q3, [%7], %8;\n\t"
        "selp.u32 t0, 1, 0, q0;\n\tselp.u32 t1, 2, 0, q1;\n\tselp.u32 t2, 4, 0, q2;\n\tselp.u32 t3, 8, 0, q3;\n\t"
        "or.b32 t0, t0, t1;\n\tor.b32 t2, t2, t3;\n\tor.b32 %0, t0, t2;\n\t}"
        : "=r"(r)
        : "r"(smem_addr(b0)), "r"(p0), "r"(smem_addr(b1)), "r"(p1), "r"(smem_addr(b2)), "r"(p2), "r"(smem_addr(b3)),
          "r"(p3)
        : "memory");
    return r;
}

// ---------------------------------------------------------------------------
// Bulk async copy global -> shared, completion counted on an mbarrier.
// dst and src 16-byte aligned; bytes a multiple of 16.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads (the MMA reading an operand written with st.shared).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------

// Lets the next kernel on the stream (launched with programmatic stream
// serialization) start once every CTA of this grid has executed this.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Waits until the previous kernel on the stream has completed and its memory
// operations are visible (a no-op without programmatic serialization).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Non-bulk async copies (16 bytes, global -> shared, bypassing L1) and flags
// ---------------------------------------------------------------------------

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// Bulk prefetch of [p, p + bytes) into L2 (p 16-byte aligned, bytes a
// multiple of 16); nothing is returned and nothing waits for it.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Bring the 128-byte line holding p into L2 (no data returned, no ordering).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// 16-byte global load that the compiler keeps where it is written: it is
// neither re-issued later (to free registers) nor moved past other volatile
// instructions, so a batch of these is in flight together.
__device__ __forceinline__ uint4 ld_global_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Predicated forms: the access happens only where pred holds, with the
// predicate inside the instruction, so that unrolled code with a condition
// per element stays straight-line (a branch around an asm statement, which
// the compiler cannot predicate, is a divergence-safe branch each).
// ld_global_v4_if leaves v unchanged where pred is false.
__device__ __forceinline__ void ld_global_v4_if(uint4& v, const void* p, bool pred) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %5, 0;\n\t@q ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\n\t}"
                 : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
                 : "l"(p), "r"(static_cast<uint32_t>(pred)));
}
__device__ __forceinline__ void st_shared_v2_if(void* p, uint32_t a, uint32_t b, bool pred) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %3, 0;\n\t@q st.shared.v2.b32 [%0], {%1, %2};\n\t}" ::"r"(
                     smem_addr(p)),
                 "r"(a), "r"(b), "r"(static_cast<uint32_t>(pred))
                 : "memory");
}
__device__ __forceinline__ void st_shared_b32_if(void* p, uint32_t a, bool pred) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.shared.b32 [%0], %1;\n\t}" ::"r"(smem_addr(p)),
                 "r"(a), "r"(static_cast<uint32_t>(pred))
                 : "memory");
}
__device__ __forceinline__ void st_global_v2_if(void* p, uint32_t a, uint32_t b, bool pred) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %3, 0;\n\t@q st.global.v2.b32 [%0], {%1, %2};\n\t}" ::"l"(p),
                 "r"(a), "r"(b), "r"(static_cast<uint32_t>(pred))
                 : "memory");
}
__device__ __forceinline__ void st_global_b32_if(void* p, uint32_t a, bool pred) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.global.b32 [%0], %1;\n\t}" ::"l"(p), "r"(a),
                 "r"(static_cast<uint32_t>(pred))
                 : "memory");
}
__device__ __forceinline__ void st_global_b8_if(void* p, uint32_t a, bool pred) {
    asm volatile("{\n\t.reg .pred q;\n\t.reg .b16 h;\n\tsetp.ne.u32 q, %2, 0;\n\tcvt.u16.u32 h, %1;\n\t"
                 "@q st.global.b8 [%0], h;\n\t}" ::"l"(p),
                 "r"(a), "r"(static_cast<uint32_t>(pred))
                 : "memory");
}

// Wait until every cp.async this thread issued has landed in shared memory.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (TMEM and the 5th-generation MMA)
// ---------------------------------------------------------------------------

// Whole warp: allocate ncols TMEM columns (power of two >= 32); the TMEM
// address is written to *slot in shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(slot)),
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

// D[tmem] (+)= A[smem] * B[smem]^T, fp8 x fp8 -> fp32, both operands K-major.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Whole-warp forms: every lane of the warp executes the call with the same
// operands and one elected lane issues the instruction.  A loop run by the
// whole warp keeps the operands warp-uniform, which was measured to issue
// MMAs at about twice the rate of the same loop run by lane 0 alone.
__device__ __forceinline__ void mma_f8f6f4_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_mxf8f6f4_bs_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                     uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}
// Named (hardware) barriers: bar.arrive marks the arrival of the calling warp
// without waiting; bar.sync waits until `count` threads have arrived.
__device__ __forceinline__ void named_arrive(uint32_t id, uint32_t count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void mma_commit_warp(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_addr(bar))
        : "memory");
}

// Arrive once on bar when all prior tcgen05 async operations of this thread
// have completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp receives
// lane (taddr.lane + i), columns taddr.col .. +15.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzle layout: 8-row x 128-byte atoms, atoms 1024 bytes apart along the
// row (M/N) dimension.  Fields: start address >> 4 (bits 0-13), leading byte
// offset >> 4 (16-29, unused for this layout), stride byte offset >> 4
// (32-45), the fixed descriptor version 1 (46-48), base offset 0 (49-51),
// swizzle mode 2 = 128B (61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(16u >> 4) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// D[tmem] (+)= (A[smem] * sfa) * (B[smem] * sfb)^T, e4m3 x e4m3 -> fp32, with
// one e8m0 scale factor per 32 K values of each row of A and of B read from
// TMEM (kind::mxf8f6f4.block_scale.scale_vec::1X).  Row r of A takes its
// factor from TMEM lane r, column sfa.col + r/32; row n of B from lane n % 32
// of the quadrant the D row lies in, column sfb.col + n/32; the byte within
// the 32-bit cell is the instruction descriptor's scale-factor id.
__device__ __forceinline__ void mma_mxf8f6f4_bs(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// One 32-bit TMEM cell per thread: thread i of the warp writes lane
// taddr.lane + i, column taddr.col (the warp's own lane quadrant).
__device__ __forceinline__ void tmem_st_32x32b_x1(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Instruction descriptor, kind::mxf8f6f4 with block scaling: B's scale-factor
// id in bits 4-5, A and B e4m3 (bits 7-9, 10-12 = 0), both K-major, N >> 3 in
// bits 17-22, scale-factor type e8m0 (bit 23 = 1), M >> 4 in bits 24-28, A's
// scale-factor id in bits 29-30.
__host__ __device__ constexpr uint32_t idesc_mxf8f6f4_e4m3_e8m0(uint32_t m, uint32_t n, uint32_t sfa_id,
                                                               uint32_t sfb_id) {
    return (sfb_id << 4) | ((n >> 3) << 17) | (1u << 23) | ((m >> 4) << 24) | (sfa_id << 29);
}

// Instruction descriptor, kind::f8f6f4, dense: D fp32 (bits 4-5 = 1), A and B
// e4m3 (bits 7-9, 10-12 = 0), no negation, both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f8f6f4_e4m3(uint32_t m, uint32_t n) {
    return (1u << 4) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

}  // namespace ptx
}  // namespace fp8bs
