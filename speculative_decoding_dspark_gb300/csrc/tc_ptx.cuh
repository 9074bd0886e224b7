// tc_ptx.cuh -- inline-PTX wrappers for sm_103a: mbarriers, TMA tile loads,
// tcgen05 tensor-memory allocation, MMA, commit and loads.
//
// Written from the PTX ISA's descriptions of these instructions.  Every spin
// on an mbarrier is bounded: after `limit_ns` of wall time (globaltimer) the
// wait gives up, raises a CTA-wide abort flag and returns false.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace dspark {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but a thread whose phase is not complete may be suspended
// for up to hint_ns (it resumes as soon as the phase completes), so a long wait
// does not keep the warp scheduler busy polling.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// The bounded wait's slow path: sleep on the barrier until the phase completes,
// another thread aborts, or limit_ns has passed (then abort).  Out of line, so
// that the callers' hot loops stay free of its code: in the MMA issuer an
// inlined copy made every tcgen05.mma cost ~117 cycles of issue against ~97
// with this one out of line (64 with no wait at all).
__device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                            uint64_t limit_ns) {
    constexpr uint32_t kSleepNs = 20000;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            return false;
        }
    }
}

// Wait for the phase of parity `parity` to complete, at most limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns) {
    if (__builtin_expect(mbar_try_wait(bar, parity), 1)) return true;
    return mbar_wait_slow(bar, parity, abort_flag, limit_ns);
}

// ---------------------------------------------------------------- proxies
// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (the tensor cores read operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// ---------------------------------------------------------------- elected issue
// Forms for a warp that runs its issue loop together (warp-uniform control flow,
// so the loop's state stays in uniform registers): one lane, chosen by
// elect.sync, issues the operation.  All 32 lanes must execute the call.  The
// same lane is chosen every time (the lowest active one), so commits track the
// MMAs that lane issued.

// Arm `bar` for `bytes` and start the 2-D tile load into dst.
__device__ __forceinline__ void tma_load_2d_elect(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                                  uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%2], %5;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(bytes)
        : "memory");
}

// L2 cache policies (createpolicy) for the hinted loads below.  Every line of a
// load with policy_evict_first() is a first candidate for eviction;
// policy_keep_fraction(f) marks the fraction f of the lines of an address range
// (the same lines every time) evict_last, the rest evict_first.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t policy_keep_fraction(float f) {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.L2::evict_first.b64 %0, %1;" : "=l"(pol) : "f"(f));
    return pol;
}

// As tma_load_2d_elect, with an L2 cache policy for the loaded lines.
__device__ __forceinline__ void tma_load_2d_elect_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                                       uint32_t bytes, uint64_t pol) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%2], %5;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %6;\n\t}" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(bytes), "l"(pol)
        : "memory");
}

// As tma_load_3d_elect, with an L2 cache policy for the loaded lines.
__device__ __forceinline__ void tma_load_3d_elect_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                                       int z, uint32_t bytes, uint64_t pol) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%2], %6;\n\t"
        "@e cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %7;\n\t}" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(bytes), "l"(pol)
        : "memory");
}

// Arm `bar` for `bytes` and start the 3-D tile load into dst.
__device__ __forceinline__ void tma_load_3d_elect(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                                  int z, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%2], %6;\n\t"
        "@e cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];\n\t}" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(bytes)
        : "memory");
}

// Arm `bar` for `bytes` and start two tile loads on it: a 2-D box of map_b into
// dst_b and a 3-D box of map_a into dst_a (the two operands of one k-block).
__device__ __forceinline__ void tma_load_2d_3d_elect(void* dst_b, const CUtensorMap* map_b, int xb, int yb,
                                                     void* dst_a, const CUtensorMap* map_a, int xa, int ya, int za,
                                                     uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%2], %10;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];\n\t"
        "@e cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%5], [%6, {%7, %8, %9}], [%2];\n\t}" ::"r"(smem_u32(dst_b)),
        "l"(reinterpret_cast<uint64_t>(map_b)), "r"(smem_u32(bar)), "r"(xb), "r"(yb), "r"(smem_u32(dst_a)),
        "l"(reinterpret_cast<uint64_t>(map_a)), "r"(xa), "r"(ya), "r"(za), "r"(bytes)
        : "memory");
}

// D (+)= A . B^T with both operands described in shared memory (as umma_bf16),
// issued by the elected lane.
__device__ __forceinline__ void umma_bf16_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D (+)= A . B^T with A in tensor memory (as umma_bf16_ta), issued by the elected lane.
__device__ __forceinline__ void umma_bf16_ta_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                   uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation the elected lane issued so far completes.
__device__ __forceinline__ void umma_commit_elect(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (quadrant base + i), columns col .. col+31, written to v[OFF .. OFF+31].
template <int OFF, int N>
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, float (&v)[N]) {
    static_assert(OFF + 32 <= N, "destination too small");
    uint32_t r0, r1, r2, r3, r4, r5, r6, r7, r8, r9, r10, r11, r12, r13, r14, r15;
    uint32_t r16, r17, r18, r19, r20, r21, r22, r23, r24, r25, r26, r27, r28, r29, r30, r31;
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3), "=r"(r4), "=r"(r5), "=r"(r6), "=r"(r7), "=r"(r8),
          "=r"(r9), "=r"(r10), "=r"(r11), "=r"(r12), "=r"(r13), "=r"(r14), "=r"(r15), "=r"(r16),
          "=r"(r17), "=r"(r18), "=r"(r19), "=r"(r20), "=r"(r21), "=r"(r22), "=r"(r23), "=r"(r24),
          "=r"(r25), "=r"(r26), "=r"(r27), "=r"(r28), "=r"(r29), "=r"(r30), "=r"(r31)
        : "r"(taddr)
        : "memory");
    v[OFF + 0] = __uint_as_float(r0); v[OFF + 1] = __uint_as_float(r1);
    v[OFF + 2] = __uint_as_float(r2); v[OFF + 3] = __uint_as_float(r3);
    v[OFF + 4] = __uint_as_float(r4); v[OFF + 5] = __uint_as_float(r5);
    v[OFF + 6] = __uint_as_float(r6); v[OFF + 7] = __uint_as_float(r7);
    v[OFF + 8] = __uint_as_float(r8); v[OFF + 9] = __uint_as_float(r9);
    v[OFF + 10] = __uint_as_float(r10); v[OFF + 11] = __uint_as_float(r11);
    v[OFF + 12] = __uint_as_float(r12); v[OFF + 13] = __uint_as_float(r13);
    v[OFF + 14] = __uint_as_float(r14); v[OFF + 15] = __uint_as_float(r15);
    v[OFF + 16] = __uint_as_float(r16); v[OFF + 17] = __uint_as_float(r17);
    v[OFF + 18] = __uint_as_float(r18); v[OFF + 19] = __uint_as_float(r19);
    v[OFF + 20] = __uint_as_float(r20); v[OFF + 21] = __uint_as_float(r21);
    v[OFF + 22] = __uint_as_float(r22); v[OFF + 23] = __uint_as_float(r23);
    v[OFF + 24] = __uint_as_float(r24); v[OFF + 25] = __uint_as_float(r25);
    v[OFF + 26] = __uint_as_float(r26); v[OFF + 27] = __uint_as_float(r27);
    v[OFF + 28] = __uint_as_float(r28); v[OFF + 29] = __uint_as_float(r29);
    v[OFF + 30] = __uint_as_float(r30); v[OFF + 31] = __uint_as_float(r31);
}

// 32 lanes x 16 consecutive 32-bit columns into v[OFF .. OFF+15].
template <int OFF, int N>
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, float (&v)[N]) {
    static_assert(OFF + 16 <= N, "destination too small");
    uint32_t r0, r1, r2, r3, r4, r5, r6, r7, r8, r9, r10, r11, r12, r13, r14, r15;
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3), "=r"(r4), "=r"(r5), "=r"(r6), "=r"(r7), "=r"(r8),
          "=r"(r9), "=r"(r10), "=r"(r11), "=r"(r12), "=r"(r13), "=r"(r14), "=r"(r15)
        : "r"(taddr)
        : "memory");
    v[OFF + 0] = __uint_as_float(r0); v[OFF + 1] = __uint_as_float(r1);
    v[OFF + 2] = __uint_as_float(r2); v[OFF + 3] = __uint_as_float(r3);
    v[OFF + 4] = __uint_as_float(r4); v[OFF + 5] = __uint_as_float(r5);
    v[OFF + 6] = __uint_as_float(r6); v[OFF + 7] = __uint_as_float(r7);
    v[OFF + 8] = __uint_as_float(r8); v[OFF + 9] = __uint_as_float(r9);
    v[OFF + 10] = __uint_as_float(r10); v[OFF + 11] = __uint_as_float(r11);
    v[OFF + 12] = __uint_as_float(r12); v[OFF + 13] = __uint_as_float(r13);
    v[OFF + 14] = __uint_as_float(r14); v[OFF + 15] = __uint_as_float(r15);
}

// D (+)= A . B^T with A in tensor memory (M lanes, K along the columns, two
// bf16 per 32-bit column) and B described in shared memory.
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 8 consecutive 32-bit columns of this warp's 32 lanes from v[0..7] (thread i
// of the warp writes lane quadrant base + i).
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 8 consecutive 32-bit columns into v[OFF .. OFF+7].
template <int OFF, int N>
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, float (&v)[N]) {
    static_assert(OFF + 8 <= N, "destination too small");
    uint32_t r0, r1, r2, r3, r4, r5, r6, r7;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3), "=r"(r4), "=r"(r5), "=r"(r6), "=r"(r7)
                 : "r"(taddr)
                 : "memory");
    v[OFF + 0] = __uint_as_float(r0); v[OFF + 1] = __uint_as_float(r1);
    v[OFF + 2] = __uint_as_float(r2); v[OFF + 3] = __uint_as_float(r3);
    v[OFF + 4] = __uint_as_float(r4); v[OFF + 5] = __uint_as_float(r5);
    v[OFF + 6] = __uint_as_float(r6); v[OFF + 7] = __uint_as_float(r7);
}

// Prefetch one TMA box of a 3-D tensor into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle: rows of 64 bf16 (128 bytes), 8-row atoms of 1024 bytes
// stacked along M/N (stride 1024 bytes).  Fields: start address >> 4 in bits
// 0-13, leading-dimension offset (unused by swizzled K-major tiles; 16 bytes)
// in bits 16-29, stride-dimension offset >> 4 in bits 32-45, descriptor
// version 1 in bits 46-47, swizzle mode 2 (128-byte) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 D, both K-major:
// D format in bits 4-5 (1 = f32), A format bits 7-9 and B format bits 10-12
// (1 = bf16), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

}  // namespace tc
}  // namespace dspark
