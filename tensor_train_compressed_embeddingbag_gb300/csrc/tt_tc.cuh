// tt_tc.cuh -- 5th-generation tensor-core helpers (tcgen05, sm_100 family) for
// the fp32 contractions, computed as three TF32 products ("3xTF32"):
//   x = hi(x) + lo(x),  hi = x rounded to TF32,  lo = x - hi (exact in fp32),
//   a.b ~ hi(a).hi(b) + hi(a).lo(b) + lo(a).hi(b)
// with fp32 accumulation in tensor memory; the dropped lo.lo term and the TF32
// truncation of lo leave a relative error near 2^-21 per product, far inside the
// 1e-4 parity tolerance, so the results match the FFMA path to fp32 rounding.
//
// Operand tiles live in shared memory in the canonical no-swizzle K-major layout:
// 8-row x 16-byte core matrices (8 x 4 fp32), the core matrices of one 8-row group
// consecutive along K (128 bytes apart: the descriptor's leading-dimension offset)
// and the 8-row groups (K / 4) * 128 bytes apart (its stride-dimension offset).
// One MMA consumes K = 8 (two core matrices along K); the next K step starts 256
// bytes later.  The accumulator D (M = 128 rows) occupies tensor-memory lanes
// 0..127, one row per lane, columns [base, base + N).
//
// Every wait on an mbarrier is bounded; a wait that gives up reports failure to
// the caller, which records kErrTimeout, issues no further MMA and rewrites no
// operand tile, and before freeing its tensor memory waits once more (with the
// full limit) for the MMAs already in flight.
#pragma once

#include <cstdint>

#include "tt_internal.cuh"

namespace ttemb {

constexpr int kTcM = 128;                 // rows per MMA (one per tensor-memory lane)
constexpr uint32_t kTcWaitLimit = kTcWaitPolls;  // polls of an mbarrier before giving up (default)

// Float offset of element (r, k) of an [rows][K] fp32 tile in the canonical layout.
__host__ __device__ __forceinline__ int tc_off(int r, int k, int K) {
    return (r >> 3) * (K * 8) + (k >> 2) * 32 + (r & 7) * 4 + (k & 3);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// TF32 rounding of x (round to nearest, ties away), kept in an fp32 container.
__device__ __forceinline__ float tf32_round(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// Shared-memory matrix descriptor: start address, leading (K) and stride (M/N)
// byte offsets, descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor of kind::tf32: fp32 accumulator, TF32 A and B, both K-major.
__host__ __device__ constexpr uint32_t tc_idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Warp-collective (one full warp): allocate ncols tensor-memory columns (a power of
// two >= 32); the base address is written to *slot.
__device__ __forceinline__ void tc_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_dealloc(uint32_t base, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Generic-proxy shared-memory writes become visible to the tensor core's reads.
__device__ __forceinline__ void tc_fence_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// D (+)= A . B^T for one K = 8 step; issued by a single thread.
__device__ __forceinline__ void tc_mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

// The mbarrier completes one phase when every MMA issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// Bounded wait (at most `limit` polls) for the phase with the given parity; false
// if it did not complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit = kTcWaitLimit) {
    for (uint32_t it = 0; it < limit; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// Bulk asynchronous copies (the TMA's untiled form) from global to shared memory,
// completion signalled on an mbarrier as transaction bytes.  One thread announces
// the bytes of all the copies (its arrival, before any copy is issued); then any
// thread issues copies of `bytes` contiguous bytes (both addresses 16-byte aligned,
// bytes a multiple of 16).
__device__ __forceinline__ void bulk_expect(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    bulk_expect(bar, bytes);
    bulk_copy(dst, src, bytes, bar);
}

// Warp-collective: 32 consecutive fp32 columns of this warp's 32 lanes (lane i of
// the warp gets row (taddr lane) + i).  Completes before returning.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace ttemb
