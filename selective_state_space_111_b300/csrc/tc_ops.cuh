// tc_ops.cuh -- tcgen05 (5th-generation tensor core) helpers for sm_103a:
// shared-memory operand descriptors, the kind::f16 MMA issued by one thread
// with its accumulator in tensor memory (TMEM), commit to an mbarrier, TMEM
// allocation and loads.  One CTA per MMA (cta_group::1), operands K-major
// without swizzle.
#pragma once

#include <type_traits>

#include "scan_ops.cuh"

namespace ssm {

// ---- tcgen05 (5th-generation tensor core) helpers: one CTA (cta_group::1)
// Shared-memory matrix descriptor of an operand without swizzle, in 8 x
// 16-byte core matrices (PTX ISA, tcgen05 shared memory descriptor: start
// address, leading and stride byte offsets in 16-byte units, descriptor
// version 1, base offset 0, layout type 0 = no swizzle).  K-major: a core
// matrix is 8 rows x 8 consecutive k; `lbo` bytes between core matrices
// adjacent along K, `sbo` bytes between 8-row groups.  MN-major: a core
// matrix is 8 k x 8 consecutive rows; `lbo` bytes between groups of 8 k,
// `sbo` bytes between groups of 8 rows.
__device__ __forceinline__ unsigned long long tc_desc(unsigned saddr, unsigned lbo, unsigned sbo) {
    return (unsigned long long)((saddr >> 4) & 0x3FFF) |
           ((unsigned long long)((lbo >> 4) & 0x3FFF) << 16) |
           ((unsigned long long)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}
// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, A and
// B of the same 16-bit type (bf16: 1, f16: 0), B K-major, A K-major or
// (a_mn) MN-major, M x N.
template <typename IO>
__host__ __device__ constexpr unsigned tc_idesc(int M, int N, bool a_mn = false) {
    return (1u << 4) | ((sizeof(IO) == 2 && !std::is_same<IO, __half>::value ? 1u : 0u) << 7) |
           ((sizeof(IO) == 2 && !std::is_same<IO, __half>::value ? 1u : 0u) << 10) |
           ((a_mn ? 1u : 0u) << 15) | ((unsigned)(N >> 3) << 17) | ((unsigned)(M >> 4) << 24);
}
// D[tmem] (+)= A * B^T for one K step of 16, issued by one thread
__device__ __forceinline__ void tc_mma(unsigned tmem, unsigned long long a, unsigned long long b,
                                       unsigned idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}
// the mbarrier completes one phase when every mma this thread issued before
// has finished
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_addr(bar)) : "memory");
}
// TMEM allocation of `cols` columns (a power of two >= 32) by one whole
// warp; the address lands in *slot
__device__ __forceinline__ void tc_alloc(unsigned *slot, unsigned cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_addr(slot)), "r"(cols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(unsigned taddr, unsigned cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// order this thread's generic-proxy shared-memory writes before later
// async-proxy (tensor core) reads
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 16 consecutive fp32 columns of this warp's 32 TMEM lanes (lane = thread)
__device__ __forceinline__ void tc_ld16(unsigned taddr, float (&v)[16]) {
    unsigned r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace ssm
