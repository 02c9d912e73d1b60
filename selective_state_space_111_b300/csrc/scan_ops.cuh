// scan_ops.cuh -- device helpers shared by the scan kernels (sm_103a).
//
// Packed fp32 pairs (the f32x2 FMA/MUL forms), MUFU approximations of 2^x,
// log2 x and 1/x, cp.async / bulk-copy / mbarrier wrappers, I/O conversions,
// softplus and the SiLU gate.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr int kMaxN = 16;      // states per channel held by the kernels
// Walk steps per chunk of the 16-state backward scan: the forward pass
// stores the state before every kStateChunk-th walk step for it.
#ifndef SSM_BWD16_T
#define SSM_BWD16_T 8
#endif
constexpr int kStateChunk = SSM_BWD16_T;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

typedef unsigned long long f2;  // two fp32 in one 64-bit register pair

// compile-time flag passed to generic lambdas (selects a specialised body)
template <bool V> struct BoolC {
    static constexpr bool value = V;
};

__device__ __forceinline__ f2 pk(float a, float b) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk(f2 v, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// .ca: through L1, so the CTA's own earlier stores to the workspace are seen
__device__ __forceinline__ void cp_async16_ca(void *smem, const void *gmem) {
    unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
template <typename IO> __device__ __forceinline__ IO from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ __half from_f32<__half>(float x) {
    return __float2half_rn(x);
}

// softplus and the SiLU gate.  fp32 I/O uses the accurate library functions;
// bf16 and fp16 I/O use the MUFU forms (ex2 / lg2 / rcp), whose relative
// error (about 2e-4 on delta for delta near 1e-3, far less elsewhere) is
// below the 16-bit output rounding.
template <typename IO> __device__ __forceinline__ float softplus_f(float x);
template <> __device__ __forceinline__ float softplus_f<float>(float x) {
    return x > 0.f ? x + log1pf(expf(-x)) : log1pf(expf(x));
}
template <> __device__ __forceinline__ float softplus_f<__nv_bfloat16>(float x) {
    // max(x, 0) + ln(1 + e^{-|x|}): never overflows
    float e = ex2_approx(-fabsf(x) * kLog2e);
    return fmaf(kLn2, lg2_approx(1.f + e), fmaxf(x, 0.f));
}
template <typename IO> __device__ __forceinline__ float silu_f(float z);
template <> __device__ __forceinline__ float silu_f<float>(float z) {
    return z / (1.f + expf(-z));
}
template <> __device__ __forceinline__ float silu_f<__nv_bfloat16>(float z) {
    return z * rcp_approx(1.f + ex2_approx(-z * kLog2e));
}
template <> __device__ __forceinline__ float softplus_f<__half>(float x) {
    return softplus_f<__nv_bfloat16>(x);
}
template <> __device__ __forceinline__ float silu_f<__half>(float z) {
    return silu_f<__nv_bfloat16>(z);
}


// ---- index checks of the debug build
// Built with SSM_DEBUG_BOUNDS, every global access and bulk copy of the
// forward path first checks its element offset against the extent of the
// tensor it addresses; an offset outside it sets bit 1 of the status word
// (ssm_get_status then reports SSM_ERR_BOUNDS) and the access is skipped (a
// load gives 0).  The product build compiles the checks away.
#ifdef SSM_DEBUG_BOUNDS
__device__ __forceinline__ bool dbg_in(long long i, long long n, unsigned *status) {
    if (i >= 0 && i < n) return true;
    if (status != nullptr) atomicOr(status, 2u);
    return false;
}
#define SSM_IN(i, n, status) ::ssm::dbg_in((long long)(i), (long long)(n), (status))
#else
#define SSM_IN(i, n, status) true
#endif

// ---- mbarrier and 1-D bulk copy (TMA) helpers
__device__ __forceinline__ unsigned smem_addr(const void *p) {
    return (unsigned)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
// Make initialised barriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
// Announce `bytes` more transaction bytes for the current phase (no arrival).
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Order this thread's earlier generic-proxy global stores before later
// async-proxy (bulk copy) reads of the same addresses.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// try_wait with a suspend-time hint: a thread whose phase is not complete
// sleeps in hardware (up to the hint, 100 us) instead of spinning, so
// waiting warps leave the issue slots to the others.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(100000u)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait for the phase with parity `parity` to complete: try_wait
// suspends the thread in hardware until the phase completes or a short
// system time limit passes, and the loop gives up after about two seconds
// of wall time.  Returns false on giving up (the caller reports a timeout;
// nothing in this library waits forever).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, unsigned parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > 2000000000ull) return false;
    }
}
// Global -> shared bulk copy of `bytes` (multiple of 16; both addresses
// 16-byte aligned), completing on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

}  // namespace ssm
