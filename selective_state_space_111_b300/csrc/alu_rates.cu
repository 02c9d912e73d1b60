// alu_rates.cu -- throughput microbenchmark of the three instruction kinds
// the selective scan's element update is made of (sm_103a): scalar fp32
// FMA, packed fp32x2 FMA and the MUFU 2^x approximation.  It supports the
// arithmetic roof the benchmark reports for the scan kernel (updates per SM
// per clock = min(FMA lanes / 4 operations, MUFU lanes / 1 exponential));
// it is built into its own small library, separate from libssm_scan.so,
// and only the benchmark's --alu-rates option loads it.
//
// Each kernel runs 8 independent dependency chains per thread, 256 threads
// per CTA and 4 CTAs per SM (32 warps per SM), long enough that launch
// overhead is negligible, and reports cycles from the SM's clock64 counter,
// so the result is per SM clock whatever the clock frequency.
#include <cuda_runtime.h>

namespace {

typedef unsigned long long f2;
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
    asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 16 x 8 dependent scalar FMAs per iteration
__global__ void rate_ffma(float *sink, int iters, long long *cyc) {
    float a[8];
    for (int i = 0; i < 8; ++i) a[i] = threadIdx.x * 1e-3f + i;
    const long long t0 = clock64();
    for (int k = 0; k < iters; ++k)
#pragma unroll
        for (int r = 0; r < 16; ++r)
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = fmaf(a[i], 0.9999f, 1e-4f);
    const long long t1 = clock64();
    float s = 0.f;
    for (int i = 0; i < 8; ++i) s += a[i];
    if (s == 1.2345f) sink[0] = s;
    if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// 8 x 8 dependent packed FMAs (two lanes each) per iteration
__global__ void rate_ffma2(float *sink, int iters, long long *cyc) {
    f2 a[8];
    for (int i = 0; i < 8; ++i) a[i] = pk(threadIdx.x * 1e-3f + i, 0.5f * i);
    const f2 m = pk(0.9999f, 0.9998f), c = pk(1e-4f, 2e-4f);
    const long long t0 = clock64();
    for (int k = 0; k < iters; ++k)
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = fma2(a[i], m, c);
    const long long t1 = clock64();
    float s = 0.f;
    for (int i = 0; i < 8; ++i) {
        float x, y;
        upk(a[i], x, y);
        s += x + y;
    }
    if (s == 1.2345f) sink[0] = s;
    if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// 16 x 8 dependent MUFU 2^x per iteration (each followed by one FADD so the
// argument stays bounded; the FADDs run on the FMA pipe, not the MUFU one)
__global__ void rate_ex2(float *sink, int iters, long long *cyc) {
    float a[8];
    for (int i = 0; i < 8; ++i) a[i] = -(threadIdx.x * 1e-3f + i * 1e-2f);
    const long long t0 = clock64();
    for (int k = 0; k < iters; ++k)
#pragma unroll
        for (int r = 0; r < 16; ++r)
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = ex2(a[i]) - 1.0f;
    const long long t1 = clock64();
    float s = 0.f;
    for (int i = 0; i < 8; ++i) s += a[i];
    if (s == 1.2345f) sink[0] = s;
    if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

}  // namespace

// Measures the three rates on the current device: out[0] scalar FMA,
// out[1] packed FMA (counting both lanes), out[2] MUFU 2^x -- each in
// lane operations per SM per SM clock (the slowest CTA's cycle count).
// Returns 0, or a CUDA error code.  Allocates (and frees) its own small
// device buffers.
extern "C" __attribute__((visibility("default"))) int ssm_alu_rates(double *out) {
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    const int threads = 256, per_sm = 4, grid = nsm * per_sm, iters = 2000;
    float *sink = nullptr;
    long long *cyc = nullptr;
    if (cudaMalloc(&sink, 64) != cudaSuccess) return 2;
    if (cudaMalloc(&cyc, grid * sizeof(long long)) != cudaSuccess) {
        cudaFree(sink);
        return 2;
    }
    long long *h = new long long[grid];
    void (*kern[3])(float *, int, long long *) = {rate_ffma, rate_ffma2, rate_ex2};
    const double ops_per_iter[3] = {16.0 * 8, 8.0 * 8 * 2, 16.0 * 8};
    int err = 0;
    for (int k = 0; k < 3 && !err; ++k) {
        kern[k]<<<grid, threads>>>(sink, 10, cyc);          // warm-up
        kern[k]<<<grid, threads>>>(sink, iters, cyc);
        if (cudaDeviceSynchronize() != cudaSuccess ||
            cudaMemcpy(h, cyc, grid * sizeof(long long), cudaMemcpyDeviceToHost) != cudaSuccess) {
            err = 3;
            break;
        }
        long long mx = 1;
        for (int i = 0; i < grid; ++i) mx = h[i] > mx ? h[i] : mx;
        out[k] = (double)grid * threads * iters * ops_per_iter[k] / ((double)nsm * mx);
    }
    delete[] h;
    cudaFree(sink);
    cudaFree(cyc);
    return err;
}
