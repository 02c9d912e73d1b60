// prologue_kernel.cuh -- the steps that feed the scan (sm_103a), one direction:
//   u  = silu(causal depthwise conv1d(x) + bias)      (conv_silu_kernel)
//   [dt_low; B; C] = W_x @ u,  dt = W_dt @ dt_low     (proj_kernel, twice)
// as in "Vision Mamba实战" section 2.1 and "从Transformer到Mamba" section 2.1
// (conv1d, x_proj = Linear(d_inner -> dt_rank + 2 d_state), dt_proj =
// Linear(dt_rank -> d_inner)) and "VMamba的SS2D模块详解" section 3.1 (the
// split into dt, B, C).  The projections write straight into the scan's
// layouts: B, C as [B, N, L] rows, dt as [B, D, L] rows (L contiguous), so
// nothing is transposed.  reverse = 1 runs the direction on the time-
// reversed input (v2's backward branch) and writes every output in that
// branch's scan order.
#pragma once

#include "scan_ops.cuh"

namespace ssm {
namespace pro {

// u[b][d][t] = silu(bias[d] + sum_k w[d][k] * xs[t - (K-1) + k]), xs = x or
// x reversed in time, zero before the start.  One thread per output.
template <typename IO>
__global__ void __launch_bounds__(256)
conv_silu_kernel(const IO *__restrict__ x, const float *__restrict__ w,
                 const float *__restrict__ bias, IO *__restrict__ u, int D, int L, int K,
                 int reverse) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const int d = blockIdx.y, b = blockIdx.z;
    if (t >= L) return;
    const long long row = ((long long)b * D + d) * L;
    float acc = bias ? bias[d] : 0.f;
    for (int k = 0; k < K; ++k) {
        const int ts = t - (K - 1) + k;
        if (ts >= 0) acc = fmaf(w[d * K + k], to_f32(x[row + (reverse ? L - 1 - ts : ts)]), acc);
    }
    u[row + t] = from_f32<IO>(acc / (1.f + expf(-acc)));
}

// Output rows [0, M) of one projection go to up to three destinations:
// rows [r0, r1) -> dst0, [r1, r2) -> dst1, [r2, M) -> dst2, each [B][rows][L]
// in its own dtype (fp32 for the internal dt_low, the I/O dtype otherwise).
struct ProjOut {
    void *dst[3];
    int f32[3];        // 1: fp32 destination
    int r[4];          // row boundaries: r[0] = 0 <= r[1] <= r[2] <= r[3] = M
};

constexpr int BM = 64, BN = 64, BK = 16;

// out[b][m][t] = sum_k W[m][k] * in[b][k][t]: W fp32 [M][K], in [B][K][L]
// (I/O dtype or fp32).  Tile 64 x 64 per CTA, 16-deep K slices through
// shared memory, 4 x 4 outputs per thread (fp32 FMA).
template <typename IN, typename IO>
__global__ void __launch_bounds__(256)
proj_kernel(const float *__restrict__ W, const IN *__restrict__ in, int M, int K, int L,
            ProjOut out) {
    __shared__ float sW[BK][BM + 4];
    __shared__ __align__(16) float sI[BK][BN + 4];
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int t0 = blockIdx.x * BN, m0 = blockIdx.y * BM, b = blockIdx.z;
    const IN *inb = in + (long long)b * K * L;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
        for (int r = 0; r < (BM * BK) / 256; ++r) {
            const int i = tid + r * 256, mm = i / BK, kk = i % BK;
            const int m = m0 + mm, k = k0 + kk;
            sW[kk][mm] = (m < M && k < K) ? W[(long long)m * K + k] : 0.f;
        }
#pragma unroll
        for (int r = 0; r < (BK * BN) / 256; ++r) {
            const int i = tid + r * 256, kk = i / BN, tt = i % BN;
            const int k = k0 + kk, t = t0 + tt;
            sI[kk][tt] = (k < K && t < L) ? to_f32(inb[(long long)k * L + t]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float wv[4], iv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) wv[i] = sW[kk][ty * 4 + i];
            const float4 v = *(const float4 *)&sI[kk][tx * 4];
            iv[0] = v.x;
            iv[1] = v.y;
            iv[2] = v.z;
            iv[3] = v.w;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(wv[i], iv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
        int s = 0;
        while (m >= out.r[s + 1]) ++s;
        const int rows = out.r[s + 1] - out.r[s], mr = m - out.r[s];
        const long long o = ((long long)b * rows + mr) * L;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int t = t0 + tx * 4 + j;
            if (t >= L) continue;
            if (out.f32[s]) ((float *)out.dst[s])[o + t] = acc[i][j];
            else ((IO *)out.dst[s])[o + t] = from_f32<IO>(acc[i][j]);
        }
    }
}

}  // namespace pro
}  // namespace ssm
