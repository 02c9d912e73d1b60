// prologue_kernel.cuh -- the steps that feed the scan (sm_103a), one direction:
//   u  = silu(causal depthwise conv1d(x) + bias)      (conv_silu_kernel)
//   [dt_low; B; C] = W_x @ u                          (xproj_mma_kernel / proj_*)
//   dt = W_dt @ dt_low                     (dtproj_tc_kernel / dtproj_kernel / proj_*)
// as in "Vision Mamba实战" section 2.1 and "从Transformer到Mamba" section 2.1
// (conv1d, x_proj = Linear(d_inner -> dt_rank + 2 d_state), dt_proj =
// Linear(dt_rank -> d_inner)) and "VMamba的SS2D模块详解" section 3.1 (the
// split into dt, B, C).  The projections write straight into the scan's
// layouts: B, C as [B, N, L] rows, dt as [B, D, L] rows (L contiguous), so
// nothing is transposed.  reverse = 1 runs the direction on the time-
// reversed input (v2's backward branch) and writes every output in that
// branch's scan order.
#pragma once

#include <cuda.h>

#include "scan_ops.cuh"
#include "tc_ops.cuh"

namespace ssm {
namespace pro {

// u[b][d][t] = silu(bias[d] + sum_k w[d][k] * xs[t - (K-1) + k]), xs = x or
// x reversed in time, zero before the start.  A CTA covers CONV_T positions
// of one channel: it stages xs over them plus the K - 1 halo in shared
// memory (coalesced reads, in reverse order for reverse = 1, every load in
// flight before the stores).  KT = 4 (compile time, the usual taps): each
// thread makes 4 consecutive outputs from the 8 values two 16-byte shared
// loads give, puts them back in shared memory, and the CTA stores along
// positions (coalesced); KT = 0 (any K <= 8): CONV_T / 256 outputs per
// thread, consecutive threads on consecutive positions.
constexpr int CONV_T = 2048, CONV_S = CONV_T + 8, CONV_V = (CONV_S + 255) / 256;
template <typename IO, int KT>
__global__ void __launch_bounds__(256)
conv_silu_kernel(const IO *__restrict__ x, const float *__restrict__ w,
                 const float *__restrict__ bias, IO *__restrict__ u, int D, int L, int K,
                 int reverse) {
    __shared__ __align__(16) float sx[CONV_S];  // sx[i] = xs[t0 - (K-1) + i], K <= 8
    const int t0 = blockIdx.x * CONV_T;
    const int d = blockIdx.y, b = blockIdx.z;
    const long long row = ((long long)b * D + d) * L;
    const int n_in = min(CONV_T, L - t0) + K - 1;
    float v[CONV_V];
#pragma unroll
    for (int j = 0; j < CONV_V; ++j) {
        const int i = j * 256 + threadIdx.x, ts = t0 - (K - 1) + i;
        v[j] = (i < n_in && ts >= 0) ? to_f32(x[row + (reverse ? L - 1 - ts : ts)]) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < CONV_V; ++j) {
        const int i = j * 256 + threadIdx.x;
        if (i < CONV_S) sx[i] = v[j];
    }
    constexpr int KM = KT > 0 ? KT : 8;
    float wk[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) wk[k] = (KT > 0 || k < K) ? w[d * K + k] : 0.f;
    const float bv = bias ? bias[d] : 0.f;
    __syncthreads();
    if constexpr (KT == 4) {
        // outputs go back to shared memory (after everyone has read sx),
        // then out along positions: coalesced stores
        float res[CONV_T / 1024][4];
#pragma unroll
        for (int j = 0; j < CONV_T / 1024; ++j) {
            const int tt = (j * 256 + threadIdx.x) * 4;
            const float4 lo = *(const float4 *)&sx[tt];
            const float4 hi = *(const float4 *)&sx[tt + 4];
            const float win[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
            for (int o = 0; o < 4; ++o) {
                float acc = bv;
#pragma unroll
                for (int k = 0; k < 4; ++k) acc = fmaf(wk[k], win[o + k], acc);
                res[j][o] = silu_f<IO>(acc);
            }
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < CONV_T / 1024; ++j)
            *(float4 *)&sx[(j * 256 + threadIdx.x) * 4] =
                make_float4(res[j][0], res[j][1], res[j][2], res[j][3]);
        __syncthreads();
#pragma unroll
        for (int j = 0; j < CONV_T / 256; ++j) {
            const int tt = j * 256 + threadIdx.x, t = t0 + tt;
            if (t < L) u[row + t] = from_f32<IO>(sx[tt]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < CONV_T / 256; ++j) {
            const int tt = j * 256 + threadIdx.x, t = t0 + tt;
            if (t >= L) break;
            float acc = bv;
#pragma unroll
            for (int k = 0; k < KM; ++k)
                if (k < K) acc = fmaf(wk[k], sx[tt + k], acc);
            u[row + t] = from_f32<IO>(silu_f<IO>(acc));
        }
    }
}

// The same for 16-bit I/O and K = 4 with 16-byte global accesses.  Rows of
// odd length put a row's elements at any 2-byte offset, so a CTA reads the
// 16-byte-aligned chunks that cover its window (reading at most 14 bytes
// outside it, inside the same aligned chunk) into shared memory and indexes
// them with the window's shift; it writes u the same way: whole aligned
// chunks of its CONV_T outputs as 16-byte stores, the partial chunks at
// either end element by element (nothing outside the segment is written).
// One load and one store instruction per 8 elements instead of 8 each.
constexpr int CV_CH = (CONV_T + 3 + 7) / 8 + 2;      // chunks of 8 covering a window
template <typename IO>
__global__ void __launch_bounds__(256)
conv_silu_vec_kernel(const IO *__restrict__ x, const float *__restrict__ w,
                     const float *__restrict__ bias, IO *__restrict__ u, int D, int L,
                     int reverse) {
    static_assert(sizeof(IO) == 2, "16-bit I/O");
    __shared__ __align__(16) IO sraw[CV_CH * 8];
    __shared__ __align__(16) float sx[CONV_S];   // sx[i] = xs[t0 - 3 + i]
    __shared__ __align__(16) IO sout[CONV_T + 8];
    const int t0 = blockIdx.x * CONV_T;
    const int d = blockIdx.y, b = blockIdx.z;
    const long long row = ((long long)b * D + d) * L;
    const int n_out = min(CONV_T, L - t0), n_in = n_out + 3;
    // the xs the window needs, [ts_lo, ts_hi), and where they sit in x
    const int ts_lo = max(t0 - 3, 0), ts_hi = t0 + n_out;
    const long long e_lo = reverse ? row + L - ts_hi : row + ts_lo;
    const long long e_hi = reverse ? row + L - ts_lo : row + ts_hi;
    const uintptr_t a_lo = (uintptr_t)(x + e_lo) & ~(uintptr_t)15;
    const uintptr_t a_hi = ((uintptr_t)(x + e_hi) + 15) & ~(uintptr_t)15;
    const int shift = (int)(((uintptr_t)(x + e_lo) - a_lo) / sizeof(IO));
    const int nchunk = (int)((a_hi - a_lo) / 16);
    {
        uint4 rv[(CV_CH + 255) / 256];
#pragma unroll
        for (int j = 0; j < (CV_CH + 255) / 256; ++j) {
            const int c = threadIdx.x + j * 256;
            if (c < nchunk) rv[j] = *(const uint4 *)(a_lo + 16 * (uintptr_t)c);
        }
#pragma unroll
        for (int j = 0; j < (CV_CH + 255) / 256; ++j) {
            const int c = threadIdx.x + j * 256;
            if (c < nchunk) *(uint4 *)&sraw[8 * c] = rv[j];
        }
    }
    float wk[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) wk[k] = w[d * 4 + k];
    const float bv = bias ? bias[d] : 0.f;
    __syncthreads();
    // xs[t0 - 3 + i] sits at sraw[base + step * i]
    const int step = reverse ? -1 : 1;
    const int base = reverse ? shift + ts_hi - 1 - (t0 - 3) : shift + (t0 - 3) - ts_lo;
#pragma unroll
    for (int j = 0; j < CONV_V; ++j) {
        const int i = j * 256 + threadIdx.x, ts = t0 - 3 + i;
        if (i < CONV_S) sx[i] = (i < n_in && ts >= 0) ? to_f32(sraw[base + step * i]) : 0.f;
    }
    __syncthreads();
    float res[CONV_T / 1024][4];
#pragma unroll
    for (int j = 0; j < CONV_T / 1024; ++j) {
        const int tt = (j * 256 + threadIdx.x) * 4;
        const float4 lo = *(const float4 *)&sx[tt];
        const float4 hi = *(const float4 *)&sx[tt + 4];
        const float win[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int o = 0; o < 4; ++o) {
            float acc = bv;
#pragma unroll
            for (int k = 0; k < 4; ++k) acc = fmaf(wk[k], win[o + k], acc);
            res[j][o] = silu_f<IO>(acc);
        }
    }
    // outputs as I/O values, shifted so that u's 16-byte chunks are
    // 8-element-aligned rows of sout: element tt at sout[off + tt]
    IO *q = u + row + t0;
    const int off = (int)(((uintptr_t)q & 15) / sizeof(IO));
#pragma unroll
    for (int j = 0; j < CONV_T / 1024; ++j) {
        const int tt = (j * 256 + threadIdx.x) * 4;
#pragma unroll
        for (int o = 0; o < 4; ++o) sout[off + tt + o] = from_f32<IO>(res[j][o]);
    }
    __syncthreads();
    // u[row + t0 + tt], tt < n_out: whole aligned chunks, then the ends
    const uintptr_t q_lo = (uintptr_t)q, q_hi = (uintptr_t)(q + n_out);
    const uintptr_t c_lo = (q_lo + 15) & ~(uintptr_t)15, c_hi = q_hi & ~(uintptr_t)15;
    const int head = (int)((min(c_lo, q_hi) - q_lo) / sizeof(IO));
    const int nfull = c_hi > c_lo ? (int)((c_hi - c_lo) / 16) : 0;
    const int m0 = off > 0 ? 1 : 0;          // sout row of the first whole chunk
#pragma unroll
    for (int j = 0; j < (CONV_T / 8 + 255) / 256; ++j) {
        const int c = threadIdx.x + j * 256;
        if (c < nfull)
            *(uint4 *)(c_lo + 16 * (uintptr_t)c) = *(const uint4 *)&sout[8 * (m0 + c)];
    }
    // the partial chunks: [0, head) and [head + 8 nfull, n_out)
    const int tail0 = head + 8 * nfull;
    if (threadIdx.x < head) q[threadIdx.x] = sout[off + threadIdx.x];
    else if (threadIdx.x >= 32 && threadIdx.x - 32 < n_out - tail0) {
        const int tt = tail0 + threadIdx.x - 32;
        q[tt] = sout[off + tt];
    }
}

// SS2D's conv2d ("VMamba的SS2D模块详解" section 2.1): u[b][d][h][w] =
// act(bias[d] + sum_{i,j} w[d][i][j] x[b][d][h+i-P][w+j-P]), P = (Kc-1)/2,
// zero outside the map, act = SiLU or identity.  A CTA covers RB rows of
// one channel's map: it stages rows h0-P .. h0+RB+P-1, zero-padded by P
// columns on the left and to the row stride WS on the right, in shared
// memory (warp by warp along the rows: coalesced; for rows of at most 64
// values eight rows per warp at a time, every load in flight).  KC = 3
// (compile time):
// a thread makes 4 consecutive outputs of a row from a 3 x 8 window read
// with six 16-byte shared loads (WS is a multiple of 4 floats); KC = 0
// (any odd Kc <= 7): warp r makes rows r, r + 8, ... one output per lane.
__host__ __device__ constexpr int conv2d_ws(int W, int Kc) {
    return ((W + 3) / 4) * 4 + ((Kc - 1) / 2) * 2 + 4 - (((Kc - 1) / 2) * 2) % 4;
}
template <typename IO, int KC>
__global__ void __launch_bounds__(256)
conv2d_act_kernel(const IO *__restrict__ x, const float *__restrict__ w,
                  const float *__restrict__ bias, IO *__restrict__ u, int D, int H, int W,
                  int Kc, int RB, int act) {
    extern __shared__ __align__(16) float c2_smem[];        // [RB + 2P][WS]
    const int P = (Kc - 1) / 2, WS = conv2d_ws(W, Kc);
    const int h0 = blockIdx.x * RB, d = blockIdx.y, b = blockIdx.z;
    const int rb = min(RB, H - h0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const IO *xm = x + ((long long)b * D + d) * H * W;
    if (WS <= 64) {
        // rows of at most 64: eight rows per warp at a time, all 16 loads of
        // a lane in flight before the shared stores
        for (int r0 = warp; r0 < rb + 2 * P; r0 += 64) {
            float v[8][2];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int r = r0 + 8 * k, h = h0 - P + r;
                const bool hin = r < rb + 2 * P && h >= 0 && h < H;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int ww = lane + 32 * q - P;
                    v[k][q] = (hin && ww >= 0 && ww < W) ? to_f32(xm[(long long)h * W + ww]) : 0.f;
                }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int r = r0 + 8 * k;
#pragma unroll
                for (int q = 0; q < 2; ++q)
                    if (r < rb + 2 * P && lane + 32 * q < WS) c2_smem[r * WS + lane + 32 * q] = v[k][q];
            }
        }
    } else {
        for (int r = warp; r < rb + 2 * P; r += 8) {
            const int h = h0 - P + r;
            const bool hin = h >= 0 && h < H;
            const IO *xr = xm + (long long)(hin ? h : 0) * W;
            float *dst = c2_smem + r * WS;
            for (int c0 = lane; c0 < WS; c0 += 64) {
                float v[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int ww = c0 + 32 * q - P;
                    v[q] = (hin && ww >= 0 && ww < W) ? to_f32(xr[ww]) : 0.f;
                }
#pragma unroll
                for (int q = 0; q < 2; ++q)
                    if (c0 + 32 * q < WS) dst[c0 + 32 * q] = v[q];
            }
        }
    }
    constexpr int KM = KC > 0 ? KC : 7;
    float wk[KM * KM];
#pragma unroll
    for (int i = 0; i < KM; ++i)
#pragma unroll
        for (int j = 0; j < KM; ++j)
            wk[i * KM + j] = (KC > 0 || (i < Kc && j < Kc)) ? w[(d * Kc + i) * Kc + j] : 0.f;
    const float bv = bias ? bias[d] : 0.f;
    __syncthreads();
    IO *um = u + ((long long)b * D + d) * H * W;
    if constexpr (KC == 3) {
        const int U = (W + 3) / 4;                              // 4-output units per row
        for (int q = threadIdx.x; q < rb * U; q += 256) {
            const int r = q / U, c = (q - r * U) * 4;
            float win[3][8];
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                const float4 lo = *(const float4 *)&c2_smem[(r + i) * WS + c];
                const float4 hi = *(const float4 *)&c2_smem[(r + i) * WS + c + 4];
                win[i][0] = lo.x;
                win[i][1] = lo.y;
                win[i][2] = lo.z;
                win[i][3] = lo.w;
                win[i][4] = hi.x;
                win[i][5] = hi.y;
                win[i][6] = hi.z;
                win[i][7] = hi.w;
            }
            IO *orow = um + (long long)(h0 + r) * W;
#pragma unroll
            for (int o = 0; o < 4; ++o) {
                float acc = bv;
#pragma unroll
                for (int i = 0; i < 3; ++i)
#pragma unroll
                    for (int j = 0; j < 3; ++j) acc = fmaf(wk[i * 3 + j], win[i][o + j], acc);
                if (c + o < W) orow[c + o] = from_f32<IO>(act ? silu_f<IO>(acc) : acc);
            }
        }
    } else {
        for (int r = warp; r < rb; r += 8) {
            for (int c = lane; c < W; c += 32) {
                float acc = bv;
#pragma unroll
                for (int i = 0; i < KM; ++i)
#pragma unroll
                    for (int j = 0; j < KM; ++j)
                        if (i < Kc && j < Kc)
                            acc = fmaf(wk[i * KM + j], c2_smem[(r + i) * WS + c + j], acc);
                um[(long long)(h0 + r) * W + c] = from_f32<IO>(act ? silu_f<IO>(acc) : acc);
            }
        }
    }
}

// Output rows [0, M) of one projection go to up to three destinations:
// rows [r0, r1) -> dst0, [r1, r2) -> dst1, [r2, M) -> dst2, each
// [B][rows][L] with batch stride bstride[s] elements, in its own dtype (fp32
// for the internal dt_low, the I/O dtype otherwise).  order >= 0 (SS2D):
// the input positions are an H x W map in row-major order and each output
// goes to its position in scan direction `order` ("VMamba的SS2D模块详解"
// section 2.2: 0 row-major, 1 column-major, 2 and 3 their reversals).
struct ProjOut {
    void *dst[3];
    int f32[3];        // 1: fp32 destination
    int r[4];          // row boundaries: r[0] = 0 <= r[1] <= r[2] <= r[3] = M
    long long bstride[3];
    int order, H, W;   // order < 0: positions are stored as they are
};

// scan position of map position p (row-major) in direction k
__device__ __forceinline__ int scan_pos(int k, int p, int H, int W) {
    if (k <= 0) return p;
    const int L = H * W;
    if (k == 2) return L - 1 - p;
    const int h = p / W, w = p - h * W, t = w * H + h;    // column-major
    return k == 1 ? t : L - 1 - t;
}

// stores output row m of batch element b at position t of its row, t
// already in the destination's order
template <typename IO>
__device__ __forceinline__ void proj_store_at(const ProjOut &out, int b, int m, int t, int L,
                                              float v) {
    int s = 0;
    while (m >= out.r[s + 1]) ++s;
    const long long o = (long long)b * out.bstride[s] + (long long)(m - out.r[s]) * L + t;
    if (out.f32[s]) ((float *)out.dst[s])[o] = v;
    else ((IO *)out.dst[s])[o] = from_f32<IO>(v);
}

// stores output row m, position t of batch element b
template <typename IO>
__device__ __forceinline__ void proj_store(const ProjOut &out, int b, int m, int t, int L,
                                           float v) {
    int s = 0;
    while (m >= out.r[s + 1]) ++s;
    const long long o = (long long)b * out.bstride[s] + (long long)(m - out.r[s]) * L +
                        scan_pos(out.order, t, out.H, out.W);
    if (out.f32[s]) ((float *)out.dst[s])[o] = v;
    else ((IO *)out.dst[s])[o] = from_f32<IO>(v);
}

constexpr int BM = 64, BN = 64, BK = 16;

// out[b][m][t] = sum_k W[m][k] * in[b][k][t]: W fp32 [M][K], in [B][K][L]
// with batch stride ib (I/O dtype or fp32).  Tile 64 x 64 per CTA, 16-deep K slices through
// shared memory, 4 x 4 outputs per thread (fp32 FMA).
template <typename IN, typename IO, typename WT = float>
__global__ void __launch_bounds__(256)
proj_kernel(const WT *__restrict__ W, const IN *__restrict__ in, int M, int K, int L,
            long long ib, ProjOut out) {
    __shared__ float sW[BK][BM + 4];
    __shared__ __align__(16) float sI[BK][BN + 4];
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int t0 = blockIdx.x * BN, m0 = blockIdx.y * BM, b = blockIdx.z;
    const IN *inb = in + (long long)b * ib;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
        for (int r = 0; r < (BM * BK) / 256; ++r) {
            const int i = tid + r * 256, mm = i / BK, kk = i % BK;
            const int m = m0 + mm, k = k0 + kk;
            sW[kk][mm] = (m < M && k < K) ? to_f32(W[(long long)m * K + k]) : 0.f;
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
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int t = t0 + tx * 4 + j;
            if (t < L) proj_store<IO>(out, b, m, t, L, acc[i][j]);
        }
    }
}

// ---- tensor-core projection (bf16 / fp16 I/O): mma.sync m16n8k16, fp32
// accumulation.  CTA tile 64 (rows) x 64 (positions), K in slices of 32;
// 8 warps, warp w computes rows 16 (w % 4) .. +16 of positions 32 (w / 4)
// .. +32 (four 16 x 8 tiles).  Operands are staged in shared memory in the
// I/O type (weights converted from fp32): W as [row][k], the input
// transposed as [position][k], so every fragment register is one aligned
// 32-bit load (fragment layouts of the PTX ISA's mma.m16n8k16).
constexpr int TK = 32, TKP = TK + 8;         // K slice, padded row (bank spread)

template <typename IO> __device__ __forceinline__ void mma16816(float (&c)[4], const unsigned (&a)[4],
                                                                 const unsigned (&b)[2]);
template <> __device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&c)[4],
                                                                    const unsigned (&a)[4],
                                                                    const unsigned (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
template <> __device__ __forceinline__ void mma16816<__half>(float (&c)[4], const unsigned (&a)[4],
                                                             const unsigned (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

template <typename IN, typename IO, typename WT = float>
__global__ void __launch_bounds__(256)
proj_mma_kernel(const WT *__restrict__ W, const IN *__restrict__ in, int M, int K, int L,
                long long ib, ProjOut out) {
    __shared__ __align__(16) IO sW[BM][TKP];        // [row][k]
    __shared__ __align__(16) IO sI[BN][TKP];        // [position][k]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tg = lane & 3;
    const int wm = (warp % 4) * 16, wn = (warp / 4) * 32;
    const int t0 = blockIdx.x * BN, m0 = blockIdx.y * BM, b = blockIdx.z;
    const IN *inb = in + (long long)b * ib;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += TK) {
        // W slice: 64 x 32 (k fastest: coalesced fp32 reads)
#pragma unroll
        for (int r = 0; r < (BM * TK) / 256; ++r) {
            const int i = tid + r * 256, mm = i / TK, kk = i % TK;
            const int m = m0 + mm, k = k0 + kk;
            sW[mm][kk] = from_f32<IO>((m < M && k < K) ? to_f32(W[(long long)m * K + k]) : 0.f);
        }
        // input slice: 32 x 64 (positions fastest: coalesced), stored transposed
#pragma unroll
        for (int r = 0; r < (TK * BN) / 256; ++r) {
            const int i = tid + r * 256, kk = i / BN, tt = i % BN;
            const int k = k0 + kk, t = t0 + tt;
            sI[tt][kk] = from_f32<IO>((k < K && t < L) ? to_f32(inb[(long long)k * L + t]) : 0.f);
        }
        __syncthreads();
#pragma unroll
        for (int ks = 0; ks < TK; ks += 16) {
            unsigned a[4];
            a[0] = *(const unsigned *)&sW[wm + g][ks + 2 * tg];
            a[1] = *(const unsigned *)&sW[wm + g + 8][ks + 2 * tg];
            a[2] = *(const unsigned *)&sW[wm + g][ks + 2 * tg + 8];
            a[3] = *(const unsigned *)&sW[wm + g + 8][ks + 2 * tg + 8];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                unsigned bf[2];
                bf[0] = *(const unsigned *)&sI[wn + nt * 8 + g][ks + 2 * tg];
                bf[1] = *(const unsigned *)&sI[wn + nt * 8 + g][ks + 2 * tg + 8];
                mma16816<IO>(acc[nt], a, bf);
            }
        }
        __syncthreads();
    }
    // c0, c1: row g, positions 2tg, 2tg+1; c2, c3: row g + 8
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int m = m0 + wm + g + 8 * half;
        if (m >= M) continue;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int t = t0 + wn + nt * 8 + 2 * tg + j;
                if (t < L) proj_store<IO>(out, b, m, t, L, acc[nt][2 * half + j]);
            }
    }
}

// dt_proj with a short inner dimension (R = dt_rank <= RP, RP in {8, 16, 24,
// 32}): out[b][m][t] = sum_r W[m][r] in[b][r][t] (out's batch stride ob;
// batch element b uses weight set b mod nw, sets [M][R] one after another).  A CTA takes DTP_T
// positions (two per thread, DTP_T / 2 apart, their R inputs in registers)
// and rows [m_lo, m_hi) in chunks of 128 staged in shared memory (zero-
// padded to RP, read back as broadcast float4); stores are coalesced along
// positions.  grid.y splits the rows so that short batches still fill the
// GPU.
constexpr int DTP_T = 512, DTP_MC = 128;
template <typename IO, int RP>
__global__ void __launch_bounds__(256, 2)
dtproj_kernel(const float *__restrict__ W, const float *__restrict__ in, int M, int R, int L,
              IO *__restrict__ out, long long ob, int nw) {
    __shared__ __align__(16) float sW[DTP_MC * RP];
    const int b = blockIdx.z;
    W += (long long)(b % nw) * M * R;                        // this z group's weight set
    const int t_a = blockIdx.x * DTP_T + threadIdx.x, t_b = t_a + DTP_T / 2;
    const int per = (M + gridDim.y - 1) / gridDim.y;
    const int m_lo = blockIdx.y * per, m_hi = min(M, m_lo + per);
    float va[RP], vb[RP];
#pragma unroll
    for (int r = 0; r < RP; ++r) {
        const float *src = in + ((long long)b * R + r) * L;
        va[r] = (r < R && t_a < L) ? src[t_a] : 0.f;
        vb[r] = (r < R && t_b < L) ? src[t_b] : 0.f;
    }
    for (int m0 = m_lo; m0 < m_hi; m0 += DTP_MC) {
        const int mc = min(DTP_MC, m_hi - m0);
        __syncthreads();
        float wv[DTP_MC * RP / 256];                     // all in flight, then stored
#pragma unroll
        for (int j = 0; j < DTP_MC * RP / 256; ++j) {
            const int i = j * 256 + threadIdx.x, mm = i / RP, r = i % RP;
            wv[j] = (mm < mc && r < R) ? W[(long long)(m0 + mm) * R + r] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < DTP_MC * RP / 256; ++j) sW[j * 256 + threadIdx.x] = wv[j];
        __syncthreads();
        // two rows at a time: four independent accumulation chains
        for (int mm = 0; mm < mc; mm += 2) {
            const bool two = mm + 1 < mc;
            const float4 *w0 = (const float4 *)&sW[mm * RP];
            const float4 *w1 = (const float4 *)&sW[(two ? mm + 1 : mm) * RP];
            float a0 = 0.f, b0 = 0.f, a1 = 0.f, b1 = 0.f;
#pragma unroll
            for (int q = 0; q < RP / 4; ++q) {
                const float4 x0 = w0[q], x1 = w1[q];
                a0 = fmaf(x0.x, va[4 * q], a0);
                b0 = fmaf(x0.x, vb[4 * q], b0);
                a1 = fmaf(x1.x, va[4 * q], a1);
                b1 = fmaf(x1.x, vb[4 * q], b1);
                a0 = fmaf(x0.y, va[4 * q + 1], a0);
                b0 = fmaf(x0.y, vb[4 * q + 1], b0);
                a1 = fmaf(x1.y, va[4 * q + 1], a1);
                b1 = fmaf(x1.y, vb[4 * q + 1], b1);
                a0 = fmaf(x0.z, va[4 * q + 2], a0);
                b0 = fmaf(x0.z, vb[4 * q + 2], b0);
                a1 = fmaf(x1.z, va[4 * q + 2], a1);
                b1 = fmaf(x1.z, vb[4 * q + 2], b1);
                a0 = fmaf(x0.w, va[4 * q + 3], a0);
                b0 = fmaf(x0.w, vb[4 * q + 3], b0);
                a1 = fmaf(x1.w, va[4 * q + 3], a1);
                b1 = fmaf(x1.w, vb[4 * q + 3], b1);
            }
            IO *o = out + (long long)b * ob + (long long)(m0 + mm) * L;
            if (t_a < L) o[t_a] = from_f32<IO>(a0);
            if (t_b < L) o[t_b] = from_f32<IO>(b0);
            if (two) {
                if (t_a < L) o[L + t_a] = from_f32<IO>(a1);
                if (t_b < L) o[L + t_b] = from_f32<IO>(b1);
            }
        }
    }
}

// dt_proj on tensor cores for 16-bit I/O: out[b][m][t] = sum_r W[m][r]
// in[b][r][t] (out's batch stride ob; weight set b mod nw) with W and the fp32 dt_low rounded to tf32 (10-bit mantissa,
// below the 16-bit output's own rounding) and fp32 accumulation, mma.sync
// m16n8k8.  A CTA takes DTC_T positions and DTC_RB rows: it stages the
// input tile [RP][DTC_T] and its W rows [DTC_RB][RP] (zero-padded to RP)
// once, then for each block of 64 rows runs the mma (warp w: rows
// 16 (w % 4) .. +16, positions 64 (w / 4) .. +64) and writes the block
// through a shared fp32 tile so that the global stores run along
// positions.
constexpr int DTC_T = 128, DTC_RB = 128, DTC_OS = DTC_T + 8;
__device__ __forceinline__ unsigned to_tf32(float f) {
    unsigned r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(f));
    return r;
}
__device__ __forceinline__ void mma1688_tf32(float (&c)[4], const unsigned (&a)[4],
                                             const unsigned (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
template <int RP> constexpr size_t dtproj_tc_smem_bytes() {
    return ((size_t)DTC_RB * (RP + 4) + (size_t)RP * DTC_OS + 64 * (size_t)DTC_OS) * 4;
}
template <typename IO, int RP>
__global__ void __launch_bounds__(256)
dtproj_tc_kernel(const float *__restrict__ W, const float *__restrict__ in, int M, int R, int L,
                 IO *__restrict__ out, long long ob, int nw) {
    constexpr int WS = RP + 4, IS = DTC_OS;     // word strides: conflict-free fragment loads
    extern __shared__ __align__(16) unsigned char dtc_smem[];
    unsigned *sW = (unsigned *)dtc_smem;        // [DTC_RB][WS]
    unsigned *sI = sW + DTC_RB * WS;            // [RP][IS]
    float *sO = (float *)(sI + RP * IS);        // [64][DTC_OS]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tg = lane & 3;
    const int wm = (warp % 4) * 16, wn = (warp / 4) * 64;
    const int t0 = blockIdx.x * DTC_T, b = blockIdx.z;
    const int m_lo = blockIdx.y * DTC_RB, mc = min(DTC_RB, M - m_lo);
    W += (long long)(b % nw) * M * R;                        // this z group's weight set
    {
        float iv[RP * DTC_T / 256], wv[RP * DTC_RB / 256];
#pragma unroll
        for (int j = 0; j < RP * DTC_T / 256; ++j) {
            const int i = j * 256 + tid, r = i / DTC_T, tt = i % DTC_T, t = t0 + tt;
            iv[j] = (r < R && t < L) ? in[((long long)b * R + r) * L + t] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < RP * DTC_RB / 256; ++j) {
            const int i = j * 256 + tid, mm = i / RP, r = i % RP;
            wv[j] = (mm < mc && r < R) ? W[(long long)(m_lo + mm) * R + r] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < RP * DTC_T / 256; ++j) {
            const int i = j * 256 + tid;
            sI[(i / DTC_T) * IS + i % DTC_T] = to_tf32(iv[j]);
        }
#pragma unroll
        for (int j = 0; j < RP * DTC_RB / 256; ++j) {
            const int i = j * 256 + tid;
            sW[(i / RP) * WS + i % RP] = to_tf32(wv[j]);
        }
    }
    __syncthreads();
    for (int mb = 0; mb < mc; mb += 64) {
        float acc[8][4] = {};
#pragma unroll
        for (int ks = 0; ks < RP; ks += 8) {
            // A (row): a0 (g, tg), a1 (g + 8, tg), a2 (g, tg + 4), a3 (g + 8, tg + 4)
            const unsigned *wr = sW + (mb + wm + g) * WS + ks + tg;
            const unsigned a[4] = {wr[0], wr[8 * WS], wr[4], wr[8 * WS + 4]};
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                // B (col): b0 (k = tg, n = g), b1 (k = tg + 4, n = g)
                const unsigned *col = sI + (ks + tg) * IS + wn + nt * 8 + g;
                const unsigned bf[2] = {col[0], col[4 * IS]};
                mma1688_tf32(acc[nt], a, bf);
            }
        }
        // c0, c1: row g, positions 2tg, 2tg+1; c2, c3: row g + 8
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int half = 0; half < 2; ++half)
                *(float2 *)&sO[(wm + g + 8 * half) * DTC_OS + wn + nt * 8 + 2 * tg] =
                    make_float2(acc[nt][2 * half], acc[nt][2 * half + 1]);
        __syncthreads();
        const int rows = min(64, mc - mb);
        for (int i = tid; i < rows * DTC_T; i += 256) {
            const int m = i / DTC_T, tt = i % DTC_T, t = t0 + tt;
            if (t < L)
                out[(long long)b * ob + (long long)(m_lo + mb + m) * L + t] =
                    from_f32<IO>(sO[m * DTC_OS + tt]);
        }
        __syncthreads();
    }
}

// ---- the whole 1-D prologue of one direction in one kernel (16-bit I/O,
// K = 4 conv taps, x_proj rows M = R + 2N <= 64, dt_rank R <= RP <= 32):
//   u = silu(conv1d(x) + bias), [dt_low; B; C] = W_x u, dt = W_dt dt_low
// ("从Transformer到Mamba" section 2.1: conv1d, x_proj, dt_proj in that
// order; "VMamba的SS2D模块详解" section 3.1: the split into dt, B and C).
// A CTA takes FP_T positions (walk order) of one batch element and every
// channel, in slices of FP_KS channels:
//   * the slice's x window (FP_T + 3 positions per channel) and W_x
//     columns are fetched one slice ahead into registers (raw loads from
//     clamped in-range addresses; masks and conversion at commit);
//   * thread = (position, 8 channels): the conv + SiLU of 8 channels at one
//     position, stored to u (along positions: coalesced) and as one 16-byte
//     row of the tensor-core operand [position][channel] in shared memory;
//   * the x_proj contribution of the slice accumulates in registers
//     (mma.sync m16n8k16, fp32 accumulation; warp w: rows 16 (w % 4) .. +16,
//     positions 32 (w / 4) .. +32);
//   * after the last slice B and C leave through a shared fp32 tile along
//     positions, dt_low stays in shared memory (rounded to tf32), and dt_proj
//     runs there in blocks of 64 rows (mma.sync m16n8k8 tf32, fp32
//     accumulation), dt stored along positions.
// So u is written once and never read back, and dt_low never leaves the
// CTA (the three-kernel path reads u again and round-trips dt_low).
#ifndef SSM_FP_MINB
#define SSM_FP_MINB 2            // CTAs per SM the register allocation allows for
#endif
constexpr int FP_T = 64, FP_KS = 32, FP_NT = 256;
constexpr int FP_XS = FP_T + 4;                  // x window row: positions t0-3 .. t0+63 (+pad)
constexpr int FP_IP = FP_KS + 8;                 // operand row [position][channel] (bank spread)
constexpr int FP_OP = FP_T + 8;                  // x_proj result row (fp32)
constexpr int FP_XV = (FP_KS * FP_XS + FP_NT - 1) / FP_NT;   // x values per thread and slice
constexpr int FP_WV = 64 * FP_KS / FP_NT;                    // W_x values per thread and slice
constexpr int FP_OS = FP_T + 4;                  // dt block row (fp32)
constexpr int FP_IS = FP_T + 8;                  // dt_low (tf32) row
// one slice's buffers: x window, operand [position][channel], W_x
// columns, conv taps and bias (two of them: slice s + 1 is staged while
// the mma of slice s still reads its own)
__host__ __device__ constexpr int fp_slice_bytes() {
    return FP_KS * FP_XS * 4 + 2 * 64 * FP_IP * 2 + FP_KS * 5 * 4;
}
template <int RP> __host__ __device__ constexpr int fp_region() {
    // slice buffers, or (after the slices) dt_proj's W block, dt_low and
    // output block; conv weights and bias at the end of the slice buffers
    constexpr int a = 2 * fp_slice_bytes();
    constexpr int c = 64 * (RP + 4) * 4 + RP * FP_IS * 4 + 64 * FP_OS * 4;
    return ((a > c ? a : c) + 15) / 16 * 16;
}
template <int RP> __host__ __device__ constexpr size_t fused_prologue_smem_bytes() {
    return (size_t)fp_region<RP>() + (size_t)64 * FP_OP * 4;
}

template <typename IO, int RP>
__global__ void __launch_bounds__(FP_NT, SSM_FP_MINB)
fused_prologue_kernel(const IO *__restrict__ x, const float *__restrict__ cw,
                      const float *__restrict__ cb, const float *__restrict__ Wx,
                      const float *__restrict__ Wdt, int D, int L, int N, int R, int reverse,
                      IO *__restrict__ u, IO *__restrict__ dt, IO *__restrict__ Bm,
                      IO *__restrict__ Cm) {
    static_assert(sizeof(IO) == 2, "16-bit I/O");
    extern __shared__ __align__(16) unsigned char fp_smem[];
    // slice phase: buffer set k of slice s = k (mod 2)
    auto sx = [&](int k) { return (float *)(fp_smem + k * fp_slice_bytes()); };   // [FP_KS][FP_XS]
    auto sI = [&](int k) { return (IO *)(sx(k) + FP_KS * FP_XS); };               // [FP_T][FP_IP]
    auto sW = [&](int k) { return sI(k) + FP_T * FP_IP; };                        // [64][FP_IP]
    auto sCW = [&](int k) { return (float *)(sW(k) + 64 * FP_IP); };             // [FP_KS][4]
    auto sCB = [&](int k) { return sCW(k) + FP_KS * 4; };                         // [FP_KS]
    // dt_proj phase (the same bytes)
    constexpr int WS = RP + 4;
    unsigned *sWd = (unsigned *)fp_smem;                       // [64][WS] tf32
    unsigned *sDL = sWd + 64 * WS;                             // [RP][FP_IS] tf32
    float *sOut = (float *)(sDL + RP * FP_IS);                 // [64][FP_OS]
    float *sO = (float *)(fp_smem + fp_region<RP>());          // [64][FP_OP]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tg = lane & 3;
    const int wm = (warp % 4) * 16, wn = (warp / 4) * 32;
    const int t0 = blockIdx.x * FP_T, b = blockIdx.y;
    const int M = R + 2 * N, nsl = (D + FP_KS - 1) / FP_KS;
    const long long xb = (long long)b * D * L;

    // this thread's share of a slice: x window element i = tid + j * FP_NT
    // (channel i / FP_XS, position i % FP_XS of the window), W_x element
    // i = tid + j * FP_NT (row i / FP_KS, channel i % FP_KS).  Offsets and
    // masks that do not depend on the slice are formed once.
    int xo[FP_XV];                    // offset in x of the element, slice 0 (clamped in range)
    unsigned xok = 0;                 // bit j: position inside the window and the sequence
    // channel within the slice of element j (>= FP_KS: not an element)
    auto xcc = [&](int j) {
        const int i = tid + j * FP_NT;
        return i < FP_KS * FP_XS ? i / FP_XS : FP_KS;
    };
#pragma unroll
    for (int j = 0; j < FP_XV; ++j) {
        const int i = tid + j * FP_NT, cc = i / FP_XS, pp = i % FP_XS, ts = t0 - 3 + pp;
        const int tc = min(max(ts, 0), L - 1);
        xo[j] = min(cc, FP_KS - 1) * L + (reverse ? L - 1 - tc : tc);
        if (i < FP_KS * FP_XS && pp < FP_T + 3 && ts >= 0 && ts < L) xok |= 1u << j;
    }
    const int wk = tid % FP_KS;       // W_x column within the slice (rows tid / FP_KS + 8 j)
    const IO *xbp = x + xb;
    IO rx[FP_XV];
    float rw[FP_WV], rc = 0.f;
    auto fetch = [&](int s) {
        const int c0 = s * FP_KS;
        const int cmax = D - 1 - c0;              // last channel of the slice inside D
        const IO *xs = xbp + (long long)c0 * L;
#pragma unroll
        for (int j = 0; j < FP_XV; ++j) {
            // clamp the channel into range (masked at commit)
            const int o = xcc(j) <= cmax ? xo[j] : xo[j] - (min(xcc(j), FP_KS - 1) - cmax) * L;
            rx[j] = xs[o];
        }
        const int kc = min(c0 + wk, D - 1);
#pragma unroll
        for (int j = 0; j < FP_WV; ++j) {
            const int m = min(tid / FP_KS + j * (FP_NT / FP_KS), M - 1);
            rw[j] = Wx[(long long)m * D + kc];
        }
        if (tid < FP_KS * 5) {                       // 4 taps and the bias of each channel
            const int c = min(c0 + tid % FP_KS, D - 1), q = tid / FP_KS;
            rc = q < 4 ? cw[(long long)c * 4 + q] : (cb ? cb[c] : 0.f);
        }
    };
    auto commit = [&](int s) {
        const int c0 = s * FP_KS, cmax = D - 1 - c0, k = s & 1;
        float *x_s = sx(k);
#pragma unroll
        for (int j = 0; j < FP_XV; ++j) {
            const int i = tid + j * FP_NT;
            if (i < FP_KS * FP_XS) x_s[i] = ((xok >> j) & 1u) && xcc(j) <= cmax ? to_f32(rx[j]) : 0.f;
        }
        const bool kin = wk <= cmax;
        IO *w_s = sW(k);
#pragma unroll
        for (int j = 0; j < FP_WV; ++j) {
            const int m = tid / FP_KS + j * (FP_NT / FP_KS);
            w_s[m * FP_IP + wk] = from_f32<IO>((m < M && kin) ? rw[j] : 0.f);
        }
        if (tid < FP_KS * 5) {
            const int cc = tid % FP_KS, q = tid / FP_KS;
            const float v = cc <= cmax ? rc : 0.f;
            if (q < 4) sCW(k)[cc * 4 + q] = v;
            else sCB(k)[cc] = v;
        }
    };
    // conv + SiLU: position cp of the tile, channels cg * 8 .. cg * 8 + 7 of the slice
    const int cp = tid % FP_T, cg = tid / FP_T;
    auto conv = [&](int s) {
        const int c0 = s * FP_KS, t = t0 + cp, k = s & 1;
        const float *x_s = sx(k), *cw_s = sCW(k), *cb_s = sCB(k);
        IO res[8];
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            const int cc = cg * 8 + c8;
            const float4 w = *(const float4 *)&cw_s[cc * 4];
            const float *xr = x_s + cc * FP_XS + cp;
            float acc = cb_s[cc];
            acc = fmaf(w.x, xr[0], acc);
            acc = fmaf(w.y, xr[1], acc);
            acc = fmaf(w.z, xr[2], acc);
            acc = fmaf(w.w, xr[3], acc);
            res[c8] = from_f32<IO>(silu_f<IO>(acc));
            if (t < L && c0 + cc < D) u[xb + (long long)(c0 + cc) * L + t] = res[c8];
        }
        uint4 pk4;
        pk4.x = (unsigned)*(const unsigned short *)&res[0] |
                ((unsigned)*(const unsigned short *)&res[1] << 16);
        pk4.y = (unsigned)*(const unsigned short *)&res[2] |
                ((unsigned)*(const unsigned short *)&res[3] << 16);
        pk4.z = (unsigned)*(const unsigned short *)&res[4] |
                ((unsigned)*(const unsigned short *)&res[5] << 16);
        pk4.w = (unsigned)*(const unsigned short *)&res[6] |
                ((unsigned)*(const unsigned short *)&res[7] << 16);
        *(uint4 *)&sI(k)[cp * FP_IP + cg * 8] = pk4;
    };
    float acc[4][4] = {};
    fetch(0);
    for (int s = 0; s < nsl; ++s) {
        // slice s's buffers were last read by the mma of slice s - 2, two
        // barriers ago
        commit(s);
        __syncthreads();
        if (s + 1 < nsl) fetch(s + 1);              // in flight during this slice
        conv(s);
        __syncthreads();
        const IO *w_s = sW(s & 1), *i_s = sI(s & 1);
#pragma unroll
        for (int ks = 0; ks < FP_KS; ks += 16) {
            unsigned a[4];
            a[0] = *(const unsigned *)&w_s[(wm + g) * FP_IP + ks + 2 * tg];
            a[1] = *(const unsigned *)&w_s[(wm + g + 8) * FP_IP + ks + 2 * tg];
            a[2] = *(const unsigned *)&w_s[(wm + g) * FP_IP + ks + 2 * tg + 8];
            a[3] = *(const unsigned *)&w_s[(wm + g + 8) * FP_IP + ks + 2 * tg + 8];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                unsigned bf[2];
                const IO *col = i_s + (wn + nt * 8 + g) * FP_IP + ks + 2 * tg;
                bf[0] = *(const unsigned *)col;
                bf[1] = *(const unsigned *)(col + 8);
                mma16816<IO>(acc[nt], a, bf);
            }
        }
    }
    __syncthreads();                                  // every warp past its last mma
    // x_proj rows to shared memory: c0, c1 row g, positions 2tg, 2tg+1; c2,
    // c3 row g + 8
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h)
            *(float2 *)&sO[(wm + g + 8 * h) * FP_OP + wn + nt * 8 + 2 * tg] =
                make_float2(acc[nt][2 * h], acc[nt][2 * h + 1]);
    __syncthreads();
    // B and C (rows R .. R + 2N - 1) along positions; dt_low (rows 0 .. R-1,
    // zero to RP) to tf32
    for (int i = tid; i < 2 * N * FP_T; i += FP_NT) {
        const int mm = i / FP_T, tt = i % FP_T, t = t0 + tt;
        if (t < L) {
            const IO v = from_f32<IO>(sO[(R + mm) * FP_OP + tt]);
            if (mm < N) Bm[((long long)b * N + mm) * L + t] = v;
            else Cm[((long long)b * N + mm - N) * L + t] = v;
        }
    }
    for (int i = tid; i < RP * FP_T; i += FP_NT) {
        const int r = i / FP_T, tt = i % FP_T;
        sDL[r * FP_IS + tt] = to_tf32(r < R ? sO[r * FP_OP + tt] : 0.f);
    }
    // dt_proj in blocks of 64 rows
    for (int mb = 0; mb < D; mb += 64) {
        for (int i = tid; i < 64 * RP; i += FP_NT) {
            const int mm = i / RP, r = i % RP, m = mb + mm;
            sWd[mm * WS + r] = to_tf32((m < D && r < R) ? Wdt[(long long)m * R + r] : 0.f);
        }
        __syncthreads();
        float dacc[4][4] = {};
#pragma unroll
        for (int ks = 0; ks < RP; ks += 8) {
            // A (row): a0 (g, tg), a1 (g + 8, tg), a2 (g, tg + 4), a3 (g + 8, tg + 4)
            const unsigned *wr = sWd + (wm + g) * WS + ks + tg;
            const unsigned a[4] = {wr[0], wr[8 * WS], wr[4], wr[8 * WS + 4]};
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                // B (col): b0 (k = tg, n = g), b1 (k = tg + 4, n = g)
                const unsigned *col = sDL + (ks + tg) * FP_IS + wn + nt * 8 + g;
                const unsigned bf[2] = {col[0], col[4 * FP_IS]};
                mma1688_tf32(dacc[nt], a, bf);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                *(float2 *)&sOut[(wm + g + 8 * h) * FP_OS + wn + nt * 8 + 2 * tg] =
                    make_float2(dacc[nt][2 * h], dacc[nt][2 * h + 1]);
        __syncthreads();
        for (int i = tid; i < 64 * FP_T; i += FP_NT) {
            const int mm = i / FP_T, tt = i % FP_T, m = mb + mm, t = t0 + tt;
            if (m < D && t < L) dt[xb + (long long)m * L + t] = from_f32<IO>(sOut[mm * FP_OS + tt]);
        }
        __syncthreads();
    }
}

// Tiles of the SS2D x_proj below: XP_T positions per tile, XP_K-deep K
// slices, XP_NT threads, XP_OP the fp32 output tile's row.
constexpr int XP_T = 128, XP_K = 256, XP_OP = XP_T + 8, XP_NT = 512;

// ---- position-contiguous 16-bit rows as the MN-major A operand of tcgen05
// A slice is KS channels (k0 ..) x 128 positions (t0 ..) of a tensor x
// [nb][K][L] whose rows are contiguous along positions and whose base is
// 16-byte aligned.  Each row is copied raw by 16-byte cp.async (no
// registers): the 17 chunks from the 16-byte boundary at or below its first
// position, zero-filled past the tensor's end and for rows at or past K;
// every thread then arrives on the stage's mbarrier once its copies have
// landed (per-row bulk copies of 272 bytes measured slower on B300 at
// this piece length).  The threads then realign the raw rows in
// shared memory into the A tile, MN-major without swizzle: element (t, k) at
//   (k / 8) * MN_KSTR + (t / 8) * MN_MSTR + (k % 8) * 16 + (t % 8) * 2,
// core matrices of 8 channels x 8 consecutive positions; the descriptor's
// leading byte offset is MN_KSTR (between channel groups), its stride byte
// offset MN_MSTR (between position groups; 144 rather than 128 so that the
// 16-byte stores of 8 lanes along positions fall on distinct banks).
// Positions past the row's end hold the next row's values (or zeros): they
// only reach output positions that are not stored.
constexpr int RAW_CH = 17, RAW_ROW = RAW_CH * 16;     // chunks and bytes per raw row
constexpr unsigned MN_MSTR = 144, MN_KSTR = 16 * MN_MSTR;
__host__ __device__ constexpr int mn_tile_bytes(int KS) { return KS / 8 * (int)MN_KSTR; }

// the barrier's pending count drops by one when every cp.async this thread
// issued before has landed
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}
// tiled TMA load of the box at (x, y) (x: innermost coordinate, its byte
// offset a multiple of 16) of the tensor map into shared memory, completing
// its bytes on `bar`
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_addr(dst)), "l"((unsigned long long)tm), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void cp_async16_n(void *smem, const void *gmem, int bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(smem)),
                 "l"(gmem), "r"(bytes)
                 : "memory");
}
// the raw rows of a slice (rows row0 .. row0 + KS - 1 of x, i.e. b * K +
// k0 + r; rows r >= nrow, k >= K, are zero), positions from t0, by 16-byte
// cp.async with zero fill past the tensor's end (E elements): NT / KS
// threads per row, thread tid copies chunks tid % (NT / KS) + (NT / KS) * i
// of row tid / (NT / KS)
template <int KS, int NT, typename IO>
__device__ __forceinline__ void raw_rows_copy(unsigned char *raw, const IO *x, long long E,
                                              long long row0, int nrow, int L, int t0,
                                              int tid) {
    constexpr int TPR = NT / KS;
    static_assert(KS * TPR == NT && TPR <= RAW_CH, "threads per raw row");
    const int r = tid / TPR, c0 = tid % TPR;
    const long long cs = ((row0 + r) * L + t0) & ~7LL;
    const long long nv0 = r < nrow ? E - cs : 0;                // elements of x from cs on
    unsigned char *d = raw + r * RAW_ROW;
#pragma unroll
    for (int i = 0; i < (RAW_CH + TPR - 1) / TPR; ++i) {
        const int ch = c0 + TPR * i;
        if (i * TPR + TPR <= RAW_CH || ch < RAW_CH) {
            const long long nv = nv0 - 8 * ch;
            const int bytes = nv >= 8 ? 16 : nv > 0 ? 2 * (int)nv : 0;
            cp_async16_n(d + ch * 16, bytes > 0 ? (const void *)(x + cs + 8 * ch) : (const void *)x,
                         bytes);
        }
    }
}
// raw rows -> A tile, 16 bytes (8 positions of one channel) per step: row r
// starts s = (its first element's offset) mod 8 elements into its raw copy,
// so output words 0..3 are element pairs s + 2i of the raw chunks j, j + 1
template <int KS, int NT>
__device__ __forceinline__ void raw_rows_realign(const unsigned char *raw, unsigned char *a,
                                                 long long row0, int L, int t0, int tid) {
#pragma unroll
    for (int c = tid; c < KS * 16; c += NT) {
        const int r = c >> 4, j = c & 15;
        const unsigned s = ((unsigned)(row0 + r) * (unsigned)L + (unsigned)t0) & 7u;
        const uint4 p = *(const uint4 *)(raw + r * RAW_ROW + 16 * j);
        const uint4 q = *(const uint4 *)(raw + r * RAW_ROW + 16 * j + 16);
        // f_i = word i + s / 2 of p, q (two selects on the bits of s / 2)
        const bool h2 = s & 4, h1 = s & 2;
        const unsigned e0 = h2 ? p.z : p.x, e1 = h2 ? p.w : p.y, e2 = h2 ? q.x : p.z,
                       e3 = h2 ? q.y : p.w, e4 = h2 ? q.z : q.x, e5 = h2 ? q.w : q.y;
        const unsigned f0 = h1 ? e1 : e0, f1 = h1 ? e2 : e1, f2 = h1 ? e3 : e2,
                       f3 = h1 ? e4 : e3, f4 = h1 ? e5 : e4;
        const unsigned sel = (s & 1) ? 0x5432u : 0x3210u;
        uint4 o;
        o.x = __byte_perm(f0, f1, sel);
        o.y = __byte_perm(f1, f2, sel);
        o.z = __byte_perm(f2, f3, sel);
        o.w = __byte_perm(f3, f4, sel);
        *(uint4 *)(a + (r >> 3) * MN_KSTR + j * MN_MSTR + (r & 7) * 16) = o;
    }
}

// x_proj on the 5th-generation tensor cores (tcgen05, 16-bit I/O, M <= 64
// rows): out[b][m][t] = sum_k W[m][k] u[b][k][t] as D[t][m] = U[t][k] W[m][k]
// with MMA M = 128 positions, N = 64 rows, K = 16 per instruction and an
// fp32 accumulator of 128 lanes x 64 columns in tensor memory.  A persistent
// CTA of 16 warps (one per SM) keeps W (I/O type, zero-padded to 64 rows
// and a multiple of 128 columns) in shared memory as the B operand in the
// canonical K-major layout without swizzle (8 x 16-byte core matrices,
// 128 bytes apart along K, 8-row groups KR * 16 bytes apart).  For each
// tile of 128 positions it streams u in slices of 128 channels: the
// threads load the next slice into registers (raw values, clamped
// addresses) while the tensor core works on the current one, then store it
// transposed into one of two A buffers (core matrices: 8 positions x 8
// channels, 2048 bytes between 8-position groups); one thread issues the 8
// MMAs of the slice and commits them to that buffer's mbarrier, which the
// threads wait on before they overwrite the buffer two slices later.  After
// a tile's last slice every warp reads its TMEM quarter (32 positions x 16
// rows, tcgen05.ld) and stores along positions: coalesced, no staging tile.
constexpr int TCX_T = 128, TCX_K = 128, TCX_NT = 512;
__host__ __device__ constexpr int tcx_kr(int K) { return ((K + TCX_K - 1) / TCX_K) * TCX_K; }
inline size_t xproj_tc_smem_bytes(int K) {
    return (size_t)64 * tcx_kr(K) * 2 + 2 * (size_t)TCX_T * TCX_K * 2 + 64;
}
template <typename IO>
__global__ void __launch_bounds__(TCX_NT, 1)
xproj_tc_kernel(const float *__restrict__ W, const IO *__restrict__ in, int M, int K, int L,
                int nb, ProjOut out) {
    static_assert(sizeof(IO) == 2, "16-bit I/O");
    extern __shared__ __align__(1024) unsigned char tcx_smem[];
    constexpr int PAIRS = TCX_T * TCX_K / 2 / TCX_NT;           // k-pairs per thread and slice
    constexpr unsigned SBO_A = TCX_K / 8 * 128;                 // 2048: next 8 positions
    constexpr int A_BYTES = TCX_T * TCX_K * 2;
    const int KR = tcx_kr(K);
    const unsigned SBO_W = (unsigned)KR / 8 * 128;              // next 8 rows of W
    unsigned char *sW = tcx_smem;                               // [64 rows][KR], core matrices
    unsigned char *sA = sW + 64 * KR * 2;                       // [2][128 positions][128]
    uint64_t *bars = (uint64_t *)(sA + 2 * A_BYTES);            // one per A buffer
    unsigned *tslot = (unsigned *)(bars + 2);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // byte offset of element (row r, column k) of a K-major tile whose
    // 8-row groups are sbo bytes apart
    auto kmaj = [](int r, int k, unsigned sbo) {
        return (int)((r >> 3) * sbo) + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
    };
    if (warp == 0) tc_alloc(tslot, 64);
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_barrier_init();
    }
    // W: element (m, k), zero past row M and column K (eight element pairs
    // per thread and step, every load of a step in flight)
    for (int i0 = tid; i0 < 64 * KR / 2; i0 += 8 * TCX_NT) {
        float w0[8], w1[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * TCX_NT, m = i / (KR / 2), k = 2 * (i - m * (KR / 2));
            const bool in = i < 64 * KR / 2 && m < M;
            w0[u] = (in && k < K) ? W[(long long)m * K + k] : 0.f;
            w1[u] = (in && k + 1 < K) ? W[(long long)m * K + k + 1] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * TCX_NT, m = i / (KR / 2), k = 2 * (i - m * (KR / 2));
            if (i < 64 * KR / 2) {
                const IO a = from_f32<IO>(w0[u]), c = from_f32<IO>(w1[u]);
                *(unsigned *)(sW + kmaj(m, k, SBO_W)) =
                    (unsigned)*(const unsigned short *)&a |
                    ((unsigned)*(const unsigned short *)&c << 16);
            }
        }
    }
    fence_proxy_async_shared();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const unsigned tmem = *tslot;
    const unsigned idesc = tc_idesc<IO>(128, 64);
    // slice loader: position tt, k-pairs kp0 + 4 j of the slice
    const int ld_tt = (warp % 8) * 16 + (lane & 15);
    const int ld_kp0 = (warp / 8) * 2 + (lane >> 4);
    const int tpb = (L + TCX_T - 1) / TCX_T, ntiles = tpb * nb;
    const int nk = KR / TCX_K;
    IO r0[PAIRS], r1[PAIRS];
    int it = 0;                        // slices issued by this CTA (buffer it & 1)
    bool ok = true;                    // every wait finished in time
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int b = tile / tpb, t0 = (tile % tpb) * TCX_T;
        const int t = min(t0 + ld_tt, L - 1);
        const bool tin = t0 + ld_tt < L;
        const IO *src = in + (long long)b * K * L + t;
        auto load = [&](int k0) {
#pragma unroll
            for (int j = 0; j < PAIRS; ++j) {
                const int k = k0 + 2 * (ld_kp0 + 4 * j);
                r0[j] = src[(long long)min(k, K - 1) * L];
                r1[j] = src[(long long)min(k + 1, K - 1) * L];
            }
        };
        load(0);
        for (int ki = 0; ki < nk; ++ki, ++it) {
            const int buf = it & 1;
            unsigned char *a_s = sA + buf * A_BYTES;
            // the mma that last read this buffer (two slices ago) is done
            if (it >= 2) ok &= mbar_wait_bounded(&bars[buf], (unsigned)(((it >> 1) - 1) & 1));
            const int k0 = ki * TCX_K;
#pragma unroll
            for (int j = 0; j < PAIRS; ++j) {
                const int kk = 2 * (ld_kp0 + 4 * j), k = k0 + kk;
                const IO z = from_f32<IO>(0.f);
                const IO v0 = (tin && k < K) ? r0[j] : z, v1 = (tin && k + 1 < K) ? r1[j] : z;
                *(unsigned *)(a_s + kmaj(ld_tt, kk, SBO_A)) =
                    (unsigned)*(const unsigned short *)&v0 |
                    ((unsigned)*(const unsigned short *)&v1 << 16);
            }
            fence_proxy_async_shared();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (tid == 0) {
#pragma unroll
                for (int ks = 0; ks < TCX_K / 16; ++ks) {
                    const unsigned long long ad = tc_desc(smem_addr(a_s) + ks * 256, 128, SBO_A);
                    const unsigned long long bd =
                        tc_desc(smem_addr(sW) + (unsigned)(k0 / 8 * 128) + ks * 256, 128, SBO_W);
                    tc_mma(tmem, ad, bd, idesc, ki > 0 || ks > 0);
                }
                tc_commit(&bars[buf]);
            }
            if (ki + 1 < nk) load(k0 + TCX_K);              // in flight during the mma
        }
        // the tile's last slice (and so every earlier one) is done
        ok &= mbar_wait_bounded(&bars[(it - 1) & 1], (unsigned)(((it - 1) >> 1) & 1));
        tc_fence_after();
        {
            // warp w: TMEM lanes (positions) 32 (w % 4) .., columns (rows) 16 (w / 4) ..
            const int q4 = warp % 4, m0 = 16 * (warp / 4);
            float v[16];
            tc_ld16(tmem + ((unsigned)(32 * q4) << 16) + (unsigned)m0, v);
            const int tp = t0 + 32 * q4 + lane;
            if (tp < L) {
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    if (m0 + q < M) proj_store<IO>(out, b, m0 + q, tp, L, v[q]);
            }
        }
        // every warp has read TMEM before the next tile's first mma overwrites it
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    (void)ok;
    __syncthreads();
    if (warp == 0) tc_dealloc(tmem, 64);
}

// The block's output projection on tcgen05 (16-bit I/O, d_model <= 512,
// d_inner a multiple of 8, y and W 16-byte aligned):
// out[b][m][t] = sum_k W[m][k] y[b][k][t] ("VMamba的SS2D模块详解" section
// 2.1: out_proj = Linear(d_inner -> d_model) after the gate), as
// D[t][m] = Y[t][k] W[m][k]: MMA M = 128 positions, N in chunks of 128 rows
// (every d_model row of a tile: NCH chunks, 128 * NCH TMEM columns), K = 16
// per instruction, fp32 accumulator in tensor memory.  A persistent CTA
// walks one stream of slices (OP_K channels of one tile of 128 positions)
// over its tiles through a ring of `ns` stages, each holding a slice's raw
// y rows and its W columns and completing on its own mbarrier; ns - 1
// slices are in flight.  Warp roles:
//   * 16 worker warps: copy the raw y rows of the slice ns - 1 ahead
//     (sixteen threads per row, cp.async, each thread arriving on the stage
//     once its copies land), realign a landed slice into one of two A
//     buffers (MN-major) and signal it on that buffer's "A full" mbarrier
//     (one arrival per warp), and after a tile's last slice read TMEM
//     (warp w: lanes 32 (w % 4), a quarter of the columns), store along
//     positions and signal "TMEM free";
//   * one MMA warp: per slice, once "A full", issues the slice's 2 * NCH
//     MMAs and commits them to the A buffer's mbarrier; once the previous
//     slice's MMAs are done it refills that stage's W by tiled TMA copies
//     (tensor map `tmW`: W [d_model][d_inner], boxes of 8 channels x 128
//     rows, zero fill past d_model and d_inner; a box lands as 128 rows x 16
//     bytes, i.e. 16 core matrices of the K-major operand without swizzle,
//     so the slice's W is K-major with the 8-channel groups NR * 16 bytes
//     apart and 8-row groups 128 bytes apart), announcing the bytes with its
//     own arrival on the stage; before a tile's first MMA it waits for
//     "TMEM free" of the tile before.
// No CTA-wide barrier inside the loop: every hand-off is an mbarrier, and
// every wait is bounded.
constexpr int OP_T = 128, OP_K = 32, OP_NT = 512, OP_MAXN = 512, OP_MAXNS = 8;
constexpr int OP_THREADS = OP_NT + 32;                      // workers + the MMA warp
template <int NCH> __host__ __device__ constexpr size_t out_proj_stage_bytes() {
    return (size_t)OP_K * RAW_ROW + (size_t)NCH * 128 * OP_K * 2;
}
template <int NCH> __host__ __device__ constexpr size_t out_proj_fixed_bytes() {
    return 2 * (size_t)mn_tile_bytes(OP_K) + 8 * (5 + OP_MAXNS) + 16;
}
template <int NCH> inline int out_proj_stages(size_t smem_max) {
    const size_t fixed = out_proj_fixed_bytes<NCH>();
    if (fixed >= smem_max) return 0;
    const size_t ns = (smem_max - fixed) / out_proj_stage_bytes<NCH>();
    return ns < 3 ? 0 : (int)(ns < (size_t)OP_MAXNS ? ns : OP_MAXNS);
}
template <int NCH> inline size_t out_proj_smem_bytes(int ns) {
    return out_proj_fixed_bytes<NCH>() + (size_t)ns * out_proj_stage_bytes<NCH>();
}
template <typename IO, int NCH>
__global__ void __launch_bounds__(OP_THREADS, 1)
out_proj_tc_kernel(const __grid_constant__ CUtensorMap tmW, const IO *__restrict__ y, int Dm,
                   int Di, int L, int nb, int ns, IO *__restrict__ out) {
    static_assert(sizeof(IO) == 2, "16-bit I/O");
    extern __shared__ __align__(1024) unsigned char op_smem[];
    constexpr int NR = NCH * 128;                               // rows of the MMA's N
    constexpr int A_BYTES = mn_tile_bytes(OP_K), RAW_BYTES = OP_K * RAW_ROW;
    constexpr size_t STAGE = out_proj_stage_bytes<NCH>();
    constexpr unsigned W_LBO = NR * 16;                          // next 8 channels of W
    constexpr unsigned W_BYTES = NR * OP_K * 2;
    unsigned char *sA = op_smem;                                // [2] A tiles (MN-major)
    unsigned char *sS = sA + 2 * A_BYTES;                       // [ns] stages: raw y, W
    uint64_t *mbars = (uint64_t *)(sS + (size_t)ns * STAGE);    // MMA done, per A buffer
    uint64_t *afull = mbars + 2;                                // A written, per A buffer
    uint64_t *tfree = afull + 2;                                // TMEM read by the epilogue
    uint64_t *rbars = tfree + 1;                                // stage landed, per stage
    unsigned *tslot = (unsigned *)(rbars + OP_MAXNS);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool mma_warp = warp == OP_NT / 32;
    constexpr unsigned TCOLS = NR <= 128 ? 128 : NR <= 256 ? 256 : 512;
    if (mma_warp) tc_alloc(tslot, TCOLS);
    if (tid == 0) {
        mbar_init(&mbars[0], 1);
        mbar_init(&mbars[1], 1);
        mbar_init(&afull[0], OP_NT / 32);
        mbar_init(&afull[1], OP_NT / 32);
        mbar_init(tfree, OP_NT / 32);
        // per use: one arrival (cp.async tracking) per worker thread and the
        // MMA warp's arrival announcing the W bytes
        for (int s = 0; s < ns; ++s) mbar_init(&rbars[s], OP_NT + 1);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const unsigned tmem = *tslot;
    const int tpb = (L + OP_T - 1) / OP_T, ntiles = tpb * nb;
    const int nk = (Di + OP_K - 1) / OP_K;
    const long long E = (long long)nb * Di * L;
    bool ok = true;                    // every wait finished in time
    if (mma_warp) {
        if (lane == 0) {
            const unsigned idesc = tc_idesc<IO>(128, 128, true);
            // the W side of the copies: slice (i_ki of any tile) into stage i_st
            int i_tile = blockIdx.x, i_ki = 0, i_st = 0;
            auto issue_w = [&]() {
                if (i_tile >= ntiles) return;
                unsigned char *w_s = sS + (size_t)i_st * STAGE + RAW_BYTES;
                mbar_arrive_expect_tx(&rbars[i_st], W_BYTES);
#pragma unroll
                for (int kc = 0; kc < OP_K / 8; ++kc)
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
                        tma_load_2d(w_s + kc * W_LBO + c * 2048, &tmW, i_ki * OP_K + 8 * kc,
                                    128 * c, &rbars[i_st]);
                if (++i_st == ns) i_st = 0;
                if (++i_ki == nk) {
                    i_ki = 0;
                    i_tile += gridDim.x;
                }
            };
            for (int g = 0; g + 1 < ns; ++g) issue_w();
            int g = 0, st = 0, nt = 0;
            for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++nt) {
                // the epilogue of the tile before has read TMEM
                if (nt > 0) ok &= mbar_wait_bounded(tfree, (unsigned)((nt - 1) & 1));
                for (int ki = 0; ki < nk; ++ki, ++g) {
                    const int buf = g & 1;
                    ok &= mbar_wait_bounded(&afull[buf], (unsigned)((g >> 1) & 1));
                    tc_fence_after();
                    const unsigned a_a = smem_addr(sA + buf * A_BYTES);
                    const unsigned w_a = smem_addr(sS + (size_t)st * STAGE + RAW_BYTES);
#pragma unroll
                    for (int ks = 0; ks < OP_K / 16; ++ks) {
                        const unsigned long long ad =
                            tc_desc(a_a + ks * 2 * MN_KSTR, MN_KSTR, MN_MSTR);
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            const unsigned long long bd =
                                tc_desc(w_a + ks * 2 * W_LBO + c * 2048, W_LBO, 128);
                            tc_mma(tmem + 128 * c, ad, bd, idesc, ki > 0 || ks > 0);
                        }
                    }
                    tc_commit(&mbars[buf]);
                    // the previous slice's MMAs are done: its stage takes the
                    // W of slice g + ns - 1
                    if (g >= 1)
                        ok &= mbar_wait_bounded(&mbars[buf ^ 1], (unsigned)(((g - 1) >> 1) & 1));
                    issue_w();
                    if (++st == ns) st = 0;
                }
            }
        }
        __syncwarp();
    } else {
        // the y side of the copies: slice (i_tile, i_ki) into stage i_st
        int i_tile = blockIdx.x, i_ki = 0, i_st = 0;
        long long i_row = (long long)(i_tile / tpb) * Di;      // b * Di of i_tile
        int i_t0 = (i_tile % tpb) * OP_T;
        auto issue_y = [&]() {
            if (i_tile >= ntiles) return;
            const int k0 = i_ki * OP_K;
            raw_rows_copy<OP_K, OP_NT>(sS + (size_t)i_st * STAGE, y, E, i_row + k0, Di - k0, L,
                                       i_t0, tid);
            cp_async_arrive_noinc(&rbars[i_st]);
            if (++i_st == ns) i_st = 0;
            if (++i_ki == nk) {
                i_ki = 0;
                i_tile += gridDim.x;
                i_row = (long long)(i_tile / tpb) * Di;
                i_t0 = (i_tile % tpb) * OP_T;
            }
        };
        for (int g = 0; g + 1 < ns; ++g) issue_y();
        int g = 0, st = 0;             // slices consumed, their stage
        unsigned rpar = 0;             // phase parity of the stages' current use
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            const int b = tile / tpb, t0 = (tile % tpb) * OP_T;
            const long long row_b = (long long)b * Di;
            for (int ki = 0; ki < nk; ++ki, ++g) {
                const int buf = g & 1;
                ok &= mbar_wait_bounded(&rbars[st], rpar);
                // the MMAs that last read this A buffer (slice g - 2) are done
                if (g >= 2) ok &= mbar_wait_bounded(&mbars[buf], (unsigned)(((g - 2) >> 1) & 1));
                raw_rows_realign<OP_K, OP_NT>(sS + (size_t)st * STAGE, sA + buf * A_BYTES,
                                              row_b + ki * OP_K, L, t0, tid);
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) mbar_arrive(&afull[buf]);
                // the previous slice's MMAs are done (and so every warp has
                // realigned it): its stage takes the y rows of slice g + ns - 1
                if (g >= 1) ok &= mbar_wait_bounded(&mbars[buf ^ 1], (unsigned)(((g - 1) >> 1) & 1));
                issue_y();
                if (++st == ns) {
                    st = 0;
                    rpar ^= 1u;
                }
            }
            // the tile's last slice (and so every earlier one) is done
            ok &= mbar_wait_bounded(&mbars[(g - 1) & 1], (unsigned)(((g - 1) >> 1) & 1));
            tc_fence_after();
            // warp w: TMEM lanes (positions) 32 (w % 4) .., columns (rows)
            // (w / 4) * NR / 4 .. + NR / 4
            const int q4 = warp % 4, tp = t0 + 32 * q4 + lane;
#pragma unroll 1
            for (int h = 0; h < NR / 4 / 16; ++h) {
                const int m0 = (warp / 4) * (NR / 4) + 16 * h;
                if (m0 >= Dm) break;                               // uniform over the warp
                float v[16];
                tc_ld16(tmem + ((unsigned)(32 * q4) << 16) + (unsigned)m0, v);
                if (tp < L) {
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (m0 + q < Dm)
                            out[((long long)b * Dm + m0 + q) * L + tp] = from_f32<IO>(v[q]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tfree);
        }
        cp_async_wait_all();
    }
    (void)ok;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (mma_warp) tc_dealloc(tmem, TCOLS);
}

// SS2D x_proj for all four scan directions in one pass over u (16-bit I/O,
// K <= 256 so that one slice holds the whole inner dimension, M <= 64 rows
// per direction).  A persistent CTA of 16 warps keeps the four weight sets
// [4][64][KQ] in shared memory (the I/O type, zero-padded), stages each
// tile's u [XP_T][KQ] once, then for each direction runs the mma against
// that direction's weights (warp w: rows 16 (w % 4) .. +16, positions
// 32 (w / 4) .. +32) and stores through a shared fp32 tile to that
// direction's destinations (outs.o[k]).  A tile is a block of 8 map rows x
// 16 columns: the row-major directions store runs of 16 positions, and the
// column-major ones, walking h fastest, runs of 8 (a tile of 128
// consecutive row-major positions would scatter them one by one, H apart).
struct ProjOut4 {
    ProjOut o[4];
};
__host__ __device__ constexpr int xproj4_kq(int K) { return ((K + 15) / 16) * 16 + 8; }
inline size_t xproj4_smem_bytes(int K, size_t esize) {
    return (4 * 64 * (size_t)xproj4_kq(K) + (size_t)XP_T * xproj4_kq(K)) * esize +
           64 * (size_t)XP_OP * sizeof(float);
}
template <typename IO>
__global__ void __launch_bounds__(XP_NT, 1)
xproj4_mma_kernel(const float *__restrict__ W, const IO *__restrict__ in, int M, int K, int L,
                  int nb, ProjOut4 outs) {
    extern __shared__ __align__(16) unsigned char xq_smem[];
    constexpr int NW = XP_NT / 32;                              // 16 warps
    constexpr int PAIRS = XP_T * XP_K / 2 / XP_NT;              // covers K <= XP_K
    const int KQ = xproj4_kq(K), KR = KQ - 8;                  // KR: K rounded up to 16
    IO *sW = (IO *)xq_smem;                                    // [4][64][KQ]
    IO *sI = sW + 4 * 64 * KQ;                                 // [XP_T][KQ]
    float *sO = (float *)(sI + XP_T * KQ);                     // [64][XP_OP]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tg = lane & 3;
    const int wm = (warp % 4) * 16, wn = (warp / 4) * 32;
    for (int m = warp; m < 4 * 64; m += NW) {
        const int k4 = m / 64, mr = m % 64;
        IO *dst = sW + m * KQ;
        const float *src = W + ((long long)k4 * M + mr) * K;
        for (int k0 = 0; k0 < KQ; k0 += 128) {
            float wv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int k = k0 + q * 32 + lane;
                wv[q] = (mr < M && k < K) ? src[k] : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int k = k0 + q * 32 + lane;
                if (k < KQ) dst[k] = from_f32<IO>(wv[q]);
            }
        }
    }
    const int ld_tt = (warp % 8) * 16 + (lane & 15);            // = 16 (row in block) + column
    const int ld_kp0 = (warp / 8) * 2 + (lane >> 4);            // + 4 j
    const int H = outs.o[0].H, Wd = outs.o[0].W;
    const int tW = (Wd + 15) / 16, tpb = ((H + 7) / 8) * tW, ntiles = tpb * nb;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int b = tile / tpb, blk = tile % tpb;
        const int h0 = (blk / tW) * 8, w0 = (blk % tW) * 16;
        const int lh = h0 + ld_tt / 16, lw = w0 + ld_tt % 16;
        const bool pin = lh < H && lw < Wd;
        const IO *src = in + (long long)b * K * L + (pin ? lh * Wd + lw : 0);
        unsigned reg[PAIRS];
#pragma unroll
        for (int j = 0; j < PAIRS; ++j) {
            const int k = 2 * (ld_kp0 + 4 * j);
            const IO z = from_f32<IO>(0.f);
            const IO v0 = (pin && k < K) ? src[(long long)k * L] : z;
            const IO v1 = (pin && k + 1 < K) ? src[(long long)(k + 1) * L] : z;
            reg[j] = (unsigned)*(const unsigned short *)&v0 |
                     ((unsigned)*(const unsigned short *)&v1 << 16);
        }
        __syncthreads();                                        // previous tile's sI reads done
        unsigned *dsti = (unsigned *)sI;
#pragma unroll
        for (int j = 0; j < PAIRS; ++j) {
            const int kp = ld_kp0 + 4 * j;
            if (2 * kp < KR) dsti[ld_tt * (KQ / 2) + kp] = reg[j];
        }
        __syncthreads();
        for (int k4 = 0; k4 < 4; ++k4) {
            const IO *wk = sW + k4 * 64 * KQ;
            float acc[4][4] = {};
            for (int ks = 0; ks < KR; ks += 16) {
                unsigned a[4];
                a[0] = *(const unsigned *)&wk[(wm + g) * KQ + ks + 2 * tg];
                a[1] = *(const unsigned *)&wk[(wm + g + 8) * KQ + ks + 2 * tg];
                a[2] = *(const unsigned *)&wk[(wm + g) * KQ + ks + 2 * tg + 8];
                a[3] = *(const unsigned *)&wk[(wm + g + 8) * KQ + ks + 2 * tg + 8];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    unsigned bf[2];
                    const IO *col = sI + (wn + nt * 8 + g) * KQ + ks + 2 * tg;
                    bf[0] = *(const unsigned *)col;
                    bf[1] = *(const unsigned *)(col + 8);
                    mma16816<IO>(acc[nt], a, bf);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int half = 0; half < 2; ++half)
                    *(float2 *)&sO[(wm + g + 8 * half) * XP_OP + wn + nt * 8 + 2 * tg] =
                        make_float2(acc[nt][2 * half], acc[nt][2 * half + 1]);
            __syncthreads();
            const bool colmajor = k4 == 1 || k4 == 3;
            for (int i = tid; i < M * XP_T; i += XP_NT) {
                const int m = i / XP_T, e = i % XP_T;
                const int tt = colmajor ? (e % 8) * 16 + e / 8 : e;    // h fastest: runs in t
                const int h = h0 + tt / 16, w = w0 + tt % 16;
                if (h < H && w < Wd) {
                    const int p = h * Wd + w, c = w * H + h;
                    const int ts = k4 == 0 ? p : k4 == 1 ? c : k4 == 2 ? L - 1 - p : L - 1 - c;
                    proj_store_at<IO>(outs.o[k4], b, m, ts, L, sO[m * XP_OP + tt]);
                }
            }
            __syncthreads();                                    // sO read before the next block
        }
    }
}

}  // namespace pro
}  // namespace ssm
