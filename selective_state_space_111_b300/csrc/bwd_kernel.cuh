// bwd_kernel.cuh -- backward pass of the selective scan (S6), sm_103a.
//
// Gradients of a loss sum_t g_t * out_t for the three forms.  Per direction,
// with a_t[n] = exp(delta_t * A[n]) and G_t[n] = dLoss/dh_t[n] (the adjoint
// of the forward recurrence of "状态空间模型如何重塑视觉序列处理", section
// "选择性扫描机制的计算效率优势", read with exp(delta*A) and delta*B):
//   G_t      = gy_t * C_t + a_{t+1} * G_{t+1}                (G_L = 0)
//   dC_t     = gy_t * h_t,       dB_t = G_t * delta_t * u_t
//   du_t     = gy_t * D + sum_n G_t * delta_t * B_t
//   dA      += G_t * h_{t-1} * a_t * delta_t
//   ddelta_t = sum_n G_t * (h_{t-1} * a_t * A + B_t * u_t)
//   ddt_t    = ddelta_t * sigmoid(dt_t + bias)   (softplus' ; or ddelta_t)
// gy is the gradient of the direction's own output y (before the gate; the
// gate, the flip-add and the cross-merge are undone by the callers).
//
//   scan_bwd_kernel   CTA = 16 channels of one batch element, one direction;
//                     lane = (channel, state).  Pass 1 runs the recurrence
//                     forward and stores the state at every chunk start
//                     (chunks of T = 32 steps).  Pass 2 walks the chunks
//                     backwards: it recomputes the chunk's states in
//                     registers from the stored start, then runs the adjoint
//                     recurrence step by step.  Every direction of a call
//                     runs in the same launch (blockIdx.z) and writes its own
//                     per-position gradients (du, ddelta: summed over the 16
//                     states by shuffles); dB
//                     and dC (summed over channels) go through shared memory
//                     into one fp32 partial per CTA, reduced afterwards in a
//                     fixed order, so results are deterministic.
//   gate_bwd_kernel   gy = g * silu(z), dz = g * y * silu'(z).
//   reduce kernels    partial sums -> dA (fp32), dB, dC (I/O dtype); dD and
//                     dbias as channel sums of the fp32 maps (G * u, ddt).
#pragma once

#include "scan_ops.cuh"

namespace ssm {
namespace bwd {

constexpr int T = 32;            // steps per chunk
constexpr int NT = 256;          // threads: lane = (channel, state)
constexpr int NWARP = NT / 32;
// channels per CTA for a state capacity NM (16: two channels per warp,
// 32: one channel per warp)
template <int NM> __host__ __device__ constexpr int channels() { return NT / NM; }

// One direction of one form.  Walk step w (0..L-1) is position
// p = rev ? L-1-w : w of the position-ordered tensors (u, G, du); dt and
// B/C are read at stream index s = stream_rev ? w : p.
struct Pass {
    const void *dt;            // delta: row (b, d) at dt_off + b * dt_bstride + d * L
    long long dt_off, dt_bstride;
    const void *u;             // [B, D, L], position order
    const void *Bm, *Cm;       // row (b, n) at bc_off + b * bc_bstride + n * L
    long long bc_off, bc_bstride;
    const float *A;            // [D, N]
    const float *Dskip;        // [D] or null
    const float *bias;         // [D] or null
    const float *G;            // dLoss/dy (fp32 [B, D, L], position order)
    float gscale;              // this direction's share of G (out_scale)
    int rev, stream_rev;
    float *du;                 // fp32 [B, D, L], position order (this pass's own)
    float *ddt;                // fp32, indexed like dt (this pass's own)
    // 16-state kernel only (null elsewhere): when set, du and ddt are
    // written in the I/O dtype here instead of the fp32 maps above, and the
    // per-(batch, channel) sums of ddt and of gscale * G * u (the dbias and
    // dD terms) are written to pbias and pdD, [B][D] fp32
    void *du_io, *ddt_io;
    float *pbias, *pdD;
    float *pdB, *pdC;          // this pass's partials [ncg][B][L][NM] (stream index)
    float *pdA;                // [B][D][NM]
    float *hc;                 // chunk-start states [B][D][nch][NM] (this pass's own)
};

constexpr int kMaxPass = 4;
struct Params {
    Pass ps[kMaxPass];         // one per direction; blockIdx.z selects it
    int B, D, L, N, nch;
    int delta_softplus;
    int hc_given;              // 16-state kernel: hc already holds the chunk-start
                               // states (stored by the forward pass); no pass 1
};

__device__ __forceinline__ float sigmoid_f(float x) {
    return 1.f / (1.f + expf(-x));
}
// sigmoid for the softplus derivative: the accurate form for fp32 I/O, the
// MUFU form (ex2, rcp) for 16-bit I/O, as the forward pass's gate uses
template <typename IO> __device__ __forceinline__ float sigmoid_io(float x) {
    if constexpr (sizeof(IO) == 4) return sigmoid_f(x);
    else return rcp_approx(1.f + ex2_approx(-x * kLog2e));
}
// dynamic shared memory: dB, dC partials per warp, then the chunk's
// recomputed states (step-major: thread-contiguous rows, no bank conflicts)
template <int NM> __host__ __device__ constexpr int part_floats() { return NWARP * NM * (T + 4); }
template <int NM> __host__ __device__ constexpr int dyn_bytes() {
    return (2 * part_floats<NM>() + T * NT) * (int)sizeof(float);
}

// Sum of 8 values over the 16 lanes of a half-warp, by halving exchanges:
// after the three halving levels lane l holds value (l>>3&1)*4 + (l>>2&1)*2
// + (l>>1&1) summed over 8 lanes, and the last exchange completes the sum
// (lanes l and l^1 then hold the same total).
__device__ __forceinline__ float half_warp_sum8(const float (&v)[8], int lane) {
    const bool b8 = lane & 8, b4 = lane & 4, b2 = lane & 2;
    float w[4], x[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = b8 ? v[i] : v[i + 4];
        w[i] = (b8 ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b4 ? w[i] : w[i + 2];
        x[i] = (b4 ? w[i + 2] : w[i]) + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    const float send = b2 ? x[0] : x[1];
    const float y = (b2 ? x[1] : x[0]) + __shfl_xor_sync(0xffffffffu, send, 2);
    return y + __shfl_xor_sync(0xffffffffu, y, 1);
}

// The same over all 32 lanes (one channel per warp): after three halving
// levels lane l holds value (l>>4&1)*4 + (l>>3&1)*2 + (l>>2&1) summed over 8
// lanes; two more exchanges complete it (lanes l, l^1, l^2, l^3 agree).
__device__ __forceinline__ float warp_sum8(const float (&v)[8], int lane) {
    const bool b16 = lane & 16, b8 = lane & 8, b4 = lane & 4;
    float w[4], x[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = b16 ? v[i] : v[i + 4];
        w[i] = (b16 ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b8 ? w[i] : w[i + 2];
        x[i] = (b8 ? w[i + 2] : w[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const float send = b4 ? x[0] : x[1];
    float y = (b4 ? x[1] : x[0]) + __shfl_xor_sync(0xffffffffu, send, 4);
    y += __shfl_xor_sync(0xffffffffu, y, 2);
    return y + __shfl_xor_sync(0xffffffffu, y, 1);
}

template <typename IO, int NM>
__global__ void __launch_bounds__(NT, 2)
scan_bwd_kernel(const Params P) {
    constexpr int CH = channels<NM>();
    constexpr int TP = T + 4;                  // padded rows: 16-byte aligned, banks spread
    __shared__ __align__(16) float sD[CH][TP], sU[CH][TP], sG[CH][TP], sS[CH][TP];
    __shared__ __align__(16) float sBt[NM][TP], sCt[NM][TP];
    __shared__ float sDu[CH][T + 1], sDd[CH][T + 1];
    __shared__ float sBias[CH], sDsk[CH];           // per-channel constants
    // per-warp dB, dC partials of a chunk, [warp][state][step] (dynamic)
    extern __shared__ __align__(16) float dyn[];
    float (*sPB)[NM][TP] = reinterpret_cast<float (*)[NM][TP]>(dyn);
    float (*sPC)[NM][TP] = reinterpret_cast<float (*)[NM][TP]>(dyn + part_floats<NM>());
    float (*sH)[NT] = reinterpret_cast<float (*)[NT]>(dyn + 2 * part_floats<NM>());

    const Pass &ps = P.ps[blockIdx.z];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ch = tid / NM, n = tid % NM;
    const int b = blockIdx.y, d0 = blockIdx.x * CH, d = d0 + ch;
    const int L = P.L, D = P.D, N = P.N, nch = P.nch;
    const bool cvalid = d < D, valid = cvalid && n < N;
    const float A2 = valid ? ps.A[(long long)d * N + n] * kLog2e : 0.f;
    const float Av = valid ? ps.A[(long long)d * N + n] : 0.f;
    const IO *dtp = (const IO *)ps.dt + ps.dt_off + b * ps.dt_bstride;
    const IO *bp = (const IO *)ps.Bm + ps.bc_off + b * ps.bc_bstride;
    const IO *cp = (const IO *)ps.Cm + ps.bc_off + b * ps.bc_bstride;
    const IO *up = (const IO *)ps.u;
    float *hcp = ps.hc + (((long long)b * D + d) * nch) * NM + n;
    if (tid < CH) {
        const int dd = d0 + tid;
        sBias[tid] = (dd < D && ps.bias) ? ps.bias[dd] : 0.f;
        sDsk[tid] = (dd < D && ps.Dskip) ? ps.Dskip[dd] : 0.f;
    }
    __syncthreads();

    auto pos = [&](int w) { return ps.rev ? L - 1 - w : w; };
    auto sidx = [&](int w) { return ps.stream_rev ? w : pos(w); };
    // Chunk staging, software-pipelined: fetch() loads this thread's share
    // of chunk c (PC of the CH x T per-channel values, PB of the NM x T B/C
    // values) into registers; commit() transforms and stores it.  The next
    // chunk is fetched before the current one is computed.
    constexpr int PC = CH * T / NT, PB = NM * T / NT;
    static_assert(PC * NT == CH * T && PB * NT == NM * T, "staging split");
    float rdt[PC], ru[PC], rg[PC], rb[PB], rc[PB];
    auto fetch = [&](int c, bool full) {
#pragma unroll
        for (int r = 0; r < PC; ++r) {
            const int i = tid + r * NT, cc = i / T, j = i % T, w = c * T + j, dd = d0 + cc;
            const bool ok = w < L && dd < D;
            rdt[r] = ok ? to_f32(dtp[(long long)dd * L + sidx(w)]) : 0.f;
            ru[r] = ok ? to_f32(up[((long long)b * D + dd) * L + pos(w)]) : 0.f;
            rg[r] = (ok && full) ? ps.G[((long long)b * D + dd) * L + pos(w)] : 0.f;
        }
#pragma unroll
        for (int r = 0; r < PB; ++r) {
            const int i = tid + r * NT, nn = i / T, j = i % T, w = c * T + j;
            const bool okb = w < L && nn < N;
            const long long o = (long long)nn * L + (okb ? sidx(w) : 0);
            rb[r] = okb ? to_f32(bp[o]) : 0.f;
            rc[r] = (okb && full) ? to_f32(cp[o]) : 0.f;
        }
    };
    auto commit = [&](int c) {
#pragma unroll
        for (int r = 0; r < PC; ++r) {
            const int i = tid + r * NT, cc = i / T, j = i % T, w = c * T + j, dd = d0 + cc;
            float dl = 0.f, sg = 1.f;
            if (w < L && dd < D) {
                const float x = rdt[r] + sBias[cc];
                if (P.delta_softplus) {
                    // the forward pass's own softplus (MUFU forms for 16-bit
                    // I/O), so the recomputed states match the forward's
                    dl = softplus_f<IO>(x);
                    sg = sigmoid_io<IO>(x);
                } else {
                    dl = x;
                }
            }
            sD[cc][j] = dl;
            sS[cc][j] = sg;
            sU[cc][j] = ru[r];
            sG[cc][j] = ps.gscale * rg[r];
        }
#pragma unroll
        for (int r = 0; r < PB; ++r) {
            const int i = tid + r * NT, nn = i / T, j = i % T;
            sBt[nn][j] = rb[r];
            sCt[nn][j] = rc[r];
        }
    };

    // ---- pass 1: states at the chunk starts
    float h = 0.f;
    fetch(0, false);
    for (int c = 0; c < nch; ++c) {
        if (cvalid) hcp[(long long)c * NM] = h;
        commit(c);
        __syncthreads();
        if (c + 1 < nch) fetch(c + 1, false);
        const int len = min(T, L - c * T);
        if (len == T) {
            // full chunk: 4 steps per group from 16-byte shared loads
#pragma unroll 2
            for (int j4 = 0; j4 < T / 4; ++j4) {
                const float4 d4 = *(const float4 *)&sD[ch][4 * j4];
                const float4 u4 = *(const float4 *)&sU[ch][4 * j4];
                const float4 b4 = *(const float4 *)&sBt[n][4 * j4];
                const float dv[4] = {d4.x, d4.y, d4.z, d4.w}, uv[4] = {u4.x, u4.y, u4.z, u4.w};
                const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    h = fmaf(ex2_approx(dv[k] * A2), h, dv[k] * bv[k] * uv[k]);
            }
        } else {
            for (int j = 0; j < len; ++j) {
                const float dl = sD[ch][j];
                h = fmaf(ex2_approx(dl * A2), h, dl * sBt[n][j] * sU[ch][j]);
            }
        }
        __syncthreads();
    }

    // ---- pass 2: adjoint, chunks in reverse; steps in groups of 4
    float Gc = 0.f, dA = 0.f;
    // FULL: a whole chunk (no step beyond L)
    auto chunk = [&](auto FULL, int len, float h0) {
        constexpr bool F = decltype(FULL)::value;
        {
            float hh = h0;
#pragma unroll 1
            for (int j4 = 0; j4 < T / 4; ++j4) {
                const float4 d4 = *(const float4 *)&sD[ch][4 * j4];
                const float4 u4 = *(const float4 *)&sU[ch][4 * j4];
                const float4 b4 = *(const float4 *)&sBt[n][4 * j4];
                const float dv[4] = {d4.x, d4.y, d4.z, d4.w}, uv[4] = {u4.x, u4.y, u4.z, u4.w};
                const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (F || 4 * j4 + k < len)
                        hh = fmaf(ex2_approx(dv[k] * A2), hh, dv[k] * bv[k] * uv[k]);
                    sH[4 * j4 + k][tid] = hh;
                }
            }
        }
        // h_j of the step being undone; the reverse sweep loads h_{j-1} once,
        // as the previous state of step j and the state of step j - 1
        float hcur = F ? sH[T - 1][tid] : 0.f;
        if (!F) {
            for (int j = T - 1; j >= 0; --j)
                if (j == len - 1) hcur = sH[j][tid];
        }
#pragma unroll 1
        for (int j4 = T / 4 - 1; j4 >= 0; --j4) {
            const int j0 = 4 * j4;
            if (!F && j0 >= len) continue;             // uniform over the CTA
            const float4 d4 = *(const float4 *)&sD[ch][j0];
            const float4 u4 = *(const float4 *)&sU[ch][j0];
            const float4 g4 = *(const float4 *)&sG[ch][j0];
            const float4 b4 = *(const float4 *)&sBt[n][j0];
            const float4 c4 = *(const float4 *)&sCt[n][j0];
            const float dv[4] = {d4.x, d4.y, d4.z, d4.w}, uv[4] = {u4.x, u4.y, u4.z, u4.w};
            const float gv[4] = {g4.x, g4.y, g4.z, g4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
            const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
            float red[8], dBp[4], dCp[4];     // red: du of the 4 steps, then ddelta
#pragma unroll
            for (int k = 3; k >= 0; --k) {
                const int j = j0 + k;
                if (!F && j >= len) {
                    red[k] = red[4 + k] = dBp[k] = dCp[k] = 0.f;
                    continue;
                }
                const float dl = dv[k], uu = uv[k], gy = gv[k], bb = bv[k];
                const float a = ex2_approx(dl * A2);
                const float hp = j > 0 ? sH[j - 1][tid] : h0;
                const float g = fmaf(gy, cv[k], Gc);
                dCp[k] = gy * hcur;
                hcur = hp;
                dBp[k] = g * dl * uu;
                red[k] = g * dl * bb;
                red[4 + k] = g * fmaf(hp * a, Av, bb * uu);
                dA = fmaf(g * hp * a, dl, dA);
                Gc = a * g;
            }
            // du, ddelta of the 4 steps: sums over the channel's NM states
            if constexpr (NM == 16) {
                const float tot = half_warp_sum8(red, lane);
                if ((lane & 1) == 0) {
                    const int idx = ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
                    if (idx < 4) sDu[ch][j0 + idx] = tot;
                    else sDd[ch][j0 + idx - 4] = tot;
                }
                // dB, dC: sums over the warp's two channels (lanes < 16 keep dB)
                const bool hi = lane >= 16;
                float qv[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float send = hi ? dBp[k] : dCp[k];
                    qv[k] = (hi ? dCp[k] : dBp[k]) + __shfl_xor_sync(0xffffffffu, send, 16);
                }
                *(float4 *)(hi ? &sPC[warp][n][j0] : &sPB[warp][n][j0]) =
                    make_float4(qv[0], qv[1], qv[2], qv[3]);
            } else {
                const float tot = warp_sum8(red, lane);
                if ((lane & 3) == 0) {
                    const int idx = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
                    if (idx < 4) sDu[ch][j0 + idx] = tot;
                    else sDd[ch][j0 + idx - 4] = tot;
                }
                // one channel per warp: its dB, dC go straight to the partials
                *(float4 *)&sPB[warp][n][j0] = make_float4(dBp[0], dBp[1], dBp[2], dBp[3]);
                *(float4 *)&sPC[warp][n][j0] = make_float4(dCp[0], dCp[1], dCp[2], dCp[3]);
            }
        }
    };
    fetch(nch - 1, true);
    float hnext = cvalid ? hcp[(long long)(nch - 1) * NM] : 0.f;
    for (int c = nch - 1; c >= 0; --c) {
        commit(c);
        __syncthreads();
        const float h0 = hnext;
        if (c > 0) {
            fetch(c - 1, true);
            hnext = cvalid ? hcp[(long long)(c - 1) * NM] : 0.f;
        }
        const int len = min(T, L - c * T);
        if (len == T) chunk(BoolC<true>(), len, h0);
        else chunk(BoolC<false>(), len, h0);
        __syncthreads();
        // per-position gradients of this direction (du with the skip term)
        for (int i = tid; i < CH * T; i += NT) {
            const int cc = i / T, j = i % T, w = c * T + j, dd = d0 + cc;
            if (w < L && dd < D) {
                const long long prow = ((long long)b * D + dd) * L;
                ps.du[prow + pos(w)] = fmaf(sG[cc][j], sDsk[cc], sDu[cc][j]);
                const float gx = P.delta_softplus ? sDd[cc][j] * sS[cc][j] : sDd[cc][j];
                ps.ddt[ps.dt_off + b * ps.dt_bstride + (long long)dd * L + sidx(w)] = gx;
            }
        }
        // dB, dC partial of this CTA: sum over its warps
        for (int i = tid; i < T * NM; i += NT) {
            const int j = i / NM, nn = i % NM, w = c * T + j;
            if (w < L) {
                float sb = 0.f, sc = 0.f;
#pragma unroll
                for (int k = 0; k < NWARP; ++k) {
                    sb += sPB[k][nn][j];
                    sc += sPC[k][nn][j];
                }
                const long long o = (((long long)blockIdx.x * P.B + b) * L + sidx(w)) * NM + nn;
                ps.pdB[o] = sb;
                ps.pdC[o] = sc;
            }
        }
        __syncthreads();
    }
    if (cvalid) ps.pdA[((long long)b * D + d) * NM + n] = dA;
}

// ------------------------------------------------------------------
// scan_bwd16_kernel: the same computation for a state capacity of 16, laid
// out so that the sums over states stay in registers.  lane = (channel,
// half): the eight states half*8 .. half*8+7 of one channel, as four packed
// fp32 pairs (f32x2 MUL/FMA).  CTA = 32 channels of one batch element, one
// direction (64 threads, two warps of 16 channels); chunks of T16 steps.
//  * pass 1 runs the recurrence forward and stores the state at each chunk
//    start (hc, [B][D][nch][16]) -- skipped when the forward pass of the
//    same call already stored them there (hc_given);
//  * pass 2 walks the chunks backwards: it recomputes the chunk's states
//    from the stored start into shared memory (h_{j-1} at step j), then
//    undoes the steps in groups of KG16.  Per step a lane forms, over its
//    eight states, sum_n G B and sum_n G h a A (the first serves du and
//    ddelta alike: ddelta = sum G h a A + u * sum G B), and one xor-shuffle
//    adds the channel's other half; dA accumulates G h a delta in registers;
//  * dB and dC (sums over channels) go through a per-warp tile: each lane
//    writes its eight dB and eight dC values of each step of the group,
//    then each lane adds four columns of one step over the warp's 16
//    channels, giving one partial per warp (16 channels) and step, written
//    to the same [slot][B][L][16] partials the 256-thread kernel fills.
// Full chunks run unrolled; the group structure keeps the warp's shared
// memory synchronisation to two __syncwarp per KG16 steps.  Shared-memory
// rows are padded so that the per-step accesses of a warp (16 channels, two
// lanes each) hit distinct banks.
#ifndef SSM_BWD16_KG
#define SSM_BWD16_KG 2           // adjoint steps per dB/dC tile group (1, 2 or 4)
#endif
#ifndef SSM_BWD16_MINB
#define SSM_BWD16_MINB 4         // CTAs per SM the register allocation allows for
#endif
constexpr int T16 = kStateChunk, CH16 = 32, NT16 = 64, KG16 = SSM_BWD16_KG;
static_assert(KG16 == 1 || KG16 == 2 || KG16 == 4, "group length");
constexpr int TILE16 = 36;                                        // tile row stride (floats)
constexpr int H16_BYTES = T16 * 2 * NT16 * (int)sizeof(float4) +  // recomputed states
                          2 * KG16 * 16 * TILE16 * (int)sizeof(float);   // dB / dC tiles
static_assert(T16 % KG16 == 0, "chunk length: a multiple of the group length");

template <typename IO>
__global__ void __launch_bounds__(NT16, SSM_BWD16_MINB)
scan_bwd16_kernel(const Params P) {
    constexpr int NM = 16, S = 8, NP = S / 2, T = T16, TP = T + 1, KG = KG16;
    __shared__ __align__(16) float4 sDW[CH16][TP];   // (delta, delta, w, w), w = delta * u
    __shared__ float sS[CH16][TP], sU[CH16][TP], sG[CH16][TP];
    __shared__ __align__(16) float sB[T][NM], sC[T][NM];   // step-major: 8 states contiguous
    __shared__ float sDu[CH16][TP], sDd[CH16][TP];
    __shared__ float sBias[CH16], sDsk[CH16];
    extern __shared__ __align__(16) float4 dyn16[];
    float4 *sH4 = dyn16;                             // [T][2][NT16]: h_{j-1} of each step
    // per warp and group step, a [16 channels][TILE16] tile; row =
    // [dB 0-7 | dC 0-7 | dB 8-15 | dC 8-15]
    float *sT = reinterpret_cast<float *>(dyn16 + T * 2 * NT16);

    const Pass &ps = P.ps[blockIdx.z];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ch = tid >> 1, half = tid & 1, lch = lane >> 1;
    const int b = blockIdx.y, d0 = blockIdx.x * CH16, d = d0 + ch;
    const int L = P.L, D = P.D, N = P.N, nch = P.nch;
    const bool cvalid = d < D;
    f2 A2[NP], Av[NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        const int n0 = half * S + 2 * q;
        const float x0 = (cvalid && n0 < N) ? ps.A[(long long)d * N + n0] : 0.f;
        const float x1 = (cvalid && n0 + 1 < N) ? ps.A[(long long)d * N + n0 + 1] : 0.f;
        A2[q] = pk(x0 * kLog2e, x1 * kLog2e);
        Av[q] = pk(x0, x1);
    }
    const IO *dtp = (const IO *)ps.dt + ps.dt_off + b * ps.dt_bstride;
    const IO *bp = (const IO *)ps.Bm + ps.bc_off + b * ps.bc_bstride;
    const IO *cp = (const IO *)ps.Cm + ps.bc_off + b * ps.bc_bstride;
    const IO *up = (const IO *)ps.u;
    // this lane's eight states of the chunk-start states [B][D][nch][16]
    float *hcp = ps.hc + ((long long)b * D + d) * nch * NM + half * S;
    if (tid < CH16) {
        const int dd = d0 + tid;
        sBias[tid] = (dd < D && ps.bias) ? ps.bias[dd] : 0.f;
        sDsk[tid] = (dd < D && ps.Dskip) ? ps.Dskip[dd] : 0.f;
    }
    __syncthreads();

    auto pos = [&](int w) { return ps.rev ? L - 1 - w : w; };
    auto sidx = [&](int w) { return ps.stream_rev ? w : pos(w); };
    // staging, fetched a chunk ahead into registers, then committed.  The
    // registers hold the raw loaded values (loads from clamped in-range
    // addresses); conversion and the masks of out-of-range elements wait
    // for commit(), so no thread waits on its loads before the next chunk.
    constexpr int PC = CH16 * T / NT16, PB = NM * T / NT16;
    static_assert(PC * NT16 == CH16 * T && PB * NT16 == NM * T, "staging split");
    IO rdt[PC], ru[PC], rb[PB], rc[PB];
    float rg[PC];
    auto fetch = [&](int c, bool full) {
#pragma unroll
        for (int r = 0; r < PC; ++r) {
            const int i = tid + r * NT16, cc = i / T, j = i % T;
            const int w = min(c * T + j, L - 1), dd = min(d0 + cc, D - 1);
            const long long row = (long long)b * D + dd;
            rdt[r] = dtp[(long long)dd * L + sidx(w)];
            ru[r] = up[row * L + pos(w)];
            if (full) rg[r] = ps.G[row * L + pos(w)];
        }
#pragma unroll
        for (int r = 0; r < PB; ++r) {
            const int i = tid + r * NT16, j = i % T;
            const int nn = min(i / T, N - 1), w = min(c * T + j, L - 1);
            const long long o = (long long)nn * L + sidx(w);
            rb[r] = bp[o];
            if (full) rc[r] = cp[o];
        }
    };
    // full: the pass-2 staging (G and C fetched too)
    auto commit = [&](int c, bool full) {
#pragma unroll
        for (int r = 0; r < PC; ++r) {
            const int i = tid + r * NT16, cc = i / T, j = i % T, w = c * T + j, dd = d0 + cc;
            const bool ok = w < L && dd < D;
            float dl = 0.f, sg = 1.f;
            if (ok) {
                const float x = to_f32(rdt[r]) + sBias[cc];
                if (P.delta_softplus) {
                    dl = softplus_f<IO>(x);             // the forward pass's own forms
                    sg = sigmoid_io<IO>(x);
                } else {
                    dl = x;
                }
            }
            const float uu = ok ? to_f32(ru[r]) : 0.f;
            const float wu = dl * uu;
            sDW[cc][j] = make_float4(dl, dl, wu, wu);
            sS[cc][j] = sg;
            sU[cc][j] = uu;
            sG[cc][j] = (ok && full) ? ps.gscale * rg[r] : 0.f;
        }
#pragma unroll
        for (int r = 0; r < PB; ++r) {
            const int i = tid + r * NT16, nn = i / T, j = i % T;
            const bool okb = c * T + j < L && nn < N;
            sB[j][nn] = okb ? to_f32(rb[r]) : 0.f;
            sC[j][nn] = (okb && full) ? to_f32(rc[r]) : 0.f;
        }
    };
    // one forward step of this lane's eight states
    auto step_fwd = [&](int j, f2 (&h)[NP]) {
        const float4 dv = sDW[ch][j];
        const f2 dd = pk(dv.x, dv.y), ww = pk(dv.z, dv.w);
        const float4 b0 = *(const float4 *)&sB[j][half * S];
        const float4 b1 = *(const float4 *)&sB[j][half * S + 4];
        const f2 bq[NP] = {pk(b0.x, b0.y), pk(b0.z, b0.w), pk(b1.x, b1.y), pk(b1.z, b1.w)};
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            float a0, a1;
            upk(mul2(dd, A2[q]), a0, a1);
            h[q] = fma2(pk(ex2_approx(a0), ex2_approx(a1)), h[q], mul2(bq[q], ww));
        }
    };
    auto save_h = [&](int j, const f2 (&h)[NP]) {
        float v[S];
#pragma unroll
        for (int q = 0; q < NP; ++q) upk(h[q], v[2 * q], v[2 * q + 1]);
        sH4[(2 * j) * NT16 + tid] = make_float4(v[0], v[1], v[2], v[3]);
        sH4[(2 * j + 1) * NT16 + tid] = make_float4(v[4], v[5], v[6], v[7]);
    };

    // ---- pass 1: states at the chunk starts (unless the forward pass
    // stored them)
    if (!P.hc_given) {
        f2 h[NP];
#pragma unroll
        for (int q = 0; q < NP; ++q) h[q] = pk(0.f, 0.f);
        fetch(0, false);
        for (int c = 0; c < nch; ++c) {
            if (cvalid) {
                float v[S];
#pragma unroll
                for (int q = 0; q < NP; ++q) upk(h[q], v[2 * q], v[2 * q + 1]);
                *(float4 *)(hcp + (long long)c * NM) = make_float4(v[0], v[1], v[2], v[3]);
                *(float4 *)(hcp + (long long)c * NM + 4) = make_float4(v[4], v[5], v[6], v[7]);
            }
            commit(c, false);
            __syncthreads();
            if (c + 1 < nch) fetch(c + 1, false);
            const int len = min(T, L - c * T);
            if (len == T) {
#pragma unroll
                for (int j = 0; j < T; ++j) step_fwd(j, h);
            } else {
#pragma unroll 1
                for (int j = 0; j < len; ++j) step_fwd(j, h);
            }
            __syncthreads();
        }
    }

    // ---- pass 2: adjoint, chunks in reverse
    f2 Gc[NP], dA[NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        Gc[q] = pk(0.f, 0.f);
        dA[q] = pk(0.f, 0.f);
    }
    const int slot = blockIdx.x * 2 + warp;                      // 16-channel group
    const bool slot_ok = d0 + warp * 16 < D;
    float *tile = sT + warp * (KG * 16 * TILE16);
    // tile reduction: lane -> group step rk, columns c0 .. c0 + KG - 1 of
    // the row [dB 0-7 | dC 0-7 | dB 8-15 | dC 8-15] (KG <= 4 columns stay
    // inside one block of eight): dC when c0 & 8, states (c0 >> 4) * 8 + c0 % 8
    constexpr int LPS = 32 / KG;                 // lanes per group step
    const int rk = lane / LPS, c0 = (lane % LPS) * KG;
    float *const pdst = ((c0 & 8) ? ps.pdC : ps.pdB) +
                        ((long long)slot * P.B + b) * L * NM + (c0 >> 4) * 8 + (c0 & 7);
    auto load_h = [&](int c, f2 (&h)[NP]) {
        float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
        if (cvalid) {
            v0 = *(const float4 *)(hcp + (long long)c * NM);
            v1 = *(const float4 *)(hcp + (long long)c * NM + 4);
        }
        h[0] = pk(v0.x, v0.y);
        h[1] = pk(v0.z, v0.w);
        h[2] = pk(v1.x, v1.y);
        h[3] = pk(v1.z, v1.w);
    };
    const float dsk = sDsk[ch];                  // this lane's channel's skip weight
    float sum_bias = 0.f, sum_skip = 0.f;        // its dbias and dD terms (half 1)
    // one adjoint step; hh holds h_j of the step being undone on entry and
    // h_{j-1} on exit
    auto step_bwd = [&](int j, int k, f2 (&hh)[NP]) {
        const float4 h0v = sH4[(2 * j) * NT16 + tid], h1v = sH4[(2 * j + 1) * NT16 + tid];
        const f2 hp[NP] = {pk(h0v.x, h0v.y), pk(h0v.z, h0v.w), pk(h1v.x, h1v.y),
                           pk(h1v.z, h1v.w)};
        const float4 dv = sDW[ch][j];
        const f2 dd = pk(dv.x, dv.y), ww = pk(dv.z, dv.w);
        const float gy = sG[ch][j], uu = sU[ch][j];
        const f2 gyy = pk(gy, gy);
        const float4 b0 = *(const float4 *)&sB[j][half * S];
        const float4 b1 = *(const float4 *)&sB[j][half * S + 4];
        const float4 c0 = *(const float4 *)&sC[j][half * S];
        const float4 c1 = *(const float4 *)&sC[j][half * S + 4];
        const f2 bq[NP] = {pk(b0.x, b0.y), pk(b0.z, b0.w), pk(b1.x, b1.y), pk(b1.z, b1.w)};
        const f2 cq[NP] = {pk(c0.x, c0.y), pk(c0.z, c0.w), pk(c1.x, c1.y), pk(c1.z, c1.w)};
        f2 su = pk(0.f, 0.f), sd = pk(0.f, 0.f), dB[NP], dC[NP];
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            float a0, a1;
            upk(mul2(dd, A2[q]), a0, a1);
            const f2 a = pk(ex2_approx(a0), ex2_approx(a1));
            const f2 g = fma2(gyy, cq[q], Gc[q]);         // G_j
            dC[q] = mul2(gyy, hh[q]);                     // gy_j h_j
            dB[q] = mul2(g, ww);                          // G_j delta_j u_j
            su = fma2(g, bq[q], su);                      // sum G B
            const f2 t = mul2(g, mul2(hp[q], a));         // G h_{j-1} a_j
            dA[q] = fma2(t, dd, dA[q]);
            sd = fma2(t, Av[q], sd);                      // sum G h a A
            Gc[q] = mul2(a, g);
            hh[q] = hp[q];
        }
        // du, ddelta of the channel: this half's sums plus the other half's
        float su0, su1, sd0, sd1;
        upk(su, su0, su1);
        upk(sd, sd0, sd1);
        float SU = su0 + su1, SD = sd0 + sd1;
        SU += __shfl_xor_sync(0xffffffffu, SU, 1);
        SD += __shfl_xor_sync(0xffffffffu, SD, 1);
        // du (with the skip term) and the gradient of dt (times softplus'
        // when the forward applied softplus): both halves hold the same
        // channel sums; half 0 stores du, half 1 the dt gradient.  Both
        // accumulate the channel's dbias and dD terms.
        const float du_j = fmaf(gy, dsk, dv.x * SU);
        const float gx = fmaf(uu, SU, SD) * sS[ch][j];
        *(half ? &sDd[ch][j] : &sDu[ch][j]) = half ? gx : du_j;
        sum_bias += gx;
        sum_skip = fmaf(gy, uu, sum_skip);
        float vb[S], vc[S];
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            upk(dB[q], vb[2 * q], vb[2 * q + 1]);
            upk(dC[q], vc[2 * q], vc[2 * q + 1]);
        }
        float *row = tile + (k * 16 + lch) * TILE16 + half * 16;
        *(float4 *)(row) = make_float4(vb[0], vb[1], vb[2], vb[3]);
        *(float4 *)(row + 4) = make_float4(vb[4], vb[5], vb[6], vb[7]);
        *(float4 *)(row + 8) = make_float4(vc[0], vc[1], vc[2], vc[3]);
        *(float4 *)(row + 12) = make_float4(vc[4], vc[5], vc[6], vc[7]);
    };
    // the group's dB, dC partials: step g0 + rk, four columns over 16 channels
    auto reduce_group = [&](int c, int g0, int len) {
        __syncwarp();
        const float *col = tile + rk * 16 * TILE16 + c0;
        const int j = g0 + rk;
        float *dst = pdst + (long long)sidx(c * T + min(j, len - 1)) * NM;
        const bool st = j < len && slot_ok;
        if constexpr (KG == 4) {
            f2 a0 = pk(0.f, 0.f), a1 = a0;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float4 v = *(const float4 *)(col + r * TILE16);
                a0 = add2(a0, pk(v.x, v.y));
                a1 = add2(a1, pk(v.z, v.w));
            }
            float x0, x1, x2, x3;
            upk(a0, x0, x1);
            upk(a1, x2, x3);
            if (st) *(float4 *)dst = make_float4(x0, x1, x2, x3);
        } else if constexpr (KG == 2) {
            f2 a0 = pk(0.f, 0.f);
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float2 v = *(const float2 *)(col + r * TILE16);
                a0 = add2(a0, pk(v.x, v.y));
            }
            float x0, x1;
            upk(a0, x0, x1);
            if (st) *(float2 *)dst = make_float2(x0, x1);
        } else {
            float a0 = 0.f;
#pragma unroll
            for (int r = 0; r < 16; ++r) a0 += col[r * TILE16];
            if (st) *dst = a0;
        }
        __syncwarp();
    };
    auto chunk = [&](auto FULL, int c, int len, f2 (&hh)[NP]) {
        constexpr bool F = decltype(FULL)::value;
        // recompute: h_{j-1} of every step of the chunk, then h_{len-1}
        if (F) {
#pragma unroll
            for (int j = 0; j < T; ++j) {
                save_h(j, hh);
                step_fwd(j, hh);
            }
        } else {
#pragma unroll 1
            for (int j = 0; j < len; ++j) {
                save_h(j, hh);
                step_fwd(j, hh);
            }
        }
#pragma unroll 1
        for (int g0 = (len - 1) / KG * KG; g0 >= 0; g0 -= KG) {
#pragma unroll
            for (int k = KG - 1; k >= 0; --k)
                if (F || g0 + k < len) step_bwd(g0 + k, k, hh);
            reduce_group(c, g0, len);
        }
    };
    f2 hnext[NP];
    fetch(nch - 1, true);
    load_h(nch - 1, hnext);
    for (int c = nch - 1; c >= 0; --c) {
        commit(c, true);
        __syncthreads();
        f2 hh[NP];
#pragma unroll
        for (int q = 0; q < NP; ++q) hh[q] = hnext[q];
        if (c > 0) {
            fetch(c - 1, true);
            load_h(c - 1, hnext);
        }
        const int len = min(T, L - c * T);
        if (len == T) chunk(BoolC<true>(), c, len, hh);
        else chunk(BoolC<false>(), c, len, hh);
        __syncthreads();
        // per-position gradients of this direction
#pragma unroll
        for (int r = 0; r < PC; ++r) {
            const int i = tid + r * NT16, cc = i / T, j = i % T, w = c * T + j, dd = d0 + cc;
            if (w < L && dd < D) {
                const long long prow = ((long long)b * D + dd) * L;
                const float du = sDu[cc][j], gx = sDd[cc][j];
                const long long di = ps.dt_off + b * ps.dt_bstride + (long long)dd * L + sidx(w);
                if (ps.du_io != nullptr) ((IO *)ps.du_io)[prow + pos(w)] = from_f32<IO>(du);
                else ps.du[prow + pos(w)] = du;
                if (ps.ddt_io != nullptr) ((IO *)ps.ddt_io)[di] = from_f32<IO>(gx);
                else ps.ddt[di] = gx;
            }
        }
        __syncthreads();
    }
    // the channel's dbias and dD terms
    if (ps.pbias != nullptr && half == 1 && cvalid) {
        ps.pbias[(long long)b * D + d] = sum_bias;
        ps.pdD[(long long)b * D + d] = sum_skip;
    }
    if (cvalid) {
        float v[S];
#pragma unroll
        for (int q = 0; q < NP; ++q) upk(dA[q], v[2 * q], v[2 * q + 1]);
        float *o = ps.pdA + ((long long)b * D + d) * NM + half * S;
        *(float4 *)o = make_float4(v[0], v[1], v[2], v[3]);
        *(float4 *)(o + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
}

// out[d] = scale * sum over (b, t) of (a + a2)[b][d][t] (* u[b][d][t] when u
// is given); a, a2 at + b * a_bstride + d * L, u [B][D][L].  One CTA per channel, a
// fixed-order tree: deterministic.  dbias (a = ddelta-dt map) and dD
// (a = G, u = the scanned input).
template <typename IO>
__global__ void __launch_bounds__(256)
channel_sum_kernel(const float *__restrict__ a, const float *__restrict__ a2, long long a_bstride,
                   const IO *__restrict__ u, int B, int D, int L, float scale,
                   float *__restrict__ out) {
    __shared__ float red[256];
    const int dch = blockIdx.x;
    // four independent accumulators (positions t, t + 256, t + 512, t + 768
    // of every 1024), so four loads are in flight; combined in a fixed order
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int b = 0; b < B; ++b) {
        const long long o = b * a_bstride + (long long)dch * L;
        const IO *ur = u ? u + ((long long)b * D + dch) * L : nullptr;
        for (int t0 = threadIdx.x; t0 < L; t0 += 1024) {
            float v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int t = t0 + 256 * q;
                v[q] = 0.f;
                if (t < L) {
                    v[q] = a[o + t];
                    if (a2) v[q] += a2[o + t];
                    if (u) v[q] *= to_f32(ur[t]);
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] += v[q];
        }
    }
    red[threadIdx.x] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    __syncthreads();
    for (int s2 = 128; s2 > 0; s2 >>= 1) {
        if (threadIdx.x < s2) red[threadIdx.x] += red[threadIdx.x + s2];
        __syncthreads();
    }
    if (threadIdx.x == 0) out[dch] = scale * red[0];
}

// gy = g * silu(z) (fp32), dz = g * y * silu'(z) (I/O dtype); z == null: gy = g
template <typename IO>
__global__ void gate_bwd_kernel(const IO *__restrict__ g, const IO *__restrict__ z,
                                const IO *__restrict__ y, float *__restrict__ gy,
                                IO *__restrict__ dz, long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const float gv = to_f32(g[i]);
        if (z) {
            const float zv = to_f32(z[i]), s = sigmoid_f(zv);
            gy[i] = gv * zv * s;
            if (dz) dz[i] = from_f32<IO>(gv * to_f32(y[i]) * s * (1.f + zv * (1.f - s)));
        } else {
            gy[i] = gv;
        }
    }
}

// out[m][c][r] = in[m][r][c] for maps of R x C (fp32 or I/O), optionally
// added to a second map: out = add + transpose(in)
template <typename E>
__global__ void transpose_kernel(const E *__restrict__ in, E *__restrict__ out, int maps, int R,
                                 int C) {
    __shared__ E tile[32][33];
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int m = blockIdx.z; m < maps; m += gridDim.z) {
        const E *src = in + (long long)m * R * C;
        E *dst = out + (long long)m * R * C;
        for (int i = ty; i < 32; i += 8) {
            const int r = r0 + i, c = c0 + tx;
            if (r < R && c < C) tile[i][tx] = src[(long long)r * C + c];
        }
        __syncthreads();
        for (int i = ty; i < 32; i += 8) {
            const int c = c0 + i, r = r0 + tx;
            if (r < R && c < C) dst[(long long)c * R + r] = tile[tx][i];
        }
        __syncthreads();
    }
}

// out (I/O or fp32) = a [+ b] [+ c] elementwise, fp32 inputs
template <typename E>
__global__ void convert_kernel(const float *__restrict__ a, const float *__restrict__ b,
                               const float *__restrict__ c, E *__restrict__ out, long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        float v = a[i];
        if (b) v += b[i];
        if (c) v += c[i];
        out[i] = from_f32<E>(v);
    }
}

// dB[b][n][s] (I/O, at out + b * out_bstride) = sum over the nslot partials
// [slot][B][L][nm] (slot-major; a fixed summation order, so the result is
// the same on every run).  One launch reduces up to eight tensors (jobs,
// grid z).  CTA = 256 / (nm / 4) positions of one batch element: thread =
// (position, group of four states), 16-byte loads of the partials, twelve
// in flight, added in slot order; the sums are transposed through shared
// memory so each state's row of positions is stored contiguously.
struct BcJobs {
    const float *part[8];
    void *out[8];
    int nslot[8];
    long long out_bstride;
};
template <typename IO, int NM>
__global__ void __launch_bounds__(256)
reduce_bc_kernel(const BcJobs J, int B, int L, int N) {
    constexpr int QN = NM / 4, PS = 256 / QN;           // quads per position, positions per CTA
    constexpr int KB = 12;                               // partial loads in flight
    __shared__ float tile[NM][PS + 1];
    const float *part = J.part[blockIdx.z];
    IO *out = (IO *)J.out[blockIdx.z];
    const int nslot = J.nslot[blockIdx.z];
    const int b = blockIdx.y, s0 = blockIdx.x * PS;
    const int t = threadIdx.x, sl = t / QN, q = t % QN, s = s0 + sl;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (s < L) {
        const float4 *src = reinterpret_cast<const float4 *>(part) +
                            (((long long)b * L + s) * NM) / 4 + q;
        const long long slot_stride = (long long)B * L * NM / 4;
        for (int k0 = 0; k0 < nslot; k0 += KB) {
            float4 v[KB];
#pragma unroll
            for (int k = 0; k < KB; ++k)
                if (k0 + k < nslot) v[k] = src[(k0 + k) * slot_stride];
#pragma unroll
            for (int k = 0; k < KB; ++k) {
                if (k0 + k < nslot) {
                    acc.x += v[k].x;
                    acc.y += v[k].y;
                    acc.z += v[k].z;
                    acc.w += v[k].w;
                }
            }
        }
    }
    tile[4 * q][sl] = acc.x;
    tile[4 * q + 1][sl] = acc.y;
    tile[4 * q + 2][sl] = acc.z;
    tile[4 * q + 3][sl] = acc.w;
    __syncthreads();
    for (int i = t; i < N * PS; i += 256) {
        const int nn = i / PS, j = i % PS;
        if (s0 + j < L)
            out[b * J.out_bstride + (long long)nn * L + s0 + j] = from_f32<IO>(tile[nn][j]);
    }
}

// Parameter gradients: out = sum over nslot x B partial rows of cols
// values (per_state: [D][nm] rows whose columns past N are padding, stored
// as [D][N]); up to twelve reductions (jobs, grid y) in one launch, each
// summed in the same fixed order.
struct ParamJobs {
    const float *part[12];
    float *out[12];
    int nslot[12];
    int per_state[12];
};
__global__ void reduce_param_kernel(const ParamJobs J, int B, int D, int N, int nm) {
    const float *part = J.part[blockIdx.y];
    float *out = J.out[blockIdx.y];
    const int nslot = J.nslot[blockIdx.y], per_state = J.per_state[blockIdx.y];
    const int cols = per_state ? D * nm : D;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < cols; i += gridDim.x * blockDim.x) {
        if (per_state && i % nm >= N) continue;
        float acc = 0.f;
        for (int k = 0; k < nslot; ++k)
            for (int b = 0; b < B; ++b) acc += part[((long long)k * B + b) * cols + i];
        out[per_state ? (i / nm) * N + i % nm : i] = acc;
    }
}

}  // namespace bwd
}  // namespace ssm
