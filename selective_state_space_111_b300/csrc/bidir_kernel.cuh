// bidir_kernel.cuh -- selective-scan (S6) forward for one direction and for
// Vision Mamba's bidirectional v1/v2 (flip-add), sm_103a.
//
// Recurrence per (batch b, channel d, state n), fp32 state in registers:
//   delta_t = softplus(dt_t + bias_d)
//   h_t[n]  = exp(delta_t * A[d,n]) * h_{t-1}[n] + delta_t * B[n,t] * u_t
//   y_t     = sum_n C[n,t] * h_t[n] + D_d * u_t
// (S6 equations of the Vision Mamba overview page, section
// "选择性扫描机制的计算效率优势", read with exp(delta*A) and delta*B as the
// discretisation; softplus and A = -exp(A_log) from "VMamba的SS2D模块详解"
// sections 3.1-3.2.)  The bidirectional form ("Vision Mamba实战" section
// 2.2, "从Transformer到Mamba" sections 2.2 and 4.3) runs a second branch
// over the reversed sequence and adds its output, flipped back, to the
// forward branch's: y_t = out_scale * (y_fwd[t] + y_bwd[t]), then the gate
// y_t * silu(z_t) ("VMamba的SS2D模块详解" section 2.1).
//
// The path is bound by the arithmetic of the recurrence (per element update
// four fp32 operations and one MUFU ex2; see the roofline in the design
// notes), so the kernel is organised to spend its issue slots there:
//
//   pack_bc_kernel  B and C ([B, N, L], I/O dtype) are converted once per
//                   batch element into a packed fp32 stream BC[b][t][32] =
//                   (B_0..B_15, C_0..C_15) -- 128 bytes per position, so one
//                   chunk of positions is one contiguous, aligned range.
//   bidir_scan_kernel
//     CTA    = G channels of one batch element x NDIR branches.
//     lane   = (branch, channel, state group): S of the 16 states of one
//              channel; LPR = 16 / S lanes share a channel.  The states are
//              packed fp32 pairs updated with the f32x2 MUL/FMA forms.
//     time   = chunks of T positions.  Everything a chunk reads arrives by
//              bulk copies (TMA, cp.async.bulk) completing on mbarriers:
//              per branch one copy of the packed B/C range (2-deep ring),
//              one per dt / u / z row segment (3-deep ring, issued two
//              chunks ahead) and one per fp32 stash / accumulator segment.
//              Rows of odd length do not start on 16 bytes, so a segment
//              copies the whole 16-byte vectors covering it; TMA tensor
//              maps cannot describe such rows (their stride must be a
//              multiple of 16 bytes).
//     phases = prep  (delta, w = delta * u) once per (branch, channel, step);
//              scan  T steps per lane; the lane's partial readout per step
//                    goes to shared memory;
//              epilogue sums the partials, adds D*u, fuses the branches,
//                    gates and stores.
//              prep and epilogue run one warp per (branch, channel) row and
//              one lane per position, so row constants are warp-uniform and
//              global stores are coalesced.
//
// Flip-add without flipped copies.  At chunk c the forward branch covers
// positions [cT, cT+T) and the backward branch [L-cT-T, L-cT) (clipped),
// walking them downward.  Position p is reached by the forward branch at
// chunk p/T and by the backward branch at chunk (L-1-p)/T.  The branch that
// reaches p first leaves its output (with its D*u term) in the fp32 stash
// W[p]; the second one reads it back, fuses, gates and stores y.  When both
// reach p in the same chunk, the forward branch finalises p from the
// backward branch's partials in shared memory.
#pragma once

#include "scan_ops.cuh"

namespace ssm {

constexpr int kBC = 2 * kMaxN;   // floats per position in the packed B/C stream

struct BiBranch {
    const void *dt;        // delta tensor (I/O dtype, 16-byte aligned); row
                           // (b, d) of this branch starts at element
                           // dt_off + b * dt_bstride + d * L
    const void *u;         // [B, D, L] I/O dtype, position order
    const float *bc;       // [B, L, 32] packed B/C of this branch
    const float *A;        // [D, N]
    const float *Dskip;    // [D] or null
    const float *bias;     // [D] or null
    long long dt_off;      // elements to this branch's first row
    long long dt_bstride;  // elements between batch elements of dt
    long long dt_total;    // elements in the whole dt tensor (tail guard)
    int stream_rev;        // backward branch only: dt and B/C are stored in
                           // walk order (index L-1-p for position p)
};

// What the finalising branch does with the fused value v = out_scale *
// (y_fwd + y_bwd) of a position:
//   OUT_Y      gate with z, store y (I/O dtype);
//   OUT_ACC    store v to acc_out (fp32, no gate);
//   OUT_ADD_Y  add acc_in (fp32), gate with z, store y.
enum { OUT_Y = 0, OUT_ACC = 1, OUT_ADD_Y = 2 };

struct BiParams {
    BiBranch br[2];
    const void *z;         // [B, D, L] or null
    void *y;               // [B, D, L]
    const float *acc_in;   // [B, D, L] fp32 (OUT_ADD_Y)
    float *acc_out;        // [B, D, L] fp32 (OUT_ACC)
    float *W;              // [B, D, L] fp32 stash (two branches, several chunks)
    unsigned *status;      // device status word, or null
    long long total;       // B * D * L
    int B, D, L, N;
    int nchunks;
    int delta_softplus;
    float out_scale;
};

// ------------------------------------------------------------------ pack
// B, C: [Bt, K, N, L] (K = 1 for the sequence forms).  For direction k,
// batch b and position t: out[((k * Bt + b) * L + t) * 32 + j] = B[b,k,j,t]
// (j < 16), C[b,k,j-16,t] (j >= 16); 0 for state indices >= N.
// Block: 64 positions of one (b, k), 256 threads; block (0,0,0) also clears
// the status word so that the scan kernel of the same call can set it.
template <typename IO>
__global__ void __launch_bounds__(256)
pack_bc_kernel(const IO *__restrict__ Bm, const IO *__restrict__ Cm, float *__restrict__ out,
               int N, int L, unsigned *status) {
    __shared__ float tile[kBC][65];
    const int b = blockIdx.y, k = blockIdx.z, t0 = blockIdx.x * 64;
    const int Bt = gridDim.y, K = gridDim.z;
    if (status != nullptr && blockIdx.x == 0 && b == 0 && k == 0 && threadIdx.x == 0) *status = 0;
    for (int i = threadIdx.x; i < kBC * 64; i += 256) {
        const int j = i >> 6, tt = i & 63, t = t0 + tt, n = j & (kMaxN - 1);
        float v = 0.f;
        if (t < L && n < N) {
            const IO *src = j < kMaxN ? Bm : Cm;
            v = to_f32(src[(((long long)b * K + k) * N + n) * L + t]);
        }
        tile[j][tt] = v;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 64 * kBC; i += 256) {
        const int tt = i >> 5, j = i & 31, t = t0 + tt;
        if (t < L) out[(((long long)k * Bt + b) * L + t) * kBC + j] = tile[j][tt];
    }
}

// ------------------------------------------------------------------ transpose
// out[m][c][r] = in[m][r][c] for maps m of R x C elements (32 x 32 tiles).
template <typename E>
__global__ void __launch_bounds__(256)
transpose_maps_kernel(const E *__restrict__ in, E *__restrict__ out, int maps, int R, int C) {
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

// ------------------------------------------------------------------ layout
template <typename IO, int S, int NDIR, int G, int T>
struct BiLayout {
    static constexpr int LPR = kMaxN / S;
    static constexpr int NT = NDIR * G * LPR;
    static constexpr int VEC = 16 / (int)sizeof(IO);       // elements per 16 B
    static constexpr int NRAW = 3;                         // raw ring depth
    static constexpr int NBC = 2;                          // B/C ring depth
    static constexpr int RC = T + 2 * VEC;                 // raw row capacity
    static constexpr int RAW_ROW = RC * (int)sizeof(IO);   // bytes
    static constexpr int RAW_DIR = 3 * G * RAW_ROW;        // dt[G], u[G], z[G]
    static constexpr int RAW_STAGE = NDIR * RAW_DIR;
    static constexpr int W_CAP = T + 8;                    // fp32 covering capacity
    static constexpr int W_ROW = W_CAP * 4;
    static constexpr int BC_DIR = T * kBC * 4;
    static constexpr int BC_STAGE = NDIR * BC_DIR;
    static constexpr int DW_ROW = T * 16 + 16;             // float4 per step, padded
    static constexpr int YP_ROW = (T * LPR + LPR) * 4;     // padded: banks spread

    static constexpr int off_bc = 0;                       // 128-byte aligned
    static constexpr int off_raw = off_bc + NBC * BC_STAGE;
    static constexpr int off_w = off_raw + NRAW * RAW_STAGE;
    static constexpr int off_dw = off_w + 2 * NDIR * G * W_ROW;   // stash, acc_in
    static constexpr int off_yp = off_dw + NDIR * G * DW_ROW;
    static constexpr int off_bar = (off_yp + NDIR * G * YP_ROW + 7) & ~7;
    static constexpr int bytes = off_bar + (NBC + NRAW + 1) * 8;

    static_assert(T % 8 == 0 && T % VEC == 0, "T must be a multiple of 8");
    static_assert(RAW_ROW % 16 == 0 && W_ROW % 16 == 0 && DW_ROW % 16 == 0, "alignment");
    static_assert(S == 4 || S == 8 || S == 16, "S must be 4, 8 or 16");
    static_assert(NT % 32 == 0, "a CTA must be whole warps");

    __device__ static IO *raw(char *sm, int stage, int d, int k, int r) {
        return (IO *)(sm + off_raw + stage * RAW_STAGE + d * RAW_DIR + (k * G + r) * RAW_ROW);
    }
};

// Positions [lo, lo + len) of branch d at chunk c (both branches have the
// same len at every chunk).
__device__ __forceinline__ void chunk_geom(int c, int d, int L, int T, int &lo, int &len) {
    if (d == 0) {
        lo = c * T;
        len = min(T, L - lo);
    } else {
        const int hi = L - c * T;
        lo = max(0, hi - T);
        len = hi - lo;
    }
}

// Stage elements [a, e) of the row that starts at element `rowbase` of a
// global array of `total` elements into dst_row, so that element a + q lands
// at dst_row[(rowbase + a) % VEC + q]: one bulk copy of the whole 16-byte
// vectors covering the range (announced on `bar` first), and element-wise
// copies for a last vector of the array that is not whole.
template <typename E>
__device__ __forceinline__ void stage_bulk(E *dst_row, const E *src, long long rowbase, int a,
                                           int e, long long total, uint64_t *bar) {
    constexpr int VEC = 16 / (int)sizeof(E);
    if (e <= a) return;
    const long long e0 = rowbase + a, e1 = rowbase + e;
    const long long v0 = e0 / VEC;
    const long long v1 = (e1 + VEC - 1) / VEC;
    const long long vfull = total / VEC;
    const long long vb = v1 < vfull ? v1 : vfull;
    if (vb > v0) {
        const unsigned bytes = (unsigned)((vb - v0) * 16);
        mbar_expect_tx(bar, bytes);
        bulk_g2s(dst_row, src + v0 * VEC, bytes, bar);
    }
    for (long long x = (vb > v0 ? vb : v0) * VEC; x < e1; ++x) dst_row[x - v0 * VEC] = src[x];
}

// ------------------------------------------------------------------ kernel
template <typename IO, int S, int NDIR, int G, int T, int OUT>
__global__ void __launch_bounds__(BiLayout<IO, S, NDIR, G, T>::NT)
bidir_scan_kernel(const BiParams P) {
    using LY = BiLayout<IO, S, NDIR, G, T>;
    constexpr int LPR = LY::LPR;
    constexpr int NT = LY::NT;
    constexpr int NW = NT / 32;
    constexpr int VEC = LY::VEC;
    constexpr int NP = S / 2;                  // packed state pairs per lane
    constexpr int U = 4;                       // scan unroll (steps)
    constexpr bool USE_W = NDIR == 2 || OUT == OUT_ADD_Y;

    extern __shared__ __align__(128) char sm[];
    uint64_t *bc_bar = (uint64_t *)(sm + LY::off_bar);     // [NBC], one arrival
    uint64_t *raw_bar = bc_bar + LY::NBC;                    // [NRAW], NT arrivals
    uint64_t *w_bar = raw_bar + LY::NRAW;                    // [1], NT arrivals
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.y;
    const int d0 = blockIdx.x * G;
    const int L = P.L, D = P.D, N = P.N;
    const long long bD = (long long)b * D;

    // ---- scan role of this lane
    const int s_dir = tid / (G * LPR);
    const int s_row = (tid / LPR) % G;
    const int s_sg = tid % LPR;
    const int s_ch = d0 + s_row;
    f2 A2[NP], h[NP];
    {
        const float *A = P.br[s_dir].A;
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            const int n0 = s_sg * S + 2 * q;
            const bool ok = s_ch < D;
            const float a0 = (ok && n0 < N) ? A[(long long)s_ch * N + n0] * kLog2e : 0.f;
            const float a1 = (ok && n0 + 1 < N) ? A[(long long)s_ch * N + n0 + 1] * kLog2e : 0.f;
            A2[q] = pk(a0, a1);
            h[q] = pk(0.f, 0.f);
        }
    }

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < LY::NBC; ++s) mbar_init(&bc_bar[s], 1);
#pragma unroll
        for (int s = 0; s < LY::NRAW; ++s) mbar_init(&raw_bar[s], NT);
        mbar_init(w_bar, NT);
        fence_barrier_init();
    }
    __syncthreads();

    // ---- chunk sub-ranges (positions)
    // first stream index (dt, B/C) of branch d at chunk c
    auto stream_lo = [&](int c, int d, int lo) { return P.br[d].stream_rev ? c * T : lo; };
    // positions branch d finalises at chunk c
    auto final_range = [&](int c, int d, int lo, int len, int &a, int &e) {
        a = lo;
        e = lo + len;
        if (NDIR == 2) {
            if (d == 0) a = max(lo, L - (c + 1) * T);
            else e = min(lo + len, c * T);
        }
    };
    // positions whose other branch reached them at an earlier chunk
    auto stash_range = [&](int c, int d, int lo, int len, int &a, int &e) {
        a = lo;
        e = lo + len;
        if (d == 0) a = max(lo, L - c * T);
        else e = min(lo + len, c * T);
    };

    // ---- staging: bulk copies (TMA) completing on mbarriers
    auto issue_bc = [&](int c) {
        if (tid != 0 || c >= P.nchunks) return;
        const int st = c % LY::NBC;
        int lo, len;
        chunk_geom(c, 0, L, T, lo, len);
        mbar_arrive_expect_tx(&bc_bar[st], (unsigned)(NDIR * len * kBC * 4));
#pragma unroll
        for (int d = 0; d < NDIR; ++d) {
            chunk_geom(c, d, L, T, lo, len);
            bulk_g2s(sm + LY::off_bc + st * LY::BC_STAGE + d * LY::BC_DIR,
                     P.br[d].bc + ((long long)b * L + stream_lo(c, d, lo)) * kBC,
                     (unsigned)(len * kBC * 4), &bc_bar[st]);
        }
    };
    // dt, u and z rows of chunk c: one segment per (branch, tensor, channel)
    auto issue_raw = [&](int c) {
        if (c >= P.nchunks) return;
        const int st = c % LY::NRAW;
        uint64_t *bar = &raw_bar[st];
        for (int sg = tid; sg < NDIR * 3 * G; sg += NT) {
            const int r = sg % G;
            const int k = (sg / G) % 3;
            const int d = sg / (3 * G);
            const int ch = d0 + r;
            if (ch >= D) continue;
            int lo, len, a, e;
            chunk_geom(c, d, L, T, lo, len);
            const BiBranch &br = P.br[d];
            if (k == 0) {
                a = stream_lo(c, d, lo);
                stage_bulk<IO>(LY::raw(sm, st, d, 0, r), (const IO *)br.dt,
                               br.dt_off + b * br.dt_bstride + (long long)ch * L, a, a + len,
                               br.dt_total, bar);
            } else if (k == 1) {
                stage_bulk<IO>(LY::raw(sm, st, d, 1, r), (const IO *)br.u, (bD + ch) * L, lo,
                               lo + len, P.total, bar);
            } else if (OUT != OUT_ACC && P.z != nullptr) {
                final_range(c, d, lo, len, a, e);
                stage_bulk<IO>(LY::raw(sm, st, d, 2, r), (const IO *)P.z, (bD + ch) * L, a, e,
                               P.total, bar);
            }
        }
        mbar_arrive(bar);
    };
    // fp32 rows of chunk c: the stash W over the second-arrival range and,
    // for OUT_ADD_Y, acc_in over the final range
    auto issue_w = [&](int c) {
        if constexpr (!USE_W) return;
        if (c >= P.nchunks) return;
        for (int sg = tid; sg < 2 * NDIR * G; sg += NT) {
            const int r = sg % G;
            const int d = (sg / G) % NDIR;
            const int which = sg / (G * NDIR);
            const int ch = d0 + r;
            if (ch >= D) continue;
            int lo, len, a, e;
            chunk_geom(c, d, L, T, lo, len);
            float *dst = (float *)(sm + LY::off_w + ((which * NDIR + d) * G + r) * LY::W_ROW);
            if (which == 0) {
                if (NDIR == 1) continue;
                stash_range(c, d, lo, len, a, e);
                stage_bulk<float>(dst, P.W, (bD + ch) * L, a, e, P.total, w_bar);
            } else if (OUT == OUT_ADD_Y) {
                final_range(c, d, lo, len, a, e);
                stage_bulk<float>(dst, P.acc_in, (bD + ch) * L, a, e, P.total, w_bar);
            }
        }
        mbar_arrive(w_bar);
    };

    // ---- prep: (delta, delta, w, w) per (branch, channel, walk step);
    // one warp per (branch, channel) row, one lane per position
    auto prep = [&](int c) {
        const int st = c % LY::NRAW;
        for (int row = warp; row < NDIR * G; row += NW) {
            const int d = row / G, r = row % G;
            const int ch = d0 + r;
            int lo, len;
            chunk_geom(c, d, L, T, lo, len);
            float4 *dwr = (float4 *)(sm + LY::off_dw + row * LY::DW_ROW);
            if (ch >= D) {
                for (int q = lane; q < len; q += 32) dwr[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                continue;
            }
            const BiBranch &br = P.br[d];
            const float bias = br.bias ? br.bias[ch] : 0.f;
            const bool srev = br.stream_rev != 0;
            const IO *rdt = LY::raw(sm, st, d, 0, r) +
                            (int)((br.dt_off + b * br.dt_bstride + (long long)ch * L +
                                   stream_lo(c, d, lo)) & (VEC - 1));
            const IO *ru = LY::raw(sm, st, d, 1, r) + (int)(((bD + ch) * L + lo) & (VEC - 1));
            for (int q = lane; q < len; q += 32) {
                const int j = d ? len - 1 - q : q;
                const float x = to_f32(rdt[srev ? j : q]) + bias;
                const float dl = P.delta_softplus ? softplus_f<IO>(x) : x;
                const float w = dl * to_f32(ru[q]);
                dwr[j] = make_float4(dl, dl, w, w);
            }
        }
    };

    // ---- scan of one chunk by this lane
    auto scan = [&](int c) -> bool {
        const int stb = c % LY::NBC;
        const bool ok = mbar_wait_bounded(&bc_bar[stb], (unsigned)((c / LY::NBC) & 1));
        int lo, len;
        chunk_geom(c, s_dir, L, T, lo, len);
        const char *dwp = sm + LY::off_dw + (s_dir * G + s_row) * LY::DW_ROW;
        const float *bcp = (const float *)(sm + LY::off_bc + stb * LY::BC_STAGE +
                                           s_dir * LY::BC_DIR) + s_sg * S;
        int bstep = kBC;
        if (s_dir == 1 && !P.br[1].stream_rev) {   // backward walk over a
            bcp += (len - 1) * kBC;                 // position-ordered stream
            bstep = -kBC;
        }
        float *ypp = (float *)(sm + LY::off_yp + (s_dir * G + s_row) * LY::YP_ROW) + s_sg;
        auto step = [&](int j) {
            const float4 v = *(const float4 *)(dwp + j * 16);
            const f2 dd = pk(v.x, v.y), ww = pk(v.z, v.w);
            const float *bj = bcp + j * bstep;
            f2 bq[NP], cq[NP];
#pragma unroll
            for (int k = 0; k < S / 4; ++k) {
                const float4 vb = *(const float4 *)(bj + 4 * k);
                const float4 vc = *(const float4 *)(bj + kMaxN + 4 * k);
                bq[2 * k] = pk(vb.x, vb.y);
                bq[2 * k + 1] = pk(vb.z, vb.w);
                cq[2 * k] = pk(vc.x, vc.y);
                cq[2 * k + 1] = pk(vc.z, vc.w);
            }
            f2 y2;
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                float a0, a1;
                upk(mul2(dd, A2[q]), a0, a1);
                const f2 e = pk(ex2_approx(a0), ex2_approx(a1));
                h[q] = fma2(e, h[q], mul2(bq[q], ww));
                y2 = (q == 0) ? mul2(cq[q], h[q]) : fma2(cq[q], h[q], y2);
            }
            float ylo, yhi;
            upk(y2, ylo, yhi);
            ypp[j * LPR] = ylo + yhi;
        };
        int j = 0;
        for (; j + U <= len; j += U) {
#pragma unroll
            for (int jj = 0; jj < U; ++jj) step(j + jj);
        }
        for (; j < len; ++j) step(j);
        return ok;
    };

    // sum of the LPR partial readouts at walk step j of a row
    auto ypsum = [&](const float *yrow, int j) -> float {
        const float *ps = yrow + j * LPR;
        if constexpr (LPR == 4) {
            const float4 v = *(const float4 *)ps;
            return (v.x + v.y) + (v.z + v.w);
        } else if constexpr (LPR == 2) {
            const float2 v = *(const float2 *)ps;
            return v.x + v.y;
        } else {
            return ps[0];
        }
    };

    // ---- epilogue of one chunk; one warp per (branch, channel) row
    auto epilogue = [&](int c) {
        const int st = c % LY::NRAW;
        int lo0, len, lo1 = 0;
        chunk_geom(c, 0, L, T, lo0, len);
        if (NDIR == 2) chunk_geom(c, 1, L, T, lo1, len);
        for (int row = warp; row < NDIR * G; row += NW) {
            const int d = row / G, r = row % G;
            const int ch = d0 + r;
            if (ch >= D) continue;
            const long long rowbase = (bD + ch) * L;
            const int lo = d ? lo1 : lo0;
            const BiBranch &br = P.br[d];
            const float dsk = br.Dskip ? br.Dskip[ch] : 0.f;
            const float *yown = (const float *)(sm + LY::off_yp + row * LY::YP_ROW);
            const IO *ru = LY::raw(sm, st, d, 1, r) + (int)((rowbase + lo) & (VEC - 1)) ;
            int fa, fe, wa, we;
            final_range(c, d, lo, len, fa, fe);
            stash_range(c, d, lo, len, wa, we);
            const IO *rz = LY::raw(sm, st, d, 2, r) + (int)((rowbase + fa) & (VEC - 1));
            const float *wst = (const float *)(sm + LY::off_w + row * LY::W_ROW) +
                               (int)((rowbase + wa) & 3);
            const float *acc = (const float *)(sm + LY::off_w + (NDIR * G + row) * LY::W_ROW) +
                               (int)((rowbase + fa) & 3);
            // the backward branch's row, for positions both reach in this chunk
            const float *yoth = (const float *)(sm + LY::off_yp + ((NDIR - 1) * G + r) * LY::YP_ROW);
            const float dsko = (NDIR == 2 && P.br[NDIR - 1].Dskip) ? P.br[NDIR - 1].Dskip[ch] : 0.f;
            const IO *ruo = LY::raw(sm, st, NDIR - 1, 1, r) + (int)((rowbase + lo1) & (VEC - 1));
            for (int q = lane; q < len; q += 32) {
                const int p = lo + q;
                // 0: first arrival (stash), 1: second arrival (stash holds
                // the other branch), 2: both in this chunk, 3: left to branch 0
                int cls = 1;
                if (NDIR == 2) {
                    if (d == 0) cls = (p < L - (c + 1) * T) ? 0 : (p >= L - c * T ? 1 : 2);
                    else cls = (p >= (c + 1) * T) ? 0 : (p < c * T ? 1 : 3);
                }
                if (cls == 3) continue;
                const int j = d ? len - 1 - q : q;
                const float yv = fmaf(dsk, to_f32(ru[q]), ypsum(yown, j));
                if (NDIR == 2 && cls == 0) {
                    P.W[rowbase + p] = yv;
                    continue;
                }
                float v = yv;
                if (NDIR == 2) {
                    const float other =
                        cls == 1 ? wst[p - wa]
                                 : fmaf(dsko, to_f32(ruo[p - lo1]), ypsum(yoth, L - 1 - p - c * T));
                    v = P.out_scale * (yv + other);
                }
                if (OUT == OUT_ACC) {
                    P.acc_out[rowbase + p] = v;
                    continue;
                }
                if (OUT == OUT_ADD_Y) v += acc[p - fa];
                if (P.z) v *= silu_f<IO>(to_f32(rz[p - fa]));
                ((IO *)P.y)[rowbase + p] = from_f32<IO>(v);
            }
        }
        // the stash stores must precede the bulk copies that read them back
        if (NDIR == 2) fence_proxy_async_global();
    };

    // ---- pipeline.  Ring depths: raw 3 (issued two chunks ahead), B/C 2,
    // fp32 rows 1 (issued after the previous chunk's epilogue).
    bool ok = true;
    issue_bc(0);
    issue_bc(1);
    issue_raw(0);
    issue_raw(1);
    issue_raw(2);
    issue_w(0);
    ok &= mbar_wait_bounded(&raw_bar[0], 0u);
    prep(0);
    __syncthreads();
    for (int c = 0; c < P.nchunks; ++c) {
        ok &= scan(c);
        if (c + 1 < P.nchunks)
            ok &= mbar_wait_bounded(&raw_bar[(c + 1) % LY::NRAW], (unsigned)(((c + 1) / LY::NRAW) & 1));
        if (USE_W) ok &= mbar_wait_bounded(w_bar, (unsigned)(c & 1));
        if (__syncthreads_or(!ok)) {
            // a bulk copy did not land in time: report, drain what was
            // issued (bounded), leave
            if (tid == 0 && P.status != nullptr) atomicOr(P.status, 1u);
            const int last_raw = min(c + 2, P.nchunks - 1);
            for (int k = max(0, last_raw - LY::NRAW + 1); k <= last_raw; ++k)
                mbar_wait_bounded(&raw_bar[k % LY::NRAW], (unsigned)((k / LY::NRAW) & 1));
            const int last_bc = min(c + 1, P.nchunks - 1);
            for (int k = max(0, last_bc - LY::NBC + 1); k <= last_bc; ++k)
                mbar_wait_bounded(&bc_bar[k % LY::NBC], (unsigned)((k / LY::NBC) & 1));
            if (USE_W) mbar_wait_bounded(w_bar, (unsigned)(c & 1));
            return;
        }
        epilogue(c);
        if (c + 1 < P.nchunks) prep(c + 1);
        __syncthreads();
        issue_bc(c + 2);
        issue_w(c + 1);
        issue_raw(c + 3);
    }
}

}  // namespace ssm
