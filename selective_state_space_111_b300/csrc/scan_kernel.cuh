// scan_kernel.cuh -- the selective-scan (S6) forward kernel for sm_103a.
//
// One kernel template serves every form of the scan:
//   * NDIR = 1: a single direction (selective_scan_fwd);
//   * NDIR = 2: a forward and a backward branch over the same positions
//     (BiMamba v1/v2 flip-add, and each half of SS2D's cross-scan).
//
// Recurrence per (batch b, channel d, state n), fp32 state in registers:
//   delta_t = softplus(dt_t + bias_d)
//   h_t[n]  = exp(delta_t * A[d,n]) * h_{t-1}[n] + delta_t * B[n,t] * u_t
//   y_t     = sum_n C[n,t] * h_t[n] + D_d * u_t
// (S6 equations of the Vision Mamba overview page, section
// "选择性扫描机制的计算效率优势", with exp(delta*A) / delta*B discretisation;
// softplus and A = -exp(A_log) from "VMamba的SS2D模块详解" sections 3.1-3.2.)
//
// Work decomposition
//   CTA     = G channels of one batch element, all NDIR directions.
//   lane    = one (direction, channel) x S of its 16 states; LPR = 16/S
//             consecutive lanes share a channel.  The states live in
//             registers as packed fp32 pairs and are updated with the
//             f32x2 FMA/MUL forms; exp uses the MUFU ex2 unit.
//   time    = walked in chunks of T steps.  Inputs for chunk c+2 are in
//             flight (cp.async, 16-byte vectors) while chunk c is scanned.
//   per chunk: convert  raw dt/u/B/C -> fp32 (delta, delta, w=delta*u, w)
//                        and B/C as [step][n] in shared memory (once per
//                        (row, step), shared by the LPR lanes and all rows);
//              scan     each lane runs T steps over its S states and writes
//                        its partial readout per step;
//              epilogue per position: sum the lanes' partials, add D*u,
//                        fuse the two branches, gate, store.
//
// Directions and the flip-add fusion ("Vision Mamba实战" section 2.2,
// "从Transformer到Mamba" sections 2.2/4.3).  Positions p in [0, L) are in
// "pair order".  The forward branch walks p upward, the backward branch
// walks p downward from L-1; at chunk c they cover
//   fwd: [cT, cT+T)        bwd: [L-cT-T, L-cT)      (clipped to [0, L)).
// A position is reached by both branches, at chunks floor(p/T) (fwd) and
// floor((L-1-p)/T) (bwd).  The branch that gets there second finalises it:
// it takes the other branch's output from shared memory when both reach it
// in the same chunk, and otherwise from the fp32 slot W[p] in which the
// first branch left it.  No flipped copy of any tensor is ever made: the
// flip is the direction of the walk.
//
// Position -> memory maps.  u (x), z, y and W are addressed through
//   MAP_ROW: offset(p) = p                  (sequence / row-major map)
//   MAP_COL: offset(p) = (p % H) * W + p / H (column-major walk of an H x W
//                                             map, SS2D directions 1 and 3)
// Each branch's delta / B / C stream is contiguous in its own order:
//   stream_rev = 0: stream index = p        (BiMamba: original token order)
//   stream_rev = 1: stream index = L-1-p    (SS2D reversed directions, whose
//                                            streams are in scan order)
//
// Output modes
//   MODE_FINAL  : y = out_scale * (y_fwd + y_bwd), gated, stored to y.
//   MODE_ACCOUT : the fused value is stored to W (fp32) instead of y
//                 (SS2D row-major pair, first launch).
//   MODE_ACCIN  : W already holds the other pair's sum; the first branch to
//                 reach p adds its output into W, the second reads W, adds
//                 its own output, gates and stores y (SS2D column pair).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr int kMaxN = 16;      // states per channel held by the kernel
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum { MAP_ROW = 0, MAP_COL = 1 };
enum { MODE_FINAL = 0, MODE_ACCOUT = 1, MODE_ACCIN = 2 };

// ------------------------------------------------------------------ params
struct DirArgs {
    const void *dt;        // delta tensor base (16-byte aligned)
    long long dt_off;      // element offset of this direction's slice
    long long dt_bs;       // element offset of (b, d): dt_off + b*dt_bs + d*L
    const void *Bm;        // B tensor base (16-byte aligned)
    const void *Cm;
    long long bc_off;      // element offset of this direction's slice
    long long bc_bs;       // element offset of (b, n): bc_off + b*bc_bs + n*L
    long long dt_total;    // elements in the whole delta tensor (tail guard)
    long long bc_total;    // elements in each whole B / C tensor
    const float *A;        // [D, N] (already offset to this direction)
    const float *Dskip;    // [D] or null
    const float *bias;     // [D] or null
    const void *u;         // [B, D, L] in position space (u or u_b)
    int stream_rev;
};

struct KParams {
    DirArgs dir[2];
    const void *z;         // [B, D, L] or null
    void *y;               // [B, D, L]
    float *W;              // [B, D, L] fp32 workspace (null if not needed)
    long long u_total;     // elements in u / z / y / W
    int B, D, L, N, H, Wd; // H, Wd: map size for MAP_COL
    int nchunks;
    int delta_softplus;
    float out_scale;
};

// ------------------------------------------------------------------ helpers
typedef unsigned long long f2;  // two fp32 in one 64-bit register pair

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
template <typename IO> __device__ __forceinline__ IO from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// softplus and the SiLU gate.  fp32 I/O uses the accurate library functions;
// bf16 I/O uses the MUFU forms (ex2 / lg2 / rcp), whose relative error
// (about 2e-4 on delta for delta near 1e-3, far less elsewhere) is two orders
// of magnitude below the bf16 output rounding.
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

// ------------------------------------------------------------------ layout
// Shared-memory layout, sizes in bytes; every region 16-byte aligned.
template <typename IO, int S, int NDIR, int G, int T>
struct Smem {
    static constexpr int VEC = 16 / (int)sizeof(IO);        // elements per 16 B
    static constexpr int RC = T + VEC;                      // raw row capacity
    static constexpr int RAW_ROW = RC * (int)sizeof(IO);    // bytes (16-aligned)
    static constexpr int LPR = kMaxN / S;
    // raw rows per direction and stage: dt[G], u[G], z[G], B[16], C[16]
    static constexpr int RAW_ROWS = 3 * G + 2 * kMaxN;
    static constexpr int RAW_DIR = RAW_ROWS * RAW_ROW;
    static constexpr int RAW_STAGE = NDIR * RAW_DIR;
    static constexpr int W_ROW = (T + 4) * 4;               // fp32, VEC 4
    static constexpr int DW_ROW = T * 16 + 16;              // float4 / step, padded
    static constexpr int BC_DIR = T * 2 * kMaxN * 4;        // [T][B0..15 C0..15]
    static constexpr int Y_ROW = T * LPR * 4 + 16;          // [T][LPR] fp32, padded

    static constexpr int off_raw = 0;                       // [2 stages]
    static constexpr int off_w = off_raw + 2 * RAW_STAGE;   // [NDIR][G] rows
    static constexpr int off_dw = off_w + NDIR * G * W_ROW; // [NDIR][G]
    static constexpr int off_bc = off_dw + NDIR * G * DW_ROW;
    static constexpr int off_y = off_bc + NDIR * BC_DIR;
    static constexpr int bytes = off_y + NDIR * G * Y_ROW;

    // raw rows inside a stage/direction
    static constexpr int R_DT = 0, R_U = G, R_Z = 2 * G, R_B = 3 * G, R_C = 3 * G + kMaxN;
    __device__ static char *raw_row(char *sm, int stage, int d, int row) {
        return sm + off_raw + stage * RAW_STAGE + d * RAW_DIR + row * RAW_ROW;
    }
};

// Chunk geometry of direction d at chunk c.
struct Range {
    int lo, len;        // positions [lo, lo + len)
    int s_lo;           // first stream index of the chunk
};
__device__ __forceinline__ Range chunk_range(int d, int c, int L, int T, int stream_rev) {
    Range r;
    if (d == 0) {
        r.lo = c * T;
        r.len = min(T, L - r.lo);
    } else {
        int hi = L - c * T;
        r.lo = max(0, hi - T);
        r.len = hi - r.lo;
    }
    r.s_lo = stream_rev ? (L - r.lo - r.len) : r.lo;
    return r;
}

// Copy elements [e0, e0 + len) of a global array with `total` elements into
// a shared row so that element e0 + i lands at row[(e0 % VEC) + i].  Whole
// 16-byte vectors are copied (cp.async); a vector reaching past the end of
// the array is copied element by element.  `part`/`nparts` spread the
// vectors over the threads that share the segment.
template <typename E, bool VIA_L1 = false>
__device__ __forceinline__ void stage_segment(E *row, const E *src, long long e0, int len,
                                              long long total, int part, int nparts) {
    constexpr int VEC = 16 / (int)sizeof(E);
    if (len <= 0) return;
    long long v0 = e0 / VEC;
    long long v1 = (e0 + len + VEC - 1) / VEC;
    for (long long v = v0 + part; v < v1; v += nparts) {
        E *dst = row + (v - v0) * VEC;
        const E *s = src + v * VEC;
        if ((v + 1) * VEC <= total) {
            if (VIA_L1) cp_async16_ca(dst, s);
            else cp_async16(dst, s);
        } else {
            for (int k = 0; k < VEC && v * VEC + k < total; ++k) dst[k] = s[k];
        }
    }
}

// Offset in u/z/y/W of position p of row (b, d).
template <int MAP>
__device__ __forceinline__ long long pos_offset(const KParams &P, long long rowbase, int p) {
    if (MAP == MAP_ROW) return rowbase + p;
    return rowbase + (long long)(p % P.H) * P.Wd + p / P.H;
}

// The sub-ranges whose z (finalise) and W (second arrival) are needed at
// chunk c for direction d.  Both are contiguous within the chunk.
struct Sub { int a, b; };
__device__ __forceinline__ Sub final_sub(int NDIR, int d, int c, int L, int T, Range r) {
    Sub s{r.lo, r.lo + r.len};
    if (NDIR == 1) return s;
    if (d == 0) s.a = max(r.lo, L - (c + 1) * T);        // bwd reached p at chunk <= c
    else s.b = min(r.lo + r.len, c * T);                  // fwd reached p at chunk < c
    if (s.b < s.a) s.b = s.a;
    return s;
}
__device__ __forceinline__ Sub second_sub(int NDIR, int MODE, int d, int c, int L, int T, Range r) {
    Sub s{r.lo, r.lo + r.len};
    if (MODE == MODE_ACCIN) return s;                     // every arrival reads W
    if (NDIR == 1) { s.b = s.a; return s; }
    if (d == 0) s.a = max(r.lo, L - c * T);               // bwd reached p at chunk < c
    else s.b = min(r.lo + r.len, c * T);                  // fwd reached p at chunk < c
    if (s.b < s.a) s.b = s.a;
    return s;
}

// ------------------------------------------------------------------ kernel
template <typename IO, int S, int NDIR, int G, int T, int MAP, int MODE>
__global__ void __launch_bounds__(NDIR * G * (kMaxN / S))
scan_kernel(const KParams P) {
    using SM = Smem<IO, S, NDIR, G, T>;
    constexpr int LPR = kMaxN / S;
    constexpr int NT = NDIR * G * LPR;
    constexpr int VEC = SM::VEC;
    constexpr int NP = S / 2;              // packed pairs per lane
    static_assert(S % 4 == 0 && T % 4 == 0, "S and T must be multiples of 4");

    extern __shared__ __align__(16) char sm[];
    const int tid = threadIdx.x;
    const int b = blockIdx.y;
    const int d0 = blockIdx.x * G;         // first channel of this CTA
    const int L = P.L;
    const int N = P.N;

    // ---- lane role in the scan
    const int s_dir = tid / (G * LPR);
    const int s_rem = tid % (G * LPR);
    const int s_row = s_rem / LPR;
    const int s_sg = s_rem % LPR;
    const int s_ch = d0 + s_row;
    f2 A2[NP], h[NP];
    {
        const float *A = P.dir[s_dir].A;
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            int n0 = s_sg * S + 2 * q;
            float a0 = (s_ch < P.D && n0 < N) ? A[(long long)s_ch * N + n0] * kLog2e : 0.f;
            float a1 = (s_ch < P.D && n0 + 1 < N) ? A[(long long)s_ch * N + n0 + 1] * kLog2e : 0.f;
            A2[q] = pk(a0, a1);
            h[q] = pk(0.f, 0.f);
        }
    }

    // ---- staging of chunk c into raw stage (c & 1)
    auto issue_raw = [&](int c) {
        if (c >= P.nchunks) return;
        const int st = c & 1;
        // segments: per dir: G dt rows, G u rows, G z rows, N B rows, N C rows
        constexpr int SEG_PER_DIR = 3 * G + 2 * kMaxN;
        constexpr int NVEC = (T + VEC - 1) / VEC + 1;       // vectors per segment
        for (int item = tid; item < NDIR * SEG_PER_DIR * NVEC; item += NT) {
            const int part = item % NVEC;
            const int seg = item / NVEC;
            const int d = seg / SEG_PER_DIR;
            const int k = seg % SEG_PER_DIR;
            const DirArgs &A = P.dir[d];
            const Range r = chunk_range(d, c, L, T, A.stream_rev);
            const IO *srcbase;
            long long e0, total;
            int len;
            if (k < G) {                                  // delta stream
                int ch = d0 + k;
                if (ch >= P.D) continue;
                srcbase = (const IO *)A.dt;
                e0 = A.dt_off + (long long)b * A.dt_bs + (long long)ch * L + r.s_lo;
                len = r.len;
                total = A.dt_total;
            } else if (k < 2 * G) {                       // u (position space)
                if (MAP != MAP_ROW) continue;
                int ch = d0 + (k - G);
                if (ch >= P.D) continue;
                srcbase = (const IO *)A.u;
                e0 = ((long long)b * P.D + ch) * L + r.lo;
                len = r.len;
                total = P.u_total;
            } else if (k < 3 * G) {                       // z, finalised sub-range
                if (MAP != MAP_ROW || MODE == MODE_ACCOUT || P.z == nullptr) continue;
                int ch = d0 + (k - 2 * G);
                if (ch >= P.D) continue;
                Sub s = final_sub(NDIR, d, c, L, T, r);
                srcbase = (const IO *)P.z;
                e0 = ((long long)b * P.D + ch) * L + s.a;
                len = s.b - s.a;
                total = P.u_total;
            } else {                                      // B or C rows
                int kk = k - 3 * G;
                int n = kk % kMaxN;
                if (n >= N) continue;
                srcbase = (const IO *)(kk < kMaxN ? A.Bm : A.Cm);
                e0 = A.bc_off + (long long)b * A.bc_bs + (long long)n * L + r.s_lo;
                len = r.len;
                total = A.bc_total;
            }
            IO *row = (IO *)SM::raw_row(sm, st, d, k);
            stage_segment<IO>(row, srcbase, e0, len, total, part, NVEC);
        }
    };
    // W prefetch for chunk c (fp32), rows laid out [d][row]
    auto issue_w = [&](int c) {
        if (MODE == MODE_FINAL && NDIR == 1) return;
        if (MAP != MAP_ROW || c >= P.nchunks) return;
        constexpr int NVEC = (T + 3) / 4 + 1;
        for (int item = tid; item < NDIR * G * NVEC; item += NT) {
            const int part = item % NVEC;
            const int seg = item / NVEC;
            const int d = seg / G, rr = seg % G;
            const int ch = d0 + rr;
            if (ch >= P.D) continue;
            const Range r = chunk_range(d, c, L, T, P.dir[d].stream_rev);
            Sub s = second_sub(NDIR, MODE, d, c, L, T, r);
            float *row = (float *)(sm + SM::off_w + (d * G + rr) * SM::W_ROW);
            stage_segment<float, true>(row, P.W, ((long long)b * P.D + ch) * L + s.a, s.b - s.a,
                                 P.u_total, part, NVEC);
        }
    };

    // ---- convert raw chunk c -> (delta, delta, w, w) and B/C as fp32
    auto convert = [&](int c) {
        const int st = c & 1;
        const int len4 = (min(T, L - c * T) + 3) & ~3;    // same length both dirs
        // delta / w
        for (int item = tid; item < NDIR * G * len4; item += NT) {
            const int j = item % len4;
            const int rr = (item / len4) % G;
            const int d = item / (len4 * G);
            const DirArgs &A = P.dir[d];
            const Range r = chunk_range(d, c, L, T, A.stream_rev);
            const int ch = d0 + rr;
            float dl = 0.f, w = 0.f;
            if (ch < P.D && j < r.len) {
                const bool rev_walk = (d == 1);
                const int si = (rev_walk && !A.stream_rev) ? r.len - 1 - j : j;
                const long long e_dt = A.dt_off + (long long)b * A.dt_bs + (long long)ch * L + r.s_lo;
                const IO *rdt = (const IO *)SM::raw_row(sm, st, d, SM::R_DT + rr);
                float x = to_f32(rdt[(int)(e_dt % VEC) + si]);
                if (A.bias) x += A.bias[ch];
                dl = P.delta_softplus ? softplus_f<IO>(x) : x;
                const int p = rev_walk ? r.lo + r.len - 1 - j : r.lo + j;
                float uu;
                if (MAP == MAP_ROW) {
                    const long long e_u = ((long long)b * P.D + ch) * L + r.lo;
                    const IO *ru = (const IO *)SM::raw_row(sm, st, d, SM::R_U + rr);
                    uu = to_f32(ru[(int)(e_u % VEC) + (p - r.lo)]);
                } else {
                    uu = to_f32(((const IO *)A.u)[pos_offset<MAP>(P, ((long long)b * P.D + ch) * L, p)]);
                }
                w = dl * uu;
            }
            float4 *dst = (float4 *)(sm + SM::off_dw + (d * G + rr) * SM::DW_ROW) + j;
            *dst = make_float4(dl, dl, w, w);
        }
        // B / C: items (d, j, which, n4) -> 4 consecutive states
        for (int item = tid; item < NDIR * len4 * 8; item += NT) {
            const int n4 = item % 4;
            const int which = (item / 4) % 2;             // 0 = B, 1 = C
            const int j = (item / 8) % len4;
            const int d = item / (8 * len4);
            const DirArgs &A = P.dir[d];
            const Range r = chunk_range(d, c, L, T, A.stream_rev);
            float v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int n = n4 * 4 + k;
                v[k] = 0.f;
                if (n < N && j < r.len) {
                    const bool rev_walk = (d == 1);
                    const int si = (rev_walk && !A.stream_rev) ? r.len - 1 - j : j;
                    const long long e = A.bc_off + (long long)b * A.bc_bs + (long long)n * L + r.s_lo;
                    const IO *rw = (const IO *)SM::raw_row(sm, st, d, (which ? SM::R_C : SM::R_B) + n);
                    v[k] = to_f32(rw[(int)(e % VEC) + si]);
                }
            }
            float4 *dst = (float4 *)(sm + SM::off_bc + d * SM::BC_DIR) + j * 8 + which * 4 + n4;
            *dst = make_float4(v[0], v[1], v[2], v[3]);
        }
    };

    // ---- the scan over one chunk
    auto scan = [&](int c) {
        const int len4 = (min(T, L - c * T) + 3) & ~3;
        const char *dwp = sm + SM::off_dw + (s_dir * G + s_row) * SM::DW_ROW;
        const char *bcp = sm + SM::off_bc + s_dir * SM::BC_DIR;
        float *yp = (float *)(sm + SM::off_y + (s_dir * G + s_row) * SM::Y_ROW) + s_sg;
        for (int j0 = 0; j0 < len4; j0 += 4) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int j = j0 + jj;
                f2 dd, ww, bq[NP], cq[NP];
                {
                    const float4 v = *(const float4 *)(dwp + j * 16);
                    dd = pk(v.x, v.y);
                    ww = pk(v.z, v.w);
                }
#pragma unroll
                for (int q = 0; q < NP; q += 2) {
                    const float4 vb = *(const float4 *)(bcp + j * 128 + (s_sg * S + 2 * q) * 4);
                    const float4 vc = *(const float4 *)(bcp + j * 128 + 64 + (s_sg * S + 2 * q) * 4);
                    bq[q] = pk(vb.x, vb.y);
                    bq[q + 1] = pk(vb.z, vb.w);
                    cq[q] = pk(vc.x, vc.y);
                    cq[q + 1] = pk(vc.z, vc.w);
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
                yp[j * LPR] = ylo + yhi;
            }
        }
    };

    // ---- epilogue of chunk c
    auto epilogue = [&](int c) {
        const int st = c & 1;
        const int clen = min(T, L - c * T);
        for (int item = tid; item < NDIR * G * clen; item += NT) {
            const int q = item % clen;
            const int rr = (item / clen) % G;
            const int d = item / (clen * G);
            const int ch = d0 + rr;
            if (ch >= P.D) continue;
            const DirArgs &A = P.dir[d];
            const Range r = chunk_range(d, c, L, T, A.stream_rev);
            const int p = r.lo + q;
            const long long rowbase = ((long long)b * P.D + ch) * L;
            // this branch's output at p
            auto branch_out = [&](int dd, const Range &rg, int pp) -> float {
                const int j = (dd == 0) ? pp - rg.lo : rg.lo + rg.len - 1 - pp;
                const float *ps = (const float *)(sm + SM::off_y + (dd * G + rr) * SM::Y_ROW) + j * LPR;
                float v;
                if constexpr (LPR == 4) {
                    const float4 part = *(const float4 *)ps;
                    v = (part.x + part.y) + (part.z + part.w);
                } else {
                    const float2 part = *(const float2 *)ps;
                    v = part.x + part.y;
                }
                const DirArgs &AD = P.dir[dd];
                if (AD.Dskip) {
                    float uu;
                    if (MAP == MAP_ROW) {
                        const long long e_u = rowbase + rg.lo;
                        const IO *ru = (const IO *)SM::raw_row(sm, st, dd, SM::R_U + rr);
                        uu = to_f32(ru[(int)(e_u % VEC) + (pp - rg.lo)]);
                    } else {
                        uu = to_f32(((const IO *)AD.u)[pos_offset<MAP>(P, rowbase, pp)]);
                    }
                    v = fmaf(AD.Dskip[ch], uu, v);
                }
                return v;
            };
            const float yv = branch_out(d, r, p);
            // classify
            int other_chunk;          // chunk at which the other branch reaches p
            if (NDIR == 1) other_chunk = c;
            else other_chunk = (d == 0) ? (L - 1 - p) / T : p / T;
            if (NDIR == 2 && d == 1 && other_chunk == c) continue;   // fwd side finalises
            // W value at p (second arrival or ACCIN)
            auto w_at = [&]() -> float {
                if (MAP == MAP_ROW) {
                    Sub s = second_sub(NDIR, MODE, d, c, L, T, r);
                    const long long e = rowbase + s.a;
                    const float *rw = (const float *)(sm + SM::off_w + (d * G + rr) * SM::W_ROW);
                    return rw[(int)(e % 4) + (p - s.a)];
                }
                return P.W[pos_offset<MAP>(P, rowbase, p)];
            };
            const long long off = pos_offset<MAP>(P, rowbase, p);
            if (NDIR == 2 && other_chunk > c) {          // first arrival
                if (MODE == MODE_ACCIN) P.W[off] = w_at() + yv;
                else P.W[off] = yv;
                continue;
            }
            float v;
            if (NDIR == 1) {
                v = yv;
            } else {
                float other;
                if (other_chunk == c) {
                    const Range rb = chunk_range(1, c, L, T, P.dir[1].stream_rev);
                    other = branch_out(1, rb, p);
                } else {
                    other = 0.f;   // taken from W below
                }
                if (MODE == MODE_ACCIN) {
                    v = yv + other + w_at();
                } else {
                    if (other_chunk < c) other = w_at();
                    v = P.out_scale * (yv + other);
                }
            }
            if (MODE == MODE_ACCOUT) {
                P.W[off] = v;
                continue;
            }
            if (P.z) {
                float zz;
                if (MAP == MAP_ROW) {
                    Sub s = final_sub(NDIR, d, c, L, T, r);
                    const long long e = rowbase + s.a;
                    const IO *rz = (const IO *)SM::raw_row(sm, st, d, SM::R_Z + rr);
                    zz = to_f32(rz[(int)(e % VEC) + (p - s.a)]);
                } else {
                    zz = to_f32(((const IO *)P.z)[off]);
                }
                v *= silu_f<IO>(zz);
            }
            ((IO *)P.y)[off] = from_f32<IO>(v);
        }
    };

    // ---- pipeline
    issue_raw(0);
    cp_async_commit();
    issue_raw(1);
    issue_w(0);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    convert(0);
    __syncthreads();
    for (int c = 0; c < P.nchunks; ++c) {
        scan(c);
        cp_async_wait<0>();               // raw(c+1) and W(c) have landed
        __syncthreads();
        epilogue(c);
        if (c + 1 < P.nchunks) convert(c + 1);
        __syncthreads();
        issue_raw(c + 2);
        issue_w(c + 1);
        cp_async_commit();
    }
}

}  // namespace ssm
