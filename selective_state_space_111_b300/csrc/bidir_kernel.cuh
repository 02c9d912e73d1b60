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
// four fp32 operations and one MUFU ex2), so the kernel is organised to
// spend its issue slots there:
//
//   pack_bc_kernel  B and C ([B, N, L], I/O dtype) are converted once per
//                   batch element into a packed fp32 stream BC[b][t][2NM] =
//                   (B_0..B_{NM-1}, C_0..C_{NM-1}) for a state capacity NM of
//                   16 or 32 (128 or 256 bytes per position), so one chunk of
//                   positions is one contiguous, aligned range that a single
//                   bulk copy (cp.async.bulk) moves to shared memory.
//   bidir_scan_kernel
//     CTA  = R channels of one batch element x NDIR branches, T = 32
//            positions per chunk, in three warp roles linked by full/empty
//            mbarrier rings:
//     scan warps      lane = (branch, channel, group of S states); the states
//                     are packed fp32 pairs (f32x2 MUL/FMA); per step the
//                     lane's partial readout goes to shared memory;
//     prep warps      lane = walk step; dt and u are read element by element
//                     (32 consecutive positions per row, coalesced) one chunk
//                     ahead; delta = softplus(dt + bias) and w = delta * u
//                     are computed once per (branch, channel, step);
//     epilogue warps  lane = position; sum the partial readouts, add D * u,
//                     fuse the branches, gate and store (coalesced); one lane
//                     issues the B/C bulk copies.
//     Every wait is bounded in time; on expiry the kernel sets the status
//     word and all roles stop.
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

// State capacity NM (16 or 32, a template parameter): the packed B/C stream
// holds 2 * NM floats per position (B_0..B_{NM-1}, C_0..C_{NM-1}).

#ifndef SSM_SCAN_BLOCK
#define SSM_SCAN_BLOCK 4         // scan steps per block (loads, then ex2, then recurrences)
#endif

struct BiBranch {
    const void *dt;        // delta tensor (I/O dtype); row
                           // (b, d) of this branch starts at element
                           // dt_off + b * dt_bstride + d * L
    const void *u;         // [B, D, L] I/O dtype, position order
    const float *bc;       // [B, L, 32] packed B/C of this branch
    const float *A;        // [D, N]
    const float *Dskip;    // [D] or null
    const float *bias;     // [D] or null
    long long dt_off;      // elements to this branch's first row
    long long dt_bstride;  // elements between batch elements of dt
    int stream_rev;        // backward branch only: dt and B/C are stored in
                           // walk order (index L-1-p for position p)
    int u_stream_rev;      // backward branch only: u is stored in walk order too
};

// What the finalising branch does with the fused value v = out_scale *
// (y_fwd + y_bwd) of a position:
//   OUT_Y      gate with z, store y (I/O dtype);
//   OUT_ACC    store v to acc_out (fp32, no gate);
//   OUT_ADD_Y  add acc_in (fp32), gate with z, store y;
//   OUT_Y_PRE  as OUT_Y, and also store v itself (before the gate) to ypre
//              (I/O dtype): the pre-gate output the backward pass needs.
enum { OUT_Y = 0, OUT_ACC = 1, OUT_ADD_Y = 2, OUT_Y_PRE = 3 };

struct BiParams {
    BiBranch br[2];
    const void *z;         // [B, D, L] or null
    void *y;               // [B, D, L]
    void *ypre;            // [B, D, L] (OUT_Y_PRE)
    const float *acc_in;   // [B, D, L] fp32 (OUT_ADD_Y)
    float *acc_out;        // [B, D, L] fp32 (OUT_ACC)
    float *W;              // [B, D, L] fp32 stash (two branches, several chunks)
    float *last_state[2];  // per branch: final state [B, D, N] fp32, or null
    // per branch: the state before every kStateChunk-th walk step, [B, D,
    // ceil(L / kStateChunk), 16] fp32 (walk chunk k holds the state after
    // walk steps 0 .. k * kStateChunk - 1), or null; state capacity 16
    // only.  The backward pass starts its recomputation from these.
    float *chunk_state[2];
    unsigned *status;      // device status word, or null
    int B, D, L, N;
    int nchunks;
    int delta_softplus;
    float out_scale;
    int withhold_bc;       // test hook: chunk whose B/C copy is never issued (-1: none)
    // extents (elements) for the debug build's index checks: each branch's
    // dt tensor and packed B/C buffer from their base pointers, the [B, D, L]
    // tensors (u, u_b, z, y, W, acc_in, acc_out), A [D, N]
    long long dt_elems[2], bc_elems[2], io_elems, a_elems;
};

// ------------------------------------------------------------------ pack
// B, C: [Bt, K, N, L] (K = 1 for the sequence forms).  For direction k,
// batch b and position t: out[((k * Bt + b) * L + t) * 2NM + j] = B[b,k,j,t]
// (j < NM), C[b,k,j-NM,t] (j >= NM); 0 for state indices >= N.
// Block: pack_pt<NM>() positions of one (b, k) (256 for 16 states, 128 for
// 32: 8192 values, 32 loads per thread in flight), 256 threads; block
// (0,0,0) also clears the status word so that the scan kernel of the same
// call can set it.
// With Bm1 given, grid z = 2 packs two separate sets (v2's two branches) in
// one launch: z = 0 the first (Bm, Cm -> out), z = 1 the second (Bm1, Cm1 ->
// out1), each with K = 1.
template <int NM> __host__ __device__ constexpr int pack_pt() { return 8192 / (2 * NM); }
template <typename IO, int NM>
__global__ void __launch_bounds__(256)
pack_bc_kernel(const IO *__restrict__ Bm, const IO *__restrict__ Cm, float *__restrict__ out,
               int N, int L, unsigned *status, const IO *__restrict__ Bm1 = nullptr,
               const IO *__restrict__ Cm1 = nullptr, float *__restrict__ out1 = nullptr) {
    // extents of B, C (each [Bt, K, N, L]) and of the packed output
    // [K, Bt, L, 2NM] (per set when two sets are packed), for the debug checks
    const long long in_elems = (long long)gridDim.y * (Bm1 != nullptr ? 1 : gridDim.z) * N * L;
    const long long out_elems = (long long)(Bm1 != nullptr ? 1 : gridDim.z) * gridDim.y * L * 2 * NM;
    (void)in_elems;                  // read by the debug build's checks only
    (void)out_elems;
    constexpr int kBC = 2 * NM, PT = pack_pt<NM>();
    __shared__ float tile[kBC][PT + 1];
    const int b = blockIdx.y, t0 = blockIdx.x * PT;
    int k = blockIdx.z, K = gridDim.z;
    const int Bt = gridDim.y;
    if (status != nullptr && blockIdx.x == 0 && b == 0 && blockIdx.z == 0 && threadIdx.x == 0)
        *status = 0;
    if (Bm1 != nullptr) {
        if (k == 1) {
            Bm = Bm1;
            Cm = Cm1;
            out = out1;
        }
        k = 0;
        K = 1;
    }
    float v[kBC * PT / 256];
#pragma unroll
    for (int r = 0; r < kBC * PT / 256; ++r) {
        const int i = threadIdx.x + r * 256, j = i / PT, tt = i % PT, t = t0 + tt;
        const int n = j & (NM - 1);
        v[r] = 0.f;
        if (t < L && n < N) {
            const IO *src = j < NM ? Bm : Cm;
            const long long o = (((long long)b * K + k) * N + n) * L + t;
            if (SSM_IN(o, in_elems, status)) v[r] = to_f32(src[o]);
        }
    }
#pragma unroll
    for (int r = 0; r < kBC * PT / 256; ++r) {
        const int i = threadIdx.x + r * 256;
        tile[i / PT][i % PT] = v[r];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < PT * kBC; i += 256) {
        const int tt = i / kBC, j = i % kBC, t = t0 + tt;
        const long long o = (((long long)k * Bt + b) * L + t) * kBC + j;
        if (t < L && SSM_IN(o, out_elems, status)) out[o] = tile[j][tt];
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

// out[m][c][r] = in[m][r][c] for maps small enough to sit whole in shared
// memory (R x (C + 1) elements, at most 48 KB): a CTA takes whole maps, so a
// map is read and written as one contiguous run (warp w, lane l: rows
// w, w + 8, ... in, columns w, w + 8, ... out; the padded row keeps the
// column reads free of bank conflicts).  SMALL (R, C <= 64): the loads are
// unrolled so that all of a thread's are in flight at once.
template <typename E, bool SMALL>
__global__ void __launch_bounds__(256)
transpose_whole_maps_kernel(const E *__restrict__ in, E *__restrict__ out, int maps, int R,
                            int C) {
    extern __shared__ __align__(16) unsigned char tw_smem[];
    E *tile = (E *)tw_smem;                                  // [R][C + 1]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int m = blockIdx.x; m < maps; m += gridDim.x) {
        const E *src = in + (long long)m * R * C;
        E *dst = out + (long long)m * R * C;
        if constexpr (SMALL) {
            // R, C <= 64: a thread's 16 elements, every load in flight
            // before the shared stores
            E v[8][2];
#pragma unroll
            for (int k = 0; k < 8; ++k)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int r = warp + 8 * k, c = lane + 32 * q;
                    if (r < R && c < C) v[k][q] = src[r * C + c];
                }
#pragma unroll
            for (int k = 0; k < 8; ++k)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int r = warp + 8 * k, c = lane + 32 * q;
                    if (r < R && c < C) tile[r * (C + 1) + c] = v[k][q];
                }
        } else {
            for (int r = warp; r < R; r += 8)
                for (int c = lane; c < C; c += 32)
                    tile[r * (C + 1) + c] = src[(long long)r * C + c];
        }
        __syncthreads();
        for (int c = warp; c < C; c += 8)
            for (int r = lane; r < R; r += 32) dst[(long long)c * R + r] = tile[r * (C + 1) + c];
        __syncthreads();
    }
}

// ------------------------------------------------------------------ layout
// One CTA = R channels of one batch element x NDIR branches, in warps with
// three roles linked by full/empty mbarrier rings (T = 32 positions per
// chunk, one lane per position in the prep and epilogue roles):
//   scan warps  (NSW)  lane = (branch, channel, state group)
//   prep warps  (NPW)  16 rows each: delta and w = delta*u from dt, u
//   epi warps   (NEW)  16 rows each (both branches of 16/NDIR channels):
//                      readout sums, D*u, fusion, gate, stores; lane 0 of
//                      the first epilogue warp also issues the B/C copies
template <typename IO, int S, int NDIR, int R, int NM = kMaxN>
struct WsLayout {
    static constexpr int T = 32;
    static constexpr int kBC = 2 * NM;                      // floats per packed position
    static constexpr int LPR = NM / S;
    static constexpr int ROWS = NDIR * R;                   // (branch, channel) rows
    static constexpr int NSW = ROWS * LPR / 32;
    static constexpr int NPW = ROWS / 16;
    static constexpr int NEW = ROWS / 16;
    static constexpr int CPE = 16 / NDIR;                   // channels per epilogue warp
    static constexpr int NT = (NSW + NPW + NEW) * 32;
    static constexpr int NBC = 2;                           // B/C ring
    static constexpr int BC_DIR = T * kBC * 4;
    static constexpr int BC_STAGE = NDIR * BC_DIR;
    static constexpr int DW_ROW = T * 16 + 16;              // float4 per step, padded
    static constexpr int DW_STAGE = ROWS * DW_ROW;
    // partial readouts stored per (row, step): lanes of more than two per
    // channel sum pairs with a shuffle first, so the stage stays small
    static constexpr int YP = LPR > 2 ? 2 : LPR;
    static constexpr int YP_ROW = (T * YP + YP) * 4;        // padded: banks spread
    static constexpr int YP_STAGE = ROWS * YP_ROW;
    static constexpr int U_STAGE = ROWS * T * (int)sizeof(IO);   // u in walk order
    static constexpr int off_bc = 0;                        // 128-byte aligned
    static constexpr int off_dw = off_bc + NBC * BC_STAGE;
    static constexpr int off_yp = off_dw + 2 * DW_STAGE;
    static constexpr int NU = R < 16 ? 2 : 4;               // u ring (prep -> epilogue)
    static constexpr int off_u = off_yp + 2 * YP_STAGE;
    static constexpr int off_bar = (off_u + NU * U_STAGE + 7) & ~7;
    // bc_full[NBC], dw_full[2], dw_empty[2], yp_full[2], yp_empty[2], u_empty[NU]
    static constexpr int NBAR = NBC + 8 + NU;
    static constexpr int off_flag = off_bar + NBAR * 8;
    static constexpr int off_tab = off_flag + 16;             // D and bias per row
    static constexpr int bytes = off_tab + 2 * ROWS * 4;     // D, then bias

    static_assert(S == 4 || S == 8 || S == 16, "S must be 4, 8 or 16");
    static_assert(NM == 16 || NM == 32, "state capacity 16 or 32");
    static_assert((ROWS * LPR) % 32 == 0 && ROWS % 16 == 0, "whole warps per role");
    static_assert(R % 16 == 0 || (R == 8 && NDIR == 2),
                  "a prep warp takes 16 channels of one branch, or 8 of each");
    // CTAs per SM that the shared memory allows (228 KB per SM, 1 KB
    // reserved per CTA), and registers per thread so that they all fit:
    // each of the 4 schedulers of an SM has its own 16 K registers and holds
    // up to ceil(CPS * NT / 128) warps
    static constexpr int CPS_SMEM = 233472 / (bytes + 1024);
    static constexpr int CPS = CPS_SMEM < 64 * 32 / NT ? CPS_SMEM : 64 * 32 / NT;
    static constexpr int WPS = (CPS * NT / 32 + 3) / 4;
    static constexpr int MAX_REGS = (16384 / (32 * WPS)) / 8 * 8 > 255 ? 255 : (16384 / (32 * WPS)) / 8 * 8;
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

// ------------------------------------------------------------------ kernel
template <typename IO, int S, int NDIR, int R, int OUT, int NM = kMaxN>
__global__ void __maxnreg__((WsLayout<IO, S, NDIR, R, NM>::MAX_REGS))
bidir_scan_kernel(const BiParams P) {
    using LY = WsLayout<IO, S, NDIR, R, NM>;
    constexpr int kBC = LY::kBC;
    constexpr int T = LY::T;
    constexpr int LPR = LY::LPR;
    constexpr int NSW = LY::NSW, NPW = LY::NPW;
    constexpr int NP = S / 2;                  // packed state pairs per lane
    constexpr int UB = SSM_SCAN_BLOCK;         // scan block (steps)

    extern __shared__ __align__(128) char sm[];
    uint64_t *bar = (uint64_t *)(sm + LY::off_bar);
    uint64_t *bc_full = bar;                   // count 1 (+ transaction bytes)
    uint64_t *dw_full = bar + LY::NBC;         // count NPW*32
    uint64_t *dw_empty = dw_full + 2;          // count NSW*32
    uint64_t *yp_full = dw_empty + 2;          // count NSW*32
    uint64_t *yp_empty = yp_full + 2;          // count NEW*32
    uint64_t *u_empty = yp_empty + 2;          // count NEW*32 (u ring, NU deep)
    volatile int *abort_flag = (volatile int *)(sm + LY::off_flag);
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.y;
    const int d0 = blockIdx.x * R;
    const int L = P.L, D = P.D;
    const int nch = P.nchunks;
    const long long bD = (long long)b * D;

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < LY::NBC; ++s) mbar_init(&bc_full[s], 1);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            mbar_init(&dw_full[s], NPW * 32);
            mbar_init(&dw_empty[s], NSW * 32);
            mbar_init(&yp_full[s], NSW * 32);
            mbar_init(&yp_empty[s], LY::NEW * 32);
        }
#pragma unroll
        for (int s = 0; s < LY::NU; ++s) mbar_init(&u_empty[s], LY::NEW * 32);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // a bounded wait that ran out: every role stops at its next check
    auto give_up = [&]() {
        *abort_flag = 1;
        if (P.status != nullptr) atomicOr(P.status, 1u);
    };
    auto wait = [&](uint64_t *bar_, int parity) -> bool {
        if (mbar_wait_bounded(bar_, (unsigned)parity)) return true;
        give_up();
        return false;
    };
    auto stream_lo = [&](int c, int d, int lo) { return P.br[d].stream_rev ? c * T : lo; };

    if (warp < NSW) {
        // ================================================================ scan
        const int s_dir = tid / (R * LPR);
        const int s_row = (tid / LPR) % R;
        const int s_sg = tid % LPR;
        const int s_ch = d0 + s_row;
        const int N = P.N;
        f2 A2[NP], h[NP];
        {
            const float *A = P.br[s_dir].A;
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const int n0 = s_sg * S + 2 * q;
                const bool ok = s_ch < D;
                const bool in0 = ok && n0 < N && SSM_IN((long long)s_ch * N + n0, P.a_elems, P.status);
                const bool in1 =
                    ok && n0 + 1 < N && SSM_IN((long long)s_ch * N + n0 + 1, P.a_elems, P.status);
                const float a0 = in0 ? A[(long long)s_ch * N + n0] * kLog2e : 0.f;
                const float a1 = in1 ? A[(long long)s_ch * N + n0 + 1] * kLog2e : 0.f;
                A2[q] = pk(a0, a1);
                h[q] = pk(0.f, 0.f);
            }
        }
        const bool walk_down = s_dir == 1 && !P.br[1].stream_rev;
        // this lane's eight states of the chunk-state output (16 states)
        float *cs = (NM == kMaxN && s_ch < D) ? P.chunk_state[s_dir] : nullptr;
        const long long cs_chunks = (L + kStateChunk - 1) / kStateChunk;
        const long long cs_off = ((bD + s_ch) * cs_chunks) * NM + s_sg * S;
        const long long cs_elems = (long long)P.B * D * cs_chunks * NM;
        (void)cs_elems;
        if (cs != nullptr) cs += cs_off;
        for (int c = 0; c < nch; ++c) {
            const int s2 = c & 1, sb = c % LY::NBC;
            if (*abort_flag || !wait(&dw_full[s2], (c >> 1) & 1) ||
                !wait(&bc_full[sb], (c / LY::NBC) & 1) || !wait(&yp_empty[s2], ((c >> 1) & 1) ^ 1))
                return;
            int lo, len;
            chunk_geom(c, s_dir, L, T, lo, len);
            const char *dwp = sm + LY::off_dw + s2 * LY::DW_STAGE + (s_dir * R + s_row) * LY::DW_ROW;
            const float *bcp = (const float *)(sm + LY::off_bc + sb * LY::BC_STAGE +
                                               s_dir * LY::BC_DIR) + s_sg * S;
            int bstep = kBC;
            if (walk_down) {                   // backward walk over a position-ordered stream
                bcp += (len - 1) * kBC;
                bstep = -kBC;
            }
            float *ypp = (float *)(sm + LY::off_yp + s2 * LY::YP_STAGE +
                                   (s_dir * R + s_row) * LY::YP_ROW) + s_sg / (LPR / LY::YP);
            // the chunk's shared-memory reads and writes stay inside their
            // stages (debug build; a chunk that fails is not scanned)
            if (!SSM_IN((dwp - sm) - LY::off_dw + (len - 1) * 16 + 15, 2 * LY::DW_STAGE, P.status) ||
                !SSM_IN((const char *)(bcp + (bstep < 0 ? (len - 1) * bstep : 0)) - sm - LY::off_bc,
                        LY::NBC * LY::BC_STAGE, P.status) ||
                !SSM_IN((const char *)(bcp + (bstep > 0 ? (len - 1) * bstep : 0) + NM + S) - sm -
                            LY::off_bc - 1,
                        LY::NBC * LY::BC_STAGE, P.status) ||
                !SSM_IN((const char *)(ypp + (len - 1) * LY::YP) - sm - LY::off_yp + 3,
                        2 * LY::YP_STAGE, P.status))
                len = 0;
            // partial readout of one step to shared memory (more than two
            // lanes per channel: pair sums, stored by the even lanes)
            auto put = [&](int j, float yv) {
                if constexpr (LPR > LY::YP) {
                    yv += __shfl_xor_sync(0xffffffffu, yv, 1);
                    if ((s_sg & 1) == 0) ypp[j * LY::YP] = yv;
                } else {
                    ypp[j * LY::YP] = yv;
                }
            };
            // UB steps at a time, in three passes so that independent work
            // is adjacent for the scheduler: (1) every shared-memory load of
            // the block; (2) every decay e = 2^(delta*A*log2e) (MUFU) and
            // input B*w of the block -- independent of the state; (3) the
            // state recurrences and readouts, then the partial stores.
            auto block = [&](int j0) {
                float4 dv[UB], bv[UB][S / 4], cv[UB][S / 4];
#pragma unroll
                for (int jj = 0; jj < UB; ++jj) {
                    dv[jj] = *(const float4 *)(dwp + (j0 + jj) * 16);
                    const float *bj = bcp + (j0 + jj) * bstep;
#pragma unroll
                    for (int k = 0; k < S / 4; ++k) {
                        bv[jj][k] = *(const float4 *)(bj + 4 * k);
                        cv[jj][k] = *(const float4 *)(bj + NM + 4 * k);
                    }
                }
                f2 e[UB][NP], bw[UB][NP];
#pragma unroll
                for (int jj = 0; jj < UB; ++jj) {
                    const f2 dd = pk(dv[jj].x, dv[jj].y), ww = pk(dv[jj].z, dv[jj].w);
#pragma unroll
                    for (int q = 0; q < NP; ++q) {
                        const float4 &vb = bv[jj][q / 2];
                        const f2 bq = (q & 1) ? pk(vb.z, vb.w) : pk(vb.x, vb.y);
                        float a0, a1;
                        upk(mul2(dd, A2[q]), a0, a1);
                        e[jj][q] = pk(ex2_approx(a0), ex2_approx(a1));
                        bw[jj][q] = mul2(bq, ww);
                    }
                }
                // recurrences in state-pair-major order (the independent h
                // chains sit next to each other) with two readout
                // accumulators per step, so no chain is longer than UB
                f2 ya[UB], yb[UB];
#pragma unroll
                for (int jj = 0; jj < UB; ++jj) {
                    ya[jj] = pk(0.f, 0.f);
                    yb[jj] = pk(0.f, 0.f);
                }
#pragma unroll
                for (int q = 0; q < NP; ++q) {
#pragma unroll
                    for (int jj = 0; jj < UB; ++jj) {
                        const float4 &vc = cv[jj][q / 2];
                        const f2 cq = (q & 1) ? pk(vc.z, vc.w) : pk(vc.x, vc.y);
                        h[q] = fma2(e[jj][q], h[q], bw[jj][q]);
                        if (q & 1) yb[jj] = fma2(cq, h[q], yb[jj]);
                        else ya[jj] = fma2(cq, h[q], ya[jj]);
                    }
                }
                float ys[UB];
#pragma unroll
                for (int jj = 0; jj < UB; ++jj) {
                    float ylo, yhi;
                    upk(add2(ya[jj], yb[jj]), ylo, yhi);
                    ys[jj] = ylo + yhi;
                }
#pragma unroll
                for (int jj = 0; jj < UB; ++jj) put(j0 + jj, ys[jj]);
            };
            // one step (the chunk's tail); the readout is summed in the
            // block's order (even and odd state pairs apart, then together),
            // so every step of every path rounds alike
            auto step = [&](int j) {
                const float4 v = *(const float4 *)(dwp + j * 16);
                const f2 dd = pk(v.x, v.y), ww = pk(v.z, v.w);
                const float *bj = bcp + j * bstep;
                f2 ya = pk(0.f, 0.f), yb = pk(0.f, 0.f);
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    const float2 vb = *(const float2 *)(bj + 2 * q);
                    const float2 vc = *(const float2 *)(bj + NM + 2 * q);
                    float a0, a1;
                    upk(mul2(dd, A2[q]), a0, a1);
                    const f2 ee = pk(ex2_approx(a0), ex2_approx(a1));
                    h[q] = fma2(ee, h[q], mul2(pk(vb.x, vb.y), ww));
                    if (q & 1) yb = fma2(pk(vc.x, vc.y), h[q], yb);
                    else ya = fma2(pk(vc.x, vc.y), h[q], ya);
                }
                float ylo, yhi;
                upk(NP > 1 ? add2(ya, yb) : ya, ylo, yhi);
                put(j, ylo + yhi);
            };
            if constexpr (NM == kMaxN && T % kStateChunk == 0 && kStateChunk % UB == 0) {
                if (cs != nullptr) {
                    // walk chunks of kStateChunk steps: store the state at
                    // the start of each, then scan it
#pragma unroll 1
                    for (int j0 = 0; j0 < len; j0 += kStateChunk) {
                        const long long k = (long long)c * (T / kStateChunk) + j0 / kStateChunk;
                        float v[2 * NP];
#pragma unroll
                        for (int q = 0; q < NP; ++q) upk(h[q], v[2 * q], v[2 * q + 1]);
                        if (SSM_IN(cs_off + k * NM + S - 1, cs_elems, P.status)) {
#pragma unroll
                            for (int q = 0; q < NP / 2; ++q)
                                *(float4 *)(cs + k * NM + 4 * q) =
                                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                        }
                        const int j1 = min(len, j0 + kStateChunk);
                        int j = j0;
                        for (; j + UB <= j1; j += UB) block(j);
                        for (; j < j1; ++j) step(j);
                    }
                    mbar_arrive(&dw_empty[s2]);
                    mbar_arrive(&yp_full[s2]);
                    continue;
                }
            }
            int j = 0;
            for (; j + UB <= len; j += UB) block(j);
            for (; j < len; ++j) step(j);
            mbar_arrive(&dw_empty[s2]);
            mbar_arrive(&yp_full[s2]);
        }
        // the state after the branch's last step (position L-1 forward,
        // position 0 for the backward walk)
        float *ls = P.last_state[s_dir];
        if (ls != nullptr && s_ch < D) {
            const long long lo = ((long long)b * D + s_ch) * N;
            ls += lo;
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const int n0 = s_sg * S + 2 * q;
                float a0, a1;
                upk(h[q], a0, a1);
                if (n0 < N && SSM_IN(lo + n0, (long long)P.B * D * N, P.status)) ls[n0] = a0;
                if (n0 + 1 < N && SSM_IN(lo + n0 + 1, (long long)P.B * D * N, P.status))
                    ls[n0 + 1] = a1;
            }
        }
    } else if (warp < NSW + NPW) {
        // ================================================================ prep
        // 16 rows of one branch; lane = walk step j of the chunk
        // rows pw*16 .. pw*16+15 of the (branch, channel) row space, in NG
        // groups of GR channels of one branch (NG = 2 when R = 8)
        constexpr int GR = R < 16 ? R : 16;
        constexpr int NG = 16 / GR;
        const int pw = warp - NSW;
        int gd[NG], gn[NG];
        bool gsrev[NG], gusr[NG];
        const IO *gdt[NG], *gu[NG];
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const int row = pw * 16 + g * GR;
            const int d = row / R, r0 = row % R;
            const BiBranch &br = P.br[d];
            gd[g] = d;
            gsrev[g] = br.stream_rev != 0;
            gusr[g] = br.u_stream_rev != 0;
            gn[g] = min(GR, D - (d0 + r0));                  // valid channels
            // first row of the group in dt and u; row i is i * L further on
            // (offsets within the rows stay below D * L < 2^31)
            gdt[g] = (const IO *)br.dt + br.dt_off + b * br.dt_bstride + (long long)(d0 + r0) * L;
            gu[g] = (const IO *)br.u + (bD + d0 + r0) * L;
        }
        // this warp's 16 biases in shared memory
        float *bias_tab = (float *)(sm + LY::off_tab) + LY::ROWS + pw * 16;
        if (lane < 16) {
            const int row = pw * 16 + lane;
            const int d = row / R, ch = d0 + row % R;
            bias_tab[lane] = (ch < D && P.br[d].bias) ? P.br[d].bias[ch] : 0.f;
        }
        __syncwarp();
        bool all_rows = true;
#pragma unroll
        for (int g = 0; g < NG; ++g) all_rows = all_rows && gn[g] == GR;
        // dt and u of chunk c for this lane's walk step, all 32 loads in
        // flight together; fetched one chunk ahead of their use (their
        // latency hides behind this role's wait for a free stage)
        IO xdt[16], xu[16];
        auto fetch = [&](int c) {
            const int j = lane;
            int p[NG], si[NG], len = 0;
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                int lo;
                chunk_geom(c, gd[g], L, T, lo, len);
                const int pos = gd[g] ? lo + len - 1 - j : lo + j;   // position of walk step j
                si[g] = gsrev[g] ? c * T + j : pos;                  // dt stream index
                p[g] = gusr[g] ? c * T + j : pos;                    // u index
            }
            // element offsets from the tensors' bases (the debug build's checks)
            auto dt_in = [&](int g, int ii) {
                return SSM_IN((gdt[g] - (const IO *)P.br[gd[g]].dt) + ii * L + si[g],
                              P.br[gd[g]].dt ? P.dt_elems[gd[g]] : 0, P.status);
            };
            auto u_in = [&](int g, int ii) {
                return SSM_IN((gu[g] - (const IO *)P.br[gd[g]].u) + ii * L + p[g], P.io_elems,
                              P.status);
            };
            if (len == T && all_rows) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int g = i / GR, ii = i % GR;
                    xdt[i] = dt_in(g, ii) ? __ldg(gdt[g] + (ii * L + si[g])) : from_f32<IO>(0.f);
                    xu[i] = u_in(g, ii) ? __ldg(gu[g] + (ii * L + p[g])) : from_f32<IO>(0.f);
                }
            } else {
                const bool act = j < len;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int g = i / GR, ii = i % GR;
                    const bool ok = act && ii < gn[g];
                    xdt[i] = (ok && dt_in(g, ii)) ? __ldg(gdt[g] + (ii * L + si[g]))
                                                  : from_f32<IO>(0.f);
                    xu[i] = (ok && u_in(g, ii)) ? __ldg(gu[g] + (ii * L + p[g])) : from_f32<IO>(0.f);
                }
            }
        };
        // delta and w of 16 rows to shared memory; SP: softplus, FULL: a
        // whole chunk of 16 valid rows (no per-row predicates)
        auto emit = [&](auto SP, auto FULL, const IO *cdt, const IO *cu, float4 *dwl, IO *usl,
                        bool act) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float x = to_f32(cdt[i]) + bias_tab[i];
                float dl = decltype(SP)::value ? softplus_f<IO>(x) : x;
                if (!decltype(FULL)::value) dl = (i % GR) < gn[i / GR] ? dl : 0.f;
                const float w = dl * to_f32(cu[i]);
                if (decltype(FULL)::value || act) {
                    dwl[i * (LY::DW_ROW / 16)] = make_float4(dl, dl, w, w);
                    usl[i * T] = cu[i];
                }
            }
        };
        fetch(0);
        for (int c = 0; c < nch; ++c) {
            const int s2 = c & 1;
            int lo, len;
            chunk_geom(c, 0, L, T, lo, len);
            const int j = lane;
            const bool act = j < len;
            const int su = c % LY::NU;
            if (*abort_flag || !wait(&dw_empty[s2], ((c >> 1) & 1) ^ 1) ||
                !wait(&u_empty[su], ((c / LY::NU) & 1) ^ 1))
                return;
            // shared-memory stores only: they cannot alias the global loads
            // in flight, so each row is computed and stored in turn
            float4 *dwl = (float4 *)(sm + LY::off_dw + s2 * LY::DW_STAGE) +
                          (pw * 16) * (LY::DW_ROW / 16) + j;
            IO *usl = (IO *)(sm + LY::off_u + su * LY::U_STAGE) + (pw * 16) * T + j;
            const bool full = len == T && all_rows;
            if (P.delta_softplus) {
                if (full) emit(BoolC<true>(), BoolC<true>(), xdt, xu, dwl, usl, act);
                else emit(BoolC<true>(), BoolC<false>(), xdt, xu, dwl, usl, act);
            } else {
                if (full) emit(BoolC<false>(), BoolC<true>(), xdt, xu, dwl, usl, act);
                else emit(BoolC<false>(), BoolC<false>(), xdt, xu, dwl, usl, act);
            }
            mbar_arrive(&dw_full[s2]);
            if (c + 1 < nch) fetch(c + 1);
        }
    } else {
        // ================================================================ epilogue
        // both branches of CPE channels; lane = position offset q in the chunk
        constexpr int CPE = LY::CPE;
        const int ew = warp - NSW - NPW;
        const int c0 = ew * CPE;                               // first channel (in CTA)
        // per-channel constants in shared memory (this warp's channels)
        float *dsk_tab = (float *)(sm + LY::off_tab) + ew * NDIR * CPE;   // [NDIR][CPE]
        if (lane < NDIR * CPE) {
            const int d = lane / CPE, ch = d0 + c0 + lane % CPE;
            dsk_tab[lane] = (ch < D && P.br[d].Dskip) ? P.br[d].Dskip[ch] : 0.f;
        }
        __syncwarp();
        // channel c0's row in each [B, D, L] tensor; channel c0 + i is i * L
        // further on (offsets within the rows stay below D * L < 2^31)
        const long long rowb0 = (bD + d0 + c0) * L;
        const IO *zrow = P.z ? (const IO *)P.z + rowb0 : nullptr;
        float *Wrow = P.W ? P.W + rowb0 : nullptr;
        IO *yrow = P.y ? (IO *)P.y + rowb0 : nullptr;
        IO *yprow = (OUT == OUT_Y_PRE && P.ypre) ? (IO *)P.ypre + rowb0 : nullptr;
        float *aorow = P.acc_out ? P.acc_out + rowb0 : nullptr;
        const float *airow = P.acc_in ? P.acc_in + rowb0 : nullptr;
        const int nch_ok = min(CPE, D - (d0 + c0));           // valid channels
        auto issue_bc = [&](int c) {
            if (c >= nch || c == P.withhold_bc) return;
            const int st = c % LY::NBC;
            int lo, len;
            chunk_geom(c, 0, L, T, lo, len);
            mbar_arrive_expect_tx(&bc_full[st], (unsigned)(NDIR * len * kBC * 4));
#pragma unroll
            for (int d = 0; d < NDIR; ++d) {
                chunk_geom(c, d, L, T, lo, len);
                const long long so = ((long long)b * L + stream_lo(c, d, lo)) * kBC;
                // source range inside the packed buffer, destination inside
                // the stage (a copy that fails either is not issued)
                if (!SSM_IN(so, P.bc_elems[d], P.status) ||
                    !SSM_IN(so + (long long)len * kBC - 1, P.bc_elems[d], P.status) ||
                    !SSM_IN(LY::off_bc + st * LY::BC_STAGE + d * LY::BC_DIR + len * kBC * 4 - 1,
                            LY::off_bc + LY::NBC * LY::BC_STAGE, P.status))
                    continue;
                bulk_g2s(sm + LY::off_bc + st * LY::BC_STAGE + d * LY::BC_DIR, P.br[d].bc + so,
                         (unsigned)(len * kBC * 4), &bc_full[st]);
            }
        };
        const bool producer = ew == 0 && lane == 0;
        if (producer) {
            issue_bc(0);
            issue_bc(1);
        }
        const int q = lane;
        // classes of this lane's position in branch d at chunk c:
        // 0 first arrival (stash), 1 second arrival (the stash holds the other
        // branch), 2 both in this chunk, 3 left to branch 0
        auto classify = [&](int c, int d, int p) -> int {
            if (NDIR == 1) return 1;
            if (d == 0) return (p < L - (c + 1) * T) ? 0 : (p >= L - c * T ? 1 : 2);
            return (p >= (c + 1) * T) ? 0 : (p < c * T ? 1 : 3);
        };
        // the same for a whole chunk (both branches): 0 every position is a
        // first arrival, 1 every position is finalised here, 2 the middle of
        // the sequence (classes mixed)
        auto kind = [&](int c) -> int {
            if (NDIR == 1) return 1;
            if ((2LL * c + 2) * T <= L) return 0;
            if (2LL * c * T >= L) return 1;
            return 2;
        };
        // z, the stash and acc_in of the positions a lane finalises at chunk
        // c, fetched one chunk ahead (raw values, converted at use, all in
        // flight together).  u comes from the prep warps through shared
        // memory (its stage is released by this role).
        IO zr[NDIR][CPE];
        float wr[NDIR][CPE], ar[NDIR][CPE];
        auto load_items = [&](auto FULL, int c, int kd, int lo0, int lo1, int len) {
            const bool act = q < len;
#pragma unroll
            for (int d = 0; d < NDIR; ++d) {
                const int p = (d ? lo1 : lo0) + q;
                const int k = kd == 1 ? 1 : classify(c, d, p);
                const bool fin = decltype(FULL)::value || (act && (k == 1 || k == 2));
                const bool stash = NDIR == 2 && (decltype(FULL)::value || k == 1);
#pragma unroll
                for (int i = 0; i < CPE; ++i) {
                    const bool ok = fin && (decltype(FULL)::value || i < nch_ok);
                    const int o = i * L + p;
                    const bool in = ok && SSM_IN(rowb0 + o, P.io_elems, P.status);
                    zr[d][i] = (in && OUT != OUT_ACC && zrow != nullptr) ? __ldg(zrow + o)
                                                                          : from_f32<IO>(0.f);
                    wr[d][i] = (in && stash) ? Wrow[o] : 0.f;
                    ar[d][i] = (OUT == OUT_ADD_Y && in) ? __ldg(airow + o) : 0.f;
                }
            }
        };
        auto prefetch = [&](int c) {
            const int kd = kind(c);
            if (kd == 0) return;                    // nothing to read back
            int lo0, len, lo1 = 0;
            chunk_geom(c, 0, L, T, lo0, len);
            if (NDIR == 2) chunk_geom(c, 1, L, T, lo1, len);
            if (kd == 1 && len == T && nch_ok == CPE) load_items(BoolC<true>(), c, kd, lo0, lo1, len);
            else load_items(BoolC<false>(), c, kd, lo0, lo1, len);
        };
        prefetch(0);
        for (int c = 0; c < nch; ++c) {
            const int s2 = c & 1;
            int lo0, len, lo1 = 0;
            chunk_geom(c, 0, L, T, lo0, len);
            if (NDIR == 2) chunk_geom(c, 1, L, T, lo1, len);
            const bool act = q < len;
            if (*abort_flag || !wait(&yp_full[s2], (c >> 1) & 1)) {
                // the producer waits (bounded) for the B/C copies it issued
                if (producer)
                    for (int k = c; k < min(c + LY::NBC, nch); ++k)
                        if (k != P.withhold_bc)
                            mbar_wait_bounded(&bc_full[k % LY::NBC], (unsigned)((k / LY::NBC) & 1));
                return;
            }
            // scan(c) is done: its B/C stage is free for chunk c + NBC
            if (producer) issue_bc(c + LY::NBC);
            const float *yp = (const float *)(sm + LY::off_yp + s2 * LY::YP_STAGE);
            const IO *us = (const IO *)(sm + LY::off_u + (c % LY::NU) * LY::U_STAGE);
            auto ypsum = [&](int row, int jj) -> float {
                const float *ps = yp + row * (LY::YP_ROW / 4) + jj * LY::YP;
                if constexpr (LY::YP == 4) {
                    const float4 v = *(const float4 *)ps;
                    return (v.x + v.y) + (v.z + v.w);
                } else if constexpr (LY::YP == 2) {
                    const float2 v = *(const float2 *)ps;
                    return v.x + v.y;
                } else {
                    return ps[0];
                }
            };
            // output of branch d, channel c0 + i at walk step jw, with D * u
            auto own = [&](int d, int i, int jw) -> float {
                const int row = d * R + c0 + i;
                return fmaf(dsk_tab[d * CPE + i], to_f32(us[row * T + jw]), ypsum(row, jw));
            };
            const int kd = kind(c);
            // each item is stored as soon as it is formed (few registers);
            // the u stage is released after the chunk's last read of it
            if (kd == 0) {
                // every position is a first arrival (so the chunk is full):
                // both branches leave their outputs in the stash
#pragma unroll
                for (int d = 0; d < NDIR; ++d) {
                    const int p = (d ? lo1 : lo0) + q;
#pragma unroll
                    for (int i = 0; i < CPE; ++i)
                        if (i < nch_ok && SSM_IN(rowb0 + i * L + p, P.io_elems, P.status))
                            Wrow[i * L + p] = own(d, i, d ? T - 1 - q : q);
                }
                mbar_arrive(&u_empty[c % LY::NU]);
            } else if (kd == 1) {
                // every position is finalised here (single direction, or
                // the other branch's output is in the stash)
                const bool gate = OUT != OUT_ACC && zrow != nullptr;
                const bool full = len == T && nch_ok == CPE;
#pragma unroll
                for (int d = 0; d < NDIR; ++d) {
                    const int jw = act ? (d ? len - 1 - q : q) : 0;
                    const int p = (d ? lo1 : lo0) + q;
#pragma unroll
                    for (int i = 0; i < CPE; ++i) {
                        float v = own(d, i, jw);
                        if (NDIR == 2) v = P.out_scale * (v + wr[d][i]);
                        if (OUT == OUT_ADD_Y) v += ar[d][i];
                        const float pre = v;
                        if (gate) v *= silu_f<IO>(to_f32(zr[d][i]));
                        if ((full || (act && i < nch_ok)) &&
                            SSM_IN(rowb0 + i * L + p, P.io_elems, P.status)) {
                            if (OUT == OUT_ACC) aorow[i * L + p] = v;
                            else yrow[i * L + p] = from_f32<IO>(v);
                            if (OUT == OUT_Y_PRE) yprow[i * L + p] = from_f32<IO>(pre);
                        }
                    }
                }
                mbar_arrive(&u_empty[c % LY::NU]);
            } else {
                // the middle of the sequence: classes differ between lanes
                float vv[NDIR][CPE];     // the stash value (first arrival) or the output
                float pv[NDIR][CPE];     // OUT_Y_PRE: the output before the gate
                int kk[NDIR];
#pragma unroll
                for (int d = 0; d < NDIR; ++d) {
                    const int lo = d ? lo1 : lo0;
                    const int p = lo + q;
                    const int k = classify(c, d, p);
                    kk[d] = k;
                    const int jw = act ? (d ? len - 1 - q : q) : 0;     // walk step of p
                    float ow[CPE];
#pragma unroll
                    for (int i = 0; i < CPE; ++i) ow[i] = own(d, i, jw);
                    if (NDIR == 2 && d == 0 && __any_sync(0xffffffffu, k == 2)) {
                        // both branches reach p in this chunk: the backward
                        // branch's output from its rows
                        const int jb = k == 2 ? L - 1 - p - c * T : 0;
#pragma unroll
                        for (int i = 0; i < CPE; ++i)
                            if (k == 2) wr[d][i] = own(NDIR - 1, i, jb);
                    }
#pragma unroll
                    for (int i = 0; i < CPE; ++i) {
                        float v = ow[i];
                        if (NDIR == 2) v = k == 0 ? v : P.out_scale * (v + wr[d][i]);
                        if (OUT == OUT_ADD_Y) v += ar[d][i];
                        if (OUT == OUT_Y_PRE) pv[d][i] = v;
                        if (OUT != OUT_ACC && zrow != nullptr && !(NDIR == 2 && k == 0))
                            v *= silu_f<IO>(to_f32(zr[d][i]));
                        vv[d][i] = v;
                    }
                }
                mbar_arrive(&u_empty[c % LY::NU]);
#pragma unroll
                for (int d = 0; d < NDIR; ++d) {
                    const int p = (d ? lo1 : lo0) + q;
                    const int k = kk[d];
                    const bool live = act && k != 3;
                    const bool fin = live && (NDIR == 1 || k != 0);
#pragma unroll
                    for (int i = 0; i < CPE; ++i) {
                        const int o = i * L + p;
                        const bool ok = i < nch_ok && (!(live || fin) ||
                                                       SSM_IN(rowb0 + o, P.io_elems, P.status));
                        if (NDIR == 2 && ok && live && k == 0) Wrow[o] = vv[d][i];
                        if (ok && fin) {
                            if (OUT == OUT_ACC) aorow[o] = vv[d][i];
                            else yrow[o] = from_f32<IO>(vv[d][i]);
                            if (OUT == OUT_Y_PRE) yprow[o] = from_f32<IO>(pv[d][i]);
                        }
                    }
                }
            }
            mbar_arrive(&yp_empty[s2]);
            // the stash stores of this chunk must precede this warp's loads
            // of the next one
            __syncwarp();
            if (c + 1 < nch) prefetch(c + 1);
        }
    }
}

}  // namespace ssm
