// ssm_scan_api.cu -- the C ABI declared in include/ssm_scan.h.
//
// Each entry point validates its arguments on the host, fills the kernel's
// parameter block and launches the scan kernel(s) on the caller's stream.
// Nothing is allocated.  The one piece of state kept between calls is the
// fixed scratch array of the allocation-free entry point and its per-device
// address.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "bidir_kernel.cuh"
#include "internal.h"
#include "ssm_scan.h"

// Scratch of bimamba_scan_fwd_v2_noalloc: a fixed device array of the
// library's image (internal linkage), held by every GPU that loads the
// library until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[SSM_STATIC_SCRATCH_BYTES];

namespace {

bool aligned(const void *p, unsigned a) { return ((uintptr_t)p % a) == 0; }

// 2^31 - 1 bounds every per-dimension index the kernels form in 32 bits.
bool fits(long long v) { return v >= 0 && v <= 0x7fffffffLL; }

ssm_status check_common(ssm_dtype dt, int B, int D, int L, int N) {
    if (dt != SSM_F32 && dt != SSM_BF16 && dt != SSM_F16) return SSM_ERR_INVALID_ARG;
    if (B < 0 || D < 0 || L < 0 || N <= 0) return SSM_ERR_INVALID_ARG;
    if (N > 2 * ssm::kMaxN) return SSM_ERR_UNSUPPORTED;      // up to 32 states
    if (B > 65535) return SSM_ERR_UNSUPPORTED;                 // grid.y
    if (!fits((long long)D * L) || !fits((long long)N * L)) return SSM_ERR_UNSUPPORTED;
    return SSM_OK;
}

// I/O tensors are read and written element by element, so they need only
// their element's alignment; the bulk copies read the workspace alone.
unsigned io_align(ssm_dtype dt) { return dt == SSM_F32 ? 4u : 2u; }
bool io_ok(ssm_dtype dt, const void *p) { return p != nullptr && aligned(p, io_align(dt)); }
bool opt_io_ok(ssm_dtype dt, const void *p) { return p == nullptr || aligned(p, io_align(dt)); }
bool f32_ok(const float *p) { return p != nullptr && aligned(p, 4); }
bool opt_f32_ok(const float *p) { return p == nullptr || aligned(p, 4); }

// ---- single / bidirectional path (bidir_kernel.cuh)
// Workspace: [256-byte header: status word][packed B/C of the forward
// branch][packed B/C of the backward branch (v2)][fp32 stash W (two
// branches, more than one chunk)].  Every region starts on 128 bytes.
constexpr size_t kHeaderBytes = 256;
#ifndef SSM_BI_S
#define SSM_BI_S 8
#endif
#ifndef SSM_BI_G2
#define SSM_BI_G2 16
#endif
#ifndef SSM_BI_G1
#define SSM_BI_G1 32
#endif
constexpr int kBiT = 32;                   // positions per chunk
constexpr int kBiS = SSM_BI_S;             // states per lane
constexpr int kBiG2 = SSM_BI_G2;           // channels per CTA, two branches
constexpr int kBiG1 = SSM_BI_G1;           // channels per CTA, one branch

int bi_chunks(int L) { return (L + kBiT - 1) / kBiT; }
// state capacity of the kernels that handle N states (16 or 32)
int nm_of(int N) { return N <= ssm::kMaxN ? ssm::kMaxN : 2 * ssm::kMaxN; }
size_t bc_bytes(int B, int L, int nm) { return (size_t)B * L * 2 * nm * sizeof(float); }

struct BiWs {
    size_t bc0, bc1, w, total;
};
// bc_sets: 1 (single, v1) or 2 (v2); stash only with two branches.
BiWs bi_ws(int bc_sets, int ndir, int B, int D, int L, int nm) {
    BiWs w;
    size_t off = kHeaderBytes;
    w.bc0 = off;
    off += bc_bytes(B, L, nm);
    w.bc1 = w.bc0;
    if (bc_sets == 2) {
        w.bc1 = off;
        off += bc_bytes(B, L, nm);
    }
    w.w = 0;
    if (ndir == 2 && bi_chunks(L) > 1) {
        w.w = off;
        off += (size_t)B * D * L * sizeof(float);
    }
    w.total = off;
    return w;
}

template <typename IO, int NM>
ssm_status launch_pack(const void *Bm, const void *Cm, float *out, int B, int N, int L,
                       unsigned *status, cudaStream_t st, int K = 1) {
    constexpr int PT = ssm::pack_pt<NM>();
    dim3 grid((L + PT - 1) / PT, B, K);
    ssm::pack_bc_kernel<IO, NM><<<grid, 256, 0, st>>>((const IO *)Bm, (const IO *)Cm, out, N, L,
                                                  status);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// Profiling hook (ssm_set_profile_events): events recorded around the last
// scan-kernel launch of each call made on this host thread.
thread_local cudaEvent_t t_prof_begin = nullptr, t_prof_end = nullptr;
// Override of the two-branch CTA shape (ssm_set_cta_channels): 0, 8 or 16.
thread_local int t_cta_channels = 0;
// Test hook (ssm_test_withhold_copy): chunk whose B/C copy the next call on
// this host thread withholds, to exercise the bounded waits.
thread_local int t_withhold = -1;
// Test hook of the debug build (ssm_test_shrink_extents): elements the next
// scan-kernel launch on this host thread takes off the [B, D, L] extent its
// index checks use.
thread_local long long t_shrink = 0;
// Chunk-state capture (ssm_internal::set_chunk_state_capture), per direction.
thread_local float *t_capture[4] = {nullptr, nullptr, nullptr, nullptr};

// A saved backward context (ssm_set_bwd_context) on this host thread, for
// a sequence form with d_state <= 16 and no internal capture active: the
// call also stores its chunk-start states and (with a gate) its pre-gate
// output there, in the layout the backward calls read.
ssm_status apply_bwd_context(ssm::BiParams &P, int ndir, ssm_dtype dt) {
    if (P.N > ssm::kMaxN || t_capture[0] != nullptr || t_capture[1] != nullptr) return SSM_OK;
    size_t cb = 0;
    char *ctx = (char *)ssm_internal::bwd_context(&cb);
    if (ctx == nullptr) return SSM_OK;
    const ssm_internal::CtxLayout cl =
        ssm_internal::ctx_layout(ndir, dt == SSM_F32 ? 4u : 2u, P.B, P.D, P.L);
    if (cb < cl.total || !aligned(ctx, 16)) return SSM_ERR_WORKSPACE;
    for (int k = 0; k < ndir; ++k) P.chunk_state[k] = (float *)(ctx + cl.hc[k]);
    P.ypre = P.z ? (void *)(ctx + cl.ypre) : nullptr;
    return SSM_OK;
}

template <typename IO, int S, int NDIR, int G, int OUT, int NM>
ssm_status launch_bidir(const ssm::BiParams &P, cudaStream_t st, bool last = true) {
    using LY = ssm::WsLayout<IO, S, NDIR, G, NM>;
    auto *kern = &ssm::bidir_scan_kernel<IO, S, NDIR, G, OUT, NM>;
    // Raising the dynamic shared-memory limit and asking for the largest
    // shared-memory carveout are cheap and idempotent; without the carveout
    // the driver may pick one that fits fewer CTAs per SM.
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::bytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess) {
        cudaGetLastError();
        return SSM_ERR_CUDA;
    }
    // the packed B/C chunks are bulk copies from base + a multiple of 128
    // bytes, so their bases must be 16-byte aligned (checked, never assumed);
    // every other tensor is accessed element by element
    for (int d = 0; d < NDIR; ++d)
        if (!aligned(P.br[d].bc, 16)) return SSM_ERR_INVALID_ARG;
    dim3 grid((P.D + G - 1) / G, P.B);
    const bool prof = last && t_prof_begin != nullptr && t_prof_end != nullptr;
    ssm::BiParams Q = P;
    Q.withhold_bc = t_withhold;
    t_withhold = -1;
    Q.io_elems = t_shrink < Q.io_elems ? Q.io_elems - t_shrink : 0;
    t_shrink = 0;
    if (prof && cudaEventRecord(t_prof_begin, st) != cudaSuccess) {
        cudaGetLastError();
        return SSM_ERR_CUDA;
    }
    kern<<<grid, LY::NT, LY::bytes, st>>>(Q);
    if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
    if (prof && cudaEventRecord(t_prof_end, st) != cudaSuccess) {
        cudaGetLastError();
        return SSM_ERR_CUDA;
    }
    return SSM_OK;
}

// Channels per CTA of the two-branch kernel: 16, or 8 when that leaves
// fewer (branch, channel) rows on the busiest SM -- small B * D, where CTAs
// of 16 channels leave SMs idle.  An SM holds LY::CPS CTAs at a time; a
// busier SM runs them in waves.
template <typename IO, int G, int NM>
long long busiest_sm_rows(int B, int D, int nsm) {
    constexpr int cps = ssm::WsLayout<IO, kBiS, 2, G, NM>::CPS;
    const long long ctas = (long long)((D + G - 1) / G) * B;
    const long long per = (ctas + nsm - 1) / nsm;
    const long long slots = per <= cps ? per : (per + cps - 1) / cps * cps;
    return slots * G;
}
template <typename IO, int NM>
bool narrow_ctas(int B, int D) {
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        nsm <= 0) {
        cudaGetLastError();
        return false;
    }
    return busiest_sm_rows<IO, 8, NM>(B, D, nsm) < busiest_sm_rows<IO, kBiG2, NM>(B, D, nsm);
}
template <typename IO, int OUT, int NM>
ssm_status launch_two_branch(const ssm::BiParams &P, cudaStream_t st, bool last = true) {
    const bool narrow = t_cta_channels == 8 ? true
                        : t_cta_channels == 16 ? false
                                               : narrow_ctas<IO, NM>(P.B, P.D);
    if (narrow) return launch_bidir<IO, kBiS, 2, 8, OUT, NM>(P, st, last);
    return launch_bidir<IO, kBiS, 2, kBiG2, OUT, NM>(P, st, last);
}

// Packs B/C (one or two sets), then runs the scan kernel.
template <typename IO, int NDIR, int NM>
ssm_status run_bidir_nm(ssm::BiParams P, const void *Bm, const void *Cm, const void *Bm_b,
                        const void *Cm_b, bool two_sets, cudaStream_t st) {
    ssm_status s;
    if (two_sets) {
        // both branches' B/C sets in one launch (grid z = 2)
        constexpr int PT = ssm::pack_pt<NM>();
        ssm::pack_bc_kernel<IO, NM><<<dim3((P.L + PT - 1) / PT, P.B, 2), 256, 0, st>>>(
            (const IO *)Bm, (const IO *)Cm, const_cast<float *>(P.br[0].bc), P.N, P.L, P.status,
            (const IO *)Bm_b, (const IO *)Cm_b, const_cast<float *>(P.br[1].bc));
        s = cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
    } else {
        s = launch_pack<IO, NM>(Bm, Cm, const_cast<float *>(P.br[0].bc), P.B, P.N, P.L,
                                P.status, st);
    }
    if (s != SSM_OK) return s;
    if constexpr (NM == ssm::kMaxN) {
        if (P.ypre != nullptr) {
            if (NDIR == 2) return launch_two_branch<IO, ssm::OUT_Y_PRE, NM>(P, st);
            return launch_bidir<IO, kBiS, 1, kBiG1, ssm::OUT_Y_PRE, NM>(P, st);
        }
    }
    if (NDIR == 2) return launch_two_branch<IO, ssm::OUT_Y, NM>(P, st);
    return launch_bidir<IO, kBiS, 1, kBiG1, ssm::OUT_Y, NM>(P, st);
}
template <typename IO, int NDIR>
ssm_status run_bidir(ssm::BiParams P, const void *Bm, const void *Cm, const void *Bm_b,
                     const void *Cm_b, bool two_sets, cudaStream_t st) {
    if (P.N <= ssm::kMaxN)
        return run_bidir_nm<IO, NDIR, ssm::kMaxN>(P, Bm, Cm, Bm_b, Cm_b, two_sets, st);
    return run_bidir_nm<IO, NDIR, 2 * ssm::kMaxN>(P, Bm, Cm, Bm_b, Cm_b, two_sets, st);
}

// Shared body of v1 / v2 (v1 passes the forward tensors for both branches
// and a single B/C set).
ssm_status bidirectional(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                         const void *u_b, const void *delta, const void *delta_b,
                         const float *A, const float *A_b, const void *Bm, const void *Cm,
                         const void *Bm_b, const void *Cm_b, const float *Dskip,
                         const float *D_b, const void *z, const float *bias,
                         const float *bias_b, int delta_softplus, float out_scale, void *y,
                         void *ws, size_t ws_bytes, bool two_sets, cudaStream_t stream,
                         float *ls = nullptr, bool scan_order = false) {
    ssm_status s = check_common(dt, B, D, L, N);
    if (s != SSM_OK) return s;
    if (!opt_f32_ok(ls)) return SSM_ERR_INVALID_ARG;
    if (!io_ok(dt, u) || !opt_io_ok(dt, u_b) || !io_ok(dt, delta) || !io_ok(dt, delta_b) ||
        !io_ok(dt, Bm) || !io_ok(dt, Cm) || !io_ok(dt, Bm_b) || !io_ok(dt, Cm_b) ||
        !opt_io_ok(dt, z) || !io_ok(dt, y) ||
        !f32_ok(A) || !f32_ok(A_b) || !opt_f32_ok(Dskip) || !opt_f32_ok(D_b) ||
        !opt_f32_ok(bias) || !opt_f32_ok(bias_b))
        return SSM_ERR_INVALID_ARG;
    if ((long long)B * D * L == 0) return SSM_OK;
    const BiWs lay = bi_ws(two_sets ? 2 : 1, 2, B, D, L, nm_of(N));
    if (ws == nullptr || ws_bytes < lay.total || !aligned(ws, 16)) return SSM_ERR_WORKSPACE;
    char *wsb = (char *)ws;
    ssm::BiParams P{};
    const long long DL = (long long)D * L;
    P.br[0] = {delta, u, (const float *)(wsb + lay.bc0), A, Dskip, bias, 0, DL, 0};
    P.br[1] = {delta_b, u_b ? u_b : u, (const float *)(wsb + lay.bc1), A_b, D_b, bias_b,
               0, DL, 0};
    if (scan_order) {
        // the backward set is given in its own walk order (reversed time)
        P.br[1].stream_rev = 1;
        P.br[1].u_stream_rev = u_b != nullptr;
    }
    P.z = z;
    P.y = y;
    P.W = lay.w ? (float *)(wsb + lay.w) : nullptr;
    const long long BDN = (long long)B * D * N;
    P.last_state[0] = ls;                               // [2][B][D][N]
    P.last_state[1] = ls ? ls + BDN : nullptr;
    P.chunk_state[0] = t_capture[0];
    P.chunk_state[1] = t_capture[1];
    P.status = (unsigned *)wsb;
    P.B = B;
    P.D = D;
    P.L = L;
    P.N = N;
    P.nchunks = bi_chunks(L);
    P.delta_softplus = delta_softplus ? 1 : 0;
    P.out_scale = out_scale;
    P.dt_elems[0] = P.dt_elems[1] = P.io_elems = (long long)B * D * L;
    P.bc_elems[0] = P.bc_elems[1] = (long long)B * L * 2 * nm_of(N);
    P.a_elems = (long long)D * N;
    if ((s = apply_bwd_context(P, 2, dt)) != SSM_OK) return s;
    if (dt == SSM_F32) return run_bidir<float, 2>(P, Bm, Cm, Bm_b, Cm_b, two_sets, stream);
    if (dt == SSM_F16) return run_bidir<__half, 2>(P, Bm, Cm, Bm_b, Cm_b, two_sets, stream);
    return run_bidir<__nv_bfloat16, 2>(P, Bm, Cm, Bm_b, Cm_b, two_sets, stream);
}

// ---- SS2D (VMamba cross-scan / cross-merge)
// Directions 0/2 walk the map row-major forward/backward and 1/3 walk it
// column-major forward/backward; each direction's delta and B/C are in its
// own scan order.  The column pair runs on the map transposed per channel
// (x^T), so both pairs are contiguous sequences of L = H * W positions:
//   1. pack B/C of the four directions;          2. x^T = transpose(x);
//   3. column pair (1, 3) on x^T -> Wt = y1 + y3 (fp32, column-major);
//   4. Wa = transpose(Wt);
//   5. row pair (0, 2) on x: y = gate(y0 + y2 + Wa, z).
// Workspace: [header][packed B/C, 4 directions][x^T][R1][R2] where R1 is
// the column pair's stash and then Wa, and R2 is Wt and then the row pair's
// stash.
struct SsWs {
    size_t bc, xt, r1, r2, total;
};
size_t round128(size_t v) { return (v + 127) & ~(size_t)127; }
SsWs ss2d_ws(ssm_dtype dt, int B, int D, int L, int nm) {
    const size_t es = dt == SSM_F32 ? 4 : 2;
    const size_t n = (size_t)B * D * L;
    SsWs w;
    w.bc = kHeaderBytes;
    w.xt = w.bc + 4 * bc_bytes(B, L, nm);
    w.r1 = w.xt + round128(n * es);
    w.r2 = w.r1 + round128(n * 4);
    w.total = w.r2 + round128(n * 4);
    return w;
}

template <typename E>
ssm_status launch_transpose(const E *in, E *out, int maps, int R, int C, cudaStream_t st) {
    const size_t whole = (size_t)R * (C + 1) * sizeof(E);
    if (whole <= 48 * 1024) {
        // whole maps per CTA: each map one contiguous read and write
        const int grid = maps < 65535 ? maps : 65535;
        if (R <= 64 && C <= 64)
            ssm::transpose_whole_maps_kernel<E, true><<<grid, 256, whole, st>>>(in, out, maps, R,
                                                                                C);
        else
            ssm::transpose_whole_maps_kernel<E, false><<<grid, 256, whole, st>>>(in, out, maps, R,
                                                                                 C);
    } else {
        dim3 grid((C + 31) / 32, (R + 31) / 32, maps < 65535 ? maps : 65535);
        ssm::transpose_maps_kernel<E><<<grid, 256, 0, st>>>(in, out, maps, R, C);
    }
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename IO, int NM>
ssm_status ss2d_run_nm(int B, int D, int H, int W, int N, const void *x, const void *delta,
                    const float *A, const void *Bm, const void *Cm, const float *Dskip,
                    const void *z, const float *bias, int delta_softplus, void *y, char *wsb,
                    const SsWs &lay, cudaStream_t st, float *ls) {
    const long long BDN = (long long)B * D * N;          // last_state: [4][B][D][N]
    auto lsk = [&](int k) { return ls ? ls + k * BDN : nullptr; };
    const int L = H * W;
    const long long DL = (long long)D * L;
    float *bcK = (float *)(wsb + lay.bc);
    IO *xt = (IO *)(wsb + lay.xt);
    float *r1 = (float *)(wsb + lay.r1), *r2 = (float *)(wsb + lay.r2);
    unsigned *status = (unsigned *)wsb;
    ssm_status s = launch_pack<IO, NM>(Bm, Cm, bcK, B, N, L, status, st, 4);
    if (s != SSM_OK) return s;
    s = launch_transpose<IO>((const IO *)x, xt, B * D, H, W, st);
    if (s != SSM_OK) return s;
    auto branch = [&](int k, const void *u, int rev) {
        ssm::BiBranch br;
        br.dt = delta;
        br.dt_off = k * DL;
        br.u = u;
        br.bc = bcK + (long long)k * B * L * 2 * NM;
        br.A = A + (long long)k * D * N;
        br.Dskip = Dskip ? Dskip + (long long)k * D : nullptr;
        br.bias = bias ? bias + (long long)k * D : nullptr;
        br.dt_bstride = 4 * DL;
        br.stream_rev = rev;
        return br;
    };
    // extents from each branch's base pointers (dt, B/C and A are the whole
    // four-direction tensors, offset per direction)
    auto extents = [&](ssm::BiParams &Q, int k0, int k1) {
        Q.dt_elems[0] = (long long)B * 4 * DL;             // offset through dt_off
        Q.dt_elems[1] = (long long)B * 4 * DL;
        Q.bc_elems[0] = (long long)(4 - k0) * B * L * 2 * NM;
        Q.bc_elems[1] = (long long)(4 - k1) * B * L * 2 * NM;
        Q.io_elems = (long long)B * DL;
        Q.a_elems = (long long)D * N;
    };
    ssm::BiParams P{};
    P.status = status;
    P.B = B;
    P.D = D;
    P.L = L;
    P.N = N;
    P.nchunks = bi_chunks(L);
    P.delta_softplus = delta_softplus ? 1 : 0;
    P.out_scale = 1.f;
    // column pair on x^T: the fused sum goes to Wt (R2), stash in R1
    P.br[0] = branch(1, xt, 0);
    P.br[1] = branch(3, xt, 1);
    extents(P, 1, 3);
    P.W = r1;
    P.acc_out = r2;
    P.last_state[0] = lsk(1);
    P.last_state[1] = lsk(3);
    P.chunk_state[0] = t_capture[1];
    P.chunk_state[1] = t_capture[3];
    s = launch_two_branch<IO, ssm::OUT_ACC, NM>(P, st, false);
    if (s != SSM_OK) return s;
    // Wa (R1) = Wt (R2) transposed back to H x W
    s = launch_transpose<float>(r2, r1, B * D, W, H, st);
    if (s != SSM_OK) return s;
    // row pair on x: y = gate(y0 + y2 + Wa), stash in R2
    P.br[0] = branch(0, x, 0);
    P.br[1] = branch(2, x, 1);
    extents(P, 0, 2);
    P.z = z;
    P.y = y;
    P.W = r2;
    P.acc_in = r1;
    P.acc_out = nullptr;
    P.last_state[0] = lsk(0);
    P.last_state[1] = lsk(2);
    P.chunk_state[0] = t_capture[0];
    P.chunk_state[1] = t_capture[2];
    return launch_two_branch<IO, ssm::OUT_ADD_Y, NM>(P, st);
}
template <typename IO>
ssm_status ss2d_run(int B, int D, int H, int W, int N, const void *x, const void *delta,
                    const float *A, const void *Bm, const void *Cm, const float *Dskip,
                    const void *z, const float *bias, int delta_softplus, void *y, char *wsb,
                    const SsWs &lay, cudaStream_t st, float *ls) {
    if (N <= ssm::kMaxN)
        return ss2d_run_nm<IO, ssm::kMaxN>(B, D, H, W, N, x, delta, A, Bm, Cm, Dskip, z, bias,
                                           delta_softplus, y, wsb, lay, st, ls);
    return ss2d_run_nm<IO, 2 * ssm::kMaxN>(B, D, H, W, N, x, delta, A, Bm, Cm, Dskip, z, bias,
                                           delta_softplus, y, wsb, lay, st, ls);
}

// ---- fixed scratch of the allocation-free entry point
// The array itself (g_static_scratch) is declared at file scope above this
// namespace; in host code its name is only a host-side stand-in, so the
// kernel is given the device address that cudaGetSymbolAddress reports for
// the current device (looked up once per device, on that device's first
// call).
constexpr int kMaxDevices = 256;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices];

ssm_status static_scratch(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SSM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return SSM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return SSM_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SSM_OK;
}

ssm_status single_impl(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                       const void *delta, const float *A, const void *Bm, const void *Cm,
                       const float *Dskip, const void *z, const float *delta_bias,
                       int delta_softplus, void *y, void *workspace, size_t ws_bytes,
                       ssm_stream_t stream, float *ls) {
    ssm_status s = check_common(dt, B, D, L, N);
    if (s != SSM_OK) return s;
    if (!opt_f32_ok(ls)) return SSM_ERR_INVALID_ARG;
    if (!io_ok(dt, u) || !io_ok(dt, delta) || !io_ok(dt, Bm) || !io_ok(dt, Cm) ||
        !opt_io_ok(dt, z) || !io_ok(dt, y) || !f32_ok(A) || !opt_f32_ok(Dskip) ||
        !opt_f32_ok(delta_bias))
        return SSM_ERR_INVALID_ARG;
    if ((long long)B * D * L == 0) return SSM_OK;
    const BiWs lay = bi_ws(1, 1, B, D, L, nm_of(N));
    if (workspace == nullptr || ws_bytes < lay.total || !aligned(workspace, 16))
        return SSM_ERR_WORKSPACE;
    char *wsb = (char *)workspace;
    ssm::BiParams P{};
    P.br[0] = {delta, u, (const float *)(wsb + lay.bc0), A, Dskip, delta_bias, 0,
               (long long)D * L, 0};
    P.br[1] = P.br[0];
    P.z = z;
    P.y = y;
    P.W = nullptr;
    P.last_state[0] = ls;
    P.last_state[1] = nullptr;
    P.chunk_state[0] = t_capture[0];
    P.status = (unsigned *)wsb;
    P.B = B;
    P.D = D;
    P.L = L;
    P.N = N;
    P.nchunks = bi_chunks(L);
    P.delta_softplus = delta_softplus ? 1 : 0;
    P.out_scale = 1.f;
    P.dt_elems[0] = P.dt_elems[1] = P.io_elems = (long long)B * D * L;
    P.bc_elems[0] = P.bc_elems[1] = (long long)B * L * 2 * nm_of(N);
    P.a_elems = (long long)D * N;
    if ((s = apply_bwd_context(P, 1, dt)) != SSM_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    if (dt == SSM_F32) return run_bidir<float, 1>(P, Bm, Cm, Bm, Cm, false, st);
    if (dt == SSM_F16) return run_bidir<__half, 1>(P, Bm, Cm, Bm, Cm, false, st);
    return run_bidir<__nv_bfloat16, 1>(P, Bm, Cm, Bm, Cm, false, st);
}

ssm_status ss2d_impl(ssm_dtype dt, int B, int D, int H, int W, int N, int K, const void *x,
                     const void *delta, const float *A, const void *Bm, const void *Cm,
                     const float *Dskip, const void *z, const float *delta_bias,
                     int delta_softplus, void *y, void *workspace, size_t ws_bytes,
                     ssm_stream_t stream, float *ls) {
    if (H < 0 || W < 0 || !opt_f32_ok(ls)) return SSM_ERR_INVALID_ARG;
    if (K != 4) return SSM_ERR_UNSUPPORTED;
    if (!fits((long long)H * W)) return SSM_ERR_UNSUPPORTED;
    const int L = H * W;
    ssm_status s = check_common(dt, B, D, L, N);
    if (s != SSM_OK) return s;
    if (!fits((long long)K * D * L) || !fits((long long)K * N * L)) return SSM_ERR_UNSUPPORTED;
    if (!io_ok(dt, x) || !io_ok(dt, delta) || !io_ok(dt, Bm) || !io_ok(dt, Cm) ||
        !opt_io_ok(dt, z) || !io_ok(dt, y) || !f32_ok(A) || !opt_f32_ok(Dskip) ||
        !opt_f32_ok(delta_bias))
        return SSM_ERR_INVALID_ARG;
    if ((long long)B * D * L == 0) return SSM_OK;
    const SsWs lay = ss2d_ws(dt, B, D, L, nm_of(N));
    if (workspace == nullptr || ws_bytes < lay.total || !aligned(workspace, 16))
        return SSM_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    if (dt == SSM_F32)
        return ss2d_run<float>(B, D, H, W, N, x, delta, A, Bm, Cm, Dskip, z, delta_bias,
                               delta_softplus, y, (char *)workspace, lay, st, ls);
    if (dt == SSM_F16)
        return ss2d_run<__half>(B, D, H, W, N, x, delta, A, Bm, Cm, Dskip, z, delta_bias,
                                delta_softplus, y, (char *)workspace, lay, st, ls);
    return ss2d_run<__nv_bfloat16>(B, D, H, W, N, x, delta, A, Bm, Cm, Dskip, z, delta_bias,
                                   delta_softplus, y, (char *)workspace, lay, st, ls);
}

}  // namespace

void ssm_internal::set_chunk_state_capture(float *const *hc) {
    for (int k = 0; k < 4; ++k) t_capture[k] = hc ? hc[k] : nullptr;
}

extern "C" {

ssm_status selective_scan_fwd(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                              const void *delta, const float *A, const void *Bm,
                              const void *Cm, const float *Dskip, const void *z,
                              const float *delta_bias, int delta_softplus, void *y,
                              void *workspace, size_t ws_bytes, ssm_stream_t stream) {
    return single_impl(dt, B, D, L, N, u, delta, A, Bm, Cm, Dskip, z, delta_bias,
                       delta_softplus, y, workspace, ws_bytes, stream, nullptr);
}

ssm_status selective_scan_fwd_ls(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                                 const void *delta, const float *A, const void *Bm,
                                 const void *Cm, const float *Dskip, const void *z,
                                 const float *delta_bias, int delta_softplus, void *y,
                                 float *last_state, void *workspace, size_t ws_bytes,
                                 ssm_stream_t stream) {
    if (last_state == nullptr) return SSM_ERR_INVALID_ARG;
    return single_impl(dt, B, D, L, N, u, delta, A, Bm, Cm, Dskip, z, delta_bias,
                       delta_softplus, y, workspace, ws_bytes, stream, last_state);
}

ssm_status bimamba_scan_fwd_v1(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                               const void *delta, const float *A, const float *A_b,
                               const void *Bm, const void *Cm, const float *Dskip,
                               const void *z, const float *delta_bias, int delta_softplus,
                               float out_scale, void *y, void *workspace, size_t ws_bytes,
                               ssm_stream_t stream) {
    return bidirectional(dt, B, D, L, N, u, nullptr, delta, delta, A, A_b, Bm, Cm, Bm, Cm,
                         Dskip, Dskip, z, delta_bias, delta_bias, delta_softplus, out_scale, y,
                         workspace, ws_bytes, false, (cudaStream_t)stream);
}

ssm_status bimamba_scan_fwd_v2(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                               const void *u_b, const void *delta, const void *delta_b,
                               const float *A, const float *A_b, const void *Bm,
                               const void *Cm, const void *Bm_b, const void *Cm_b,
                               const float *Dskip, const float *D_b, const void *z,
                               const float *delta_bias, const float *delta_bias_b,
                               int delta_softplus, float out_scale, void *y, void *workspace,
                               size_t ws_bytes, ssm_stream_t stream) {
    return bidirectional(dt, B, D, L, N, u, u_b, delta, delta_b, A, A_b, Bm, Cm, Bm_b, Cm_b,
                         Dskip, D_b, z, delta_bias, delta_bias_b, delta_softplus, out_scale, y,
                         workspace, ws_bytes, true, (cudaStream_t)stream);
}

ssm_status bimamba_scan_fwd_v1_ls(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                                  const void *delta, const float *A, const float *A_b,
                                  const void *Bm, const void *Cm, const float *Dskip,
                                  const void *z, const float *delta_bias, int delta_softplus,
                                  float out_scale, void *y, float *last_state, void *workspace,
                                  size_t ws_bytes, ssm_stream_t stream) {
    if (last_state == nullptr) return SSM_ERR_INVALID_ARG;
    return bidirectional(dt, B, D, L, N, u, nullptr, delta, delta, A, A_b, Bm, Cm, Bm, Cm,
                         Dskip, Dskip, z, delta_bias, delta_bias, delta_softplus, out_scale, y,
                         workspace, ws_bytes, false, (cudaStream_t)stream, last_state);
}

ssm_status bimamba_scan_fwd_v2_ls(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                                  const void *u_b, const void *delta, const void *delta_b,
                                  const float *A, const float *A_b, const void *Bm,
                                  const void *Cm, const void *Bm_b, const void *Cm_b,
                                  const float *Dskip, const float *D_b, const void *z,
                                  const float *delta_bias, const float *delta_bias_b,
                                  int delta_softplus, float out_scale, void *y,
                                  float *last_state, void *workspace, size_t ws_bytes,
                                  ssm_stream_t stream) {
    if (last_state == nullptr) return SSM_ERR_INVALID_ARG;
    return bidirectional(dt, B, D, L, N, u, u_b, delta, delta_b, A, A_b, Bm, Cm, Bm_b, Cm_b,
                         Dskip, D_b, z, delta_bias, delta_bias_b, delta_softplus, out_scale, y,
                         workspace, ws_bytes, true, (cudaStream_t)stream, last_state);
}

ssm_status bimamba_scan_fwd_v2_so(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                                  const void *u_b, const void *delta, const void *delta_b,
                                  const float *A, const float *A_b, const void *Bm,
                                  const void *Cm, const void *Bm_b, const void *Cm_b,
                                  const float *Dskip, const float *D_b, const void *z,
                                  const float *delta_bias, const float *delta_bias_b,
                                  int delta_softplus, float out_scale, void *y,
                                  float *last_state, void *workspace, size_t ws_bytes,
                                  ssm_stream_t stream) {
    return bidirectional(dt, B, D, L, N, u, u_b, delta, delta_b, A, A_b, Bm, Cm, Bm_b, Cm_b,
                         Dskip, D_b, z, delta_bias, delta_bias_b, delta_softplus, out_scale, y,
                         workspace, ws_bytes, true, (cudaStream_t)stream, last_state, true);
}

ssm_status bimamba_scan_fwd_v2_noalloc(ssm_dtype dt, int B, int D, int L, int N,
                                       const void *u, const void *u_b, const void *delta,
                                       const void *delta_b, const float *A, const float *A_b,
                                       const void *Bm, const void *Cm, const void *Bm_b,
                                       const void *Cm_b, const float *Dskip, const float *D_b,
                                       const void *z, const float *delta_bias,
                                       const float *delta_bias_b, int delta_softplus,
                                       float out_scale, void *y, ssm_stream_t stream) {
    ssm_status s = check_common(dt, B, D, L, N);
    if (s != SSM_OK) return s;
    // argument errors are reported before the scratch limit
    if (!io_ok(dt, u) || !opt_io_ok(dt, u_b) || !io_ok(dt, delta) || !io_ok(dt, delta_b) ||
        !io_ok(dt, Bm) || !io_ok(dt, Cm) || !io_ok(dt, Bm_b) || !io_ok(dt, Cm_b) ||
        !opt_io_ok(dt, z) || !io_ok(dt, y) || !f32_ok(A) || !f32_ok(A_b) ||
        !opt_f32_ok(Dskip) || !opt_f32_ok(D_b) || !opt_f32_ok(delta_bias) ||
        !opt_f32_ok(delta_bias_b))
        return SSM_ERR_INVALID_ARG;
    if (bi_ws(2, 2, B, D, L, nm_of(N)).total > SSM_STATIC_SCRATCH_BYTES)
        return SSM_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    s = static_scratch(&scratch);
    if (s != SSM_OK) return s;
    return bidirectional(dt, B, D, L, N, u, u_b, delta, delta_b, A, A_b, Bm, Cm, Bm_b, Cm_b,
                         Dskip, D_b, z, delta_bias, delta_bias_b, delta_softplus, out_scale, y,
                         scratch, SSM_STATIC_SCRATCH_BYTES, true, (cudaStream_t)stream);
}

ssm_status ss2d_scan_fwd(ssm_dtype dt, int B, int D, int H, int W, int N, int K,
                         const void *x, const void *delta, const float *A, const void *Bm,
                         const void *Cm, const float *Dskip, const void *z,
                         const float *delta_bias, int delta_softplus, void *y,
                         void *workspace, size_t ws_bytes, ssm_stream_t stream) {
    return ss2d_impl(dt, B, D, H, W, N, K, x, delta, A, Bm, Cm, Dskip, z, delta_bias,
                     delta_softplus, y, workspace, ws_bytes, stream, nullptr);
}

ssm_status ss2d_scan_fwd_ls(ssm_dtype dt, int B, int D, int H, int W, int N, int K,
                            const void *x, const void *delta, const float *A, const void *Bm,
                            const void *Cm, const float *Dskip, const void *z,
                            const float *delta_bias, int delta_softplus, void *y,
                            float *last_state, void *workspace, size_t ws_bytes,
                            ssm_stream_t stream) {
    if (last_state == nullptr) return SSM_ERR_INVALID_ARG;
    return ss2d_impl(dt, B, D, H, W, N, K, x, delta, A, Bm, Cm, Dskip, z, delta_bias,
                     delta_softplus, y, workspace, ws_bytes, stream, last_state);
}

size_t ssm_workspace_bytes(ssm_op op, ssm_dtype dt, int B, int D, int L_or_HW, int N, int K) {
    if (dt != SSM_F32 && dt != SSM_BF16 && dt != SSM_F16) return (size_t)-1;
    if (B < 0 || D < 0 || L_or_HW < 0 || N <= 0 || N > 2 * ssm::kMaxN) return (size_t)-1;
    const int nm = nm_of(N);
    switch (op) {
    case SSM_OP_SELECTIVE_SCAN:
        return bi_ws(1, 1, B, D, L_or_HW, nm).total;
    case SSM_OP_BIMAMBA_V1:
        return bi_ws(1, 2, B, D, L_or_HW, nm).total;
    case SSM_OP_BIMAMBA_V2:
        return bi_ws(2, 2, B, D, L_or_HW, nm).total;
    case SSM_OP_SS2D:
        if (K != 4) return (size_t)-1;
        return ss2d_ws(dt, B, D, L_or_HW, nm).total;
    }
    return (size_t)-1;
}

ssm_status ssm_get_status(const void *workspace, ssm_stream_t stream, ssm_status *out) {
    if (workspace == nullptr || out == nullptr) return SSM_ERR_INVALID_ARG;
    unsigned word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost,
                        (cudaStream_t)stream) != cudaSuccess ||
        cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) {
        cudaGetLastError();
        return SSM_ERR_CUDA;
    }
    *out = (word & 2u) ? SSM_ERR_BOUNDS : word ? SSM_ERR_TIMEOUT : SSM_OK;
    return SSM_OK;
}

const char *ssm_status_string(ssm_status s) {
    switch (s) {
    case SSM_OK: return "ok";
    case SSM_ERR_INVALID_ARG: return "invalid argument";
    case SSM_ERR_UNSUPPORTED: return "unsupported size or option";
    case SSM_ERR_CUDA: return "CUDA launch error";
    case SSM_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SSM_ERR_TIMEOUT: return "a kernel's bounded wait for its own copies ran out";
    case SSM_ERR_SCRATCH_LIMIT:
        return "problem needs more scratch than the library's fixed 64 MiB array";
    case SSM_ERR_BOUNDS:
        return "an index outside its tensor was caught and skipped (debug build)";
    }
    return "unknown status";
}

void ssm_test_withhold_copy(int chunk) { t_withhold = chunk; }

void ssm_test_shrink_extents(long long elems) { t_shrink = elems > 0 ? elems : 0; }

void ssm_set_cta_channels(int channels) {
    t_cta_channels = (channels == 8 || channels == 16) ? channels : 0;
}

void ssm_set_profile_events(void *begin, void *end) {
    t_prof_begin = (cudaEvent_t)begin;
    t_prof_end = (cudaEvent_t)end;
}

const char *ssm_version(void) { return "0.2.0"; }

}  // extern "C"
