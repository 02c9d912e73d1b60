// ssm_scan_api.cu -- the C ABI declared in include/ssm_scan.h.
//
// Each entry point validates its arguments on the host, fills the kernel's
// parameter block and launches the scan kernel(s) on the caller's stream.
// Nothing is allocated.  The one piece of state kept between calls is the
// fixed scratch array of the allocation-free entry point and its per-device
// address.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "scan_kernel.cuh"
#include "ssm_scan.h"

namespace {

using ssm::KParams;
using ssm::DirArgs;

constexpr int kChunk = 32;      // time steps per chunk (T)
constexpr int kRows = 16;       // channels per CTA (G)

bool aligned(const void *p, unsigned a) { return ((uintptr_t)p % a) == 0; }

// 2^31 - 1 bounds every per-dimension index the kernel forms in 32 bits.
bool fits(long long v) { return v >= 0 && v <= 0x7fffffffLL; }

int chunks_of(int L) { return (L + kChunk - 1) / kChunk; }

template <typename IO, int S, int NDIR, int MAP, int MODE>
ssm_status launch(const KParams &P, cudaStream_t stream) {
    using SM = ssm::Smem<IO, S, NDIR, kRows, kChunk>;
    constexpr int NT = NDIR * kRows * (ssm::kMaxN / S);
    auto *kern = &ssm::scan_kernel<IO, S, NDIR, kRows, kChunk, MAP, MODE>;
    // Raising the dynamic shared-memory limit is cheap and idempotent.
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::bytes) !=
        cudaSuccess) {
        cudaGetLastError();
        return SSM_ERR_CUDA;
    }
    dim3 grid((P.D + kRows - 1) / kRows, P.B);
    kern<<<grid, NT, SM::bytes, stream>>>(P);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// Pick the states-per-lane variant: 4 states per lane (more threads) unless
// the problem has enough rows to keep every SM busy with 8 per lane.
int pick_S(long long rows, int ndir) {
    const long long lanes8 = rows * ndir * 2;     // threads at S = 8
    return lanes8 >= 148LL * 384 ? 8 : 4;
}

template <int NDIR, int MAP, int MODE>
ssm_status dispatch(ssm_dtype dt, const KParams &P, cudaStream_t st) {
    const int S = pick_S((long long)P.B * P.D, NDIR);
    if (dt == SSM_F32) {
        return S == 8 ? launch<float, 8, NDIR, MAP, MODE>(P, st)
                      : launch<float, 4, NDIR, MAP, MODE>(P, st);
    }
    return S == 8 ? launch<__nv_bfloat16, 8, NDIR, MAP, MODE>(P, st)
                  : launch<__nv_bfloat16, 4, NDIR, MAP, MODE>(P, st);
}

ssm_status check_common(ssm_dtype dt, int B, int D, int L, int N) {
    if (dt != SSM_F32 && dt != SSM_BF16) return SSM_ERR_INVALID_ARG;
    if (B < 0 || D < 0 || L < 0 || N <= 0) return SSM_ERR_INVALID_ARG;
    if (N > ssm::kMaxN) return SSM_ERR_UNSUPPORTED;
    if (B > 65535) return SSM_ERR_UNSUPPORTED;                 // grid.y
    if (!fits((long long)D * L) || !fits((long long)N * L)) return SSM_ERR_UNSUPPORTED;
    return SSM_OK;
}

bool io_ok(const void *p) { return p != nullptr && aligned(p, 16); }
bool opt_io_ok(const void *p) { return p == nullptr || aligned(p, 16); }
bool f32_ok(const float *p) { return p != nullptr && aligned(p, 4); }
bool opt_f32_ok(const float *p) { return p == nullptr || aligned(p, 4); }

size_t bidir_ws(int B, int D, int L) {
    return chunks_of(L) > 1 ? (size_t)B * D * L * sizeof(float) : 0;
}

void fill_dir(DirArgs &a, const void *dt, long long dt_off, long long dt_bs, long long dt_total,
              const void *Bm, const void *Cm, long long bc_off, long long bc_bs,
              long long bc_total, const float *A, const float *Dskip, const float *bias,
              const void *u, int stream_rev) {
    a.dt = dt;
    a.dt_off = dt_off;
    a.dt_bs = dt_bs;
    a.dt_total = dt_total;
    a.Bm = Bm;
    a.Cm = Cm;
    a.bc_off = bc_off;
    a.bc_bs = bc_bs;
    a.bc_total = bc_total;
    a.A = A;
    a.Dskip = Dskip;
    a.bias = bias;
    a.u = u;
    a.stream_rev = stream_rev;
}

// Shared body of v1 / v2 (v1 passes the forward tensors for both branches).
ssm_status bidirectional(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                         const void *u_b, const void *delta, const void *delta_b,
                         const float *A, const float *A_b, const void *Bm, const void *Cm,
                         const void *Bm_b, const void *Cm_b, const float *Dskip,
                         const float *D_b, const void *z, const float *bias,
                         const float *bias_b, int delta_softplus, float out_scale, void *y,
                         void *ws, size_t ws_bytes, cudaStream_t stream) {
    ssm_status s = check_common(dt, B, D, L, N);
    if (s != SSM_OK) return s;
    if (!io_ok(u) || !opt_io_ok(u_b) || !io_ok(delta) || !io_ok(delta_b) || !io_ok(Bm) ||
        !io_ok(Cm) || !io_ok(Bm_b) || !io_ok(Cm_b) || !opt_io_ok(z) || !io_ok(y) ||
        !f32_ok(A) || !f32_ok(A_b) || !opt_f32_ok(Dskip) || !opt_f32_ok(D_b) ||
        !opt_f32_ok(bias) || !opt_f32_ok(bias_b))
        return SSM_ERR_INVALID_ARG;
    const size_t need = bidir_ws(B, D, L);
    if (need > 0 && (ws == nullptr || ws_bytes < need || !aligned(ws, 16)))
        return SSM_ERR_WORKSPACE;
    if ((long long)B * D * L == 0) return SSM_OK;
    const long long tot = (long long)B * D * L, bct = (long long)B * N * L;
    KParams P{};
    fill_dir(P.dir[0], delta, 0, (long long)D * L, tot, Bm, Cm, 0, (long long)N * L, bct, A,
             Dskip, bias, u, 0);
    fill_dir(P.dir[1], delta_b, 0, (long long)D * L, tot, Bm_b, Cm_b, 0, (long long)N * L, bct,
             A_b, D_b, bias_b, u_b ? u_b : u, 0);
    P.z = z;
    P.y = y;
    P.W = (float *)ws;
    P.u_total = tot;
    P.B = B;
    P.D = D;
    P.L = L;
    P.N = N;
    P.H = 1;
    P.Wd = L;
    P.nchunks = chunks_of(L);
    P.delta_softplus = delta_softplus ? 1 : 0;
    P.out_scale = out_scale;
    return dispatch<2, ssm::MAP_ROW, ssm::MODE_FINAL>(dt, P, stream);
}

// ---- fixed scratch of the allocation-free entry point
// The array lives in the library's device image; in host code its name is
// only a host-side stand-in, so the kernel is given the device address that
// cudaGetSymbolAddress reports for the current device (looked up once per
// device, on that device's first call).
constexpr int kMaxDevices = 256;
__device__ __align__(256) unsigned char g_static_scratch[SSM_STATIC_SCRATCH_BYTES];
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

}  // namespace

extern "C" {

ssm_status selective_scan_fwd(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                              const void *delta, const float *A, const void *Bm,
                              const void *Cm, const float *Dskip, const void *z,
                              const float *delta_bias, int delta_softplus, void *y,
                              void *workspace, size_t ws_bytes, ssm_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    ssm_status s = check_common(dt, B, D, L, N);
    if (s != SSM_OK) return s;
    if (!io_ok(u) || !io_ok(delta) || !io_ok(Bm) || !io_ok(Cm) || !opt_io_ok(z) ||
        !io_ok(y) || !f32_ok(A) || !opt_f32_ok(Dskip) || !opt_f32_ok(delta_bias))
        return SSM_ERR_INVALID_ARG;
    if ((long long)B * D * L == 0) return SSM_OK;
    const long long tot = (long long)B * D * L, bct = (long long)B * N * L;
    KParams P{};
    fill_dir(P.dir[0], delta, 0, (long long)D * L, tot, Bm, Cm, 0, (long long)N * L, bct, A,
             Dskip, delta_bias, u, 0);
    P.dir[1] = P.dir[0];
    P.z = z;
    P.y = y;
    P.W = nullptr;
    P.u_total = tot;
    P.B = B;
    P.D = D;
    P.L = L;
    P.N = N;
    P.H = 1;
    P.Wd = L;
    P.nchunks = chunks_of(L);
    P.delta_softplus = delta_softplus ? 1 : 0;
    P.out_scale = 1.f;
    return dispatch<1, ssm::MAP_ROW, ssm::MODE_FINAL>(dt, P, (cudaStream_t)stream);
}

ssm_status bimamba_scan_fwd_v1(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                               const void *delta, const float *A, const float *A_b,
                               const void *Bm, const void *Cm, const float *Dskip,
                               const void *z, const float *delta_bias, int delta_softplus,
                               float out_scale, void *y, void *workspace, size_t ws_bytes,
                               ssm_stream_t stream) {
    return bidirectional(dt, B, D, L, N, u, nullptr, delta, delta, A, A_b, Bm, Cm, Bm, Cm,
                         Dskip, Dskip, z, delta_bias, delta_bias, delta_softplus, out_scale, y,
                         workspace, ws_bytes, (cudaStream_t)stream);
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
                         workspace, ws_bytes, (cudaStream_t)stream);
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
    if (bidir_ws(B, D, L) > SSM_STATIC_SCRATCH_BYTES) return SSM_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    s = static_scratch(&scratch);
    if (s != SSM_OK) return s;
    return bidirectional(dt, B, D, L, N, u, u_b, delta, delta_b, A, A_b, Bm, Cm, Bm_b, Cm_b,
                         Dskip, D_b, z, delta_bias, delta_bias_b, delta_softplus, out_scale, y,
                         scratch, SSM_STATIC_SCRATCH_BYTES, (cudaStream_t)stream);
}

ssm_status ss2d_scan_fwd(ssm_dtype dt, int B, int D, int H, int W, int N, int K,
                         const void *x, const void *delta, const float *A, const void *Bm,
                         const void *Cm, const float *Dskip, const void *z,
                         const float *delta_bias, int delta_softplus, void *y,
                         void *workspace, size_t ws_bytes, ssm_stream_t stream) {
    if (H < 0 || W < 0) return SSM_ERR_INVALID_ARG;
    if (K != 4) return SSM_ERR_UNSUPPORTED;
    if (!fits((long long)H * W)) return SSM_ERR_UNSUPPORTED;
    const int L = H * W;
    ssm_status s = check_common(dt, B, D, L, N);
    if (s != SSM_OK) return s;
    if (!fits((long long)K * D * L) || !fits((long long)K * N * L)) return SSM_ERR_UNSUPPORTED;
    if (!io_ok(x) || !io_ok(delta) || !io_ok(Bm) || !io_ok(Cm) || !opt_io_ok(z) ||
        !io_ok(y) || !f32_ok(A) || !opt_f32_ok(Dskip) || !opt_f32_ok(delta_bias))
        return SSM_ERR_INVALID_ARG;
    const size_t need = ssm_workspace_bytes(SSM_OP_SS2D, dt, B, D, L, N, K);
    if (need > 0 && (workspace == nullptr || ws_bytes < need || !aligned(workspace, 16)))
        return SSM_ERR_WORKSPACE;
    if ((long long)B * D * L == 0) return SSM_OK;
    const long long DL = (long long)D * L, NL = (long long)N * L;
    const long long dtot = (long long)B * K * DL, bct = (long long)B * K * NL;
    auto dir = [&](DirArgs &a, int k, int stream_rev) {
        fill_dir(a, delta, k * DL, K * DL, dtot, Bm, Cm, k * NL, K * NL, bct,
                 A + (long long)k * D * N, Dskip ? Dskip + (long long)k * D : nullptr,
                 delta_bias ? delta_bias + (long long)k * D : nullptr, x, stream_rev);
    };
    KParams P{};
    P.z = z;
    P.y = y;
    P.W = (float *)workspace;
    P.u_total = (long long)B * DL;
    P.B = B;
    P.D = D;
    P.L = L;
    P.N = N;
    P.H = H;
    P.Wd = W;
    P.nchunks = chunks_of(L);
    P.delta_softplus = delta_softplus ? 1 : 0;
    P.out_scale = 1.f;
    // Row-major pair: directions 0 (forward) and 2 (reversed), fused sum to W.
    dir(P.dir[0], 0, 0);
    dir(P.dir[1], 2, 1);
    s = dispatch<2, ssm::MAP_ROW, ssm::MODE_ACCOUT>(dt, P, (cudaStream_t)stream);
    if (s != SSM_OK) return s;
    // Column-major pair: directions 1 and 3; adds W, gates and stores y.
    dir(P.dir[0], 1, 0);
    dir(P.dir[1], 3, 1);
    return dispatch<2, ssm::MAP_COL, ssm::MODE_ACCIN>(dt, P, (cudaStream_t)stream);
}

size_t ssm_workspace_bytes(ssm_op op, ssm_dtype dt, int B, int D, int L_or_HW, int N, int K) {
    (void)N;
    if (dt != SSM_F32 && dt != SSM_BF16) return (size_t)-1;
    if (B < 0 || D < 0 || L_or_HW < 0) return (size_t)-1;
    switch (op) {
    case SSM_OP_SELECTIVE_SCAN:
        return 0;
    case SSM_OP_BIMAMBA_V1:
    case SSM_OP_BIMAMBA_V2:
        return bidir_ws(B, D, L_or_HW);
    case SSM_OP_SS2D:
        if (K != 4) return (size_t)-1;
        return (size_t)B * D * L_or_HW * sizeof(float);
    }
    return (size_t)-1;
}

const char *ssm_status_string(ssm_status s) {
    switch (s) {
    case SSM_OK: return "ok";
    case SSM_ERR_INVALID_ARG: return "invalid argument";
    case SSM_ERR_UNSUPPORTED: return "unsupported size or option";
    case SSM_ERR_CUDA: return "CUDA launch error";
    case SSM_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SSM_ERR_SCRATCH_LIMIT:
        return "problem needs more scratch than the library's fixed 64 MiB array";
    }
    return "unknown status";
}

const char *ssm_version(void) { return "0.1.0"; }

}  // extern "C"
