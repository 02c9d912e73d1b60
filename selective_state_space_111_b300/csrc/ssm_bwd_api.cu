// ssm_bwd_api.cu -- the backward entry points declared in include/ssm_scan.h.
//
// Each call: (1) recomputes the pre-gate output y with the forward entry
// point (only when z is given), (2) gy = dout * silu(z) and dz, (3) one
// scan_bwd_kernel launch for all directions, each writing its own fp32
// per-position gradients and per-CTA partial sums of the parameter
// gradients, (4) fixed-order sums and reductions, and conversion to the
// output dtypes.  Nothing is allocated; everything lives in the
// caller's workspace (ssm_bwd_workspace_bytes).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bwd_kernel.cuh"
#include "internal.h"
#include "ssm_scan.h"

namespace {

using ssm::bwd::Pass;

bool aligned(const void *p, unsigned a) { return ((uintptr_t)p % a) == 0; }
bool fits(long long v) { return v >= 0 && v <= 0x7fffffffLL; }
unsigned esz(ssm_dtype dt) { return dt == SSM_F32 ? 4u : 2u; }
bool io_ok(ssm_dtype dt, const void *p) { return p != nullptr && aligned(p, esz(dt)); }
bool opt_io(ssm_dtype dt, const void *p) { return p == nullptr || aligned(p, esz(dt)); }
bool f32_ok(const float *p) { return p != nullptr && aligned(p, 4); }
bool opt_f32(const float *p) { return p == nullptr || aligned(p, 4); }

ssm_status check_sizes(ssm_dtype dt, int B, int D, int L, int N) {
    if (dt != SSM_F32 && dt != SSM_BF16 && dt != SSM_F16) return SSM_ERR_INVALID_ARG;
    if (B < 0 || D < 0 || L < 0 || N <= 0) return SSM_ERR_INVALID_ARG;
    if (N > 2 * ssm::kMaxN) return SSM_ERR_UNSUPPORTED;      // up to 32 states
    if (B > 65535) return SSM_ERR_UNSUPPORTED;
    if (!fits((long long)D * L) || !fits((long long)N * L)) return SSM_ERR_UNSUPPORTED;
    return SSM_OK;
}

size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

// state capacity (16 or 32) and channels per backward CTA for N states
int nm_of(int N) { return N <= ssm::kMaxN ? ssm::kMaxN : 2 * ssm::kMaxN; }
int ch_of(int N) { return ssm::bwd::NT / nm_of(N); }
// steps per chunk of the backward scan (the 16-state kernel's chunks are
// shorter: its recomputed states take eight floats per thread and step)
int chunk_of(int N) { return N <= ssm::kMaxN ? ssm::bwd::T16 : ssm::bwd::T; }
int nch_of(int L, int N) { return (L + chunk_of(N) - 1) / chunk_of(N); }

template <typename IO> constexpr ssm_dtype dtype_of() { return SSM_BF16; }
template <> constexpr ssm_dtype dtype_of<float>() { return SSM_F32; }
template <> constexpr ssm_dtype dtype_of<__half>() { return SSM_F16; }

// Workspace of one backward call; every region starts on 256 bytes.
struct BwdWs {
    size_t fwd, ypre, G, GT, xT, du, ddt, hc, pdB, pdC, pdA, pbias, pdD, total;
    size_t fwd_bytes;
};
// op: 0 single, 1 v1, 2 v2, 3 SS2D.  du and ddt hold one fp32 map per
// direction (SS2D's ddt is [B][4][D][L], like delta).
BwdWs bwd_ws(int op, ssm_dtype dt, int B, int D, int L, int N, bool sep_ub) {
    (void)sep_ub;
    const size_t n = (size_t)B * D * L;
    const int npass = op == 0 ? 1 : op == 3 ? 4 : 2;
    const int nm = nm_of(N), ncg = (D + ch_of(N) - 1) / ch_of(N);
    const int nch = nch_of(L, N);
    BwdWs w{};
    size_t off = 256;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += up256(bytes);
        return o;
    };
    const ssm_op fop = op == 0 ? SSM_OP_SELECTIVE_SCAN
                       : op == 1 ? SSM_OP_BIMAMBA_V1
                       : op == 2 ? SSM_OP_BIMAMBA_V2
                                 : SSM_OP_SS2D;
    w.fwd_bytes = ssm_workspace_bytes(fop, dt, B, D, L, N, 4);
    w.fwd = take(w.fwd_bytes);
    w.ypre = take(n * esz(dt));
    w.G = take(n * 4);
    w.GT = op == 3 ? take(n * 4) : 0;
    w.xT = op == 3 ? take(n * esz(dt)) : 0;
    w.du = take(n * 4 * npass);
    w.ddt = take(n * 4 * npass);
    // chunk-start states: one region per direction (they run concurrently)
    w.hc = take((size_t)npass * B * D * nch * nm * 4);
    const size_t part = (size_t)npass * ncg * B * L * nm * 4;
    w.pdB = take(part);
    w.pdC = take(part);
    w.pdA = take((size_t)npass * B * D * nm * 4);
    // per-(direction, batch, channel) sums of ddt and G * u (16 states)
    w.pbias = take((size_t)npass * B * D * 4);
    w.pdD = take((size_t)npass * B * D * 4);
    w.total = off;
    return w;
}

int grid1d(long long n) {
    long long g = (n + 255) / 256;
    return (int)(g < 1 ? 1 : g > 148 * 16 ? 148 * 16 : g);
}

ssm_status last_error() {
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// One scan_bwd_kernel launch for all directions (grid: channel groups x
// batch x directions).
template <typename IO, int NM>
ssm_status launch_passes_nm(const Pass *ps, int npass, int B, int D, int L, int N, int sp,
                            bool hc_given, cudaStream_t st) {
    ssm::bwd::Params P{};
    for (int k = 0; k < npass; ++k) P.ps[k] = ps[k];
    P.B = B;
    P.D = D;
    P.L = L;
    P.N = N;
    P.nch = nch_of(L, N);
    P.delta_softplus = sp ? 1 : 0;
    P.hc_given = (NM == ssm::kMaxN && hc_given) ? 1 : 0;
    if constexpr (NM == ssm::kMaxN) {
        // 16 states: eight per thread, 32 channels per CTA
        constexpr int dyn = ssm::bwd::H16_BYTES;
        dim3 grid((D + ssm::bwd::CH16 - 1) / ssm::bwd::CH16, B, npass);
        auto *kern = &ssm::bwd::scan_bwd16_kernel<IO>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) !=
            cudaSuccess) {
            cudaGetLastError();
            return SSM_ERR_CUDA;
        }
        kern<<<grid, ssm::bwd::NT16, dyn, st>>>(P);
        return last_error();
    } else {
        constexpr int CH = ssm::bwd::channels<NM>();
        constexpr int dyn = ssm::bwd::dyn_bytes<NM>();
        dim3 grid((D + CH - 1) / CH, B, npass);
        auto *kern = &ssm::bwd::scan_bwd_kernel<IO, NM>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) !=
            cudaSuccess) {
            cudaGetLastError();
            return SSM_ERR_CUDA;
        }
        kern<<<grid, ssm::bwd::NT, dyn, st>>>(P);
        return last_error();
    }
}
// hc_given: the forward pass of this call stored the chunk-start states
// (16 states only)
template <typename IO>
ssm_status launch_passes(const Pass *ps, int npass, int B, int D, int L, int N, int sp,
                         bool hc_given, cudaStream_t st) {
    if (N <= ssm::kMaxN)
        return launch_passes_nm<IO, ssm::kMaxN>(ps, npass, B, D, L, N, sp, hc_given, st);
    return launch_passes_nm<IO, 2 * ssm::kMaxN>(ps, npass, B, D, L, N, sp, false, st);
}

// Saved backward context of this host thread (ssm_set_bwd_context).
thread_local void *t_ctx = nullptr;
thread_local size_t t_ctx_bytes = 0;

// Scope in which the forward calls of this host thread also store their
// chunk-start states for the 16-state backward kernel.
struct CaptureScope {
    explicit CaptureScope(float *const *hc) { ssm_internal::set_chunk_state_capture(hc); }
    ~CaptureScope() { ssm_internal::set_chunk_state_capture(nullptr); }
    CaptureScope(const CaptureScope &) = delete;
    CaptureScope &operator=(const CaptureScope &) = delete;
};

template <typename IO>
ssm_status gate_bwd(const void *g, const void *z, const void *y, float *G, void *dz, long long n,
                    cudaStream_t st) {
    ssm::bwd::gate_bwd_kernel<IO><<<grid1d(n), 256, 0, st>>>(
        (const IO *)g, (const IO *)z, (const IO *)y, G, (IO *)dz, n);
    return last_error();
}

template <typename E>
ssm_status transpose(const E *in, E *out, int maps, int R, int C, cudaStream_t st) {
    dim3 grid((C + 31) / 32, (R + 31) / 32, maps < 65535 ? maps : 65535);
    ssm::bwd::transpose_kernel<E><<<grid, 256, 0, st>>>(in, out, maps, R, C);
    return last_error();
}

template <typename E>
ssm_status convert(const float *a, const float *b, const float *c, void *out, long long n,
                   cudaStream_t st) {
    ssm::bwd::convert_kernel<E><<<grid1d(n), 256, 0, st>>>(a, b, c, (E *)out, n);
    return last_error();
}

template <typename IO>
ssm_status reduce_bc(const ssm::bwd::BcJobs &J, int njobs, int B, int L, int N,
                     cudaStream_t st) {
    if (B == 0 || L == 0 || njobs == 0) return SSM_OK;
    if (N <= ssm::kMaxN) {
        constexpr int PS = 256 / (ssm::kMaxN / 4);
        ssm::bwd::reduce_bc_kernel<IO, ssm::kMaxN>
            <<<dim3((L + PS - 1) / PS, B, njobs), 256, 0, st>>>(J, B, L, N);
    } else {
        constexpr int PS = 256 / (2 * ssm::kMaxN / 4);
        ssm::bwd::reduce_bc_kernel<IO, 2 * ssm::kMaxN>
            <<<dim3((L + PS - 1) / PS, B, njobs), 256, 0, st>>>(J, B, L, N);
    }
    return last_error();
}

// out[d] = scale * sum over (b, t) of (a [+ a2]) [* u], see channel_sum_kernel
template <typename IO>
ssm_status channel_sum(const float *a, const float *a2, long long a_bstride, const void *u,
                       int B, int D, int L, float scale, float *out, cudaStream_t st) {
    if (out == nullptr) return SSM_OK;
    ssm::bwd::channel_sum_kernel<IO><<<D, 256, 0, st>>>(a, a2, a_bstride, (const IO *)u, B, D, L,
                                                         scale, out);
    return last_error();
}

// Parameter-gradient reductions gathered for one launch (null outputs are
// skipped).
struct ParamList {
    ssm::bwd::ParamJobs J{};
    int n = 0;
    bool per_state_any = false;
    void add(const float *part, int nslot, bool per_state, float *out) {
        if (out == nullptr) return;
        J.part[n] = part;
        J.out[n] = out;
        J.nslot[n] = nslot;
        J.per_state[n] = per_state ? 1 : 0;
        per_state_any = per_state_any || per_state;
        ++n;
    }
};
ssm_status reduce_params(const ParamList &pl, int B, int D, int N, cudaStream_t st) {
    if (pl.n == 0) return SSM_OK;
    const int cols = pl.per_state_any ? D * nm_of(N) : D;
    dim3 grid(grid1d(cols), pl.n);
    ssm::bwd::reduce_param_kernel<<<grid, 256, 0, st>>>(pl.J, B, D, N, nm_of(N));
    return last_error();
}

#define TRY(x)                              \
    do {                                    \
        const ssm_status s_ = (x);          \
        if (s_ != SSM_OK) return s_;        \
    } while (0)

// The common tail: partials of pass p live at slot offset p * ncg.
struct Parts {
    const float *pdB, *pdC, *pdA;
    int ncg, B, D, L, N;
    const float *dB_slot(int p) const { return pdB + (size_t)p * ncg * B * L * nm_of(N); }
    const float *dC_slot(int p) const { return pdC + (size_t)p * ncg * B * L * nm_of(N); }
    const float *dA_slot(int p) const { return pdA + (size_t)p * B * D * nm_of(N); }
};

Parts parts_of(char *ws, const BwdWs &w, int B, int D, int L, int N) {
    Parts q;
    q.pdB = (const float *)(ws + w.pdB);
    q.pdC = (const float *)(ws + w.pdC);
    q.pdA = (const float *)(ws + w.pdA);
    q.ncg = (D + ch_of(N) - 1) / ch_of(N);
    q.B = B;
    q.D = D;
    q.L = L;
    q.N = N;
    return q;
}

// Pass p's parameter and scratch pointers into the workspace.
Pass base_pass(char *ws, const BwdWs &w, int p, int B, int D, int L, int N) {
    Pass ps{};
    const int nm = nm_of(N), ncg = (D + ch_of(N) - 1) / ch_of(N);
    ps.pdB = (float *)(ws + w.pdB) + (size_t)p * ncg * B * L * nm;
    ps.pdC = (float *)(ws + w.pdC) + (size_t)p * ncg * B * L * nm;
    ps.pdA = (float *)(ws + w.pdA) + (size_t)p * B * D * nm;
    ps.hc = (float *)(ws + w.hc) + (size_t)p * B * D * nch_of(L, N) * nm;
    ps.G = (const float *)(ws + w.G);
    ps.gscale = 1.f;
    if (N <= ssm::kMaxN) {
        // the 16-state kernel sums dbias and dD itself
        ps.pbias = (float *)(ws + w.pbias) + (size_t)p * B * D;
        ps.pdD = (float *)(ws + w.pdD) + (size_t)p * B * D;
    }
    return ps;
}

// ---- the sequence forms (single, v1, v2)
template <typename IO>
ssm_status seq_bwd(int op, int B, int D, int L, int N, const void *u, const void *u_b,
                   const void *delta, const void *delta_b, const float *A, const float *A_b,
                   const void *Bm, const void *Cm, const void *Bm_b, const void *Cm_b,
                   const float *Dskip, const float *D_b, const void *z, const float *bias,
                   const float *bias_b, int sp, float out_scale, const void *dout, void *du,
                   void *du_b, void *ddelta, void *ddelta_b, float *dA, float *dA_b, void *dB,
                   void *dC, void *dB_b, void *dC_b, float *dD, float *dD_b, void *dz,
                   float *dbias, float *dbias_b, char *ws, const BwdWs &w, cudaStream_t st) {
    const ssm_dtype dt = dtype_of<IO>();
    const long long n = (long long)B * D * L;
    float *G = (float *)(ws + w.G);
    float *du0 = (float *)(ws + w.du), *du1 = du0 + n;      // per direction
    float *dt0 = (float *)(ws + w.ddt), *dt1 = dt0 + n;
    // (1) the forward pass: the pre-gate output (for dz) and, with 16
    // states, the chunk-start states of every direction (the backward
    // kernel then skips its own forward sweep) -- or, with a saved context
    // (16 states), both as the forward call left them
    void *ypre = ws + w.ypre;
    void *fws = ws + w.fwd;
    const bool capture = N <= ssm::kMaxN;
    const bool from_ctx = capture && t_ctx != nullptr;
    ssm_internal::CtxLayout cl{};
    if (from_ctx) {
        cl = ssm_internal::ctx_layout(op == 0 ? 1 : 2, esz(dt), B, D, L);
        if (t_ctx_bytes < cl.total || !aligned(t_ctx, 16)) return SSM_ERR_WORKSPACE;
        ypre = (char *)t_ctx + cl.ypre;
    }
    if (!from_ctx && (z != nullptr || capture)) {
        float *hc[4] = {base_pass(ws, w, 0, B, D, L, N).hc,
                        op == 0 ? nullptr : base_pass(ws, w, 1, B, D, L, N).hc, nullptr, nullptr};
        CaptureScope scope(capture ? hc : nullptr);
        ssm_stream_t sst = (ssm_stream_t)st;
        if (op == 0)
            TRY(selective_scan_fwd(dt, B, D, L, N, u, delta, A, Bm, Cm, Dskip, nullptr, bias, sp,
                                   ypre, fws, w.fwd_bytes, sst));
        else if (op == 1)
            TRY(bimamba_scan_fwd_v1(dt, B, D, L, N, u, delta, A, A_b, Bm, Cm, Dskip, nullptr,
                                    bias, sp, out_scale, ypre, fws, w.fwd_bytes, sst));
        else
            TRY(bimamba_scan_fwd_v2(dt, B, D, L, N, u, u_b, delta, delta_b, A, A_b, Bm, Cm,
                                    Bm_b, Cm_b, Dskip, D_b, nullptr, bias, bias_b, sp,
                                    out_scale, ypre, fws, w.fwd_bytes, sst));
    }
    // (2) gy and dz
    TRY(gate_bwd<IO>(dout, z, ypre, G, dz, n, st));
    // (3) one pass per direction
    const long long DL = (long long)D * L, NL = (long long)N * L;
    Pass p0 = base_pass(ws, w, 0, B, D, L, N);
    p0.dt = delta;
    p0.dt_off = 0;
    p0.dt_bstride = DL;
    p0.u = u;
    p0.Bm = Bm;
    p0.Cm = Cm;
    p0.bc_off = 0;
    p0.bc_bstride = NL;
    p0.A = A;
    p0.Dskip = Dskip;
    p0.bias = bias;
    p0.gscale = op == 0 ? 1.f : out_scale;
    p0.rev = 0;
    p0.stream_rev = 0;
    p0.du = du0;
    p0.ddt = dt0;
    if (from_ctx) p0.hc = (float *)((char *)t_ctx + cl.hc[0]);
    // 16 states: a direction that owns its du or ddelta writes it in the
    // I/O dtype directly; tensors the two branches share are summed from
    // the fp32 maps below
    const bool fused = N <= ssm::kMaxN;
    const bool du_own = op == 0 || (op == 2 && u_b != nullptr), ddt_own = op != 1;
    if (fused) {
        p0.du_io = du_own ? du : nullptr;
        p0.ddt_io = ddt_own ? ddelta : nullptr;
    }
    Pass pp[2] = {p0, p0};
    if (op != 0) {
        Pass p1 = p0;
        Pass q = base_pass(ws, w, 1, B, D, L, N);
        p1.pdB = q.pdB;
        p1.pdC = q.pdC;
        p1.pdA = q.pdA;
        p1.hc = from_ctx ? (float *)((char *)t_ctx + cl.hc[1]) : q.hc;
        p1.pbias = q.pbias;
        p1.pdD = q.pdD;
        p1.du_io = fused && du_own ? du_b : nullptr;
        p1.ddt_io = fused && ddt_own ? ddelta_b : nullptr;
        p1.dt = op == 2 ? delta_b : delta;
        p1.u = (op == 2 && u_b) ? u_b : u;
        p1.Bm = op == 2 ? Bm_b : Bm;
        p1.Cm = op == 2 ? Cm_b : Cm;
        p1.A = A_b;
        p1.Dskip = op == 2 ? D_b : Dskip;
        p1.bias = op == 2 ? bias_b : bias;
        p1.rev = 1;
        p1.du = du1;
        p1.ddt = dt1;
        pp[1] = p1;
    }
    TRY(launch_passes<IO>(pp, op == 0 ? 1 : 2, B, D, L, N, sp, capture, st));
    // (4) outputs: shared tensors sum both branches' gradients
    const bool shared_u = op == 1 || (op == 2 && u_b == nullptr);
    if (!(fused && du_own)) {
        TRY(convert<IO>(du0, shared_u ? du1 : nullptr, nullptr, du, n, st));
        if (op == 2 && u_b != nullptr) TRY(convert<IO>(du1, nullptr, nullptr, du_b, n, st));
    }
    if (!(fused && ddt_own)) {
        TRY(convert<IO>(dt0, op == 1 ? dt1 : nullptr, nullptr, ddelta, n, st));
        if (op == 2) TRY(convert<IO>(dt1, nullptr, nullptr, ddelta_b, n, st));
    }
    const Parts q = parts_of(ws, w, B, D, L, N);
    const int shared_bc = op == 1 ? 2 : 1;      // v1: both passes add into dB, dC
    {
        // dB, dC (and for v2 dB_b, dC_b) in one launch
        ssm::bwd::BcJobs J{};
        J.out_bstride = NL;
        const float *parts[4] = {q.dB_slot(0), q.dC_slot(0), op == 2 ? q.dB_slot(1) : nullptr,
                                 op == 2 ? q.dC_slot(1) : nullptr};
        void *outs[4] = {dB, dC, dB_b, dC_b};
        for (int j = 0; j < (op == 2 ? 4 : 2); ++j) {
            J.part[j] = parts[j];
            J.out[j] = outs[j];
            J.nslot[j] = j < 2 ? shared_bc * q.ncg : q.ncg;
        }
        TRY(reduce_bc<IO>(J, op == 2 ? 4 : 2, B, L, N, st));
    }
    // dA of each direction; with 16 states also dD and dbias from the
    // kernel's per-(direction, batch) channel sums -- one launch
    ParamList pl;
    pl.add(q.dA_slot(0), 1, true, dA);
    if (op != 0) pl.add(q.dA_slot(1), 1, true, dA_b);
    // dD: each branch's skip term is D * u_t at every position, so
    // dD = gscale * sum G u (v1: both branches, shared D); dbias = sum ddt
    const float gs = op == 0 ? 1.f : out_scale;
    if (fused) {
        // (G already carries gscale; v1 adds both directions)
        const float *pb = p0.pbias, *pd = p0.pdD;
        const int nsum = op == 1 ? 2 : 1;
        if (Dskip) pl.add(pd, nsum, false, dD);
        pl.add(pb, nsum, false, dbias);
        if (op == 2) {
            if (D_b) pl.add(pd + (size_t)B * D, 1, false, dD_b);
            pl.add(pb + (size_t)B * D, 1, false, dbias_b);
        }
        return reduce_params(pl, B, D, N, st);
    }
    TRY(reduce_params(pl, B, D, N, st));
    if (Dskip) TRY(channel_sum<IO>(G, nullptr, DL, u, B, D, L, op == 1 ? 2.f * gs : gs, dD, st));
    TRY(channel_sum<IO>(dt0, op == 1 ? dt1 : nullptr, DL, nullptr, B, D, L, 1.f, dbias, st));
    if (op == 2) {
        if (D_b) TRY(channel_sum<IO>(G, nullptr, DL, u_b ? u_b : u, B, D, L, gs, dD_b, st));
        TRY(channel_sum<IO>(dt1, nullptr, DL, nullptr, B, D, L, 1.f, dbias_b, st));
    }
    return SSM_OK;
}

// ---- SS2D: directions 0/2 walk x row-major (forward / reversed), 1/3 walk
// x^T (column-major of x); each direction's delta, B and C are in its scan
// order, so the reversed directions read them by walk step.
template <typename IO>
ssm_status ss2d_bwd_run(int B, int D, int H, int W, int N, const void *x, const void *delta,
                        const float *A, const void *Bm, const void *Cm, const float *Dskip,
                        const void *z, const float *bias, int sp, const void *dout, void *dx,
                        void *ddelta, float *dA, void *dB, void *dC, float *dD, void *dz,
                        float *dbias, char *ws, const BwdWs &w, cudaStream_t st) {
    const ssm_dtype dt = dtype_of<IO>();
    const int L = H * W, K = 4;
    const long long n = (long long)B * D * L;
    void *ypre = ws + w.ypre;
    // the forward pass: the pre-gate output (for dz) and, with 16 states,
    // the chunk-start states of the four directions
    const bool capture = N <= ssm::kMaxN;
    if (z != nullptr || capture) {
        float *hc[4];
        for (int k = 0; k < K; ++k) hc[k] = base_pass(ws, w, k, B, D, L, N).hc;
        CaptureScope scope(capture ? hc : nullptr);
        TRY(ss2d_scan_fwd(dt, B, D, H, W, N, K, x, delta, A, Bm, Cm, Dskip, nullptr, bias, sp,
                          ypre, ws + w.fwd, w.fwd_bytes, (ssm_stream_t)st));
    }
    float *G = (float *)(ws + w.G), *GT = (float *)(ws + w.GT);
    IO *xT = (IO *)(ws + w.xT);
    TRY(gate_bwd<IO>(dout, z, ypre, G, dz, n, st));
    TRY(transpose<float>(G, GT, B * D, H, W, st));
    TRY(transpose<IO>((const IO *)x, xT, B * D, H, W, st));
    const long long DL = (long long)D * L, NL = (long long)N * L;
    float *du = (float *)(ws + w.du);                 // [4][B][D][L], one map per direction
    Pass pp[4];
    for (int k = 0; k < K; ++k) {
        Pass ps = base_pass(ws, w, k, B, D, L, N);
        const bool col = k == 1 || k == 3;
        ps.dt = delta;
        ps.dt_off = k * DL;
        ps.dt_bstride = K * DL;
        ps.Bm = Bm;
        ps.Cm = Cm;
        ps.bc_off = k * NL;
        ps.bc_bstride = K * NL;
        ps.A = A + (long long)k * D * N;
        ps.Dskip = Dskip ? Dskip + (long long)k * D : nullptr;
        ps.bias = bias ? bias + (long long)k * D : nullptr;
        ps.u = col ? (const void *)xT : x;
        ps.G = col ? GT : G;
        ps.rev = k >= 2;
        ps.stream_rev = k >= 2;
        ps.du = du + k * n;
        ps.ddt = (float *)(ws + w.ddt);
        if (capture) ps.ddt_io = ddelta;        // each direction owns its ddelta slice
        pp[k] = ps;
    }
    TRY(launch_passes<IO>(pp, K, B, D, L, N, sp, capture, st));
    // dx = row pair (0, 2) + the column pair (1, 3) transposed back; G^T's
    // space is free now
    TRY(convert<float>(du + n, du + 3 * n, nullptr, du + n, n, st));
    TRY(transpose<float>(du + n, GT, B * D, W, H, st));
    TRY(convert<IO>(du, du + 2 * n, GT, dx, n, st));
    if (!capture)
        TRY(convert<IO>((const float *)(ws + w.ddt), nullptr, nullptr, ddelta, n * K, st));
    const Parts q = parts_of(ws, w, B, D, L, N);
    {
        // the four directions' dB and dC in one launch
        ssm::bwd::BcJobs J{};
        J.out_bstride = K * NL;
        for (int k = 0; k < K; ++k) {
            J.part[2 * k] = q.dB_slot(k);
            J.out[2 * k] = (IO *)dB + k * NL;
            J.part[2 * k + 1] = q.dC_slot(k);
            J.out[2 * k + 1] = (IO *)dC + k * NL;
            J.nslot[2 * k] = J.nslot[2 * k + 1] = q.ncg;
        }
        TRY(reduce_bc<IO>(J, 2 * K, B, L, N, st));
    }
    ParamList pl;
    for (int k = 0; k < K; ++k) {
        pl.add(q.dA_slot(k), 1, true, dA + (long long)k * D * N);
        if (capture) {
            // the kernel's channel sums: every direction visits every
            // position once, so its sum of G * x is dD_k
            if (Dskip) pl.add(pp[k].pdD, 1, false, dD ? dD + k * D : nullptr);
            pl.add(pp[k].pbias, 1, false, dbias ? dbias + k * D : nullptr);
            continue;
        }
        // every direction visits every position once: dD_k = sum G x
        if (Dskip)
            TRY(channel_sum<IO>(G, nullptr, DL, x, B, D, L, 1.f, dD ? dD + k * D : nullptr, st));
        TRY(channel_sum<IO>((const float *)(ws + w.ddt) + k * DL, nullptr, K * DL, nullptr, B, D,
                            L, 1.f, dbias ? dbias + k * D : nullptr, st));
    }
    return reduce_params(pl, B, D, N, st);
}

}  // namespace

void *ssm_internal::bwd_context(size_t *bytes) {
    if (bytes) *bytes = t_ctx_bytes;
    return t_ctx;
}

ssm_internal::CtxLayout ssm_internal::ctx_layout(int ndir, unsigned esize, int B, int D, int L) {
    CtxLayout c{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += (bytes + 255) / 256 * 256;
        return at;
    };
    const size_t n = (size_t)B * D * L;
    c.ypre = take(n * esize);
    for (int k = 0; k < ndir; ++k)
        c.hc[k] = take((size_t)B * D * nch_of(L, ssm::kMaxN) * ssm::kMaxN * sizeof(float));
    c.total = off;
    return c;
}

extern "C" {

void ssm_set_bwd_context(void *ctx, size_t ctx_bytes) {
    t_ctx = ctx;
    t_ctx_bytes = ctx ? ctx_bytes : 0;
}

size_t ssm_bwd_context_bytes(ssm_op op, ssm_dtype dt, int B, int D, int L, int N) {
    if (dt != SSM_F32 && dt != SSM_BF16 && dt != SSM_F16) return (size_t)-1;
    if (B < 0 || D < 0 || L < 0 || N <= 0 || N > 2 * ssm::kMaxN) return (size_t)-1;
    int ndir;
    switch (op) {
    case SSM_OP_SELECTIVE_SCAN: ndir = 1; break;
    case SSM_OP_BIMAMBA_V1:
    case SSM_OP_BIMAMBA_V2: ndir = 2; break;
    default: return (size_t)-1;
    }
    if (N > ssm::kMaxN || (long long)B * D * L == 0) return 0;
    return ssm_internal::ctx_layout(ndir, esz(dt), B, D, L).total;
}

size_t ssm_bwd_workspace_bytes(ssm_op op, ssm_dtype dt, int B, int D, int L_or_HW, int N, int K,
                               int separate_u_b) {
    if (dt != SSM_F32 && dt != SSM_BF16 && dt != SSM_F16) return (size_t)-1;
    if (B < 0 || D < 0 || L_or_HW < 0 || N <= 0 || N > 2 * ssm::kMaxN) return (size_t)-1;
    int o;
    switch (op) {
    case SSM_OP_SELECTIVE_SCAN: o = 0; break;
    case SSM_OP_BIMAMBA_V1: o = 1; break;
    case SSM_OP_BIMAMBA_V2: o = 2; break;
    case SSM_OP_SS2D:
        if (K != 4) return (size_t)-1;
        o = 3;
        break;
    default: return (size_t)-1;
    }
    if ((long long)B * D * L_or_HW == 0) return 0;
    return bwd_ws(o, dt, B, D, L_or_HW, N, separate_u_b != 0).total;
}

ssm_status selective_scan_bwd(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                              const void *delta, const float *A, const void *Bm, const void *Cm,
                              const float *Dskip, const void *z, const float *delta_bias,
                              int delta_softplus, const void *dout, void *du, void *ddelta,
                              float *dA, void *dB, void *dC, float *dD, void *dz,
                              float *ddelta_bias, void *workspace, size_t ws_bytes,
                              ssm_stream_t stream) {
    TRY(check_sizes(dt, B, D, L, N));
    if (!io_ok(dt, u) || !io_ok(dt, delta) || !io_ok(dt, Bm) || !io_ok(dt, Cm) ||
        !opt_io(dt, z) || !io_ok(dt, dout) || !io_ok(dt, du) || !io_ok(dt, ddelta) ||
        !io_ok(dt, dB) || !io_ok(dt, dC) || !opt_io(dt, dz) || !f32_ok(A) || !f32_ok(dA) ||
        !opt_f32(Dskip) || !opt_f32(dD) || !opt_f32(delta_bias) || !opt_f32(ddelta_bias) ||
        (z != nullptr && dz == nullptr))
        return SSM_ERR_INVALID_ARG;
    if ((long long)B * D * L == 0) return SSM_OK;
    const BwdWs w = bwd_ws(0, dt, B, D, L, N, false);
    if (workspace == nullptr || ws_bytes < w.total || !aligned(workspace, 16))
        return SSM_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    char *ws = (char *)workspace;
    auto run = [&](auto tag) {
        using IO = decltype(tag);
        return seq_bwd<IO>(0, B, D, L, N, u, nullptr, delta, nullptr, A, nullptr, Bm, Cm,
                           nullptr, nullptr, Dskip, nullptr, z, delta_bias, nullptr,
                           delta_softplus, 1.f, dout, du, nullptr, ddelta, nullptr, dA, nullptr,
                           dB, dC, nullptr, nullptr, dD, nullptr, dz, ddelta_bias, nullptr, ws,
                           w, st);
    };
    return dt == SSM_F32 ? run(float()) : dt == SSM_F16 ? run(__half()) : run(__nv_bfloat16());
}

ssm_status bimamba_scan_bwd_v1(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                               const void *delta, const float *A, const float *A_b,
                               const void *Bm, const void *Cm, const float *Dskip,
                               const void *z, const float *delta_bias, int delta_softplus,
                               float out_scale, const void *dout, void *du, void *ddelta,
                               float *dA, float *dA_b, void *dB, void *dC, float *dD, void *dz,
                               float *ddelta_bias, void *workspace, size_t ws_bytes,
                               ssm_stream_t stream) {
    TRY(check_sizes(dt, B, D, L, N));
    if (!io_ok(dt, u) || !io_ok(dt, delta) || !io_ok(dt, Bm) || !io_ok(dt, Cm) ||
        !opt_io(dt, z) || !io_ok(dt, dout) || !io_ok(dt, du) || !io_ok(dt, ddelta) ||
        !io_ok(dt, dB) || !io_ok(dt, dC) || !opt_io(dt, dz) || !f32_ok(A) || !f32_ok(A_b) ||
        !f32_ok(dA) || !f32_ok(dA_b) || !opt_f32(Dskip) || !opt_f32(dD) ||
        !opt_f32(delta_bias) || !opt_f32(ddelta_bias) || (z != nullptr && dz == nullptr))
        return SSM_ERR_INVALID_ARG;
    if ((long long)B * D * L == 0) return SSM_OK;
    const BwdWs w = bwd_ws(1, dt, B, D, L, N, false);
    if (workspace == nullptr || ws_bytes < w.total || !aligned(workspace, 16))
        return SSM_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    char *ws = (char *)workspace;
    auto run = [&](auto tag) {
        using IO = decltype(tag);
        return seq_bwd<IO>(1, B, D, L, N, u, nullptr, delta, nullptr, A, A_b, Bm, Cm, nullptr,
                           nullptr, Dskip, nullptr, z, delta_bias, nullptr, delta_softplus,
                           out_scale, dout, du, nullptr, ddelta, nullptr, dA, dA_b, dB, dC,
                           nullptr, nullptr, dD, nullptr, dz, ddelta_bias, nullptr, ws, w, st);
    };
    return dt == SSM_F32 ? run(float()) : dt == SSM_F16 ? run(__half()) : run(__nv_bfloat16());
}

ssm_status bimamba_scan_bwd_v2(ssm_dtype dt, int B, int D, int L, int N, const void *u,
                               const void *u_b, const void *delta, const void *delta_b,
                               const float *A, const float *A_b, const void *Bm,
                               const void *Cm, const void *Bm_b, const void *Cm_b,
                               const float *Dskip, const float *D_b, const void *z,
                               const float *delta_bias, const float *delta_bias_b,
                               int delta_softplus, float out_scale, const void *dout, void *du,
                               void *du_b, void *ddelta, void *ddelta_b, float *dA,
                               float *dA_b, void *dB, void *dC, void *dB_b, void *dC_b,
                               float *dD, float *dD_b, void *dz, float *ddelta_bias,
                               float *ddelta_bias_b, void *workspace, size_t ws_bytes,
                               ssm_stream_t stream) {
    TRY(check_sizes(dt, B, D, L, N));
    if (!io_ok(dt, u) || !opt_io(dt, u_b) || !io_ok(dt, delta) || !io_ok(dt, delta_b) ||
        !io_ok(dt, Bm) || !io_ok(dt, Cm) || !io_ok(dt, Bm_b) || !io_ok(dt, Cm_b) ||
        !opt_io(dt, z) || !io_ok(dt, dout) || !io_ok(dt, du) || !io_ok(dt, ddelta) ||
        !io_ok(dt, ddelta_b) || !io_ok(dt, dB) || !io_ok(dt, dC) || !io_ok(dt, dB_b) ||
        !io_ok(dt, dC_b) || !opt_io(dt, dz) || !f32_ok(A) || !f32_ok(A_b) || !f32_ok(dA) ||
        !f32_ok(dA_b) || !opt_f32(Dskip) || !opt_f32(D_b) || !opt_f32(dD) || !opt_f32(dD_b) ||
        !opt_f32(delta_bias) || !opt_f32(delta_bias_b) || !opt_f32(ddelta_bias) ||
        !opt_f32(ddelta_bias_b) || (z != nullptr && dz == nullptr) ||
        (u_b != nullptr && !io_ok(dt, du_b)))
        return SSM_ERR_INVALID_ARG;
    if ((long long)B * D * L == 0) return SSM_OK;
    const BwdWs w = bwd_ws(2, dt, B, D, L, N, u_b != nullptr);
    if (workspace == nullptr || ws_bytes < w.total || !aligned(workspace, 16))
        return SSM_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    char *ws = (char *)workspace;
    auto run = [&](auto tag) {
        using IO = decltype(tag);
        return seq_bwd<IO>(2, B, D, L, N, u, u_b, delta, delta_b, A, A_b, Bm, Cm, Bm_b, Cm_b,
                           Dskip, D_b, z, delta_bias, delta_bias_b, delta_softplus, out_scale,
                           dout, du, du_b, ddelta, ddelta_b, dA, dA_b, dB, dC, dB_b, dC_b, dD,
                           dD_b, dz, ddelta_bias, ddelta_bias_b, ws, w, st);
    };
    return dt == SSM_F32 ? run(float()) : dt == SSM_F16 ? run(__half()) : run(__nv_bfloat16());
}

ssm_status ss2d_scan_bwd(ssm_dtype dt, int B, int D, int H, int W, int N, int K, const void *x,
                         const void *delta, const float *A, const void *Bm, const void *Cm,
                         const float *Dskip, const void *z, const float *delta_bias,
                         int delta_softplus, const void *dout, void *dx, void *ddelta,
                         float *dA, void *dB, void *dC, float *dD, void *dz,
                         float *ddelta_bias, void *workspace, size_t ws_bytes,
                         ssm_stream_t stream) {
    if (H < 0 || W < 0) return SSM_ERR_INVALID_ARG;
    if (K != 4) return SSM_ERR_UNSUPPORTED;
    if (!fits((long long)H * W)) return SSM_ERR_UNSUPPORTED;
    const int L = H * W;
    TRY(check_sizes(dt, B, D, L, N));
    if (!fits((long long)K * D * L) || !fits((long long)K * N * L)) return SSM_ERR_UNSUPPORTED;
    if (!io_ok(dt, x) || !io_ok(dt, delta) || !io_ok(dt, Bm) || !io_ok(dt, Cm) ||
        !opt_io(dt, z) || !io_ok(dt, dout) || !io_ok(dt, dx) || !io_ok(dt, ddelta) ||
        !io_ok(dt, dB) || !io_ok(dt, dC) || !opt_io(dt, dz) || !f32_ok(A) || !f32_ok(dA) ||
        !opt_f32(Dskip) || !opt_f32(dD) || !opt_f32(delta_bias) || !opt_f32(ddelta_bias) ||
        (z != nullptr && dz == nullptr))
        return SSM_ERR_INVALID_ARG;
    if ((long long)B * D * L == 0) return SSM_OK;
    const BwdWs w = bwd_ws(3, dt, B, D, L, N, false);
    if (workspace == nullptr || ws_bytes < w.total || !aligned(workspace, 16))
        return SSM_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    char *ws = (char *)workspace;
    auto run = [&](auto tag) {
        using IO = decltype(tag);
        return ss2d_bwd_run<IO>(B, D, H, W, N, x, delta, A, Bm, Cm, Dskip, z, delta_bias,
                                delta_softplus, dout, dx, ddelta, dA, dB, dC, dD, dz,
                                ddelta_bias, ws, w, st);
    };
    return dt == SSM_F32 ? run(float()) : dt == SSM_F16 ? run(__half()) : run(__nv_bfloat16());
}

}  // extern "C"
