// ssm_prologue_api.cu -- mamba_prologue_fwd and ss2d_prologue_fwd
// (include/ssm_scan.h): one direction's conv1d + SiLU, x_proj split and
// dt_proj, or SS2D's conv2d (+ SiLU) and its four directions' x_proj and
// dt_proj, producing the scan's inputs in the scan's own layouts.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "prologue_kernel.cuh"
#include "ssm_scan.h"

namespace {

bool aligned(const void *p, unsigned a) { return ((uintptr_t)p % a) == 0; }
unsigned esz(ssm_dtype dt) { return dt == SSM_F32 ? 4u : 2u; }
bool io_ok(ssm_dtype dt, const void *p) { return p != nullptr && aligned(p, esz(dt)); }
bool f32_ok(const float *p) { return p != nullptr && aligned(p, 4); }
bool opt_f32(const float *p) { return p == nullptr || aligned(p, 4); }

ssm_status last_error() {
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// Per-host-thread choice of the 1-D prologue's kernels
// (ssm_set_prologue_fused): 1 automatic, 0 always the three-kernel path, 2
// the fused kernel wherever it applies.
thread_local int t_fused = 1;
// Automatic choice: the fused kernel below this sequence length.  Measured on
// B300 (bf16, 50k positions per call): fused / three-kernel time 0.39-0.44
// at L = 197, 0.65-0.78 at 512, 0.91-1.13 at 1024, 1.10-1.42 from 2048 up
// (the three-kernel conv streams long rows with wide CTAs; short rows
// leave most of its threads idle).
constexpr int kFusedMaxL = 1024;
// shared memory a CTA may opt into on sm_100-class GPUs (227 KB)
constexpr size_t kSmemOptin = 227 * 1024;

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

// generic tiled projection: fp32 FMA for fp32 I/O, mma.sync for 16-bit I/O
// (weights fp32, or WT)
template <typename IN, typename IO, typename WT = float>
void launch_proj(dim3 grid, const WT *W, const IN *in, int M, int K, int L, long long ib,
                 ssm::pro::ProjOut o, cudaStream_t st) {
    if constexpr (sizeof(IO) == 4)
        ssm::pro::proj_kernel<IN, IO, WT><<<grid, 256, 0, st>>>(W, in, M, K, L, ib, o);
    else
        ssm::pro::proj_mma_kernel<IN, IO, WT><<<grid, 256, 0, st>>>(W, in, M, K, L, ib, o);
}

// x_proj: the weights-stationary tcgen05 kernel when its rows (<= 64) and W
// (in shared memory) fit, else the generic tiled one
template <typename IO>
ssm_status x_proj(int B, int M, int K, int L, const float *W, const IO *u, ssm::pro::ProjOut o,
                  cudaStream_t st) {
    using namespace ssm::pro;
    if constexpr (sizeof(IO) == 2) {
        const size_t smem = xproj_tc_smem_bytes(K);
        if (M <= 64 && smem <= kSmemOptin) {
            if (cudaFuncSetAttribute(xproj_tc_kernel<IO>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem) != cudaSuccess)
                return SSM_ERR_CUDA;
            const long long tiles = (long long)B * ((L + TCX_T - 1) / TCX_T);
            const int grid = (int)std::min<long long>(tiles, sm_count());
            xproj_tc_kernel<IO><<<grid, TCX_NT, smem, st>>>(W, u, M, K, L, B, o);
            return last_error();
        }
    }
    launch_proj<IO, IO>(dim3((L + BN - 1) / BN, (M + BM - 1) / BM, B), W, u, M, K, L,
                        (long long)K * L, o, st);
    return last_error();
}

// dt_proj: the register-blocked FMA kernel for dt_rank <= 32, else the
// generic tiled one
template <typename IO, int RP>
ssm_status launch_dtproj(int B, int D, int R, int L, const float *W, const float *dt_low, IO *dt,
                         long long ob, int nw, cudaStream_t st) {
    using namespace ssm::pro;
    if constexpr (sizeof(IO) == 2) {
        // tensor cores (tf32 operands, fp32 accumulation)
        constexpr size_t smem = dtproj_tc_smem_bytes<RP>();
        if (cudaFuncSetAttribute(dtproj_tc_kernel<IO, RP>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return SSM_ERR_CUDA;
        dtproj_tc_kernel<IO, RP><<<dim3((L + DTC_T - 1) / DTC_T, (D + DTC_RB - 1) / DTC_RB, B),
                                   256, smem, st>>>(W, dt_low, D, R, L, dt, ob, nw);
    } else {
        // fp32 I/O: fp32 FMA
        const int tiles = (L + DTP_T - 1) / DTP_T;
        const long long want = 4LL * sm_count();
        int split = (int)std::min<long long>(
            (want + (long long)tiles * B - 1) / ((long long)tiles * B), (D + DTP_MC - 1) / DTP_MC);
        split = std::max(split, 1);
        dtproj_kernel<IO, RP><<<dim3(tiles, split, B), 256, 0, st>>>(W, dt_low, D, R, L, dt, ob,
                                                                     nw);
    }
    return last_error();
}

// dt_proj of nw weight sets (scan directions): dt_low [B][nw][R][L] ->
// dt [B][nw][D][L] with W [nw][D][R]; the register-blocked kernels for
// dt_rank <= 32 (one launch, the (batch, set) pairs along grid z), else the
// generic tiled one per set
template <typename IO>
ssm_status dt_proj(int B, int nw, int D, int R, int L, const float *W, const float *dt_low,
                   IO *dt, cudaStream_t st) {
    using namespace ssm::pro;
    const long long ob = (long long)D * L;
    const int Bz = B * nw;
    if (R <= 8) return launch_dtproj<IO, 8>(Bz, D, R, L, W, dt_low, dt, ob, nw, st);
    if (R <= 16) return launch_dtproj<IO, 16>(Bz, D, R, L, W, dt_low, dt, ob, nw, st);
    if (R <= 24) return launch_dtproj<IO, 24>(Bz, D, R, L, W, dt_low, dt, ob, nw, st);
    if (R <= 32) return launch_dtproj<IO, 32>(Bz, D, R, L, W, dt_low, dt, ob, nw, st);
    for (int k = 0; k < nw; ++k) {
        ProjOut o{};
        o.dst[0] = dt + (long long)k * D * L;
        o.r[0] = 0;
        o.r[1] = D;
        o.r[2] = D;
        o.r[3] = D;
        o.bstride[0] = (long long)nw * D * L;
        o.order = -1;
        launch_proj<float, IO>(dim3((L + BN - 1) / BN, (D + BM - 1) / BM, B),
                               W + (long long)k * D * R, dt_low + (long long)k * R * L, D, R, L,
                               (long long)nw * R * L, o, st);
        if (last_error() != SSM_OK) return SSM_ERR_CUDA;
    }
    return SSM_OK;
}

// the fused one-kernel prologue (16-bit I/O, 4 taps, x_proj rows <= 64,
// dt_rank <= RP)
template <typename IO, int RP>
ssm_status launch_fused(int B, int D, int L, int N, int R, const void *x, const float *conv_w,
                        const float *conv_b, const float *W_x, const float *W_dt, int reverse,
                        void *u, void *dt, void *Bm, void *Cm, cudaStream_t st) {
    using namespace ssm::pro;
    constexpr size_t smem = fused_prologue_smem_bytes<RP>();
    if (cudaFuncSetAttribute(fused_prologue_kernel<IO, RP>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return SSM_ERR_CUDA;
    fused_prologue_kernel<IO, RP><<<dim3((L + FP_T - 1) / FP_T, B), FP_NT, smem, st>>>(
        (const IO *)x, conv_w, conv_b, W_x, W_dt, D, L, N, R, reverse ? 1 : 0, (IO *)u, (IO *)dt,
        (IO *)Bm, (IO *)Cm);
    return last_error();
}

template <typename IO>
ssm_status run(int B, int D, int L, int N, int R, int K, const void *x, const float *conv_w,
               const float *conv_b, const float *W_x, const float *W_dt, int reverse, void *u,
               void *dt, void *Bm, void *Cm, float *dt_low, cudaStream_t st) {
    using namespace ssm::pro;
    if constexpr (sizeof(IO) == 2) {
        if (K == 4 && R + 2 * N <= 64 && R <= 32 &&
            (t_fused == 2 || (t_fused == 1 && L < kFusedMaxL))) {
            if (R <= 8)
                return launch_fused<IO, 8>(B, D, L, N, R, x, conv_w, conv_b, W_x, W_dt, reverse,
                                           u, dt, Bm, Cm, st);
            if (R <= 16)
                return launch_fused<IO, 16>(B, D, L, N, R, x, conv_w, conv_b, W_x, W_dt, reverse,
                                            u, dt, Bm, Cm, st);
            if (R <= 24)
                return launch_fused<IO, 24>(B, D, L, N, R, x, conv_w, conv_b, W_x, W_dt, reverse,
                                            u, dt, Bm, Cm, st);
            return launch_fused<IO, 32>(B, D, L, N, R, x, conv_w, conv_b, W_x, W_dt, reverse, u,
                                        dt, Bm, Cm, st);
        }
    }
    const dim3 cgrid((L + CONV_T - 1) / CONV_T, D, B);
    bool done = false;
    if constexpr (sizeof(IO) == 2) {
        if (K == 4) {
            conv_silu_vec_kernel<IO><<<cgrid, 256, 0, st>>>((const IO *)x, conv_w, conv_b,
                                                            (IO *)u, D, L, reverse ? 1 : 0);
            done = true;
        }
    }
    if (done) {
    } else if (K == 4)
        conv_silu_kernel<IO, 4><<<cgrid, 256, 0, st>>>((const IO *)x, conv_w, conv_b, (IO *)u, D,
                                                       L, K, reverse ? 1 : 0);
    else
        conv_silu_kernel<IO, 0><<<cgrid, 256, 0, st>>>((const IO *)x, conv_w, conv_b, (IO *)u, D,
                                                       L, K, reverse ? 1 : 0);
    if (last_error() != SSM_OK) return SSM_ERR_CUDA;
    // x_proj: rows [0, R) -> dt_low (fp32), [R, R+N) -> B, [R+N, R+2N) -> C
    const int M = R + 2 * N;
    ProjOut o1{};
    o1.dst[0] = dt_low;
    o1.dst[1] = Bm;
    o1.dst[2] = Cm;
    o1.f32[0] = 1;
    o1.r[0] = 0;
    o1.r[1] = R;
    o1.r[2] = R + N;
    o1.r[3] = M;
    o1.bstride[0] = (long long)R * L;
    o1.bstride[1] = o1.bstride[2] = (long long)N * L;
    o1.order = -1;
    if (x_proj<IO>(B, M, D, L, W_x, (const IO *)u, o1, st) != SSM_OK) return SSM_ERR_CUDA;
    // dt_proj: all D rows -> dt
    return dt_proj<IO>(B, 1, D, R, L, W_dt, dt_low, (IO *)dt, st);
}

// rows of the map per conv2d CTA (about 2048 outputs) and its shared bytes
int c2_rows(int H, int W) { return std::max(1, std::min(H, 2048 / std::max(W, 1))); }
size_t c2_smem(int H, int W, int Kc) {
    const int P = (Kc - 1) / 2;
    return (size_t)(c2_rows(H, W) + 2 * P) * ssm::pro::conv2d_ws(W, Kc) * sizeof(float);
}

// SS2D: conv2d (+ SiLU), then for each of the four directions x_proj
// (outputs scattered to that direction's scan order) and dt_proj
template <typename IO>
ssm_status run_ss2d(int B, int D, int H, int W, int N, int R, int Kc, const void *x,
                    const float *conv_w, const float *conv_b, const float *W_x,
                    const float *W_dt, int act, void *u, void *delta, void *Bm, void *Cm,
                    float *dt_low, cudaStream_t st) {
    using namespace ssm::pro;
    const int L = H * W, RB = c2_rows(H, W);
    const size_t smem = c2_smem(H, W, Kc);
    const dim3 cgrid((H + RB - 1) / RB, D, B);
    if (Kc == 3) {
        if (cudaFuncSetAttribute(conv2d_act_kernel<IO, 3>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return SSM_ERR_CUDA;
        conv2d_act_kernel<IO, 3><<<cgrid, 256, smem, st>>>((const IO *)x, conv_w, conv_b, (IO *)u,
                                                          D, H, W, Kc, RB, act);
    } else {
        if (cudaFuncSetAttribute(conv2d_act_kernel<IO, 0>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return SSM_ERR_CUDA;
        conv2d_act_kernel<IO, 0><<<cgrid, 256, smem, st>>>((const IO *)x, conv_w, conv_b, (IO *)u,
                                                          D, H, W, Kc, RB, act);
    }
    if (last_error() != SSM_OK) return SSM_ERR_CUDA;
    // x_proj of the four directions: dt_low [B][4][R][L] (workspace), B, C
    // [B][4][N][L], each output at its position in that direction's order
    const int M = R + 2 * N;
    ProjOut4 outs{};
    for (int k = 0; k < 4; ++k) {
        ProjOut &o = outs.o[k];
        o.dst[0] = dt_low + (long long)k * R * L;
        o.dst[1] = (IO *)Bm + (long long)k * N * L;
        o.dst[2] = (IO *)Cm + (long long)k * N * L;
        o.f32[0] = 1;
        o.r[0] = 0;
        o.r[1] = R;
        o.r[2] = R + N;
        o.r[3] = M;
        o.bstride[0] = 4LL * R * L;
        o.bstride[1] = o.bstride[2] = 4LL * N * L;
        o.order = k;
        o.H = H;
        o.W = W;
    }
    bool done = false;
    if constexpr (sizeof(IO) == 2) {
        // one pass over u for all four directions
        const size_t xs = xproj4_smem_bytes(D, sizeof(IO));
        if (M <= 64 && D <= XP_K && xs <= 227 * 1024) {
            if (cudaFuncSetAttribute(xproj4_mma_kernel<IO>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)xs) != cudaSuccess)
                return SSM_ERR_CUDA;
            // tiles of 8 map rows x 16 columns
            const long long tiles = (long long)B * ((H + 7) / 8) * ((W + 15) / 16);
            const int grid = (int)std::min<long long>(tiles, sm_count());
            xproj4_mma_kernel<IO><<<grid, XP_NT, xs, st>>>(W_x, (const IO *)u, M, D, L, B, outs);
            if (last_error() != SSM_OK) return SSM_ERR_CUDA;
            done = true;
        }
    }
    if (!done)
        for (int k = 0; k < 4; ++k)
            if (x_proj<IO>(B, M, D, L, W_x + (long long)k * M * D, (const IO *)u, outs.o[k], st) !=
                SSM_OK)
                return SSM_ERR_CUDA;
    // dt_proj of the four directions in one launch
    return dt_proj<IO>(B, 4, D, R, L, W_dt, dt_low, (IO *)delta, st);
}


// out_proj: the tcgen05 kernel for 16-bit I/O and d_model <= 512 (NCH
// chunks of 128 rows), else the generic tiled projection
// The driver's tensor-map encoder, looked up once through the runtime (the
// library does not link the driver library itself).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return (PFN_cuTensorMapEncodeTiled_v12000)p;
    }();
    return fn;
}

// Tensor map of W [Dm][Di] (16-bit, 16-byte aligned, Di a multiple of 8)
// for boxes of 8 channels x 128 rows, no swizzle, zero fill out of range.
// A map describes memory by address and sizes only, so the last one made on
// this host thread is reused for the same W address, sizes and dtype.
struct WMapCache {
    const void *W = nullptr;
    int Dm = 0, Di = 0, f16 = 0;
    CUtensorMap map;
};
thread_local WMapCache t_wmap;
template <typename IO>
bool out_proj_w_map(CUtensorMap *m, const IO *W, int Dm, int Di) {
    const int f16 = std::is_same<IO, __half>::value ? 1 : 0;
    if (t_wmap.W == (const void *)W && t_wmap.Dm == Dm && t_wmap.Di == Di && t_wmap.f16 == f16) {
        *m = t_wmap.map;
        return true;
    }
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)Di, (cuuint64_t)Dm};
    const cuuint64_t strides[1] = {(cuuint64_t)Di * sizeof(IO)};
    const cuuint32_t box[2] = {8, 128}, estr[2] = {1, 1};
    const CUtensorMapDataType t = std::is_same<IO, __half>::value
                                      ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (enc(m, t, 2, (void *)W, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    t_wmap.W = W;
    t_wmap.Dm = Dm;
    t_wmap.Di = Di;
    t_wmap.f16 = f16;
    t_wmap.map = *m;
    return true;
}

template <typename IO, int NCH>
ssm_status launch_out_proj(int B, int Di, int Dm, int L, const void *y, const CUtensorMap &tmW,
                           void *out, cudaStream_t st) {
    using namespace ssm::pro;
    const int ns = out_proj_stages<NCH>(kSmemOptin);
    const size_t smem = out_proj_smem_bytes<NCH>(ns);
    if (cudaFuncSetAttribute(out_proj_tc_kernel<IO, NCH>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return SSM_ERR_CUDA;
    const long long tiles = (long long)B * ((L + OP_T - 1) / OP_T);
    const int grid = (int)std::min<long long>(tiles, sm_count());
    out_proj_tc_kernel<IO, NCH><<<grid, OP_THREADS, smem, st>>>(tmW, (const IO *)y, Dm, Di, L,
                                                                B, ns, (IO *)out);
    return last_error();
}
template <typename IO>
ssm_status out_proj_run(int B, int Di, int Dm, int L, const void *y, const void *Wv, void *out,
                        cudaStream_t st) {
    using namespace ssm::pro;
    const IO *W = (const IO *)Wv;
    if constexpr (sizeof(IO) == 2) {
        // W goes through a tensor map (base 16-byte aligned, row pitch Di * 2
        // bytes a multiple of 16) and y is copied as 16-byte chunks (16-byte
        // aligned); without a tensor-map encoder the tiled kernel runs
        CUtensorMap tmW;
        if (Di % 8 == 0 && aligned(W, 16) && aligned(y, 16) && Dm <= OP_MAXN &&
            out_proj_w_map<IO>(&tmW, W, Dm, Di)) {
            if (Dm <= 128) return launch_out_proj<IO, 1>(B, Di, Dm, L, y, tmW, out, st);
            if (Dm <= 256) return launch_out_proj<IO, 2>(B, Di, Dm, L, y, tmW, out, st);
            if (Dm <= 384) return launch_out_proj<IO, 3>(B, Di, Dm, L, y, tmW, out, st);
            return launch_out_proj<IO, 4>(B, Di, Dm, L, y, tmW, out, st);
        }
    }
    ProjOut o{};
    o.dst[0] = out;
    o.r[0] = 0;
    o.r[1] = o.r[2] = o.r[3] = Dm;
    o.bstride[0] = (long long)Dm * L;
    o.order = -1;
    launch_proj<IO, IO, IO>(dim3((L + BN - 1) / BN, (Dm + BM - 1) / BM, B), W, (const IO *)y, Dm,
                            Di, L, (long long)Di * L, o, st);
    return last_error();
}

}  // namespace

extern "C" {

void ssm_set_prologue_fused(int mode) { t_fused = (mode == 0 || mode == 2) ? mode : 1; }

size_t ssm_prologue_workspace_bytes(int B, int L, int R) {
    if (B < 0 || L < 0 || R <= 0) return (size_t)-1;
    return (size_t)B * R * L * sizeof(float);
}

ssm_status mamba_prologue_fwd(ssm_dtype dt, int B, int D, int L, int N, int R, int K,
                              const void *x, const float *conv_w, const float *conv_b,
                              const float *W_x, const float *W_dt, int reverse, void *u,
                              void *delta, void *Bm, void *Cm, void *workspace,
                              size_t ws_bytes, ssm_stream_t stream) {
    if (dt != SSM_F32 && dt != SSM_BF16 && dt != SSM_F16) return SSM_ERR_INVALID_ARG;
    if (B < 0 || D < 0 || L < 0 || N <= 0 || R <= 0 || K <= 0) return SSM_ERR_INVALID_ARG;
    if (N > 32 || K > 8 || B > 65535 || D > 65535) return SSM_ERR_UNSUPPORTED;
    if ((long long)D * L > 0x7fffffffLL || (long long)(R + 2 * N) * L > 0x7fffffffLL)
        return SSM_ERR_UNSUPPORTED;
    if (!io_ok(dt, x) || !f32_ok(conv_w) || !opt_f32(conv_b) || !f32_ok(W_x) || !f32_ok(W_dt) ||
        !io_ok(dt, u) || !io_ok(dt, delta) || !io_ok(dt, Bm) || !io_ok(dt, Cm))
        return SSM_ERR_INVALID_ARG;
    if ((long long)B * D * L == 0) return SSM_OK;
    if (workspace == nullptr || ws_bytes < ssm_prologue_workspace_bytes(B, L, R) ||
        !aligned(workspace, 16))
        return SSM_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    float *dt_low = (float *)workspace;
    if (dt == SSM_F32)
        return run<float>(B, D, L, N, R, K, x, conv_w, conv_b, W_x, W_dt, reverse, u, delta, Bm,
                          Cm, dt_low, st);
    if (dt == SSM_F16)
        return run<__half>(B, D, L, N, R, K, x, conv_w, conv_b, W_x, W_dt, reverse, u, delta, Bm,
                           Cm, dt_low, st);
    return run<__nv_bfloat16>(B, D, L, N, R, K, x, conv_w, conv_b, W_x, W_dt, reverse, u, delta,
                              Bm, Cm, dt_low, st);
}

size_t ss2d_prologue_workspace_bytes(int B, int H, int W, int R) {
    if (B < 0 || H < 0 || W < 0 || R <= 0) return (size_t)-1;
    return (size_t)B * 4 * R * H * W * sizeof(float);
}

ssm_status ss2d_prologue_fwd(ssm_dtype dt, int B, int D, int H, int W, int N, int R, int Kc,
                             const void *x, const float *conv_w, const float *conv_b,
                             const float *W_x, const float *W_dt, int silu_act, void *u,
                             void *delta, void *Bm, void *Cm, void *workspace, size_t ws_bytes,
                             ssm_stream_t stream) {
    if (dt != SSM_F32 && dt != SSM_BF16 && dt != SSM_F16) return SSM_ERR_INVALID_ARG;
    if (B < 0 || D < 0 || H < 0 || W < 0 || N <= 0 || R <= 0 || Kc <= 0 || Kc % 2 == 0)
        return SSM_ERR_INVALID_ARG;
    if (N > 32 || Kc > 7 || B > 16383 || D > 65535) return SSM_ERR_UNSUPPORTED;
    const long long L = (long long)H * W;
    if ((long long)D * L > 0x7fffffffLL || (long long)(R + 2 * N) * L > 0x7fffffffLL ||
        4LL * D * L > 0x7fffffffLL || c2_smem(H, W, Kc) > 200 * 1024)
        return SSM_ERR_UNSUPPORTED;
    if (!io_ok(dt, x) || !f32_ok(conv_w) || !opt_f32(conv_b) || !f32_ok(W_x) || !f32_ok(W_dt) ||
        !io_ok(dt, u) || !io_ok(dt, delta) || !io_ok(dt, Bm) || !io_ok(dt, Cm))
        return SSM_ERR_INVALID_ARG;
    if ((long long)B * D * L == 0) return SSM_OK;
    if (workspace == nullptr || ws_bytes < ss2d_prologue_workspace_bytes(B, H, W, R) ||
        !aligned(workspace, 16))
        return SSM_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    float *dt_low = (float *)workspace;
    const int act = silu_act ? 1 : 0;
    if (dt == SSM_F32)
        return run_ss2d<float>(B, D, H, W, N, R, Kc, x, conv_w, conv_b, W_x, W_dt, act, u, delta,
                               Bm, Cm, dt_low, st);
    if (dt == SSM_F16)
        return run_ss2d<__half>(B, D, H, W, N, R, Kc, x, conv_w, conv_b, W_x, W_dt, act, u, delta,
                                Bm, Cm, dt_low, st);
    return run_ss2d<__nv_bfloat16>(B, D, H, W, N, R, Kc, x, conv_w, conv_b, W_x, W_dt, act, u,
                                   delta, Bm, Cm, dt_low, st);
}

ssm_status out_proj_fwd(ssm_dtype dt, int B, int Di, int Dm, int L, const void *y,
                        const void *W_out, void *out, ssm_stream_t stream) {
    if (dt != SSM_F32 && dt != SSM_BF16 && dt != SSM_F16) return SSM_ERR_INVALID_ARG;
    if (B < 0 || Di <= 0 || Dm <= 0 || L < 0) return SSM_ERR_INVALID_ARG;
    if (B > 65535 || (long long)Di * L > 0x7fffffffLL || (long long)Dm * L > 0x7fffffffLL ||
        (long long)Dm * Di > 0x7fffffffLL)
        return SSM_ERR_UNSUPPORTED;
    if (!io_ok(dt, y) || !io_ok(dt, W_out) || !io_ok(dt, out)) return SSM_ERR_INVALID_ARG;
    if ((long long)B * L == 0) return SSM_OK;
    cudaStream_t st = (cudaStream_t)stream;
    if (dt == SSM_F32) return out_proj_run<float>(B, Di, Dm, L, y, W_out, out, st);
    if (dt == SSM_F16) return out_proj_run<__half>(B, Di, Dm, L, y, W_out, out, st);
    return out_proj_run<__nv_bfloat16>(B, Di, Dm, L, y, W_out, out, st);
}

}  // extern "C"
