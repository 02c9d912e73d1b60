// ssm_prologue_api.cu -- mamba_prologue_fwd (include/ssm_scan.h): one
// direction's conv1d + SiLU, x_proj split and dt_proj, producing the
// scan's inputs u, dt, B, C in the scan's own layouts.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

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

template <typename IO>
ssm_status run(int B, int D, int L, int N, int R, int K, const void *x, const float *conv_w,
               const float *conv_b, const float *W_x, const float *W_dt, int reverse, void *u,
               void *dt, void *Bm, void *Cm, float *dt_low, cudaStream_t st) {
    using namespace ssm::pro;
    conv_silu_kernel<IO><<<dim3((L + 255) / 256, D, B), 256, 0, st>>>(
        (const IO *)x, conv_w, conv_b, (IO *)u, D, L, K, reverse ? 1 : 0);
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
    proj_kernel<IO, IO><<<dim3((L + BN - 1) / BN, (M + BM - 1) / BM, B), 256, 0, st>>>(
        W_x, (const IO *)u, M, D, L, o1);
    if (last_error() != SSM_OK) return SSM_ERR_CUDA;
    // dt_proj: all D rows -> dt
    ProjOut o2{};
    o2.dst[0] = dt;
    o2.r[0] = 0;
    o2.r[1] = D;
    o2.r[2] = D;
    o2.r[3] = D;
    proj_kernel<float, IO><<<dim3((L + BN - 1) / BN, (D + BM - 1) / BM, B), 256, 0, st>>>(
        W_dt, dt_low, D, R, L, o2);
    return last_error();
}

}  // namespace

extern "C" {

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

}  // extern "C"
