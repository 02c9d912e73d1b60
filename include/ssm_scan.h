/*
 * ssm_scan.h -- C ABI of the B300 (sm_103a) selective-scan library.
 *
 * The library computes the Mamba selective scan (S6) forward pass in three
 * forms: one direction, Vision Mamba's bidirectional v1/v2 with flip-add
 * fusion, and VMamba's SS2D four-way cross-scan with cross-merge.  Every step
 * runs in the library's own CUDA kernels; there is no host fallback.
 *
 * Per (batch b, channel d, state n) and time t, with h_{-1} = 0:
 *   delta_t = softplus(dt_t + delta_bias[d])   (dt_t + delta_bias[d] if
 *                                               delta_softplus == 0)
 *   h_t[n]  = exp(delta_t * A[d,n]) * h_{t-1}[n] + delta_t * B[n,t] * u_t
 *   y_t     = sum_n C[n,t] * h_t[n] + Dskip[d] * u_t
 * and the output is gated, y_t * silu(z_t), when z is given.
 * Sources: the S6 equations in "状态空间模型如何重塑视觉序列处理" (Vision Mamba
 * overview), section "选择性扫描机制的计算效率优势" (discretisation read as
 * exp(delta*A) for A and delta*B for B); delta = softplus(dt_proj(x)) and
 * A = -exp(A_log) in "VMamba的SS2D模块详解", sections 3.1 and 3.2; the
 * tensor shapes in "Vision Mamba实战", section 1.
 *
 * Common conventions
 *  - All tensor pointers are DEVICE pointers to contiguous, caller-owned
 *    memory.  I/O tensors (u, delta, B, C, z, y and the per-branch copies)
 *    use the dtype `dt` (fp32, bf16 or fp16); A, Dskip and delta_bias are
 *    fp32.
 *  - Every pointer must be aligned to its element type (2 bytes for bf16
 *    and fp16, 4 for fp32); I/O tensors may start anywhere else, e.g. at an offset
 *    into a larger buffer.  Only the workspace needs 16 bytes.
 *  - Optional pointers may be NULL: Dskip -> 0, z -> no gate,
 *    delta_bias -> 0 (and u_b -> u for v2).
 *  - `y` must not alias any input.  State and arithmetic are fp32; bf16
 *    and fp16 outputs are rounded to nearest even.
 *  - `workspace` is device memory of at least ssm_workspace_bytes(...)
 *    bytes for the same arguments, 16-byte aligned (NULL is fine when that
 *    is 0).  It holds a status word, the B and C tensors repacked per
 *    position for the kernels, and (bidirectional forms) the fp32 outputs
 *    of the branch that reaches a position first.  Its contents need no
 *    initialisation and are garbage afterwards, except the status word read
 *    by ssm_get_status.  Two calls in flight at once must not share a
 *    workspace.
 *  - Calls are asynchronous on `stream` (0 = the legacy default stream).
 *    The library allocates nothing.  Its only state outside the caller's
 *    buffers is the fixed scratch array that bimamba_scan_fwd_v2_noalloc
 *    uses and six per-host-thread settings, each changed only by its own
 *    setter and applying to later calls made on that host thread: the
 *    profiling events (ssm_set_profile_events), the CTA-shape override
 *    (ssm_set_cta_channels), the prologue's kernel choice
 *    (ssm_set_prologue_fused), the saved backward context
 *    (ssm_set_bwd_context) and the one-launch test hooks
 *    (ssm_test_withhold_copy, ssm_test_shrink_extents).  (The backward
 *    calls also set, and clear before returning, a per-thread request that
 *    the forward run inside them store its chunk-start states; and
 *    out_proj_fwd keeps, per host thread, the TMA tensor map it last made,
 *    reused for the same W_out address, sizes and dtype.)
 *  - Errors: SSM_ERR_INVALID_ARG for a bad size, NULL required pointer or
 *    misaligned pointer; SSM_ERR_UNSUPPORTED for N > 32, K != 4 or sizes
 *    beyond the 32-bit index range; SSM_ERR_WORKSPACE when ws_bytes is too
 *    small; SSM_ERR_CUDA when a launch fails (cudaGetLastError is consumed);
 *    SSM_ERR_SCRATCH_LIMIT when a problem is too large for the fixed scratch
 *    of bimamba_scan_fwd_v2_noalloc;
 *    SSM_ERR_TIMEOUT (through ssm_get_status, after the call's kernels ran)
 *    when a kernel's bounded wait for its own bulk copies ran out; its
 *    output is then incomplete.  SSM_ERR_BOUNDS (through ssm_get_status)
 *    only from a build with SSM_DEBUG_BOUNDS defined (libssm_scan_debug.so):
 *    a forward kernel caught an element offset outside the tensor it
 *    addresses and skipped that access; the product build never checks.
 *    Every check happens before any launch: an error means nothing ran.
 *  - A call with B == 0, D == 0 or L == 0 is valid and launches nothing.
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

typedef struct CUstream_st *ssm_stream_t; /* same type as cudaStream_t */

typedef enum { SSM_F32 = 0, SSM_BF16 = 1, SSM_F16 = 2 } ssm_dtype;

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1,
    SSM_ERR_UNSUPPORTED = 2,
    SSM_ERR_CUDA = 3,
    SSM_ERR_WORKSPACE = 4,
    SSM_ERR_SCRATCH_LIMIT = 5,
    SSM_ERR_TIMEOUT = 6,
    SSM_ERR_BOUNDS = 7
} ssm_status;

typedef enum {
    SSM_OP_SELECTIVE_SCAN = 0,
    SSM_OP_BIMAMBA_V1 = 1,
    SSM_OP_BIMAMBA_V2 = 2,
    SSM_OP_SS2D = 3
} ssm_op;

/*
 * One direction.
 *   u, delta, z, y : [B, D, L]      A : [D, N]      Bm, Cm : [B, N, L]
 *   Dskip, delta_bias : [D]
 */
SSM_API ssm_status selective_scan_fwd(ssm_dtype dt, int B, int D, int L, int N,
                              const void *u, const void *delta, const float *A,
                              const void *Bm, const void *Cm,
                              const float *Dskip, const void *z,
                              const float *delta_bias, int delta_softplus,
                              void *y, void *workspace, size_t ws_bytes,
                              ssm_stream_t stream);

/*
 * BiMamba v1 ("从Transformer到Mamba" section 2.1; "Vision Mamba实战"
 * sections 1 and 2.2): delta, B, C, Dskip and delta_bias are shared by the
 * two branches; only A (forward) and A_b (backward) differ.  The backward
 * branch scans the sequence reversed in time, and its output is flipped
 * back before the fusion
 *   y_t = out_scale * (y_fwd[t] + y_bwd[t]),   then the gate.
 * (out_scale = 1 is the plain flip-add of the pages; 0.5 averages.)
 * Every tensor is in ORIGINAL token order; the kernel reads the backward
 * branch reversed.  Shapes as selective_scan_fwd, A_b : [D, N].
 */
SSM_API ssm_status bimamba_scan_fwd_v1(ssm_dtype dt, int B, int D, int L, int N,
                               const void *u, const void *delta,
                               const float *A, const float *A_b,
                               const void *Bm, const void *Cm,
                               const float *Dskip, const void *z,
                               const float *delta_bias, int delta_softplus,
                               float out_scale, void *y, void *workspace,
                               size_t ws_bytes, ssm_stream_t stream);

/*
 * BiMamba v2 ("从Transformer到Mamba" sections 2.1, 2.2 and 4.3): the
 * backward branch has its own delta_b, A_b, Bm_b, Cm_b, D_b and
 * delta_bias_b (and u_b when its input differs; NULL means it scans u).
 * Fusion as v1; the pages' v2 averages, i.e. out_scale = 0.5.  All tensors
 * in ORIGINAL token order.  Shapes as v1; delta_b, u_b : [B, D, L];
 * Bm_b, Cm_b : [B, N, L]; D_b, delta_bias_b : [D].
 */
SSM_API ssm_status bimamba_scan_fwd_v2(ssm_dtype dt, int B, int D, int L, int N,
                               const void *u, const void *u_b,
                               const void *delta, const void *delta_b,
                               const float *A, const float *A_b,
                               const void *Bm, const void *Cm,
                               const void *Bm_b, const void *Cm_b,
                               const float *Dskip, const float *D_b,
                               const void *z, const float *delta_bias,
                               const float *delta_bias_b, int delta_softplus,
                               float out_scale, void *y, void *workspace,
                               size_t ws_bytes, ssm_stream_t stream);

/*
 * VMamba SS2D ("VMamba的SS2D模块详解" sections 2.1, 2.2 and 3.1), K = 4.
 * Direction k scans the H x W map in order
 *   k=0 row-major, k=1 column-major, k=2 row-major reversed,
 *   k=3 column-major reversed,
 * with its own delta_k, A_k, B_k, C_k, D_k and delta_bias_k.  The four
 * outputs are mapped back to H x W and summed (cross-merge), then gated.
 *   x, z, y : [B, D, H, W] (spatial)
 *   delta : [B, K, D, L] and Bm, Cm : [B, K, N, L] in each direction's SCAN
 *           order (L = H*W), as per-direction projections emit them
 *   A : [K, D, N];  Dskip, delta_bias : [K, D]
 * Cross-scan and cross-merge are folded into the kernels' addressing.
 */
SSM_API ssm_status ss2d_scan_fwd(ssm_dtype dt, int B, int D, int H, int W, int N,
                         int K, const void *x, const void *delta,
                         const float *A, const void *Bm, const void *Cm,
                         const float *Dskip, const void *z,
                         const float *delta_bias, int delta_softplus, void *y,
                         void *workspace, size_t ws_bytes,
                         ssm_stream_t stream);

/*
 * The same four operations, also returning the final state of every
 * direction: last_state (fp32, device, required) receives h after the
 * direction's last step -- position L-1 for a forward walk, position 0 for
 * the backward branch of v1/v2, the last position of each SS2D direction's
 * scan order -- laid out [directions][B][D][N] (1, 2 or 4 directions).
 * It is the state a caller would carry into the next segment of a longer
 * sequence (chunked inference; the pages' recurrence, "状态空间模型如何重塑
 * 视觉序列处理", section "选择性扫描机制的计算效率优势", run to its end).
 * Everything else as for the calls above.
 */
SSM_API ssm_status selective_scan_fwd_ls(ssm_dtype dt, int B, int D, int L, int N,
                         const void *u, const void *delta, const float *A,
                         const void *Bm, const void *Cm, const float *Dskip,
                         const void *z, const float *delta_bias,
                         int delta_softplus, void *y, float *last_state,
                         void *workspace, size_t ws_bytes, ssm_stream_t stream);
SSM_API ssm_status bimamba_scan_fwd_v1_ls(ssm_dtype dt, int B, int D, int L, int N,
                         const void *u, const void *delta, const float *A,
                         const float *A_b, const void *Bm, const void *Cm,
                         const float *Dskip, const void *z,
                         const float *delta_bias, int delta_softplus,
                         float out_scale, void *y, float *last_state,
                         void *workspace, size_t ws_bytes, ssm_stream_t stream);
SSM_API ssm_status bimamba_scan_fwd_v2_ls(ssm_dtype dt, int B, int D, int L, int N,
                         const void *u, const void *u_b, const void *delta,
                         const void *delta_b, const float *A, const float *A_b,
                         const void *Bm, const void *Cm, const void *Bm_b,
                         const void *Cm_b, const float *Dskip, const float *D_b,
                         const void *z, const float *delta_bias,
                         const float *delta_bias_b, int delta_softplus,
                         float out_scale, void *y, float *last_state,
                         void *workspace, size_t ws_bytes, ssm_stream_t stream);
SSM_API ssm_status ss2d_scan_fwd_ls(ssm_dtype dt, int B, int D, int H, int W, int N,
                         int K, const void *x, const void *delta,
                         const float *A, const void *Bm, const void *Cm,
                         const float *Dskip, const void *z,
                         const float *delta_bias, int delta_softplus, void *y,
                         float *last_state, void *workspace, size_t ws_bytes,
                         ssm_stream_t stream);

/*
 * v2 with the backward set in its own scan order: delta_b, Bm_b, Cm_b (and
 * u_b when given) are time-reversed -- element t of a row is position L-1-t
 * -- as produced when the backward branch's projections run on the flipped
 * sequence ("Vision Mamba实战", section 2.2, flips the input before the
 * backward scan).  u (shared, u_b == NULL), z and y stay in original order;
 * the result equals bimamba_scan_fwd_v2 on the un-reversed tensors, without
 * materialising the flips.  last_state may be NULL (else as *_fwd_ls).
 */
SSM_API ssm_status bimamba_scan_fwd_v2_so(ssm_dtype dt, int B, int D, int L, int N,
                         const void *u, const void *u_b, const void *delta,
                         const void *delta_b, const float *A, const float *A_b,
                         const void *Bm, const void *Cm, const void *Bm_b,
                         const void *Cm_b, const float *Dskip, const float *D_b,
                         const void *z, const float *delta_bias,
                         const float *delta_bias_b, int delta_softplus,
                         float out_scale, void *y, float *last_state,
                         void *workspace, size_t ws_bytes, ssm_stream_t stream);

/*
 * Status of the last call that used `workspace`, once the work queued on
 * `stream` before this call has finished (the call synchronises `stream`):
 * *out = SSM_OK, or SSM_ERR_TIMEOUT when a kernel gave up a bounded wait.
 * For selective_scan_fwd and bimamba_scan_fwd_v1/_v2 only.  Returns
 * SSM_ERR_CUDA if the copy of the status word fails.
 */
SSM_API ssm_status ssm_get_status(const void *workspace, ssm_stream_t stream,
                                  ssm_status *out);

/*
 * Workspace bytes the call with these sizes needs (0 when none).
 * `L_or_HW` is L, or H*W for SS2D; K is ignored except for SS2D.
 * Returns (size_t)-1 for invalid sizes.
 */
SSM_API size_t ssm_workspace_bytes(ssm_op op, ssm_dtype dt, int B, int D,
                           int L_or_HW, int N, int K);

/*
 * Allocation-free variant of bimamba_scan_fwd_v2.  The pages have no
 * counterpart for this entry point: it exists for callers that cannot
 * allocate device memory themselves, for example a plugin inside a host
 * framework that owns the device allocator and hands its plugins only their
 * input and output buffers, or real-time code that must not call cudaMalloc
 * (which can synchronise the device) once it is running.
 *
 * Arguments, layouts, results and errors are those of bimamba_scan_fwd_v2,
 * without `workspace` / `ws_bytes`.  Instead of a caller workspace, the call
 * uses a scratch array of SSM_STATIC_SCRATCH_BYTES bytes that the library
 * declares as a file-scope static __device__ array, so every GPU that loads
 * the library holds those bytes until the process exits.
 *  - Argument errors (SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED) are checked
 *    first; then problems whose workspace (ssm_workspace_bytes(
 *    SSM_OP_BIMAMBA_V2, ...)) exceeds SSM_STATIC_SCRATCH_BYTES return
 *    SSM_ERR_SCRATCH_LIMIT before anything runs.
 *  - The status word that ssm_get_status reads for the other calls lives in
 *    the scratch array here, which the caller cannot address: a bounded wait
 *    that runs out inside this call (SSM_ERR_TIMEOUT for the other calls)
 *    is not observable through this entry point.  The call still returns,
 *    the device stays usable and the next call runs normally, but the
 *    output of the timed-out call is incomplete.
 *  - The first call on a device (the one current on the calling thread,
 *    which must be the device `stream` belongs to) looks up the array's
 *    device address, once; make that first call before any stream capture.
 *  - The call allocates nothing, on the host or the device.
 *  - Every call on a device shares the one array, and the array keeps the
 *    previous call's contents.  The kernel writes each scratch slot before
 *    it reads it, so nothing needs clearing between calls; but calls whose
 *    executions overlap on the GPU (different streams, or different host
 *    threads) race on the array and give wrong results.  Serialise them.
 */
#define SSM_STATIC_SCRATCH_BYTES ((size_t)64 << 20)

SSM_API ssm_status bimamba_scan_fwd_v2_noalloc(
    ssm_dtype dt, int B, int D, int L, int N, const void *u, const void *u_b,
    const void *delta, const void *delta_b, const float *A, const float *A_b,
    const void *Bm, const void *Cm, const void *Bm_b, const void *Cm_b,
    const float *Dskip, const float *D_b, const void *z,
    const float *delta_bias, const float *delta_bias_b, int delta_softplus,
    float out_scale, void *y, ssm_stream_t stream);

/* Static description of a status code (never NULL). */
SSM_API const char *ssm_status_string(ssm_status s);

/*
 * Profiling hook.  `begin` and `end` are cudaEvent_t handles (or both NULL
 * to switch the hook off).  While set, every call made on this host thread
 * records `begin` immediately before and `end` immediately after its scan
 * kernel on the call's stream -- for ss2d_scan_fwd the row-pair scan, the
 * last of its two -- so that cudaEventElapsedTime gives that kernel's
 * duration.  The events stay owned by the caller.
 */
SSM_API void ssm_set_profile_events(void *begin, void *end);

/* ---------------------------------------------------------------------------
 * Backward pass.  Gradients of the loss sum(dout * out) for the output `out`
 * of the matching forward call with the same arguments: the adjoint of the
 * recurrence above (G_t = gy_t C_t + exp(delta_{t+1} A) G_{t+1}, then dC, dB,
 * du, dA, ddelta from G and the states), of the softplus, the gate, the
 * flip-add and the cross-merge.  The pages discuss training through the
 * scan and checking its gradients ("Vision Mamba实战", section 4;
 * "从Transformer到Mamba", section 4.2) but print no backward formula; this
 * is the exact derivative of the forward definition.
 *
 * Gradient outputs are device buffers with their input's shape: du, ddelta,
 * dB, dC, dz (and the _b and dx variants) in the I/O dtype; dA, dD and
 * ddelta_bias fp32.  Every output is overwritten.  dz is required when z is
 * given (ignored otherwise); dD is written only when Dskip is given;
 * ddelta_bias (and the _b variants) may be NULL.  Parameter gradients sum
 * over every batch element and position (and, for v1, both branches);
 * partial sums are reduced in a fixed order, so results are deterministic.
 * `workspace`: at least ssm_bwd_workspace_bytes(...) bytes, 16-byte
 * aligned, contents irrelevant.  State and arithmetic are fp32.  Errors as
 * for the forward calls; SSM_ERR_WORKSPACE when it is too small.
 * ------------------------------------------------------------------------- */
SSM_API ssm_status selective_scan_bwd(ssm_dtype dt, int B, int D, int L, int N,
                         const void *u, const void *delta, const float *A,
                         const void *Bm, const void *Cm, const float *Dskip,
                         const void *z, const float *delta_bias,
                         int delta_softplus, const void *dout, void *du,
                         void *ddelta, float *dA, void *dB, void *dC, float *dD,
                         void *dz, float *ddelta_bias, void *workspace,
                         size_t ws_bytes, ssm_stream_t stream);

/* v1: delta, B, C, Dskip and delta_bias are shared by both branches, so their
 * gradients sum both; dA and dA_b belong to A and A_b. */
SSM_API ssm_status bimamba_scan_bwd_v1(ssm_dtype dt, int B, int D, int L, int N,
                         const void *u, const void *delta, const float *A,
                         const float *A_b, const void *Bm, const void *Cm,
                         const float *Dskip, const void *z,
                         const float *delta_bias, int delta_softplus,
                         float out_scale, const void *dout, void *du,
                         void *ddelta, float *dA, float *dA_b, void *dB, void *dC,
                         float *dD, void *dz, float *ddelta_bias,
                         void *workspace, size_t ws_bytes, ssm_stream_t stream);

/* v2: one gradient per tensor of each set.  u_b == NULL (shared u): du sums
 * both branches and du_b is ignored; otherwise du_b is required. */
SSM_API ssm_status bimamba_scan_bwd_v2(ssm_dtype dt, int B, int D, int L, int N,
                         const void *u, const void *u_b, const void *delta,
                         const void *delta_b, const float *A, const float *A_b,
                         const void *Bm, const void *Cm, const void *Bm_b,
                         const void *Cm_b, const float *Dskip, const float *D_b,
                         const void *z, const float *delta_bias,
                         const float *delta_bias_b, int delta_softplus,
                         float out_scale, const void *dout, void *du, void *du_b,
                         void *ddelta, void *ddelta_b, float *dA, float *dA_b,
                         void *dB, void *dC, void *dB_b, void *dC_b, float *dD,
                         float *dD_b, void *dz, float *ddelta_bias,
                         float *ddelta_bias_b, void *workspace, size_t ws_bytes,
                         ssm_stream_t stream);

/* SS2D, K = 4: dx [B,D,H,W]; ddelta [B,4,D,L], dB/dC [B,4,N,L] in each
 * direction's scan order; dA [4,D,N]; dD and ddelta_bias [4,D]. */
SSM_API ssm_status ss2d_scan_bwd(ssm_dtype dt, int B, int D, int H, int W, int N,
                         int K, const void *x, const void *delta, const float *A,
                         const void *Bm, const void *Cm, const float *Dskip,
                         const void *z, const float *delta_bias,
                         int delta_softplus, const void *dout, void *dx,
                         void *ddelta, float *dA, void *dB, void *dC, float *dD,
                         void *dz, float *ddelta_bias, void *workspace,
                         size_t ws_bytes, ssm_stream_t stream);

/* Workspace bytes of the backward call with these sizes (0 when B*D*L is 0;
 * (size_t)-1 for invalid sizes).  separate_u_b: v2 called with u_b != NULL. */
SSM_API size_t ssm_bwd_workspace_bytes(ssm_op op, ssm_dtype dt, int B, int D,
                                       int L_or_HW, int N, int K,
                                       int separate_u_b);

/* ---------------------------------------------------------------------------
 * Saved backward context.  Each backward call above first runs the forward
 * pass again: the gate's derivative needs the pre-gate output y, and with
 * d_state <= 16 the backward kernel starts from the states the forward
 * pass had before every eighth step.  That is the recompute side of the
 * memory / compute trade-off ("Vision Mamba实战" section 4 recomputes
 * activations under gradient checkpointing to save memory).  A training
 * loop that can spend the memory keeps both from its own forward call:
 *
 *   ssm_set_bwd_context(ctx, ctx_bytes)   on the host thread making the calls
 *   forward call                          also stores y before the gate and
 *                                         the chunk-start states in ctx
 *   ... (other calls, each layer with its own context)
 *   ssm_set_bwd_context(ctx, ctx_bytes)   the same buffer again
 *   backward call, same inputs            reads ctx instead of running the
 *                                         forward pass
 *   ssm_set_bwd_context(NULL, 0)
 *
 * It applies to selective_scan_fwd / _bwd, bimamba_scan_fwd_v1 / _bwd_v1
 * and bimamba_scan_fwd_v2 (and its _ls, _so and _noalloc variants) /
 * _bwd_v2 with d_state <= 16; SS2D calls and d_state > 16 ignore it.  The
 * caller guarantees that the backward call has the same operation, sizes,
 * dtype, inputs and gate (z given or not) as the forward call that filled
 * ctx; the library cannot check this.  `ctx`: device memory of at least
 * ssm_bwd_context_bytes(...) bytes, 16-byte aligned, owned by the caller;
 * a forward or backward call that finds it smaller or misaligned returns
 * SSM_ERR_WORKSPACE.  The setting is per host thread (the sixth per-thread
 * setting) and stays until changed.  Results are bit-identical to the
 * backward call without a context. */
SSM_API void ssm_set_bwd_context(void *ctx, size_t ctx_bytes);

/* Bytes of a saved backward context for these sizes: the pre-gate output
 * (B * D * L elements of dt) and, per direction, fp32 states [B][D][ceil(L
 * / 8)][16]; 0 when d_state > 16 or B*D*L is 0 (the context is then
 * ignored); (size_t)-1 for SS2D or invalid sizes. */
SSM_API size_t ssm_bwd_context_bytes(ssm_op op, ssm_dtype dt, int B, int D, int L, int N);

/* ---------------------------------------------------------------------------
 * Prologue: the steps that turn a block's input x into the scan's inputs,
 * for one direction ("Vision Mamba实战" section 2.1, "从Transformer到Mamba"
 * section 2.1: conv1d, x_proj, dt_proj; "VMamba的SS2D模块详解" section 3.1:
 * dt, B, C = split(x_proj(.), [dt_rank, d_state, d_state])):
 *   u[t]  = silu(conv_b[d] + sum_k conv_w[d][k] * xs[t - (K-1) + k])
 *           (depthwise, causal: xs before the start is 0)
 *   [dt_low; B; C] = W_x u        (W_x [R + 2N, D] fp32, rows in that order)
 *   delta = W_dt dt_low           (W_dt [D, R] fp32; dt_proj's bias is the
 *                                  scan's delta_bias, applied there with the
 *                                  softplus)
 * xs = x [B, D, L], or x reversed in time when reverse != 0 -- v2's backward
 * branch runs its own weights on the flipped sequence, and its outputs then
 * come out in that branch's scan order, ready for bimamba_scan_fwd_v2_so.
 * Outputs (I/O dtype, device, caller-owned): u, delta [B, D, L]; Bm, Cm
 * [B, N, L] -- the layouts the scan calls take.  N <= 32, 1 <= K <= 8.
 * workspace: ssm_prologue_workspace_bytes(B, L, R) bytes, 16-byte aligned
 * (the fp32 dt_low of the three-kernel path; the fused path below does not
 * touch it, but the size is required either way).  Kernels: with 16-bit
 * I/O, K = 4, R + 2N <= 64, R <= 32 and L < 1024 one fused kernel per call
 * (conv, x_proj and dt_proj per tile of 64 positions: u written once and
 * not read back, dt_low kept on chip; ssm_set_prologue_fused overrides the
 * choice), otherwise three launches (conv1d + SiLU, x_proj, dt_proj).
 * Arithmetic:
 * fp32 accumulation throughout; with 16-bit I/O x_proj runs on tensor
 * cores with u and W_x in the I/O type and dt_proj on tf32 operands; with
 * fp32 I/O both are fp32 FMA.  Outputs are
 * rounded to the I/O dtype.  Errors: SSM_ERR_INVALID_ARG for a bad dtype,
 * size or pointer; SSM_ERR_UNSUPPORTED for N > 32, K > 8 or sizes past the
 * 32-bit index range; SSM_ERR_WORKSPACE for a short or misaligned
 * workspace; SSM_ERR_CUDA for a launch error.  Asynchronous on `stream`.
 * ------------------------------------------------------------------------- */
SSM_API ssm_status mamba_prologue_fwd(ssm_dtype dt, int B, int D, int L, int N,
                         int R, int K, const void *x, const float *conv_w,
                         const float *conv_b, const float *W_x,
                         const float *W_dt, int reverse, void *u, void *delta,
                         void *Bm, void *Cm, void *workspace, size_t ws_bytes,
                         ssm_stream_t stream);
SSM_API size_t ssm_prologue_workspace_bytes(int B, int L, int R);

/* ---------------------------------------------------------------------------
 * SS2D prologue ("VMamba的SS2D模块详解" section 2.1: conv2d on the [B, D, H, W]
 * map before the core; section 2.2: the four scan orders; section 3.1: one
 * x_proj and one dt_proj per scan direction):
 *   u = act(conv_b[d] + sum_{i,j} conv_w[d][i][j] x[h+i-P][w+j-P])
 *       depthwise, P = (Kc-1)/2, zero outside the map, act = SiLU when
 *       silu_act != 0, else identity (the pages' simplified SS2D forward
 *       shows no activation after conv2d; the 1D path applies SiLU)
 *   for k = 0..3 (row-major, column-major, and their reversals):
 *     [dt_low; B_k; C_k] = W_x[k] xs_k,  delta_k = W_dt[k] dt_low
 *   where xs_k is u read in direction k's scan order.
 * x, u [B, D, H, W]; conv_w [D, Kc, Kc], conv_b [D] or NULL (fp32);
 * W_x [4, R + 2N, D], W_dt [4, D, R] (fp32).  Outputs, each direction in
 * its own scan order -- exactly the layouts ss2d_scan_fwd takes (u as its
 * x): delta [B, 4, D, H*W], Bm, Cm [B, 4, N, H*W].  All tensors contiguous,
 * device, caller-owned; I/O tensors in `dt`.  Kc odd, <= 7; N <= 32.
 * workspace: ss2d_prologue_workspace_bytes(B, H, W, R) bytes, 16-byte
 * aligned (the four directions' fp32 dt_low, [B, 4, R, H*W]).  B <= 16383.  Arithmetic and errors
 * as mamba_prologue_fwd (SSM_ERR_INVALID_ARG also for an even Kc;
 * SSM_ERR_UNSUPPORTED also when the conv's staging of (rows + Kc - 1) x
 * (W + Kc - 1) fp32 values passes 200 KB: W above about 17000 for Kc = 3).
 * ------------------------------------------------------------------------- */
SSM_API ssm_status ss2d_prologue_fwd(ssm_dtype dt, int B, int D, int H, int W,
                         int N, int R, int Kc, const void *x,
                         const float *conv_w, const float *conv_b,
                         const float *W_x, const float *W_dt, int silu_act,
                         void *u, void *delta, void *Bm, void *Cm,
                         void *workspace, size_t ws_bytes, ssm_stream_t stream);
SSM_API size_t ss2d_prologue_workspace_bytes(int B, int H, int W, int R);

/* ---------------------------------------------------------------------------
 * The block's output projection ("VMamba的SS2D模块详解" section 2.1: after the
 * gate y * act(z), out_proj = Linear(d_inner -> d_model), no bias):
 *   out[b][m][t] = sum_k W_out[m][k] * y[b][k][t]
 * y [B, Di, L] (the gated output of a scan call), W_out [Dm, Di] and out
 * [B, Dm, L], all in the I/O dtype; device pointers, caller-owned.
 * Arithmetic: fp32 accumulation; with 16-bit I/O, Dm <= 512, Di a multiple
 * of 8 and y and W_out 16-byte aligned on the tcgen05 tensor cores (fp32
 * accumulator in tensor memory; W_out read through a TMA tensor map that
 * the call encodes and caches per host thread), otherwise tiled (mma.sync
 * for 16-bit I/O, fp32 FMA for fp32 I/O); out is rounded to the I/O dtype.
 * The result does not depend on which kernel runs beyond fp32 summation
 * order.  No workspace.
 * Errors: SSM_ERR_INVALID_ARG for a bad dtype, size or pointer (NULL or
 * misaligned); SSM_ERR_UNSUPPORTED for B > 65535 or Di * L, Dm * L or
 * Dm * Di past the 32-bit index range; SSM_ERR_CUDA for a launch error.  Asynchronous on
 * `stream`.
 * ------------------------------------------------------------------------- */
SSM_API ssm_status out_proj_fwd(ssm_dtype dt, int B, int Di, int Dm, int L, const void *y,
                                const void *W_out, void *out, ssm_stream_t stream);

/*
 * Tuning override for the two-branch kernels (v1, v2 and both SS2D passes).
 * A CTA takes `channels` channels of one batch element, both branches:
 * 16, or 8 (about half the shared memory, so more CTAs fit an SM).  With 0,
 * the default, each call picks the one that leaves fewer (branch, channel)
 * rows on the busiest SM for its B and D -- 8 for small B * D, where CTAs of
 * 16 channels leave SMs idle.  Applies to later calls on this host thread;
 * any other value is treated as 0.  Results do not depend on it.
 */
SSM_API void ssm_set_cta_channels(int channels);

/*
 * Kernel choice of mamba_prologue_fwd where the fused kernel applies (16-bit
 * I/O, K = 4, R + 2N <= 64, R <= 32).  mode 1 (the default, and any value
 * other than 0 or 2): automatic -- the fused kernel for L < 1024, where it
 * measured faster, else the three-kernel path; 0: always the three-kernel
 * path; 2: the fused kernel at every L.  Applies to later calls on this host
 * thread.  Both paths compute the same sums with the same operand
 * roundings; results agree to accumulation order, not bit for bit.
 */
SSM_API void ssm_set_prologue_fused(int mode);

/*
 * Test hook for the failure path.  The next scan-kernel launch made on this
 * host thread never issues the bulk copy of B/C for chunk `chunk` (>= 0), so
 * the scan's bounded wait for it runs out after about two seconds; the kernel
 * then stops, sets the status word and leaves its output incomplete, and
 * ssm_get_status reports SSM_ERR_TIMEOUT.  Nothing faults or hangs.  The
 * hook applies to one launch only; -1 clears it.
 */
SSM_API void ssm_test_withhold_copy(int chunk);

/*
 * Test hook of the debug build (SSM_DEBUG_BOUNDS).  The next scan-kernel
 * launch made on this host thread checks its accesses to the [B, D, L]
 * tensors against an extent `elems` elements short of the real one, so the
 * accesses to the last `elems` elements are caught, skipped and reported
 * (SSM_ERR_BOUNDS through ssm_get_status) -- without any access leaving the
 * real tensor.  One launch only; the product build, which has no checks,
 * ignores it.
 */
SSM_API void ssm_test_shrink_extents(long long elems);

/* Library version, "major.minor.patch". */
SSM_API const char *ssm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H */
