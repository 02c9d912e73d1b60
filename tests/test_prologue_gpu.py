"""GPU parity of the prologue (conv1d + SiLU, x_proj split, dt_proj) against
the fp64 prologue oracle, and of the whole v2 inner path (prologue of each
branch, the backward one on the flipped input, then the scan-order v2
scan), link by link.

Tolerances, element by element.  u: |gpu - ref| <= tol * (1 + |ref|), tol
= 1e-4 / 1e-2 / 5e-3 for fp32 / bf16 / fp16 I/O.  dt, B and C are dot
products of rounded operands, so their rounding error scales with the sum
of the terms' magnitudes, not with the (possibly cancelling) result: each
element is held to |gpu - ref| <= tol_el * (1 + S), where S = sum_k
|W[m,k] * u[k,t]| for the rows of B and C, and S = sum_r |W_dt[d,r]| *
sum_k |W_x[r,k] * u[k,t]| for dt (the bound of its two-stage sum).  tol_el
= 1e-4 / 1e-2 / 5e-3: bf16 operands carry 2^-9 relative rounding each (W
and u: 2^-8 per product), the tf32 dt_proj 2^-11 per operand and the bf16
output 2^-9, which sum to below 7e-3 * S; fp16 to below 2.5e-3 * S; fp32
accumulation over K <= 1400 terms to below 1e-4 * S.

Full-size cases run the persistent x_proj kernels with several tiles per
CTA (Vim-S 1248^2 and a longer sequence for the 1D prologue, VMamba 56x56
for SS2D), checked over every element.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import prologue as pro

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
TOL = {"f32": 1e-4, "bf16": 1e-2, "f16": 5e-3}
TOL_EL = {"f32": 1e-4, "bf16": 1e-2, "f16": 5e-3}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_111_b300 import build
    build.build()


def weights(g, D, R, N, K):
    """Seeded prologue weights (fp32): PyTorch-like init scales."""
    u = lambda *s, a: (torch.rand(*s, generator=g) * 2 - 1) * a
    return dict(conv_w=u(D, K, a=K ** -0.5), conv_b=u(D, a=K ** -0.5),
                W_x=torch.randn(R + 2 * N, D, generator=g) * D ** -0.5,
                W_dt=torch.randn(D, R, generator=g) * R ** -0.5)


def seq_err(a, r):
    a = a.double().cpu().numpy() if hasattr(a, "cpu") else a
    return float(np.max(np.abs(a - r) / (1 + np.abs(r)))) if r.size else 0.0


def _np(a):
    return a.double().cpu().numpy() if hasattr(a, "cpu") else np.asarray(a, dtype=np.float64)


def proj_bounds(W_x, W_dt, u, R, N):
    """(S_dt, S_B, S_C): per-element sums of the terms' magnitudes of the
    two projections, from the oracle's u [B, D, L] (fp64)."""
    Wx, Wdt = np.abs(_np(W_x)), np.abs(_np(W_dt))
    S = np.einsum("mk,bkl->bml", Wx, np.abs(u))
    return np.einsum("dr,brl->bdl", Wdt, S[:, :R]), S[:, R:R + N], S[:, R + N:R + 2 * N]


def elem_err(a, r, S):
    """max over elements of |a - r| / (1 + S)."""
    a = _np(a)
    assert a.shape == r.shape == S.shape, (a.shape, r.shape, S.shape)
    return float(np.max(np.abs(a - r) / (1.0 + S))) if r.size else 0.0


def check_prologue(io, got, ref, w, R, N):
    """u element by element; dt, B, C against their per-element bounds."""
    u, dt, Bm, Cm = got
    ru, rdt, rB, rC = ref
    assert seq_err(u, ru) <= TOL[io], seq_err(u, ru)
    Sdt, SB, SC = proj_bounds(w["W_x"], w["W_dt"], ru, R, N)
    for name, a, r, S in (("dt", dt, rdt, Sdt), ("B", Bm, rB, SB), ("C", Cm, rC, SC)):
        e = elem_err(a, r, S)
        assert np.isfinite(e) and e <= TOL_EL[io], "%s: %.3g" % (name, e)


def check_ss2d_prologue(io, got, ref, w, R, N, H, W):
    """The four directions' projections against their per-element bounds
    (each direction's sequence is u in its own scan order)."""
    u, delta, Bm, Cm = got
    ru, rdelta, rB, rC = ref
    assert seq_err(u, ru) <= TOL[io], seq_err(u, ru)
    Bn, Dn = ru.shape[:2]
    uf = ru.reshape(Bn, Dn, H * W)
    dl, Bg, Cg = _np(delta), _np(Bm), _np(Cm)
    for k in range(4):
        xs = uf[..., oracle.cross_scan_index(H, W, k)]
        Sdt, SB, SC = proj_bounds(w["W_x"][k], w["W_dt"][k], xs, R, N)
        for name, a, r, S in (("delta", dl[:, k], rdelta[:, k], Sdt), ("B", Bg[:, k], rB[:, k], SB),
                              ("C", Cg[:, k], rC[:, k], SC)):
            e = elem_err(a, r, S)
            assert np.isfinite(e) and e <= TOL_EL[io], "direction %d %s: %.3g" % (k, name, e)


# (B, D, L, N, R, K); D = 1400: W_x past shared memory, the generic tiled
# x_proj; R = 40: dt_proj past 32, the generic tiled dt_proj
SHAPES = [(1, 5, 7, 4, 2, 4), (2, 70, 130, 16, 5, 4), (1, 33, 65, 32, 3, 3),
          (2, 64, 64, 16, 24, 4), (1, 1, 1, 16, 1, 4), (1, 1400, 37, 16, 6, 4),
          (1, 48, 2100, 16, 40, 4)]


@pytest.fixture(params=["fused", "three_kernel"])
def path(request):
    """The 1-D prologue's kernels for 16-bit I/O, forced: the fused
    one-kernel path (where it applies: K = 4, R + 2N <= 64, R <= 32; at
    every L) or the three-kernel path."""
    import selective_state_space_111_b300 as ssm
    ssm.set_prologue_fused(2 if request.param == "fused" else 0)
    yield request.param
    ssm.set_prologue_fused(1)


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("reverse", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_prologue_matches_oracle(io, reverse, shape, path):
    import selective_state_space_111_b300 as ssm
    if io == "f32" and path == "three_kernel":
        pytest.skip("fp32 I/O has one path")
    B, D, L, N, R, K = shape
    g = torch.Generator().manual_seed(B * 1000 + D + L + 7 * reverse)
    x = torch.randn(B, D, L, generator=g).to(DT[io])
    w = weights(g, D, R, N, K)
    wg = {k: v.cuda() for k, v in w.items()}
    u, dt, Bm, Cm = ssm.mamba_prologue_fwd(x.cuda(), wg["conv_w"], wg["conv_b"], wg["W_x"],
                                           wg["W_dt"], R, N, reverse=reverse)
    torch.cuda.synchronize()
    ref = pro.prologue(x, w["conv_w"], w["conv_b"], w["W_x"], w["W_dt"], R, N, reverse=reverse)
    check_prologue(io, (u, dt, Bm, Cm), ref, w, R, N)


# Full size.  Three-kernel path: B * ceil(L / 128) tiles of 128 positions on
# one persistent x_proj CTA per SM -- Vim-S 1248^2 (384 tiles: two or three
# per CTA, a 69-position tail) and a longer sequence (504 tiles: three or
# four per CTA, a 1-position tail).  Fused path: B * ceil(L / 64) CTAs
# (768: a 5-position tail; 1004: a 1-position tail), 24 and 4 channel slices.
FULL = [(8, 768, 6085, 16, 24, 4), (4, 128, 16001, 16, 8, 4)]


@pytest.mark.slow
@pytest.mark.parametrize("reverse", [False, True])
@pytest.mark.parametrize("shape", FULL)
def test_prologue_full_size_multi_tile(shape, reverse, path):
    import selective_state_space_111_b300 as ssm
    B, D, L, N, R, K = shape
    g = torch.Generator().manual_seed(L + 3 * reverse)
    x = torch.randn(B, D, L, generator=g).to(torch.bfloat16)
    w = weights(g, D, R, N, K)
    wg = {k: v.cuda() for k, v in w.items()}
    got = ssm.mamba_prologue_fwd(x.cuda(), wg["conv_w"], wg["conv_b"], wg["W_x"], wg["W_dt"], R,
                                 N, reverse=reverse)
    torch.cuda.synchronize()
    ref = pro.prologue(x, w["conv_w"], w["conv_b"], w["W_x"], w["W_dt"], R, N, reverse=reverse)
    check_prologue("bf16", got, ref, w, R, N)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_v2_inner_path_from_x(io):
    # prologue of each branch (the backward one on the flipped input, its
    # outputs in scan order) -> bimamba_scan_fwd_v2 with scan_order=True
    import selective_state_space_111_b300 as ssm
    B, D, L, N, R, K = 2, 40, 150, 16, 6, 4
    g = torch.Generator().manual_seed(77)
    x = torch.randn(B, D, L, generator=g).to(DT[io])
    z = torch.randn(B, D, L, generator=g).to(DT[io])
    wf, wb = weights(g, D, R, N, K), weights(g, D, R, N, K)
    A = -torch.arange(1, N + 1, dtype=torch.float32).repeat(D, 1)
    A_b = A * (1 + 0.1 * torch.rand(D, N, generator=g))
    Dk, Db = torch.rand(D, generator=g) + 0.5, torch.rand(D, generator=g) + 0.5
    bias, bias_b = torch.rand(D, generator=g) - 2.0, torch.rand(D, generator=g) - 2.0
    cu = lambda d: {k: v.cuda() for k, v in d.items()}
    gf, gb = cu(wf), cu(wb)
    xc = x.cuda()
    u, dt, Bm, Cm = ssm.mamba_prologue_fwd(xc, gf["conv_w"], gf["conv_b"], gf["W_x"], gf["W_dt"],
                                           R, N)
    ub, dtb, Bb, Cb = ssm.mamba_prologue_fwd(xc, gb["conv_w"], gb["conv_b"], gb["W_x"],
                                             gb["W_dt"], R, N, reverse=True)
    y = ssm.bimamba_scan_fwd_v2(u, dt, dtb, A.cuda(), A_b.cuda(), Bm, Cm, Bb, Cb, Dk.cuda(),
                                Db.cuda(), z.cuda(), bias.cuda(), bias_b.cuda(), ub, True, 0.5,
                                scan_order=True)
    torch.cuda.synchronize()
    # link by link: each branch's prologue against the oracle prologue
    # (per-element bounds), then the scan on the very tensors the prologues
    # produced against the oracle scan on them.  The chain from x is the
    # composition of these links; a direct comparison of y with the oracle
    # chain has no per-element bound short of one that amplifies the
    # prologue's accumulated rounding by the scan's sensitivity.
    check_prologue(io, (u, dt, Bm, Cm),
                   pro.prologue(x, wf["conv_w"], wf["conv_b"], wf["W_x"], wf["W_dt"], R, N),
                   wf, R, N)
    check_prologue(io, (ub, dtb, Bb, Cb),
                   pro.prologue(x, wb["conv_w"], wb["conv_b"], wb["W_x"], wb["W_dt"], R, N,
                                reverse=True), wb, R, N)
    ref_scan = oracle.bimamba_v2(u, dt, torch.flip(dtb, [-1]), A, A_b, Bm, Cm,
                                 torch.flip(Bb, [-1]), torch.flip(Cb, [-1]), Dk, Db, z, bias,
                                 bias_b, torch.flip(ub, [-1]), True, 0.5)
    assert seq_err(y, ref_scan) <= TOL[io]              # the scan on what it was given


# ---------------------------------------------------------------- SS2D

def ss2d_weights(g, D, R, N, Kc):
    """Seeded SS2D prologue weights (fp32): one x_proj and dt_proj per
    direction, PyTorch-like init scales."""
    u = lambda *s, a: (torch.rand(*s, generator=g) * 2 - 1) * a
    return dict(conv_w=u(D, Kc, Kc, a=1.0 / Kc), conv_b=u(D, a=1.0 / Kc),
                W_x=torch.randn(4, R + 2 * N, D, generator=g) * D ** -0.5,
                W_dt=torch.randn(4, D, R, generator=g) * R ** -0.5)


# (B, D, H, W, N, R, Kc): non-square maps, one-row and one-column maps,
# d_state 32 (x_proj past 64 rows: the generic tiled kernel), Kc 1..7,
# and the fallbacks below
SS2D_SHAPES = [(1, 5, 4, 6, 16, 2, 3), (2, 70, 9, 13, 16, 5, 3), (1, 33, 7, 5, 32, 3, 5),
               (2, 64, 16, 16, 16, 6, 3), (1, 1, 1, 1, 16, 1, 3), (1, 8, 3, 40, 16, 4, 7),
               (1, 9, 50, 1, 16, 2, 1), (1, 16, 130, 3, 16, 24, 3),
               (1, 300, 5, 6, 16, 4, 3),     # d_inner > 256: x_proj per direction, 2 slices
               (2, 12, 6, 7, 16, 36, 3)]     # dt_rank > 32: the generic dt_proj per direction


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", SS2D_SHAPES)
def test_ss2d_prologue_matches_oracle(io, shape):
    import selective_state_space_111_b300 as ssm
    B, D, H, W, N, R, Kc = shape
    act = (H + W) % 2 == 0 or io == "bf16"
    g = torch.Generator().manual_seed(B * 1000 + D + H * W + Kc)
    x = torch.randn(B, D, H, W, generator=g).to(DT[io])
    w = ss2d_weights(g, D, R, N, Kc)
    wg = {k: v.cuda() for k, v in w.items()}
    u, delta, Bm, Cm = ssm.ss2d_prologue_fwd(x.cuda(), wg["conv_w"], wg["conv_b"], wg["W_x"],
                                             wg["W_dt"], R, N, silu_act=act)
    torch.cuda.synchronize()
    ref = pro.ss2d_prologue(x, w["conv_w"], w["conv_b"], w["W_x"], w["W_dt"], R, N,
                            silu_act=act)
    check_ss2d_prologue(io, (u, delta, Bm, Cm), ref, w, R, N, H, W)


@pytest.mark.slow
def test_ss2d_prologue_full_size_multi_tile():
    # VMamba 56x56 (B 32, d_inner 192, dt_rank 6): 896 map tiles of 8 x 16
    # on one persistent CTA per SM, six or seven per CTA, ragged in W
    import selective_state_space_111_b300 as ssm
    B, D, H, W, N, R, Kc = 32, 192, 56, 56, 16, 6, 3
    g = torch.Generator().manual_seed(5656)
    x = torch.randn(B, D, H, W, generator=g).to(torch.bfloat16)
    w = ss2d_weights(g, D, R, N, Kc)
    wg = {k: v.cuda() for k, v in w.items()}
    got = ssm.ss2d_prologue_fwd(x.cuda(), wg["conv_w"], wg["conv_b"], wg["W_x"], wg["W_dt"], R, N)
    torch.cuda.synchronize()
    ref = pro.ss2d_prologue(x, w["conv_w"], w["conv_b"], w["W_x"], w["W_dt"], R, N)
    check_ss2d_prologue("bf16", got, ref, w, R, N, H, W)


def test_ss2d_prologue_without_activation_and_bias():
    import selective_state_space_111_b300 as ssm
    B, D, H, W, N, R, Kc = 2, 20, 11, 7, 16, 4, 3
    g = torch.Generator().manual_seed(91)
    x = torch.randn(B, D, H, W, generator=g)
    w = ss2d_weights(g, D, R, N, Kc)
    wg = {k: v.cuda() for k, v in w.items()}
    u, delta, Bm, Cm = ssm.ss2d_prologue_fwd(x.cuda(), wg["conv_w"], None, wg["W_x"], wg["W_dt"],
                                             R, N, silu_act=False)
    torch.cuda.synchronize()
    ref = pro.ss2d_prologue(x, w["conv_w"], None, w["W_x"], w["W_dt"], R, N, silu_act=False)
    check_ss2d_prologue("f32", (u, delta, Bm, Cm), ref, w, R, N, H, W)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_ss2d_inner_path_from_x(io):
    # conv2d + the four directions' projections -> ss2d_scan_fwd, against
    # the oracle chain
    import selective_state_space_111_b300 as ssm
    B, D, H, W, N, R, Kc = 2, 24, 9, 11, 16, 3, 3
    g = torch.Generator().manual_seed(123)
    x = torch.randn(B, D, H, W, generator=g).to(DT[io])
    z = torch.randn(B, D, H, W, generator=g).to(DT[io])
    w = ss2d_weights(g, D, R, N, Kc)
    A = -torch.arange(1, N + 1, dtype=torch.float32).repeat(4, D, 1)
    A = A * (1 + 0.1 * torch.rand(4, D, N, generator=g))
    Dk = torch.rand(4, D, generator=g) + 0.5
    bias = torch.rand(4, D, generator=g) - 2.0
    wg = {k: v.cuda() for k, v in w.items()}
    u, delta, Bm, Cm = ssm.ss2d_prologue_fwd(x.cuda(), wg["conv_w"], wg["conv_b"], wg["W_x"],
                                             wg["W_dt"], R, N)
    y = ssm.ss2d_scan_fwd(u, delta, A.cuda(), Bm, Cm, Dk.cuda(), z.cuda(), bias.cuda(), True)
    torch.cuda.synchronize()
    # link by link, as for the v2 path
    check_ss2d_prologue(io, (u, delta, Bm, Cm),
                        pro.ss2d_prologue(x, w["conv_w"], w["conv_b"], w["W_x"], w["W_dt"], R, N),
                        w, R, N, H, W)
    ref_scan = oracle.ss2d(u, delta, A, Bm, Cm, Dk, z, bias, True)
    assert seq_err(y, ref_scan) <= TOL[io]              # the scan on what it was given


def test_prologue_outputs_off_the_4_byte_grid(path):
    # outputs one element into larger buffers (2-byte aligned only): the
    # pair stores must fall back to 2-byte stores; straight through the C ABI
    from selective_state_space_111_b300 import binding
    lib = binding.lib()
    B, D, L, N, R, K = 2, 40, 301, 16, 5, 4
    g = torch.Generator().manual_seed(303)
    x = torch.randn(B, D, L, generator=g).to(torch.bfloat16)
    w = weights(g, D, R, N, K)
    wg = {k: v.cuda() for k, v in w.items()}
    xc = x.cuda()

    def shifted(*shape):
        n = int(np.prod(shape))
        return torch.zeros(n + 1, dtype=torch.bfloat16, device="cuda")[1:].view(*shape)

    u, delta, Bm, Cm = shifted(B, D, L), shifted(B, D, L), shifted(B, N, L), shifted(B, N, L)
    assert u.data_ptr() % 4 == 2
    nws = int(lib.ssm_prologue_workspace_bytes(B, L, R))
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    st = lib.mamba_prologue_fwd(1, B, D, L, N, R, K, xc.data_ptr(), wg["conv_w"].data_ptr(),
                                wg["conv_b"].data_ptr(), wg["W_x"].data_ptr(),
                                wg["W_dt"].data_ptr(), 0, u.data_ptr(), delta.data_ptr(),
                                Bm.data_ptr(), Cm.data_ptr(), ws.data_ptr(), nws,
                                torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    ref = pro.prologue(x, w["conv_w"], w["conv_b"], w["W_x"], w["W_dt"], R, N)
    check_prologue("bf16", (u, delta, Bm, Cm), ref, w, R, N)
