"""The block's output projection (out_proj_fwd) against the fp64 oracle.

out[b][m][t] = sum_k W_out[m][k] y[b][k][t] ("VMamba的SS2D模块详解" section
2.1: Linear(d_inner -> d_model) after the gate).  Inputs are rounded to the
I/O dtype once on the host, so both sides see the same operands; the check
is element by element against the sum of the terms' magnitudes, S =
sum_k |W_mk y_kt|: a dot product of K rounded operands with fp32
accumulation errs by at most (output rounding + accumulation) * S, so
|gpu - oracle| <= tol * (1 + S) with tol the I/O dtype's (1e-4 fp32, 1e-2
bf16, 5e-3 fp16).
"""
import numpy as np
import pytest
import torch

from oracle import prologue as pro

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
TOL = {"f32": 1e-4, "bf16": 1e-2, "f16": 5e-3}


def _inputs(B, Di, Dm, L, io, seed):
    g = torch.Generator().manual_seed(seed)
    y = torch.randn(B, Di, L, generator=g).to(DT[io])
    W = (torch.randn(Dm, Di, generator=g) * Di ** -0.5).to(DT[io])
    return y, W


def _check(got, y, W, io, b_rows=None):
    ref = pro.out_proj(y if b_rows is None else y[b_rows], W)
    S = np.einsum("mk,bkl->bml", np.abs(W.double().numpy()),
                  np.abs((y if b_rows is None else y[b_rows]).double().numpy()))
    a = got.double().cpu().numpy()
    if b_rows is not None:
        a = a[b_rows]
    err = float(np.max(np.abs(a - ref) / (1.0 + S))) if ref.size else 0.0
    assert np.isfinite(err) and err <= TOL[io], "%.3g > %g" % (err, TOL[io])


# (B, Di, Dm, L): the tcgen05 path with one to four 128-row chunks, ragged
# L and Dm, Di not a multiple of 64; Di not a multiple of 8 and Dm > 512 take
# the tiled path
SHAPES = [(1, 8, 5, 7), (2, 64, 128, 130), (2, 96, 200, 257), (1, 40, 384, 129),
          (2, 768, 384, 300), (1, 136, 512, 64), (2, 100, 72, 77), (1, 40, 600, 33)]


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_out_proj_matches_oracle(io, shape):
    import selective_state_space_111_b300 as ssm
    B, Di, Dm, L = shape
    y, W = _inputs(B, Di, Dm, L, io, 100 + Di + Dm + L)
    got = ssm.out_proj_fwd(y.cuda(), W.cuda())
    torch.cuda.synchronize()
    assert got.shape == (B, Dm, L)
    _check(got, y, W, io)


def test_out_proj_weights_off_the_16_byte_grid():
    # W_out one element into a larger buffer: the tiled path, same results
    import selective_state_space_111_b300 as ssm
    B, Di, Dm, L = 2, 64, 96, 50
    y, W = _inputs(B, Di, Dm, L, "bf16", 7)
    buf = torch.empty(Dm * Di + 1, dtype=torch.bfloat16, device="cuda")[1:].view(Dm, Di)
    buf.copy_(W.cuda())
    assert buf.data_ptr() % 16 != 0
    got = ssm.out_proj_fwd(y.cuda(), buf)
    torch.cuda.synchronize()
    _check(got, y, W, "bf16")


def test_out_proj_activations_off_the_16_byte_grid():
    # y one element into a larger buffer: its rows cannot be staged by
    # 16-byte copies, so the tiled path runs; same results
    import selective_state_space_111_b300 as ssm
    B, Di, Dm, L = 2, 64, 96, 50
    y, W = _inputs(B, Di, Dm, L, "bf16", 8)
    buf = torch.empty(B * Di * L + 1, dtype=torch.bfloat16, device="cuda")[1:].view(B, Di, L)
    buf.copy_(y.cuda())
    assert buf.data_ptr() % 16 != 0
    got = ssm.out_proj_fwd(buf, W.cuda())
    torch.cuda.synchronize()
    _check(got, y, W, "bf16")


def test_out_proj_full_size_vim_s():
    # Vim-S 1248^2: d_inner 768 -> d_model 384 over 8 x 6085 positions
    # (384 tiles on the persistent CTAs: two or three each, a 69-position
    # tail); two batch elements checked in full against the oracle
    import selective_state_space_111_b300 as ssm
    B, Di, Dm, L = 8, 768, 384, 6085
    y, W = _inputs(B, Di, Dm, L, "bf16", 5)
    got = ssm.out_proj_fwd(y.cuda(), W.cuda())
    torch.cuda.synchronize()
    _check(got, y, W, "bf16", b_rows=[0, 7])
