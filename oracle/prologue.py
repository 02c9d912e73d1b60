"""fp64 oracle of the scan's prologue (test infrastructure only).

TEST INFRASTRUCTURE ONLY: called by the test suite and the benchmark's
CPU-baseline leg, never by the product path, and it imports nothing from
the product package.

The steps that turn the block's input x [B, D, L] into the scan's inputs,
for one direction ("Vision Mamba实战" section 2.1 and "从Transformer到Mamba"
section 2.1: conv1d, x_proj = Linear(d_inner -> dt_rank + 2 d_state),
dt_proj = Linear(dt_rank -> d_inner); "VMamba的SS2D模块详解" section 3.1:
dt, B, C = split(x_proj(x), [dt_rank, d_state, d_state]) and
delta = softplus(dt_proj(dt)); "从Transformer到Mamba" section 2.2: the
backward branch of v2 runs the same steps with its own weights on the
flipped sequence):

  xs      = x, or x reversed in time (reverse=True: the backward branch)
  conv[t] = bias[d] + sum_k w[d][k] * xs[t - (K-1) + k]   (causal, depthwise;
            xs[<0] = 0 -- the pages print Conv1d without groups/padding;
            reading: Mamba's depthwise causal convolution)
  u       = silu(conv)
  proj    = W_x @ u          rows: dt_low [0, R), B [R, R+N), C [R+N, R+2N)
  dt      = W_dt @ dt_low    (dt_proj's bias is the scan's delta_bias; the
                              scan applies softplus)

Outputs are in scan order for reverse=True (element t is position L-1-t).

SS2D's prologue ("VMamba的SS2D模块详解" section 2.1: conv2d, the depthwise
convolution on the [B, D, H, W] map, d_conv 3 in its parameter table;
section 2.2: the four scan orders; section 3.1: one x_proj and one
dt_proj per scan direction):

  conv2d[h][w] = bias[d] + sum_{i,j} w[d][i][j] * x[h+i-P][w+j-P], P =
            (Kc-1)/2, zero outside the map (output the size of the input;
            the pages print conv2d without its arguments -- reading:
            depthwise, "same" zero padding, odd Kc)
  u       = silu(conv2d), or conv2d itself with silu=False (the pages'
            simplified SS2D forward shows no activation after conv2d; the
            1D path applies SiLU)
  xs_k    = u flattened in direction k's scan order (k = 0 row-major,
            1 column-major, 2 and 3 their reversals)
  proj_k  = W_x[k] @ xs_k, split as in the 1D case; dt_k = W_dt[k] @ dt_low_k

The block's output projection ("VMamba的SS2D模块详解" section 2.1: after the
gate y * act(z), out_proj = Linear(d_inner -> d_model); the pages show no
bias -- reading: none, as in Mamba), on the library's [B, D, L] layout:

  out[b][m][t] = sum_k W_out[m][k] * y[b][k][t]
"""
from __future__ import annotations

import numpy as np


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        import torch
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def causal_conv(x, w, b=None, reverse=False):
    """[B, D, L] pre-activation of the depthwise causal convolution."""
    x = _f64(x)
    w = _f64(w)
    if reverse:
        x = x[..., ::-1]
    Bn, Dn, L = x.shape
    K = w.shape[1]
    out = np.zeros((Bn, Dn, L))
    if b is not None:
        out += _f64(b)[None, :, None]
    for k in range(K):
        shift = K - 1 - k                       # tap k reads position t - shift
        if shift < L:
            out[..., shift:] += w[None, :, k, None] * x[..., :L - shift]
    return out


def silu(v):
    return v / (1.0 + np.exp(-v))


def prologue(x, conv_w, conv_b, W_x, W_dt, dt_rank, d_state, reverse=False):
    """Returns (u [B,D,L], dt [B,D,L], Bm [B,N,L], Cm [B,N,L])."""
    u = silu(causal_conv(x, conv_w, conv_b, reverse))
    W_x = _f64(W_x)
    proj = np.einsum("md,bdl->bml", W_x, u)
    R, N = dt_rank, d_state
    dt_low, Bm, Cm = proj[:, :R], proj[:, R:R + N], proj[:, R + N:R + 2 * N]
    dt = np.einsum("dr,brl->bdl", _f64(W_dt), dt_low)
    return u, dt, Bm, Cm


def depthwise_conv2d(x, w, b=None):
    """[B, D, H, W] pre-activation of the depthwise 2D convolution with zero
    padding (Kc-1)/2 on every side: out[h][w] = b + sum_{i,j} w[i][j] *
    x[h + i - P][w + j - P] (a correlation, as a Conv2d layer computes)."""
    x = _f64(x)
    w = _f64(w)
    Bn, Dn, H, W = x.shape
    Kc = w.shape[-1]
    P = (Kc - 1) // 2
    xp = np.zeros((Bn, Dn, H + 2 * P, W + 2 * P))
    xp[..., P:P + H, P:P + W] = x
    out = np.zeros((Bn, Dn, H, W))
    if b is not None:
        out += _f64(b)[None, :, None, None]
    for i in range(Kc):
        for j in range(Kc):
            out += w[None, :, i, j, None, None] * xp[..., i:i + H, j:j + W]
    return out


def ss2d_prologue(x, conv_w, conv_b, W_x, W_dt, dt_rank, d_state, silu_act=True):
    """Returns (u [B,D,H,W], delta [B,4,D,L], Bm [B,4,N,L], Cm [B,4,N,L]),
    the per-direction tensors in each direction's scan order (L = H W)."""
    from . import cross_scan_index
    c = depthwise_conv2d(x, conv_w, conv_b)
    u = silu(c) if silu_act else c
    Bn, Dn, H, W = u.shape
    L = H * W
    uf = u.reshape(Bn, Dn, L)
    W_x, W_dt = _f64(W_x), _f64(W_dt)
    R, N = dt_rank, d_state
    delta = np.empty((Bn, 4, Dn, L))
    Bm = np.empty((Bn, 4, N, L))
    Cm = np.empty((Bn, 4, N, L))
    for k in range(4):
        xs = uf[..., cross_scan_index(H, W, k)]
        proj = np.einsum("md,bdl->bml", W_x[k], xs)
        Bm[:, k], Cm[:, k] = proj[:, R:R + N], proj[:, R + N:R + 2 * N]
        delta[:, k] = np.einsum("dr,brl->bdl", W_dt[k], proj[:, :R])
    return u, delta, Bm, Cm


def out_proj(y, W_out):
    """[B, d_model, L] = W_out [d_model, d_inner] applied to y [B, d_inner, L]."""
    return np.einsum("mk,bkl->bml", _f64(W_out), _f64(y))
