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
