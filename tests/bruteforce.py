"""Explicit unrolled closed form of the S6 forward pass (numpy, fp64).

An independent checker for the oracle: it never runs the recurrence.  For one
sequence it evaluates, for every t,

  y_t = sum_{s<=t} sum_n C[n,t] * exp(A[n] * sum_{r=s+1..t} delta_r)
                               * delta_s * B[n,s] * u_s  +  D * u_t,

the unrolled form of h_t = exp(delta_t A) h_{t-1} + delta_t B_t u_t with
h_{-1} = 0, y_t = C_t h_t + D u_t (the S6 equations of the Vision Mamba
overview page, section "选择性扫描机制的计算效率优势", with zero-order-hold
A and Euler B).  O(L^2 N): tiny L only.
"""
import numpy as np


def softplus(x):
    x = np.asarray(x, np.float64)
    return np.where(x > 0, x + np.log1p(np.exp(-np.abs(x))), np.log1p(np.exp(np.minimum(x, 0))))


def closed_form_sequence(u, dt, A, B, C, D=0.0, bias=0.0, delta_softplus=True):
    """u, dt: [L]; A: [N]; B, C: [N, L].  Returns y: [L]."""
    u = np.asarray(u, np.float64)
    x = np.asarray(dt, np.float64) + bias
    delta = softplus(x) if delta_softplus else x
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    C = np.asarray(C, np.float64)
    L = u.shape[0]
    y = np.empty(L)
    for t in range(L):
        total = 0.0
        for s in range(t + 1):
            decay = np.exp(A * np.sum(delta[s + 1:t + 1]))   # [N]
            total += np.sum(C[:, t] * decay * delta[s] * B[:, s]) * u[s]
        y[t] = total + D * u[t]
    return y


def silu_gate(y, z):
    z = np.asarray(z, np.float64)
    return y * z / (1.0 + np.exp(-z))


def closed_form_last_state(u, dt, A, B, bias=0.0, delta_softplus=True):
    """State after the last step, unrolled (no recurrence):
    h_{L-1}[n] = sum_s exp(A[n] * sum_{r=s+1..L-1} delta_r) * delta_s * B[n,s] * u_s."""
    u = np.asarray(u, np.float64)
    x = np.asarray(dt, np.float64) + bias
    delta = softplus(x) if delta_softplus else x
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    L = u.shape[0]
    h = np.zeros(A.shape[0])
    for s in range(L):
        h += np.exp(A * np.sum(delta[s + 1:])) * delta[s] * B[:, s] * u[s]
    return h
