"""fp64 CPU oracle for the selective-scan forward pass (test infrastructure).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path never
imports this package, and this package never imports the product package.

The arithmetic lives in ``ssm_oracle.c`` (plain C, fp64, strictly sequential;
see its header for the page/section each step follows).  This module only
compiles it (gcc, once), marshals numpy arrays to fp64 and calls it.

Functions mirror the C ABI's operations:
  selective_scan(u, delta, A, B, C, D=None, z=None, delta_bias=None,
                 delta_softplus=True)                                 -> y
  bimamba_v1(u, delta, A, A_b, B, C, D=None, z=None, delta_bias=None,
             delta_softplus=True, out_scale=1.0)                      -> y
  bimamba_v2(u, delta, delta_b, A, A_b, B, C, B_b, C_b, D=None, D_b=None,
             z=None, delta_bias=None, delta_bias_b=None, u_b=None,
             delta_softplus=True, out_scale=0.5)                      -> y
  ss2d(x, delta, A, B, C, D=None, z=None, delta_bias=None,
       delta_softplus=True)                                           -> y
  cross_scan_index(H, W, k)                   -> int64 array of length H*W
and the backward pass of each form (gradients of sum(g * out) for the
incoming output gradient g), returning a dict of gradient arrays:
  selective_scan_bwd(g, ...same inputs...)    -> du, ddelta, dA, dB, dC, dD, dz, ddelta_bias
  bimamba_v1_bwd(g, ...)                      -> du, ddelta, dA, dA_b, dB, dC, dD, dz,
                                                 ddelta_bias
  bimamba_v2_bwd(g, ...)                      -> du, (du_b), ddelta, ddelta_b, dA, dA_b,
                                                 dB, dC, dB_b, dC_b, dD, dD_b, dz,
                                                 ddelta_bias, ddelta_bias_b
  ss2d_bwd(g, ...)                            -> dx, ddelta, dA, dB, dC, dD, dz,
                                                 ddelta_bias
and the final state of every direction ([directions, B, D, N]):
  selective_scan_last_state, bimamba_v1_last_state, bimamba_v2_last_state,
  ss2d_last_state (same inputs as the forward calls; C, D and z play no part)
Shapes are the ones documented in ``ssm_oracle.c``; a gradient has its
input's shape.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB = os.path.join(_HERE, "libssm_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile ssm_oracle.c into libssm_oracle.so (no fast-math: IEEE fp64)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, d = ctypes.c_int, ctypes.c_double
            lib.oracle_selective_scan.argtypes = [i, i, i, i] + [_dp] * 8 + [i, _dp]
            lib.oracle_bimamba_v1.argtypes = [i, i, i, i] + [_dp] * 9 + [i, d, _dp]
            lib.oracle_bimamba_v2.argtypes = [i, i, i, i] + [_dp] * 15 + [i, d, _dp]
            lib.oracle_ss2d.argtypes = [i, i, i, i, i, i] + [_dp] * 8 + [i, _dp]
            lib.oracle_selective_scan_bwd.argtypes = [i, i, i, i] + [_dp] * 8 + [i] + [_dp] * 9
            lib.oracle_bimamba_v1_bwd.argtypes = [i, i, i, i] + [_dp] * 9 + [i, d] + [_dp] * 10
            lib.oracle_bimamba_v2_bwd.argtypes = ([i, i, i, i] + [_dp] * 15 + [i, d] +
                                                  [_dp] * 16)
            lib.oracle_ss2d_bwd.argtypes = [i, i, i, i, i, i] + [_dp] * 8 + [i] + [_dp] * 9
            lib.oracle_last_state.argtypes = [i, i, i, i] + [_dp] * 5 + [i, _dp]
            lib.oracle_last_state.restype = ctypes.c_int
            lib.oracle_cross_scan_index.argtypes = [i, i, i, ctypes.c_long]
            lib.oracle_cross_scan_index.restype = ctypes.c_long
            for f in (lib.oracle_selective_scan, lib.oracle_bimamba_v1,
                      lib.oracle_bimamba_v2, lib.oracle_ss2d, lib.oracle_selective_scan_bwd,
                      lib.oracle_bimamba_v1_bwd, lib.oracle_bimamba_v2_bwd,
                      lib.oracle_ss2d_bwd):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a, shape=None):
    """Contiguous fp64 copy of an array-like (torch tensors go through numpy)."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: widen exactly on the torch side
        import torch  # local: only needed when tensors are passed

        a = a.detach().to("cpu", torch.float64).numpy()
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and arr.shape != tuple(shape):
        raise ValueError("expected shape %s, got %s" % (tuple(shape), arr.shape))
    return arr


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _check(rc, name):
    if rc != 0:
        raise RuntimeError("%s: bad argument or allocation failure" % name)


def selective_scan(u, delta, A, B, C, D=None, z=None, delta_bias=None,
                   delta_softplus=True):
    u = _f64(u)
    Bn, Dn, L = u.shape
    N = np.shape(A)[1]
    a = [u, _f64(delta, (Bn, Dn, L)), _f64(A, (Dn, N)), _f64(B, (Bn, N, L)),
         _f64(C, (Bn, N, L)), _f64(D, (Dn,)), _f64(z, (Bn, Dn, L)),
         _f64(delta_bias, (Dn,))]
    y = np.empty((Bn, Dn, L), np.float64)
    _check(_load().oracle_selective_scan(Bn, Dn, L, N, *map(_ptr, a),
                                         int(bool(delta_softplus)), _ptr(y)),
           "selective_scan")
    return y


def bimamba_v1(u, delta, A, A_b, B, C, D=None, z=None, delta_bias=None,
               delta_softplus=True, out_scale=1.0):
    u = _f64(u)
    Bn, Dn, L = u.shape
    N = np.shape(A)[1]
    a = [u, _f64(delta, (Bn, Dn, L)), _f64(A, (Dn, N)), _f64(A_b, (Dn, N)),
         _f64(B, (Bn, N, L)), _f64(C, (Bn, N, L)), _f64(D, (Dn,)),
         _f64(z, (Bn, Dn, L)), _f64(delta_bias, (Dn,))]
    y = np.empty((Bn, Dn, L), np.float64)
    _check(_load().oracle_bimamba_v1(Bn, Dn, L, N, *map(_ptr, a),
                                     int(bool(delta_softplus)), float(out_scale),
                                     _ptr(y)), "bimamba_v1")
    return y


def bimamba_v2(u, delta, delta_b, A, A_b, B, C, B_b, C_b, D=None, D_b=None,
               z=None, delta_bias=None, delta_bias_b=None, u_b=None,
               delta_softplus=True, out_scale=0.5):
    u = _f64(u)
    Bn, Dn, L = u.shape
    N = np.shape(A)[1]
    a = [u, _f64(u_b, (Bn, Dn, L)), _f64(delta, (Bn, Dn, L)),
         _f64(delta_b, (Bn, Dn, L)), _f64(A, (Dn, N)), _f64(A_b, (Dn, N)),
         _f64(B, (Bn, N, L)), _f64(C, (Bn, N, L)), _f64(B_b, (Bn, N, L)),
         _f64(C_b, (Bn, N, L)), _f64(D, (Dn,)), _f64(D_b, (Dn,)),
         _f64(z, (Bn, Dn, L)), _f64(delta_bias, (Dn,)), _f64(delta_bias_b, (Dn,))]
    y = np.empty((Bn, Dn, L), np.float64)
    _check(_load().oracle_bimamba_v2(Bn, Dn, L, N, *map(_ptr, a),
                                     int(bool(delta_softplus)), float(out_scale),
                                     _ptr(y)), "bimamba_v2")
    return y


def ss2d(x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True):
    x = _f64(x)
    Bn, Dn, H, W = x.shape
    K = 4
    L = H * W
    N = np.shape(A)[2]
    a = [x, _f64(delta, (Bn, K, Dn, L)), _f64(A, (K, Dn, N)),
         _f64(B, (Bn, K, N, L)), _f64(C, (Bn, K, N, L)), _f64(D, (K, Dn)),
         _f64(z, (Bn, Dn, H, W)), _f64(delta_bias, (K, Dn))]
    y = np.empty((Bn, Dn, H, W), np.float64)
    _check(_load().oracle_ss2d(Bn, Dn, H, W, N, K, *map(_ptr, a),
                               int(bool(delta_softplus)), _ptr(y)), "ss2d")
    return y


def cross_scan_index(H, W, k):
    lib = _load()
    out = np.array([lib.oracle_cross_scan_index(H, W, k, t) for t in range(H * W)],
                   dtype=np.int64)
    if (out < 0).any():
        raise ValueError("bad cross-scan arguments")
    return out


# ---------------------------------------------------------------- backward
def _out(shape, present=True):
    return np.empty(shape, np.float64) if present else None


def selective_scan_bwd(g, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                       delta_softplus=True):
    u = _f64(u)
    Bn, Dn, L = u.shape
    N = np.shape(A)[1]
    a = [u, _f64(delta, (Bn, Dn, L)), _f64(A, (Dn, N)), _f64(B, (Bn, N, L)),
         _f64(C, (Bn, N, L)), _f64(D, (Dn,)), _f64(z, (Bn, Dn, L)),
         _f64(delta_bias, (Dn,))]
    r = {"du": _out((Bn, Dn, L)), "ddelta": _out((Bn, Dn, L)), "dA": _out((Dn, N)),
         "dB": _out((Bn, N, L)), "dC": _out((Bn, N, L)), "dD": _out((Dn,), D is not None),
         "dz": _out((Bn, Dn, L), z is not None),
         "ddelta_bias": _out((Dn,), delta_bias is not None)}
    _check(_load().oracle_selective_scan_bwd(
        Bn, Dn, L, N, *map(_ptr, a), int(bool(delta_softplus)), _ptr(_f64(g, (Bn, Dn, L))),
        *[_ptr(r[k]) for k in ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias")]),
        "selective_scan_bwd")
    return {k: v for k, v in r.items() if v is not None}


def bimamba_v1_bwd(g, u, delta, A, A_b, B, C, D=None, z=None, delta_bias=None,
                   delta_softplus=True, out_scale=1.0):
    u = _f64(u)
    Bn, Dn, L = u.shape
    N = np.shape(A)[1]
    a = [u, _f64(delta, (Bn, Dn, L)), _f64(A, (Dn, N)), _f64(A_b, (Dn, N)),
         _f64(B, (Bn, N, L)), _f64(C, (Bn, N, L)), _f64(D, (Dn,)),
         _f64(z, (Bn, Dn, L)), _f64(delta_bias, (Dn,))]
    keys = ("du", "ddelta", "dA", "dA_b", "dB", "dC", "dD", "dz", "ddelta_bias")
    r = {"du": _out((Bn, Dn, L)), "ddelta": _out((Bn, Dn, L)), "dA": _out((Dn, N)),
         "dA_b": _out((Dn, N)), "dB": _out((Bn, N, L)), "dC": _out((Bn, N, L)),
         "dD": _out((Dn,), D is not None), "dz": _out((Bn, Dn, L), z is not None),
         "ddelta_bias": _out((Dn,), delta_bias is not None)}
    _check(_load().oracle_bimamba_v1_bwd(
        Bn, Dn, L, N, *map(_ptr, a), int(bool(delta_softplus)), float(out_scale),
        _ptr(_f64(g, (Bn, Dn, L))), *[_ptr(r[k]) for k in keys]), "bimamba_v1_bwd")
    return {k: v for k, v in r.items() if v is not None}


def bimamba_v2_bwd(g, u, delta, delta_b, A, A_b, B, C, B_b, C_b, D=None, D_b=None,
                   z=None, delta_bias=None, delta_bias_b=None, u_b=None,
                   delta_softplus=True, out_scale=0.5):
    u = _f64(u)
    Bn, Dn, L = u.shape
    N = np.shape(A)[1]
    a = [u, _f64(u_b, (Bn, Dn, L)), _f64(delta, (Bn, Dn, L)),
         _f64(delta_b, (Bn, Dn, L)), _f64(A, (Dn, N)), _f64(A_b, (Dn, N)),
         _f64(B, (Bn, N, L)), _f64(C, (Bn, N, L)), _f64(B_b, (Bn, N, L)),
         _f64(C_b, (Bn, N, L)), _f64(D, (Dn,)), _f64(D_b, (Dn,)),
         _f64(z, (Bn, Dn, L)), _f64(delta_bias, (Dn,)), _f64(delta_bias_b, (Dn,))]
    keys = ("du", "du_b", "ddelta", "ddelta_b", "dA", "dA_b", "dB", "dC", "dB_b", "dC_b",
            "dD", "dD_b", "dz", "ddelta_bias", "ddelta_bias_b")
    sh, shn = (Bn, Dn, L), (Bn, N, L)
    r = {"du": _out(sh), "du_b": _out(sh, u_b is not None), "ddelta": _out(sh),
         "ddelta_b": _out(sh), "dA": _out((Dn, N)), "dA_b": _out((Dn, N)),
         "dB": _out(shn), "dC": _out(shn), "dB_b": _out(shn), "dC_b": _out(shn),
         "dD": _out((Dn,), D is not None), "dD_b": _out((Dn,), D_b is not None),
         "dz": _out(sh, z is not None), "ddelta_bias": _out((Dn,), delta_bias is not None),
         "ddelta_bias_b": _out((Dn,), delta_bias_b is not None)}
    _check(_load().oracle_bimamba_v2_bwd(
        Bn, Dn, L, N, *map(_ptr, a), int(bool(delta_softplus)), float(out_scale),
        _ptr(_f64(g, sh)), *[_ptr(r[k]) for k in keys]), "bimamba_v2_bwd")
    return {k: v for k, v in r.items() if v is not None}


def ss2d_bwd(g, x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True):
    x = _f64(x)
    Bn, Dn, H, W = x.shape
    K = 4
    L = H * W
    N = np.shape(A)[2]
    a = [x, _f64(delta, (Bn, K, Dn, L)), _f64(A, (K, Dn, N)),
         _f64(B, (Bn, K, N, L)), _f64(C, (Bn, K, N, L)), _f64(D, (K, Dn)),
         _f64(z, (Bn, Dn, H, W)), _f64(delta_bias, (K, Dn))]
    keys = ("dx", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias")
    r = {"dx": _out((Bn, Dn, H, W)), "ddelta": _out((Bn, K, Dn, L)), "dA": _out((K, Dn, N)),
         "dB": _out((Bn, K, N, L)), "dC": _out((Bn, K, N, L)),
         "dD": _out((K, Dn), D is not None), "dz": _out((Bn, Dn, H, W), z is not None),
         "ddelta_bias": _out((K, Dn), delta_bias is not None)}
    _check(_load().oracle_ss2d_bwd(
        Bn, Dn, H, W, N, K, *map(_ptr, a), int(bool(delta_softplus)),
        _ptr(_f64(g, (Bn, Dn, H, W))), *[_ptr(r[k]) for k in keys]), "ss2d_bwd")
    return {k: v for k, v in r.items() if v is not None}


# ---------------------------------------------------------------- final states
def _last_state(u, delta, A, B, delta_bias, delta_softplus):
    """Final state of one direction over the rows as given: [B, D, N]."""
    u = _f64(u)
    Bn, Dn, L = u.shape
    N = np.shape(A)[1]
    out = np.empty((Bn, Dn, N), np.float64)
    a = [u, _f64(delta, (Bn, Dn, L)), _f64(A, (Dn, N)), _f64(B, (Bn, N, L)),
         _f64(delta_bias, (Dn,))]
    _check(_load().oracle_last_state(Bn, Dn, L, N, *map(_ptr, a), int(bool(delta_softplus)),
                                     _ptr(out)), "last_state")
    return out


def selective_scan_last_state(u, delta, A, B, C=None, D=None, z=None, delta_bias=None,
                              delta_softplus=True):
    return _last_state(u, delta, A, B, delta_bias, delta_softplus)[None]


def bimamba_v2_last_state(u, delta, delta_b, A, A_b, B, C, B_b, C_b, D=None, D_b=None, z=None,
                          delta_bias=None, delta_bias_b=None, u_b=None, delta_softplus=True,
                          out_scale=0.5):
    """[2, B, D, N]: the forward branch after position L-1, the backward
    branch (run on the time-reversed copies) after position 0."""
    ub = _f64(u if u_b is None else u_b)
    f = _last_state(u, delta, A, B, delta_bias, delta_softplus)
    b = _last_state(np.flip(ub, -1), np.flip(_f64(delta_b), -1), A_b, np.flip(_f64(B_b), -1),
                    delta_bias_b, delta_softplus)
    return np.stack([f, b])


def bimamba_v1_last_state(u, delta, A, A_b, B, C, D=None, z=None, delta_bias=None,
                          delta_softplus=True, out_scale=1.0):
    return bimamba_v2_last_state(u, delta, delta, A, A_b, B, C, B, C, delta_bias=delta_bias,
                                 delta_bias_b=delta_bias, delta_softplus=delta_softplus)


def ss2d_last_state(x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True):
    """[4, B, D, N]: direction k run over the image read in its scan order."""
    x = _f64(x)
    Bn, Dn, H, W = x.shape
    L = H * W
    flat = x.reshape(Bn, Dn, L)
    out = []
    for k in range(4):
        xs = flat[:, :, cross_scan_index(H, W, k)]
        out.append(_last_state(xs, _f64(delta)[:, k], _f64(A)[k], _f64(B)[:, k],
                               None if delta_bias is None else _f64(delta_bias)[k],
                               delta_softplus))
    return np.stack(out)
