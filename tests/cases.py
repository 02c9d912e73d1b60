"""Shared helpers for the parity tests: run an operation through the CUDA
library and through the fp64 oracle on the same seeded inputs."""
import numpy as np
import torch

import oracle
from selective_state_space_111_b300.synth import make_inputs  # noqa: F401

# Tolerances: |gpu - oracle| <= TOL * (1 + |oracle|), elementwise.
TOL = {"f32": 1e-4, "bf16": 1e-2, "f16": 2e-3}


def to_dev(t):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}


def run_gpu(spec, t, workspace=None, dev=None, out=None):
    """Runs the library on the host inputs `t` (copied to the GPU), or on
    the device tensors `dev` when given; `out` is an optional output."""
    import selective_state_space_111_b300 as ssm

    g = to_dev(t) if dev is None else dev
    sp = spec.delta_softplus
    kw = dict(workspace=workspace, out=out)
    if spec.op == "single":
        return ssm.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                      g["delta_bias"], sp, **kw)
    if spec.op == "v1":
        return ssm.bimamba_scan_fwd_v1(g["u"], g["delta"], g["A"], g["A_b"], g["B"], g["C"],
                                       g["D"], g["z"], g["delta_bias"], sp, g["out_scale"], **kw)
    if spec.op == "v2":
        return ssm.bimamba_scan_fwd_v2(g["u"], g["delta"], g["delta_b"], g["A"], g["A_b"], g["B"],
                                       g["C"], g["B_b"], g["C_b"], g["D"], g["D_b"], g["z"],
                                       g["delta_bias"], g["delta_bias_b"], g["u_b"], sp,
                                       g["out_scale"], **kw)
    return ssm.ss2d_scan_fwd(g["x"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                             g["delta_bias"], sp, **kw)


def run_oracle(spec, t):
    sp = spec.delta_softplus
    if spec.op == "single":
        return oracle.selective_scan(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                     t["delta_bias"], sp)
    if spec.op == "v1":
        return oracle.bimamba_v1(t["u"], t["delta"], t["A"], t["A_b"], t["B"], t["C"], t["D"],
                                 t["z"], t["delta_bias"], sp, t["out_scale"])
    if spec.op == "v2":
        return oracle.bimamba_v2(t["u"], t["delta"], t["delta_b"], t["A"], t["A_b"], t["B"],
                                 t["C"], t["B_b"], t["C_b"], t["D"], t["D_b"], t["z"],
                                 t["delta_bias"], t["delta_bias_b"], t["u_b"], sp, t["out_scale"])
    return oracle.ss2d(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                       t["delta_bias"], sp)


def row_slice(spec, t, b, d):
    """Inputs of the single (b, d) row as a B=1, D=1 problem (rows are
    independent in every operation)."""
    s = {}
    for k, v in t.items():
        if not isinstance(v, torch.Tensor):
            s[k] = v
            continue
        if spec.op == "ss2d":
            if k in ("x", "z"):
                s[k] = v[b:b + 1, d:d + 1]
            elif k == "delta":
                s[k] = v[b:b + 1, :, d:d + 1]
            elif k in ("B", "C"):
                s[k] = v[b:b + 1]
            elif k == "A":
                s[k] = v[:, d:d + 1]
            else:  # D, delta_bias [K, D]
                s[k] = v[:, d:d + 1]
        else:
            if k in ("u", "u_b", "delta", "delta_b", "z"):
                s[k] = v[b:b + 1, d:d + 1]
            elif k in ("B", "C", "B_b", "C_b"):
                s[k] = v[b:b + 1]
            elif k in ("A", "A_b"):
                s[k] = v[d:d + 1]
            else:  # D, D_b, delta_bias(_b) [D]
                s[k] = v[d:d + 1]
    return s


def max_scaled_err(y_gpu, y_ref):
    y = y_gpu.detach().double().cpu().numpy() if isinstance(y_gpu, torch.Tensor) else y_gpu
    return float(np.max(np.abs(y - y_ref) / (1.0 + np.abs(y_ref)))) if y_ref.size else 0.0
