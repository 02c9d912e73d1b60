"""GPU parity of the backward pass: the CUDA library against the fp64
oracle's backward (itself pinned by finite differences of the forward
oracle), on the same seeded inputs and the same incoming gradient.

Tolerances.  Per-position gradients (du, ddelta, dz, dx) element by element:
|gpu - ref| <= tol * (1 + |ref|).  Gradients that are sums over many rows
and positions (dA, dD, ddelta_bias, and dB, dC, summed over channels) are
compared against their own scale: max|gpu - ref| <= tol * (1 + max|ref|),
because fp32 summation of thousands of terms of both signs leaves an
absolute error proportional to the terms' size, not to the (possibly
cancelling) result.  tol = 2e-4 for fp32 I/O, 2e-2 for bf16 I/O and 1e-2
for fp16 I/O (outputs rounded to the 16-bit type, inputs and the recomputed
pre-gate output in it).
"""
import numpy as np
import pytest
import torch

import oracle
from cases import row_slice
from selective_state_space_111_b300.synth import WORKLOADS, Spec, make_inputs, seed_for

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-4, "bf16": 2e-2, "f16": 1e-2}
SEQ = {"du", "du_b", "ddelta", "ddelta_b", "dz", "dx"}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_111_b300 import build
    build.build()


def _dout(spec, t, seed):
    shape = t["x" if spec.op == "ss2d" else "u"].shape
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(t["x" if spec.op == "ss2d" else "u"].dtype)


def run_bwd_gpu(spec, t, dout):
    import selective_state_space_111_b300 as ssm
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    go = dout.cuda()
    sp = spec.delta_softplus
    if spec.op == "single":
        r = ssm.selective_scan_bwd(go, g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], sp)
    elif spec.op == "v1":
        r = ssm.bimamba_scan_bwd_v1(go, g["u"], g["delta"], g["A"], g["A_b"], g["B"], g["C"],
                                    g["D"], g["z"], g["delta_bias"], sp, g["out_scale"])
    elif spec.op == "v2":
        r = ssm.bimamba_scan_bwd_v2(go, g["u"], g["delta"], g["delta_b"], g["A"], g["A_b"],
                                    g["B"], g["C"], g["B_b"], g["C_b"], g["D"], g["D_b"], g["z"],
                                    g["delta_bias"], g["delta_bias_b"], g["u_b"], sp,
                                    g["out_scale"])
    else:
        r = ssm.ss2d_scan_bwd(go, g["x"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                              g["delta_bias"], sp)
    torch.cuda.synchronize()
    return {k: v.double().cpu().numpy() for k, v in r.items()}


def run_bwd_oracle(spec, t, dout):
    sp = spec.delta_softplus
    if spec.op == "single":
        return oracle.selective_scan_bwd(dout, t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"],
                                         t["z"], t["delta_bias"], sp)
    if spec.op == "v1":
        return oracle.bimamba_v1_bwd(dout, t["u"], t["delta"], t["A"], t["A_b"], t["B"], t["C"],
                                     t["D"], t["z"], t["delta_bias"], sp, t["out_scale"])
    if spec.op == "v2":
        return oracle.bimamba_v2_bwd(dout, t["u"], t["delta"], t["delta_b"], t["A"], t["A_b"],
                                     t["B"], t["C"], t["B_b"], t["C_b"], t["D"], t["D_b"], t["z"],
                                     t["delta_bias"], t["delta_bias_b"], t["u_b"], sp,
                                     t["out_scale"])
    return oracle.ss2d_bwd(dout, t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                           t["delta_bias"], sp)


def compare(gpu, ref, io, keys=None):
    assert set(gpu) == set(ref), (sorted(gpu), sorted(ref))
    tol = TOL[io]
    worst = {}
    for k in (keys or ref):
        a, r = gpu[k], ref[k]
        assert a.shape == r.shape, k
        if k in SEQ:
            err = float(np.max(np.abs(a - r) / (1.0 + np.abs(r)))) if r.size else 0.0
        else:
            err = float(np.max(np.abs(a - r)) / (1.0 + np.max(np.abs(r)))) if r.size else 0.0
        worst[k] = err
        assert np.isfinite(err) and err <= tol, "%s: %.3g > %g" % (k, err, tol)
    return worst


def check(spec, seed):
    t = make_inputs(spec, seed)
    dout = _dout(spec, t, seed + 1)
    return compare(run_bwd_gpu(spec, t, dout), run_bwd_oracle(spec, t, dout), spec.io)


SHAPES = [(1, 1, 1, 16), (2, 3, 33, 16), (1, 17, 64, 16), (2, 20, 97, 16), (1, 9, 40, 7),
          (2, 4, 129, 1), (2, 11, 70, 32), (1, 9, 40, 24)]   # d_state 32 and 17..32


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_single_bwd(io, shape):
    B, D, L, N = shape
    check(Spec("single", io, B=B, D=D, L=L, N=N, perturb=True), 5000 + L)


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_v1_bwd(io, shape):
    B, D, L, N = shape
    check(Spec("v1", io, B=B, D=D, L=L, N=N, perturb=True, a_b_noise=0.1, out_scale=1.0),
          6000 + L)


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("shared_u", [True, False])
def test_v2_bwd(io, shape, shared_u):
    B, D, L, N = shape
    check(Spec("v2", io, B=B, D=D, L=L, N=N, perturb=True, shared_u=shared_u, out_scale=0.5),
          7000 + L)


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (1, 2, 2, 3), (2, 3, 5, 7), (1, 17, 8, 8),
                                   (1, 4, 11, 3)])
def test_ss2d_bwd(io, shape):
    B, D, H, W = shape
    check(Spec("ss2d", io, B=B, D=D, H=H, W=W, perturb=True), 8000 + H * W)


def test_ss2d_bwd_d_state_32():
    check(Spec("ss2d", "f32", B=1, D=10, H=5, W=7, N=32, perturb=True), 8600)


@pytest.mark.parametrize("op", ["single", "v1", "v2", "ss2d"])
def test_bwd_optional_inputs_absent(op):
    # no gate, no skip, no bias, no softplus: those gradients are absent
    kw = dict(H=5, W=6) if op == "ss2d" else dict(L=77)
    spec = Spec(op, "f32", B=2, D=18, gate=False, delta_softplus=False, **kw)
    t = make_inputs(spec, 77)
    t["delta"] = t["delta"].abs() * 0.05 + 0.01
    if op == "v2":
        t["delta_b"] = t["delta_b"].abs() * 0.05 + 0.01
    for k in ("D", "D_b", "delta_bias", "delta_bias_b"):
        if k in t:
            t[k] = None
    dout = _dout(spec, t, 78)
    gpu = run_bwd_gpu(spec, t, dout)
    assert "dz" not in gpu and "dD" not in gpu and "ddelta_bias" not in gpu
    compare(gpu, run_bwd_oracle(spec, t, dout), "f32")


def test_bwd_deterministic():
    spec = Spec("v2", "bf16", B=2, D=40, L=150, perturb=True, out_scale=0.5)
    t = make_inputs(spec, 3)
    dout = _dout(spec, t, 4)
    a = run_bwd_gpu(spec, t, dout)
    b = run_bwd_gpu(spec, t, dout)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("name,nrows", [("vim_ti_224_bimamba_v2", 24),
                                        ("vim_s_1248_bimamba_v2", 12)])
def test_bwd_workload_sampled_rows(name, nrows):
    # full-size launch; the per-position gradients of a row depend on that
    # row (and its batch element's B, C) only, so the oracle recomputes
    # sampled rows one by one
    spec = WORKLOADS[name]
    seed = seed_for(name)
    t = make_inputs(spec, seed)
    dout = _dout(spec, t, seed + 1)
    gpu = run_bwd_gpu(spec, t, dout)
    rng = np.random.default_rng(seed)
    rows = {(0, 0), (spec.B - 1, spec.D - 1)}
    while len(rows) < nrows:
        rows.add((int(rng.integers(spec.B)), int(rng.integers(spec.D))))
    for b, d in sorted(rows):
        ts = row_slice(spec, t, b, d)
        ref = run_bwd_oracle(spec, ts, dout[b:b + 1, d:d + 1])
        sub = {k: gpu[k][b:b + 1, d:d + 1] for k in ("du", "ddelta", "ddelta_b", "dz")}
        compare(sub, {k: ref[k] for k in sub}, spec.io)


def _channel_rows(spec, t, d):
    """Inputs of every batch element's rows of channel d (B x 1 rows, B/C
    whole): the parameter gradients of channel d sum over exactly these."""
    s = {}
    for k, v in t.items():
        if not isinstance(v, torch.Tensor):
            s[k] = v
        elif k in ("u", "u_b", "delta", "delta_b", "z"):
            s[k] = v[:, d:d + 1]
        elif k in ("A", "A_b", "D", "D_b", "delta_bias", "delta_bias_b"):
            s[k] = v[d:d + 1]
        else:
            s[k] = v
    return s


def _batch_rows(spec, t, b):
    """Inputs of batch element b (all channels): dB and dC of b sum over
    exactly these rows."""
    return {k: (v[b:b + 1] if isinstance(v, torch.Tensor) and
                k in ("u", "u_b", "delta", "delta_b", "z", "B", "C", "B_b", "C_b") else v)
            for k, v in t.items()}


@pytest.mark.slow
def test_bwd_workload_parameter_gradients():
    # Vim-S 1248^2 v2 at full size: dA, dD and ddelta_bias of sampled
    # channels (each a sum over that channel's rows of every batch element)
    # and dB, dC of the last batch element (a sum over its 768 channels),
    # each against the oracle run on exactly the rows it sums over
    name = "vim_s_1248_bimamba_v2"
    spec = WORKLOADS[name]
    seed = seed_for(name)
    t = make_inputs(spec, seed)
    dout = _dout(spec, t, seed + 1)
    gpu = run_bwd_gpu(spec, t, dout)
    rng = np.random.default_rng(seed + 2)
    chans = sorted({0, spec.D - 1, *[int(c) for c in rng.integers(spec.D, size=4)]})
    per_channel = ("dA", "dA_b", "dD", "dD_b", "ddelta_bias", "ddelta_bias_b")
    for d in chans:
        ref = run_bwd_oracle(spec, _channel_rows(spec, t, d), dout[:, d:d + 1])
        compare({k: gpu[k][d:d + 1] for k in per_channel}, {k: ref[k] for k in per_channel},
                spec.io)
    b = spec.B - 1
    ref = run_bwd_oracle(spec, _batch_rows(spec, t, b), dout[b:b + 1])
    per_batch = ("dB", "dC", "dB_b", "dC_b")
    compare({k: gpu[k][b:b + 1] for k in per_batch}, {k: ref[k] for k in per_batch}, spec.io)
