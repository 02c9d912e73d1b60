"""Saved backward context (ssm_set_bwd_context).

A forward call made while a context is set also stores its pre-gate output
and the states before every eighth step; the backward call on the same
inputs then reads them instead of running the forward pass again.  Both
calls must give exactly what the plain calls give (the same kernels, the
same arithmetic): outputs and every gradient are compared bit for bit with
the calls made without a context, whose gradients test_bwd_gpu.py checks
against the oracle (one case here checks against the oracle directly).  A
context overwritten between the two calls must change the gradients: the
backward really reads it.
"""
import numpy as np
import pytest
import torch

from cases import run_gpu
from selective_state_space_111_b300.synth import Spec, make_inputs
from test_bwd_gpu import TOL, SEQ, _dout, run_bwd_oracle

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _spec(op, io, B, D, L, N, gate=True, shared_u=True):
    return Spec(op, io, B=B, D=D, L=L, N=N, perturb=True, gate=gate, shared_u=shared_u,
                out_scale=0.5 if op == "v2" else 1.0, a_b_noise=0.1 if op == "v1" else 0.0)


def _bwd_dev(spec, t, dout):
    """The backward call's gradients as device tensors."""
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
    return r


def _same(g0, g1):
    assert set(g0) == set(g1)
    for k in g0:
        assert torch.equal(g0[k], g1[k]), k


def _with_context(spec, t, dout, poison=False):
    import selective_state_space_111_b300 as ssm
    n = ssm.bwd_context_bytes(spec.op, DT[spec.io], spec.B, spec.D, spec.L, spec.N)
    ctx = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    ssm.set_bwd_context(ctx)
    try:
        y = run_gpu(spec, t)
        if poison:
            torch.cuda.synchronize()
            ctx.zero_()
        g = _bwd_dev(spec, t, dout)
    finally:
        ssm.set_bwd_context(None)
    return y, g


# (op, io, B, D, L, N, gate, shared_u): ragged L and channel groups, the
# three forms, every dtype, no gate, separate u_b, N below 16
CASES = [("single", "bf16", 2, 24, 77, 16, True, True),
         ("single", "f32", 1, 9, 33, 7, False, True),
         ("v1", "bf16", 2, 20, 130, 16, True, True),
         ("v2", "bf16", 2, 19, 300, 16, True, True),
         ("v2", "bf16", 2, 24, 100, 16, True, False),
         ("v2", "f32", 1, 33, 65, 16, True, True),
         ("v2", "f16", 2, 16, 40, 8, True, True),
         ("v2", "bf16", 1, 40, 9, 16, False, True)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s-%s-L%d-N%d-%s" % (
    c[0], c[1], c[4], c[5], "gate" if c[6] else "nogate"))
def test_context_calls_match_plain_calls_bit_for_bit(case):
    op, io, B, D, L, N, gate, shared_u = case
    spec = _spec(op, io, B, D, L, N, gate, shared_u)
    t = make_inputs(spec, 300 + D + L)
    dout = _dout(spec, t, 7)
    y0 = run_gpu(spec, t)
    g0 = _bwd_dev(spec, t, dout)
    y1, g1 = _with_context(spec, t, dout)
    assert torch.equal(y0, y1)
    _same(g0, g1)


def test_context_gradients_match_oracle():
    spec = _spec("v2", "bf16", 2, 20, 150, 16)
    t = make_inputs(spec, 11)
    dout = _dout(spec, t, 12)
    _, gd = _with_context(spec, t, dout)
    g = {k: v.double().cpu().numpy() for k, v in gd.items()}
    ref = run_bwd_oracle(spec, t, dout)
    tol = TOL["bf16"]
    for k, r in ref.items():
        if k not in g:
            continue
        if k in SEQ:
            err = np.max(np.abs(g[k] - r) / (1.0 + np.abs(r)))
        else:
            err = np.max(np.abs(g[k] - r)) / (1.0 + np.max(np.abs(r)))
        assert err <= tol, (k, err)


@pytest.mark.parametrize("op", ["single", "v2"])
def test_backward_reads_the_context(op):
    # zeroing the context between the calls changes the gradients that
    # depend on what it holds: ddelta and dC on the states, dz on the
    # pre-gate output (du depends on neither: its adjoint recurrence never
    # reads the forward states).  Zero states and a zero pre-gate output
    # are valid values, so nothing faults.
    spec = _spec(op, "bf16", 2, 16, 90, 16)
    t = make_inputs(spec, 21)
    dout = _dout(spec, t, 22)
    g0 = _bwd_dev(spec, t, dout)
    _, g1 = _with_context(spec, t, dout, poison=True)
    for k in ("ddelta", "dC", "dz"):
        assert not torch.equal(g0[k], g1[k]), k
    assert torch.equal(g0["du"], g1["du"])


def test_context_is_ignored_past_16_states_and_for_ss2d():
    import selective_state_space_111_b300 as ssm
    assert ssm.bwd_context_bytes("v2", torch.bfloat16, 2, 16, 50, 24) == 0
    with pytest.raises(ValueError):
        ssm.bwd_context_bytes("ss2d", torch.bfloat16, 2, 16, 50, 16)
    spec = _spec("v2", "bf16", 2, 16, 50, 24)
    t = make_inputs(spec, 31)
    dout = _dout(spec, t, 32)
    y0, g0 = run_gpu(spec, t), _bwd_dev(spec, t, dout)
    y1, g1 = _with_context(spec, t, dout)
    assert torch.equal(y0, y1)
    _same(g0, g1)
    s2 = Spec("ss2d", "bf16", B=1, D=8, H=5, W=6, N=16, perturb=True)
    t2 = make_inputs(s2, 33)
    d2 = _dout(s2, t2, 34)
    ctx = torch.empty(16, dtype=torch.uint8, device="cuda")
    y0, g0 = run_gpu(s2, t2), _bwd_dev(s2, t2, d2)
    ssm.set_bwd_context(ctx)
    try:
        y1, g1 = run_gpu(s2, t2), _bwd_dev(s2, t2, d2)
    finally:
        ssm.set_bwd_context(None)
    assert torch.equal(y0, y1)
    _same(g0, g1)


def test_too_small_a_context_is_refused():
    import selective_state_space_111_b300 as ssm
    spec = _spec("v2", "bf16", 2, 16, 64, 16)
    t = make_inputs(spec, 41)
    n = ssm.bwd_context_bytes("v2", torch.bfloat16, 2, 16, 64, 16)
    ctx = torch.empty(n - 256, dtype=torch.uint8, device="cuda")
    ssm.set_bwd_context(ctx)
    try:
        with pytest.raises(ssm.SsmError) as e:
            run_gpu(spec, t)
        assert e.value.status == 4                 # SSM_ERR_WORKSPACE
    finally:
        ssm.set_bwd_context(None)


def test_context_full_size_vim_s():
    # the bench's workload: B 8, d_inner 768, L 6085, d_state 16, bf16
    spec = _spec("v2", "bf16", 8, 768, 6085, 16)
    t = make_inputs(spec, 51)
    dout = _dout(spec, t, 52)
    y0 = run_gpu(spec, t)
    g0 = _bwd_dev(spec, t, dout)
    y1, g1 = _with_context(spec, t, dout)
    assert torch.equal(y0, y1)
    _same(g0, g1)
