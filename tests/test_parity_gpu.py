"""GPU parity: the CUDA library against the fp64 oracle, element by element,
on the same seeded inputs (tolerance |gpu - oracle| <= tol * (1 + |oracle|),
tol = 1e-4 for fp32 I/O, 1e-2 for bf16 I/O and 2e-3 for fp16 I/O)."""
import numpy as np
import pytest
import torch

from cases import TOL, max_scaled_err, row_slice, run_gpu, run_oracle
from selective_state_space_111_b300.synth import WORKLOADS, Spec, make_inputs, seed_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_111_b300 import build
    build.build()


def check(spec, seed, ref=None):
    t = make_inputs(spec, seed)
    y = run_gpu(spec, t)
    torch.cuda.synchronize()
    if ref is None:
        ref = run_oracle(spec, t)
    err = max_scaled_err(y, ref)
    assert np.isfinite(err) and err <= TOL[spec.io], "%s: max scaled error %.3g" % (spec, err)
    return y, err


# ------------------------------------------------------------ small shapes
# L spans: shorter than a chunk, one chunk, chunk +- 1, several chunks with a
# ragged tail; D spans partial CTAs; N < 16 exercises the state mask.
SHAPES = [(1, 1, 1, 16), (2, 3, 5, 16), (1, 17, 31, 16), (2, 16, 32, 16), (1, 5, 33, 16),
          (3, 20, 97, 16), (2, 40, 197, 16), (1, 9, 64, 7), (2, 4, 129, 1), (1, 33, 300, 16),
          (2, 19, 77, 32), (1, 9, 40, 24)]   # d_state 32 and a 17..32 size


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_single(io, shape):
    B, D, L, N = shape
    check(Spec("single", io, B=B, D=D, L=L, N=N, perturb=True), 1000 + L)


@pytest.fixture(params=[8, 16], ids=["cta8", "cta16"])
def cta(request):
    """Both CTA shapes of the two-branch kernels (8 or 16 channels)."""
    import selective_state_space_111_b300 as ssm
    ssm.set_cta_channels(request.param)
    yield request.param
    ssm.set_cta_channels(0)


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_v1(io, shape, cta):
    B, D, L, N = shape
    check(Spec("v1", io, B=B, D=D, L=L, N=N, perturb=True, a_b_noise=0.1, out_scale=1.0), 2000 + L)


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("shared_u", [True, False])
def test_v2(io, shape, shared_u, cta):
    B, D, L, N = shape
    check(Spec("v2", io, B=B, D=D, L=L, N=N, perturb=True, shared_u=shared_u, out_scale=0.5),
          3000 + L)


# the last two maps are too large for the whole-map transpose (> 48 KB of
# shared memory as fp32), so they take the tiled one
SS2D_SHAPES = [(1, 1, 1, 1), (1, 2, 2, 3), (2, 3, 5, 7), (1, 17, 8, 8), (2, 5, 3, 11),
               (1, 4, 11, 3), (1, 16, 14, 14), (1, 3, 56, 56), (1, 2, 120, 112),
               (1, 1, 9, 1500)]


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", SS2D_SHAPES)
def test_ss2d(io, shape, cta):
    B, D, H, W = shape
    check(Spec("ss2d", io, B=B, D=D, H=H, W=W, perturb=True), 4000 + H * W)


@pytest.mark.parametrize("op", ["single", "v1", "v2", "ss2d"])
def test_d_state_32(op, cta):
    # 32 states (the pages recommend 16-32): the 32-state kernels
    kw = dict(H=7, W=9) if op == "ss2d" else dict(L=150)
    check(Spec(op, "bf16", B=2, D=24, N=32, perturb=True,
               out_scale=0.5 if op == "v2" else 1.0, **kw), 4500)


# ------------------------------------------------------------ options
@pytest.mark.parametrize("op", ["single", "v1", "v2", "ss2d"])
def test_optional_inputs_absent(op):
    # no gate, no skip, no bias, no softplus (delta used as given)
    kw = dict(H=5, W=6) if op == "ss2d" else dict(L=77)
    spec = Spec(op, "f32", B=2, D=18, gate=False, delta_softplus=False, **kw)
    t = make_inputs(spec, 77)
    t["delta"] = t["delta"].abs() * 0.05           # keep delta positive
    if op == "v2":
        t["delta_b"] = t["delta_b"].abs() * 0.05
    for k in ("D", "D_b", "delta_bias", "delta_bias_b"):
        if k in t:
            t[k] = None
    y = run_gpu(spec, t)
    ref = run_oracle(spec, t)
    assert max_scaled_err(y, ref) <= TOL["f32"]


def test_deterministic_and_workspace_contents_irrelevant():
    spec = Spec("v2", "bf16", B=2, D=24, L=150, perturb=True, out_scale=0.5)
    t = make_inputs(spec, 5)
    from selective_state_space_111_b300 import workspace_bytes
    n = workspace_bytes("v2", torch.bfloat16, 2, 24, 150, 16)
    ws1 = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")   # NaN patterns
    ws2 = torch.zeros((n,), dtype=torch.uint8, device="cuda")
    y1 = run_gpu(spec, t, workspace=ws1)
    y2 = run_gpu(spec, t, workspace=ws2)
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("op", ["v1", "v2", "ss2d"])
def test_cta_shape_does_not_change_results(op):
    # the two CTA shapes run the same arithmetic per row: identical bits
    import selective_state_space_111_b300 as ssm
    kw = dict(H=9, W=13) if op == "ss2d" else dict(L=300)
    spec = Spec(op, "bf16", B=3, D=40, perturb=True, out_scale=0.5 if op == "v2" else 1.0, **kw)
    t = make_inputs(spec, 12)
    try:
        ssm.set_cta_channels(8)
        y8 = run_gpu(spec, t)
        ssm.set_cta_channels(16)
        y16 = run_gpu(spec, t)
    finally:
        ssm.set_cta_channels(0)
    assert torch.equal(y8, y16)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["single", "v1", "v2", "ss2d"])
def test_last_state(op, io, cta):
    # the final state of every direction against the oracle's; y unchanged
    import oracle
    import selective_state_space_111_b300 as ssm
    kw = dict(H=6, W=9) if op == "ss2d" else dict(L=133)
    spec = Spec(op, io, B=2, D=21, perturb=True, out_scale=0.5 if op == "v2" else 1.0, **kw)
    t = make_inputs(spec, 21)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    ndir = {"single": 1, "v1": 2, "v2": 2, "ss2d": 4}[op]
    ls = torch.full((ndir, 2, 21, 16), float("nan"), device="cuda")
    sp = spec.delta_softplus
    if op == "single":
        y = ssm.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], sp, last_state=ls)
        ref = oracle.selective_scan_last_state(t["u"], t["delta"], t["A"], t["B"],
                                               delta_bias=t["delta_bias"])
    elif op == "v1":
        y = ssm.bimamba_scan_fwd_v1(g["u"], g["delta"], g["A"], g["A_b"], g["B"], g["C"], g["D"],
                                    g["z"], g["delta_bias"], sp, 1.0, last_state=ls)
        ref = oracle.bimamba_v1_last_state(t["u"], t["delta"], t["A"], t["A_b"], t["B"], t["C"],
                                           delta_bias=t["delta_bias"])
    elif op == "v2":
        y = ssm.bimamba_scan_fwd_v2(g["u"], g["delta"], g["delta_b"], g["A"], g["A_b"], g["B"],
                                    g["C"], g["B_b"], g["C_b"], g["D"], g["D_b"], g["z"],
                                    g["delta_bias"], g["delta_bias_b"], g["u_b"], sp, 0.5,
                                    last_state=ls)
        ref = oracle.bimamba_v2_last_state(t["u"], t["delta"], t["delta_b"], t["A"], t["A_b"],
                                           t["B"], t["C"], t["B_b"], t["C_b"],
                                           delta_bias=t["delta_bias"],
                                           delta_bias_b=t["delta_bias_b"], u_b=t["u_b"])
    else:
        y = ssm.ss2d_scan_fwd(g["x"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                              g["delta_bias"], sp, last_state=ls)
        ref = oracle.ss2d_last_state(t["x"], t["delta"], t["A"], t["B"], t["C"],
                                     delta_bias=t["delta_bias"])
    torch.cuda.synchronize()
    assert max_scaled_err(ls, ref) <= TOL["f32"] * 10    # fp32 state, inputs as rounded
    assert max_scaled_err(y, run_oracle(spec, t)) <= TOL[io]


@pytest.mark.parametrize("shared_u", [True, False])
def test_v2_scan_order_inputs(shared_u, cta):
    # the backward set given time-reversed gives the same y (and states)
    import selective_state_space_111_b300 as ssm
    spec = Spec("v2", "bf16", B=2, D=21, L=133, perturb=True, shared_u=shared_u, out_scale=0.5)
    t = make_inputs(spec, 31)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    fl = {k: (torch.flip(g[k], dims=[-1]) if g[k] is not None else None)
          for k in ("delta_b", "B_b", "C_b", "u_b")}
    ls1 = torch.empty(2, 2, 21, 16, device="cuda")
    ls2 = torch.empty_like(ls1)
    y1 = ssm.bimamba_scan_fwd_v2(g["u"], g["delta"], g["delta_b"], g["A"], g["A_b"], g["B"],
                                 g["C"], g["B_b"], g["C_b"], g["D"], g["D_b"], g["z"],
                                 g["delta_bias"], g["delta_bias_b"], g["u_b"], True, 0.5,
                                 last_state=ls1)
    y2 = ssm.bimamba_scan_fwd_v2(g["u"], g["delta"], fl["delta_b"], g["A"], g["A_b"], g["B"],
                                 g["C"], fl["B_b"], fl["C_b"], g["D"], g["D_b"], g["z"],
                                 g["delta_bias"], g["delta_bias_b"], fl["u_b"], True, 0.5,
                                 last_state=ls2, scan_order=True)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)          # same arithmetic in the same order
    assert torch.equal(ls1, ls2)
    assert max_scaled_err(y2, run_oracle(spec, t)) <= TOL["bf16"]


def test_length_one_branches_agree():
    # With L = 1 and identical parameter sets the two branches coincide, so
    # v2 with out_scale 0.5 equals the single-direction scan.
    spec = Spec("v2", "f32", B=2, D=8, L=1, out_scale=0.5)
    t = make_inputs(spec, 9)
    for a, b in (("delta_b", "delta"), ("A_b", "A"), ("B_b", "B"), ("C_b", "C"), ("D_b", "D"),
                 ("delta_bias_b", "delta_bias")):
        t[a] = t[b].clone()
    y2 = run_gpu(spec, t)
    ys = run_gpu(Spec("single", "f32", B=2, D=8, L=1), t)
    assert torch.allclose(y2, ys, rtol=1e-6, atol=1e-6)


def _at_offset(v, k):
    """A contiguous device copy of `v` that starts k elements into a larger
    buffer (so off every vector boundary for odd k)."""
    buf = torch.zeros(v.numel() + k, dtype=v.dtype, device="cuda")
    w = buf[k:].view(v.shape)
    w.copy_(v)
    return w


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["single", "v1", "v2", "ss2d"])
def test_unaligned_io_tensors(op, io, cta):
    # every I/O tensor and the output start one element past a 16-byte
    # boundary; rows of odd length then start anywhere
    kw = dict(H=7, W=9) if op == "ss2d" else dict(L=101)
    spec = Spec(op, io, B=2, D=19, perturb=True, out_scale=0.5 if op == "v2" else 1.0, **kw)
    t = make_inputs(spec, 31)
    g = {k: (_at_offset(v.cuda(), 1) if isinstance(v, torch.Tensor) else v)
         for k, v in t.items()}
    shape = t["x" if op == "ss2d" else "u"].shape
    out = _at_offset(torch.zeros(shape, dtype=g["delta"].dtype, device="cuda"), 1)
    y = run_gpu(spec, t, dev=g, out=out)
    torch.cuda.synchronize()
    assert y.data_ptr() % 16 != 0 and g["delta"].data_ptr() % 16 != 0
    err = max_scaled_err(y, run_oracle(spec, t))
    assert err <= TOL[io], err


# ------------------------------------------------------------ the pages' workloads
def _sampled_rows(spec, seed, nrows):
    """Full-size launch; the oracle recomputes a seeded sample of whole rows."""
    t = make_inputs(spec, seed)
    y = run_gpu(spec, t).cpu()
    rng = np.random.default_rng(seed)
    rows = {(0, 0), (spec.B - 1, spec.D - 1)}
    while len(rows) < nrows:
        rows.add((int(rng.integers(spec.B)), int(rng.integers(spec.D))))
    worst = 0.0
    for b, d in sorted(rows):
        ref = run_oracle(spec, row_slice(spec, t, b, d))
        worst = max(worst, max_scaled_err(y[b:b + 1, d:d + 1], ref))
    assert worst <= TOL[spec.io], "%s: worst sampled row error %.3g" % (spec.name, worst)
    return worst


def test_workload_vim_ti_224_single_f32_full():
    name = "vim_ti_224_single_f32"
    check(WORKLOADS[name], seed_for(name))


def test_workload_vim_ti_224_bimamba_v2():
    name = "vim_ti_224_bimamba_v2"
    _sampled_rows(WORKLOADS[name], seed_for(name), 64)


def test_workload_vim_s_1248_bimamba_v2():
    name = "vim_s_1248_bimamba_v2"
    _sampled_rows(WORKLOADS[name], seed_for(name), 64)


def test_workload_vmamba_56x56_ss2d():
    name = "vmamba_56x56_ss2d"
    _sampled_rows(WORKLOADS[name], seed_for(name), 48)


@pytest.mark.parametrize("L", [4096, 16384, 65536])
def test_workload_bimamba_v1_long(L):
    name = "bimamba_v1_L%d" % L
    _sampled_rows(WORKLOADS[name], seed_for(name), 16 if L > 16384 else 32)


@pytest.mark.slow
def test_workload_bimamba_v1_L262144():
    name = "bimamba_v1_L262144"
    _sampled_rows(WORKLOADS[name], seed_for(name), 8)
