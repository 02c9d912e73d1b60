"""The index-checking debug build (libssm_scan_debug.so, SSM_DEBUG_BOUNDS).

In that build every global access and bulk copy of the forward path checks
its element offset against the extent of the tensor it addresses (and the
scan's shared-memory ranges against their stages); an offset outside is
recorded in the status word and the access is skipped.  It stands in for a
memory checker: these tests run the forward forms' edge cases through it --
ragged lengths, partial channel groups, batch offsets, N below 16 and the
32-state kernels, reversed-stream inputs, final states, SS2D on non-square
maps, tensors one element off a 16-byte boundary -- and require a clean
status word and the oracle's results.  A last test narrows the checked
extent with a test hook (no access leaves the real tensor) to show that a
violation is caught and reported.
"""
import ctypes

import pytest
import torch

from cases import TOL, max_scaled_err, run_gpu, run_oracle, to_dev
from selective_state_space_111_b300.synth import Spec, make_inputs

pytestmark = pytest.mark.gpu

BOUNDS = 7


@pytest.fixture(scope="module")
def dbg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_111_b300 import binding, build
    lib = binding._declare(ctypes.CDLL(build.build_debug()))
    saved = binding._lib
    binding._lib = lib                   # the binding's calls go to the debug build
    yield lib
    binding._lib = saved


def _workspace(spec, t):
    import selective_state_space_111_b300 as ssm
    key = "x" if spec.op == "ss2d" else "u"
    n = ssm.workspace_bytes(spec.op, t[key].dtype, spec.B, spec.D, spec.seq_len, spec.N,
                            spec.K)
    return torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")


# (op, io, B, D, L or (H, W), N): ragged L, partial channel groups, N < 16,
# the 32-state kernels, a one-chunk sequence, non-square and thin maps
CASES = [("single", "bf16", 2, 21, 97, 16), ("single", "f32", 1, 9, 33, 7),
         ("v1", "bf16", 3, 20, 130, 16), ("v1", "f16", 1, 40, 31, 16),
         ("v2", "bf16", 2, 19, 300, 16), ("v2", "f32", 2, 33, 65, 32),
         ("v2", "bf16", 1, 8, 20, 24),
         ("ss2d", "bf16", 2, 12, (7, 13), 16), ("ss2d", "f32", 1, 5, (1, 40), 16),
         ("ss2d", "bf16", 1, 17, (9, 4), 32)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s-%s-%s" % (c[0], c[1], c[4]))
def test_debug_build_clean_and_matches_oracle(dbg, case):
    import selective_state_space_111_b300 as ssm
    op, io, B, D, L, N = case
    kw = dict(H=L[0], W=L[1]) if op == "ss2d" else dict(L=L)
    spec = Spec(op, io, B=B, D=D, N=N, perturb=True, out_scale=0.5 if op == "v2" else 1.0,
                shared_u=(B % 2 == 0), a_b_noise=0.1, **kw)
    t = make_inputs(spec, 900 + D + N)
    ws = _workspace(spec, t)
    y = run_gpu(spec, t, workspace=ws)
    assert ssm.get_status(ws) == 0
    assert max_scaled_err(y, run_oracle(spec, t)) <= TOL[io]


@pytest.mark.parametrize("op", ["v1", "v2"])
def test_debug_build_final_states_and_scan_order(dbg, op):
    # last_state outputs, and (v2) the backward set given in walk order
    import oracle
    import selective_state_space_111_b300 as ssm
    spec = Spec(op, "bf16", B=2, D=24, L=77, perturb=True, shared_u=False, a_b_noise=0.1,
                out_scale=0.5 if op == "v2" else 1.0)
    t = make_inputs(spec, 41)
    g = to_dev(t)
    ws = _workspace(spec, t)
    ls = torch.empty(2, spec.B, spec.D, spec.N, device="cuda")
    if op == "v1":
        y = ssm.bimamba_scan_fwd_v1(g["u"], g["delta"], g["A"], g["A_b"], g["B"], g["C"], g["D"],
                                    g["z"], g["delta_bias"], True, 1.0, workspace=ws,
                                    last_state=ls)
        ref_ls = oracle.bimamba_v1_last_state(t["u"], t["delta"], t["A"], t["A_b"], t["B"],
                                              t["C"], t["D"], t["z"], t["delta_bias"], True, 1.0)
    else:
        rev = lambda k: torch.flip(g[k], [-1]).contiguous()
        y = ssm.bimamba_scan_fwd_v2(g["u"], g["delta"], rev("delta_b"), g["A"], g["A_b"], g["B"],
                                    g["C"], rev("B_b"), rev("C_b"), g["D"], g["D_b"], g["z"],
                                    g["delta_bias"], g["delta_bias_b"], rev("u_b"), True, 0.5,
                                    workspace=ws, last_state=ls, scan_order=True)
        ref_ls = oracle.bimamba_v2_last_state(t["u"], t["delta"], t["delta_b"], t["A"], t["A_b"],
                                              t["B"], t["C"], t["B_b"], t["C_b"], t["D"],
                                              t["D_b"], t["z"], t["delta_bias"],
                                              t["delta_bias_b"], t["u_b"], True, 0.5)
    torch.cuda.synchronize()
    assert ssm.get_status(ws) == 0
    assert max_scaled_err(y, run_oracle(spec, t)) <= TOL["bf16"]
    assert max_scaled_err(ls, ref_ls) <= 1e-3


def test_debug_build_unaligned_tensors(dbg):
    # every I/O tensor one element past a 16-byte boundary
    import selective_state_space_111_b300 as ssm
    spec = Spec("v2", "bf16", B=2, D=18, L=101, perturb=True, out_scale=0.5)
    t = make_inputs(spec, 43)

    def shifted(v):
        if not isinstance(v, torch.Tensor):
            return v
        buf = torch.empty(v.numel() + 1, dtype=v.dtype, device="cuda")[1:]
        return buf.view(v.shape).copy_(v.cuda())
    g = {k: shifted(v) for k, v in t.items()}
    assert g["u"].data_ptr() % 16 != 0
    ws = _workspace(spec, t)
    out = shifted(torch.empty_like(t["u"]))
    y = run_gpu(spec, t, workspace=ws, dev=g, out=out)
    assert ssm.get_status(ws) == 0
    assert max_scaled_err(y, run_oracle(spec, t)) <= TOL["bf16"]


def test_debug_build_reports_a_narrowed_extent(dbg):
    # the hook narrows the [B, D, L] extent the next launch checks against
    # by one row: the accesses to the last row are caught, skipped and
    # reported; the next call (hook cleared) is clean again
    import selective_state_space_111_b300 as ssm
    spec = Spec("v2", "bf16", B=2, D=16, L=90, perturb=True, out_scale=0.5)
    t = make_inputs(spec, 44)
    ws = _workspace(spec, t)
    dbg.ssm_test_shrink_extents(spec.L)
    run_gpu(spec, t, workspace=ws)
    assert ssm.get_status(ws) == BOUNDS
    assert b"debug build" in dbg.ssm_status_string(BOUNDS)
    y = run_gpu(spec, t, workspace=ws)
    assert ssm.get_status(ws) == 0
    assert max_scaled_err(y, run_oracle(spec, t)) <= TOL["bf16"]
