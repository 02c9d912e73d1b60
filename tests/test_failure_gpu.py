"""Failure detection without a GPU fault: every wait in the scan kernel is
bounded.  The test hook ssm_test_withhold_copy makes the kernel skip one
chunk's B/C bulk copy, so the scan's wait for it runs out; the kernel must
stop, set the workspace status word, and leave the context usable.  The
allocation-free entry point runs the same kernel on its fixed scratch: its
status word is not observable, but the call must return and the next call
must run normally."""
import numpy as np
import pytest
import torch

from cases import TOL, max_scaled_err, run_oracle, to_dev
from selective_state_space_111_b300.synth import Spec, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_111_b300 import build
    build.build()
    import selective_state_space_111_b300 as m
    return m


def _v2(ssm, g, ws):
    return ssm.bimamba_scan_fwd_v2(g["u"], g["delta"], g["delta_b"], g["A"], g["A_b"], g["B"],
                                   g["C"], g["B_b"], g["C_b"], g["D"], g["D_b"], g["z"],
                                   g["delta_bias"], g["delta_bias_b"], g["u_b"], True, 0.5,
                                   workspace=ws)


def test_withheld_copy_times_out_and_context_stays_usable(ssm):
    from selective_state_space_111_b300 import binding
    spec = Spec("v2", "bf16", B=1, D=16, L=300, perturb=True, out_scale=0.5)
    t = make_inputs(spec, 31)
    g = to_dev(t)
    n = ssm.workspace_bytes("v2", torch.bfloat16, 1, 16, 300, 16)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    binding.lib().ssm_test_withhold_copy(3)            # chunk 3 of 10 never arrives
    _v2(ssm, g, ws)
    assert ssm.get_status(ws) == 6                      # SSM_ERR_TIMEOUT
    # the next call (hook cleared) runs normally and is correct
    y = _v2(ssm, g, ws)
    assert ssm.get_status(ws) == 0
    ref = run_oracle(spec, t)
    assert max_scaled_err(y, ref) <= TOL["bf16"]
    assert torch.cuda.is_available() and np.isfinite(y.float().sum().item())


def test_withheld_copy_in_allocation_free_call_returns(ssm):
    import ctypes
    from selective_state_space_111_b300 import binding
    lib = binding.lib()
    spec = Spec("v2", "bf16", B=1, D=16, L=300, perturb=True, out_scale=0.5)
    t = make_inputs(spec, 32)
    g = to_dev(t)
    stream = torch.cuda.current_stream().cuda_stream

    def call(y):
        p = lambda v: None if v is None else v.data_ptr()
        return lib.bimamba_scan_fwd_v2_noalloc(
            1, 1, 16, 300, 16, p(g["u"]), p(g["u_b"]), p(g["delta"]), p(g["delta_b"]),
            p(g["A"]), p(g["A_b"]), p(g["B"]), p(g["C"]), p(g["B_b"]), p(g["C_b"]), p(g["D"]),
            p(g["D_b"]), p(g["z"]), p(g["delta_bias"]), p(g["delta_bias_b"]), 1,
            ctypes.c_float(0.5), y.data_ptr(), stream)

    lib.ssm_test_withhold_copy(3)                       # chunk 3 of 10 never arrives
    y = torch.empty_like(g["u"])
    assert call(y) == 0
    torch.cuda.synchronize()                            # returns: the waits are bounded
    y = torch.empty_like(g["u"])
    assert call(y) == 0                                 # hook cleared: a normal call
    torch.cuda.synchronize()
    assert max_scaled_err(y, run_oracle(spec, t)) <= TOL["bf16"]
