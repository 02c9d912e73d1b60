"""Failure detection without a GPU fault: every wait in the scan kernel is
bounded.  The test hook ssm_test_withhold_copy makes the kernel skip one
chunk's B/C bulk copy, so the scan's wait for it runs out; the kernel must
stop, set the workspace status word, and leave the context usable."""
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
