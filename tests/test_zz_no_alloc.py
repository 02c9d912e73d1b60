"""The allocation-free BiMamba v2 entry point (bimamba_scan_fwd_v2_noalloc).

Some callers cannot allocate device memory: a plugin inside a host framework
that owns the allocator and hands it only input and output buffers, or
real-time code that must not call cudaMalloc once running.  For them the
library offers a variant of bimamba_scan_fwd_v2 whose scratch is a fixed
array inside the library instead of a caller workspace.  These tests check,
through the C ABI, that it gives bit for bit the output of the regular entry
point (both launch the same kernels on the same inputs) on two calls in a
row -- the larger problem first, so that every scratch slot the second call
reads holds the first call's leftovers -- and that a problem too large for
the array is refused before anything runs, after the argument checks.

This file sorts last so that a run stopping at its first failure has run
every other test already; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

from cases import to_dev
from selective_state_space_111_b300.synth import Spec, make_inputs

SCRATCH_BYTES = 64 << 20
SCRATCH_LIMIT = 5
INVALID_ARG = 1


@pytest.fixture(scope="module")
def lib():
    from selective_state_space_111_b300 import build
    build.build()
    from selective_state_space_111_b300 import binding
    return binding.lib()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _call_noalloc(lib, g, y, stream):
    Bt, Dc, L = g["u"].shape
    N = g["A"].shape[1]
    code = 0 if g["u"].dtype == torch.float32 else 1
    return lib.bimamba_scan_fwd_v2_noalloc(
        code, Bt, Dc, L, N, _ptr(g["u"]), _ptr(g["u_b"]), _ptr(g["delta"]), _ptr(g["delta_b"]),
        _ptr(g["A"]), _ptr(g["A_b"]), _ptr(g["B"]), _ptr(g["C"]), _ptr(g["B_b"]),
        _ptr(g["C_b"]), _ptr(g["D"]), _ptr(g["D_b"]), _ptr(g["z"]), _ptr(g["delta_bias"]),
        _ptr(g["delta_bias_b"]), 1, ctypes.c_float(g["out_scale"]), y.data_ptr(), stream)


def _call_workspace(lib, g, y, ws, stream):
    Bt, Dc, L = g["u"].shape
    N = g["A"].shape[1]
    code = 0 if g["u"].dtype == torch.float32 else 1
    return lib.bimamba_scan_fwd_v2(
        code, Bt, Dc, L, N, _ptr(g["u"]), _ptr(g["u_b"]), _ptr(g["delta"]), _ptr(g["delta_b"]),
        _ptr(g["A"]), _ptr(g["A_b"]), _ptr(g["B"]), _ptr(g["C"]), _ptr(g["B_b"]),
        _ptr(g["C_b"]), _ptr(g["D"]), _ptr(g["D_b"]), _ptr(g["z"]), _ptr(g["delta_bias"]),
        _ptr(g["delta_bias_b"]), 1, ctypes.c_float(g["out_scale"]), y.data_ptr(),
        ws.data_ptr(), ws.numel(), stream)


@pytest.mark.gpu
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(lib, io):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    stream = torch.cuda.current_stream().cuda_stream
    # Two different problems in a row; both span many time chunks, so both
    # go through the scratch array (packed B/C and the stash), and the
    # second, smaller one finds the first one's leftovers in every slot it
    # reads.
    for k, (B, D, L) in enumerate([(3, 24, 517), (2, 40, 300)]):
        spec = Spec("v2", io, B=B, D=D, L=L, perturb=True, shared_u=(k == 0), out_scale=0.5)
        g = to_dev(make_inputs(spec, 7100 + k))
        y_ref = torch.empty_like(g["u"])
        need = lib.ssm_workspace_bytes(2, 0 if io == "f32" else 1, B, D, L, 16, 4)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        assert _call_workspace(lib, g, y_ref, ws, stream) == 0
        y = torch.full_like(g["u"], float("nan"))
        assert _call_noalloc(lib, g, y, stream) == 0
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref), "call %d: outputs differ" % k
        assert bool(torch.isfinite(y).all())


FAKE = 0x10000   # 16-byte aligned, never dereferenced: the call is refused first


def test_noalloc_refuses_problems_beyond_its_scratch(lib):
    # the stash alone (B * D * L fp32) is beyond 64 MiB
    B, D, L = 1, 1, SCRATCH_BYTES // 4 + 1
    st = lib.bimamba_scan_fwd_v2_noalloc(1, B, D, L, 16, FAKE, None, FAKE, FAKE, FAKE, FAKE,
                                         FAKE, FAKE, FAKE, FAKE, None, None, None, None, None,
                                         1, ctypes.c_float(0.5), FAKE, None)
    assert st == SCRATCH_LIMIT
    assert b"64 MiB" in lib.ssm_status_string(SCRATCH_LIMIT)
    # a missing required pointer is an argument error, whatever the size
    st = lib.bimamba_scan_fwd_v2_noalloc(1, B, D, L, 16, None, None, FAKE, FAKE, FAKE, FAKE,
                                         FAKE, FAKE, FAKE, FAKE, None, None, None, None, None,
                                         1, ctypes.c_float(0.5), FAKE, None)
    assert st == INVALID_ARG
