"""The C ABI: the library loads, exports every function include/ssm_scan.h
declares, and rejects bad arguments before touching the GPU.  CPU only: no
call here reaches a kernel launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssm_scan.h")


@pytest.fixture(scope="module")
def lib():
    from selective_state_space_111_b300 import build
    build.build()
    from selective_state_space_111_b300 import binding
    return binding.lib()


def declared_functions():
    src = open(HEADER).read()
    return re.findall(r"SSM_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)


def test_header_declares_the_operations():
    names = set(declared_functions())
    assert {"selective_scan_fwd", "bimamba_scan_fwd_v1", "bimamba_scan_fwd_v2", "ss2d_scan_fwd",
            "ssm_workspace_bytes", "ssm_get_status", "ssm_status_string", "ssm_version"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    for code in range(7):
        assert lib.ssm_status_string(code)
    assert re.match(rb"^\d+\.\d+\.\d+$", lib.ssm_version())


def test_workspace_bytes(lib):
    ws = lib.ssm_workspace_bytes
    hdr, bc = 256, 32 * 4          # status header; packed B/C: 32 fp32 per (batch, position)
    assert ws(0, 1, 8, 768, 6085, 16, 4) == hdr + 8 * 6085 * bc            # single
    assert ws(2, 1, 8, 768, 6085, 16, 4) == hdr + 2 * 8 * 6085 * bc + 8 * 768 * 6085 * 4
    assert ws(1, 1, 2, 1536, 4096, 16, 4) == hdr + 2 * 4096 * bc + 2 * 1536 * 4096 * 4
    assert ws(2, 1, 4, 8, 20, 16, 4) == hdr + 2 * 4 * 20 * bc     # one chunk: no stash
    n = 32 * 192 * 3136                                           # SS2D: B/C of 4 directions,
    assert ws(3, 1, 32, 192, 3136, 16, 4) == hdr + 4 * 32 * 3136 * bc + 2 * n + 2 * 4 * n  # x^T, 2 fp32
    assert ws(3, 1, 32, 192, 3136, 16, 2) == ctypes.c_size_t(-1).value
    assert ws(0, 7, 1, 1, 1, 16, 4) == ctypes.c_size_t(-1).value   # bad dtype


FAKE = 0x10000   # 16-byte aligned, never dereferenced: every call below fails validation


def single(lib, *, dt=1, B=1, D=1, L=8, N=16, u=FAKE, delta=FAKE, A=FAKE, Bm=FAKE, Cm=FAKE,
           Ds=None, z=None, bias=None, y=FAKE):
    return lib.selective_scan_fwd(dt, B, D, L, N, u, delta, A, Bm, Cm, Ds, z, bias, 1, y,
                                  None, 0, None)


def test_invalid_arguments_are_rejected_before_launch(lib):
    assert single(lib, N=33) == 2                   # N > 32: unsupported
    assert single(lib, N=32, y=None) == 1           # 32 states are supported: only y is missing
    assert single(lib, N=0) == 1
    assert single(lib, L=-1) == 1
    assert single(lib, dt=5) == 1
    assert single(lib, u=None) == 1                 # required pointer
    assert single(lib, u=FAKE + 1) == 1             # bf16 I/O tensor off its 2-byte grid
    assert single(lib, dt=0, u=FAKE + 2) == 1       # fp32 I/O tensor off its 4-byte grid
    assert single(lib, A=FAKE + 2) == 1             # misaligned fp32 parameter
    assert single(lib, y=None) == 1


def test_empty_problems_launch_nothing(lib):
    assert single(lib, B=0) == 0
    assert single(lib, D=0) == 0
    assert single(lib, L=0) == 0


def test_bidirectional_workspace_is_checked(lib):
    args = [1, 2, 16, 100, 16] + [FAKE] * 4 + [FAKE, FAKE] + [FAKE] * 4 + [None, None, None,
                                                                           None, None]
    # v2 with a multi-chunk L and no workspace
    st = lib.bimamba_scan_fwd_v2(*args, 1, ctypes.c_float(0.5), FAKE, None, 0, None)
    assert st == 4
    st = lib.bimamba_scan_fwd_v2(*args, 1, ctypes.c_float(0.5), FAKE, FAKE, 16, None)
    assert st == 4


def test_ss2d_requires_four_directions(lib):
    st = lib.ss2d_scan_fwd(1, 1, 1, 4, 4, 16, 2, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None,
                           1, FAKE, FAKE, 1 << 20, None)
    assert st == 2


# ---------------------------------------------------------------- backward
def test_header_declares_the_backward_operations():
    names = set(declared_functions())
    assert {"selective_scan_bwd", "bimamba_scan_bwd_v1", "bimamba_scan_bwd_v2", "ss2d_scan_bwd",
            "ssm_bwd_workspace_bytes"} <= names


def test_bwd_workspace_bytes(lib):
    wb = lib.ssm_bwd_workspace_bytes
    neg = ctypes.c_size_t(-1).value
    assert wb(0, 1, 0, 8, 100, 16, 4, 0) == 0                   # empty problem
    assert wb(0, 7, 1, 8, 100, 16, 4, 0) == neg                  # bad dtype
    assert wb(0, 1, 1, 8, 100, 33, 4, 0) == neg                  # N > 32
    assert wb(3, 1, 1, 8, 100, 16, 2, 0) == neg                  # SS2D needs K = 4
    single = wb(0, 1, 2, 40, 300, 16, 4, 0)
    v1, v2 = wb(1, 1, 2, 40, 300, 16, 4, 0), wb(2, 1, 2, 40, 300, 16, 4, 0)
    assert 0 < single < v1 <= v2 <= wb(2, 1, 2, 40, 300, 16, 4, 1)   # more passes, more scratch
    # at least the fp32 gradient of u, the chunk states and two partial sets
    n = 2 * 40 * 300
    assert single >= 4 * n + 2 * 40 * 10 * 16 * 4 + 2 * 3 * 2 * 300 * 16 * 4


def test_bwd_context_bytes(lib):
    # the saved backward context: the pre-gate output in the I/O dtype, then
    # per direction the fp32 states [B][D][ceil(L / 8)][16], each region
    # rounded up to 256 bytes
    cb = lib.ssm_bwd_context_bytes
    neg = ctypes.c_size_t(-1).value
    up = lambda x: (x + 255) // 256 * 256
    B, D, L = 2, 40, 301
    hc = up(B * D * ((L + 7) // 8) * 16 * 4)
    assert cb(0, 1, B, D, L, 16) == up(B * D * L * 2) + hc          # single, bf16
    assert cb(2, 0, B, D, L, 16) == up(B * D * L * 4) + 2 * hc      # v2, fp32
    assert cb(1, 2, B, D, L, 8) == up(B * D * L * 2) + 2 * hc       # v1, fp16, N < 16
    assert cb(2, 1, B, D, L, 24) == 0                                # past 16 states: none
    assert cb(2, 1, 0, D, L, 16) == 0                                # empty problem
    assert cb(3, 1, B, D, L, 16) == neg                              # SS2D keeps no context
    assert cb(2, 7, B, D, L, 16) == neg                              # bad dtype
    assert cb(2, 1, B, D, L, 33) == neg                              # N > 32
    lib.ssm_set_bwd_context(None, 0)                                 # clearing is always valid


def bwd_single(lib, *, dt=1, B=1, D=1, L=8, N=16, u=FAKE, z=None, dz=None, du=FAKE,
               ws=None, ws_bytes=0):
    return lib.selective_scan_bwd(dt, B, D, L, N, u, FAKE, FAKE, FAKE, FAKE, None, z, None, 1,
                                  FAKE, du, FAKE, FAKE, FAKE, FAKE, None, dz, None, ws,
                                  ws_bytes, None)


def test_bwd_invalid_arguments_are_rejected_before_launch(lib):
    assert bwd_single(lib, N=33) == 2
    assert bwd_single(lib, L=-1) == 1
    assert bwd_single(lib, u=None) == 1                     # required input
    assert bwd_single(lib, du=None) == 1                    # required gradient output
    assert bwd_single(lib, du=FAKE + 1) == 1                # misaligned bf16 output
    assert bwd_single(lib, z=FAKE) == 1                     # z given but no dz
    assert bwd_single(lib, z=FAKE, dz=FAKE) == 4            # no workspace
    assert bwd_single(lib, B=0) == 0                        # empty: nothing to do
    # SS2D: K != 4 unsupported
    st = lib.ss2d_scan_bwd(1, 1, 1, 2, 2, 16, 3, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None,
                           1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, None, 0, None)
    assert st == 2


def prologue(lib, *, dt=1, B=1, D=2, L=8, N=16, R=2, K=4, x=FAKE, ws=None, wsb=0):
    return lib.mamba_prologue_fwd(dt, B, D, L, N, R, K, x, FAKE, None, FAKE, FAKE, 0, FAKE,
                                  FAKE, FAKE, FAKE, ws, wsb, None)


def ss2d_prologue(lib, *, dt=1, B=1, D=2, H=3, W=4, N=16, R=2, Kc=3, x=FAKE, ws=None, wsb=0):
    return lib.ss2d_prologue_fwd(dt, B, D, H, W, N, R, Kc, x, FAKE, None, FAKE, FAKE, 1, FAKE,
                                 FAKE, FAKE, FAKE, ws, wsb, None)


def test_prologue_arguments_are_rejected_before_launch(lib):
    assert prologue(lib, K=9) == 2                  # more than 8 taps
    assert prologue(lib, N=33) == 2
    assert prologue(lib, R=0) == 1
    assert prologue(lib, x=None) == 1
    assert prologue(lib, x=FAKE + 1) == 1
    assert prologue(lib) == 4                       # no workspace
    assert prologue(lib, ws=FAKE, wsb=2 * 8 * 4 - 1) == 4
    assert prologue(lib, B=0) == 0                  # empty: nothing to launch
    assert lib.ssm_prologue_workspace_bytes(3, 10, 5) == 3 * 5 * 10 * 4


def test_ss2d_prologue_arguments_are_rejected_before_launch(lib):
    assert ss2d_prologue(lib, Kc=4) == 1            # even kernel: no centred padding
    assert ss2d_prologue(lib, Kc=9) == 2            # larger than 7
    assert ss2d_prologue(lib, N=33) == 2
    assert ss2d_prologue(lib, W=-1) == 1
    assert ss2d_prologue(lib, x=None) == 1
    assert ss2d_prologue(lib, x=FAKE + 1) == 1
    assert ss2d_prologue(lib, W=40000) == 2         # conv staging over its shared-memory bound
    assert ss2d_prologue(lib) == 4                  # no workspace
    assert ss2d_prologue(lib, ws=FAKE, wsb=4 * 2 * 12 * 4 - 1) == 4
    assert ss2d_prologue(lib, B=16384) == 2          # the (batch, direction) grid's z bound
    assert ss2d_prologue(lib, H=0) == 0
    assert lib.ss2d_prologue_workspace_bytes(2, 3, 4, 5) == 2 * 4 * 5 * 12 * 4   # four dt_low sets
