"""Thin Python binding of the C ABI in include/ssm_scan.h (ctypes).

Argument marshalling only: every function checks that the tensors are CUDA,
contiguous and of the right dtype, passes their device pointers and the
current CUDA stream to the library, and raises SsmError on a non-zero status.
PyTorch supplies the device memory (outputs and workspace) and the stream.
All arithmetic runs in the library's kernels; if the library is missing this
module fails to import.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libssm_scan.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        "libssm_scan.so not found next to %s; build it with "
        "`python -m selective_state_space_111_b300.build`" % __file__)

_lib = ctypes.CDLL(_LIB_PATH)

SSM_F32, SSM_BF16, SSM_F16 = 0, 1, 2
_CODES = {torch.float32: SSM_F32, torch.bfloat16: SSM_BF16, torch.float16: SSM_F16}
OPS = {"single": 0, "v1": 1, "v2": 2, "ss2d": 3}
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA launch error",
           4: "workspace", 5: "scratch limit", 6: "timeout", 7: "bounds (debug build)"}

_vp, _fp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


def _declare(lib):
    """Argument and result types of every entry point of `lib` (this
    library, or a build of the same sources with other flags)."""
    lib.selective_scan_fwd.argtypes = [_i] * 5 + [_vp] * 8 + [_i, _vp, _vp, _sz, _vp]
    lib.bimamba_scan_fwd_v1.argtypes = [_i] * 5 + [_vp] * 9 + [_i, _f, _vp, _vp, _sz, _vp]
    lib.bimamba_scan_fwd_v2.argtypes = [_i] * 5 + [_vp] * 15 + [_i, _f, _vp, _vp, _sz, _vp]
    lib.ss2d_scan_fwd.argtypes = [_i] * 7 + [_vp] * 8 + [_i, _vp, _vp, _sz, _vp]
    lib.bimamba_scan_fwd_v2_noalloc.argtypes = [_i] * 5 + [_vp] * 15 + [_i, _f, _vp, _vp]
    lib.selective_scan_fwd_ls.argtypes = [_i] * 5 + [_vp] * 8 + [_i, _vp, _vp, _vp, _sz, _vp]
    lib.bimamba_scan_fwd_v1_ls.argtypes = [_i] * 5 + [_vp] * 9 + [_i, _f, _vp, _vp, _vp, _sz, _vp]
    lib.bimamba_scan_fwd_v2_ls.argtypes = [_i] * 5 + [_vp] * 15 + [_i, _f, _vp, _vp, _vp, _sz,
                                                                     _vp]
    lib.ss2d_scan_fwd_ls.argtypes = [_i] * 7 + [_vp] * 8 + [_i, _vp, _vp, _vp, _sz, _vp]
    lib.bimamba_scan_fwd_v2_so.argtypes = [_i] * 5 + [_vp] * 15 + [_i, _f, _vp, _vp, _vp, _sz,
                                                                     _vp]
    lib.ssm_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i]
    lib.ssm_workspace_bytes.restype = _sz
    lib.ssm_get_status.argtypes = [_vp, _vp, ctypes.POINTER(_i)]
    lib.ssm_get_status.restype = _i
    lib.ssm_status_string.argtypes = [_i]
    lib.ssm_status_string.restype = ctypes.c_char_p
    lib.ssm_version.restype = ctypes.c_char_p
    lib.ssm_test_withhold_copy.argtypes = [_i]
    lib.ssm_test_withhold_copy.restype = None
    lib.ssm_test_shrink_extents.argtypes = [ctypes.c_longlong]
    lib.ssm_test_shrink_extents.restype = None
    lib.ssm_set_cta_channels.argtypes = [_i]
    lib.ssm_set_cta_channels.restype = None
    lib.ssm_set_prologue_fused.argtypes = [_i]
    lib.ssm_set_prologue_fused.restype = None
    lib.ssm_set_profile_events.argtypes = [_vp, _vp]
    lib.ssm_set_profile_events.restype = None
    lib.selective_scan_bwd.argtypes = [_i] * 5 + [_vp] * 8 + [_i] + [_vp] * 10 + [_sz, _vp]
    lib.bimamba_scan_bwd_v1.argtypes = ([_i] * 5 + [_vp] * 9 + [_i, _f] + [_vp] * 11 +
                                         [_sz, _vp])
    lib.bimamba_scan_bwd_v2.argtypes = ([_i] * 5 + [_vp] * 15 + [_i, _f] + [_vp] * 17 +
                                         [_sz, _vp])
    lib.ss2d_scan_bwd.argtypes = [_i] * 7 + [_vp] * 8 + [_i] + [_vp] * 10 + [_sz, _vp]
    lib.mamba_prologue_fwd.argtypes = [_i] * 7 + [_vp] * 5 + [_i] + [_vp] * 5 + [_sz, _vp]
    lib.mamba_prologue_fwd.restype = _i
    lib.out_proj_fwd.argtypes = [_i] * 5 + [_vp] * 4
    lib.out_proj_fwd.restype = _i
    lib.ssm_prologue_workspace_bytes.argtypes = [_i, _i, _i]
    lib.ssm_prologue_workspace_bytes.restype = _sz
    lib.ss2d_prologue_fwd.argtypes = [_i] * 8 + [_vp] * 5 + [_i] + [_vp] * 5 + [_sz, _vp]
    lib.ss2d_prologue_fwd.restype = _i
    lib.ss2d_prologue_workspace_bytes.argtypes = [_i, _i, _i, _i]
    lib.ss2d_prologue_workspace_bytes.restype = _sz
    lib.ssm_bwd_workspace_bytes.argtypes = [_i] * 8
    lib.ssm_bwd_workspace_bytes.restype = _sz
    lib.ssm_set_bwd_context.argtypes = [_vp, _sz]
    lib.ssm_set_bwd_context.restype = None
    lib.ssm_bwd_context_bytes.argtypes = [_i] * 6
    lib.ssm_bwd_context_bytes.restype = _sz
    for _fn in (lib.selective_scan_fwd, lib.bimamba_scan_fwd_v1, lib.bimamba_scan_fwd_v2,
                lib.ss2d_scan_fwd, lib.bimamba_scan_fwd_v2_noalloc, lib.selective_scan_fwd_ls,
                lib.bimamba_scan_fwd_v1_ls, lib.bimamba_scan_fwd_v2_ls, lib.ss2d_scan_fwd_ls,
                lib.bimamba_scan_fwd_v2_so,
                lib.selective_scan_bwd,
                lib.bimamba_scan_bwd_v1, lib.bimamba_scan_bwd_v2, lib.ss2d_scan_bwd):
        _fn.restype = _i
    return lib


_declare(_lib)


class SsmError(RuntimeError):
    def __init__(self, status, where):
        msg = _lib.ssm_status_string(status).decode()
        super().__init__("%s: %s (status %d)" % (where, msg, status))
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded ctypes library (for callers that pass raw pointers)."""
    return _lib


def version() -> str:
    return _lib.ssm_version().decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _CODES:
        raise TypeError("I/O tensors must be float32, bfloat16 or float16, got %s" % t.dtype)
    return _CODES[t.dtype]


def _io(t, io_dtype, name, shape=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError("%s is required" % name)
    if not t.is_cuda or not t.is_contiguous() or t.dtype != io_dtype:
        raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, io_dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s: expected shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return t.data_ptr()


def _par(t, name, shape=None, optional=False):
    return _io(t, torch.float32, name, shape, optional)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def workspace_bytes(op: str, dtype: torch.dtype, B: int, D: int, L: int, N: int, K: int = 4) -> int:
    code = _CODES[dtype]
    n = _lib.ssm_workspace_bytes(OPS[op], code, B, D, L, N, K)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid sizes")
    return int(n)


def _workspace(op, dtype, B, D, L, N, device, workspace, K=4):
    need = workspace_bytes(op, dtype, B, D, L, N, K)
    if need == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    if not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError("workspace must be a CUDA tensor of at least %d bytes" % need)
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def set_profile_events(begin=None, end=None) -> None:
    """Record `begin` / `end` (torch.cuda.Event, already created by a first
    record) around the scan kernel of every later call on this thread;
    None switches the hook off."""
    if begin is None or end is None:
        _lib.ssm_set_profile_events(None, None)
        return
    _lib.ssm_set_profile_events(ctypes.c_void_p(begin.cuda_event), ctypes.c_void_p(end.cuda_event))


def set_cta_channels(channels: int = 0) -> None:
    """Channels per CTA of the two-branch kernels for later calls on this
    thread: 8, 16, or 0 for the automatic choice."""
    _lib.ssm_set_cta_channels(int(channels))


def set_prologue_fused(mode: int = 1) -> None:
    """Kernels of mamba_prologue_fwd for later calls on this thread, where
    the fused kernel applies: 1 automatic (fused for L < 1024), 0 always
    the three-kernel path, 2 the fused kernel at every L."""
    _lib.ssm_set_prologue_fused(int(mode))


def get_status(workspace, stream=None) -> int:
    """Status word of the last call that used `workspace` (0 = ok, 6 = a
    kernel's bounded wait ran out); synchronises the stream."""
    out = _i(0)
    _check(_lib.ssm_get_status(workspace.data_ptr(), _stream(stream), ctypes.byref(out)),
           "ssm_get_status")
    return out.value


def _check(status, where):
    if status != 0:
        raise SsmError(status, where)


def selective_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None,
                       delta_softplus=True, out=None, workspace=None, stream=None,
                       last_state=None):
    """One direction.  u, delta, z: [Bt, Dc, L]; A: [Dc, N] fp32; B, C: [Bt, N, L];
    D, delta_bias: [Dc] fp32.  Returns y [Bt, Dc, L].  last_state: optional fp32
    [1, Bt, Dc, N] tensor that receives the final state."""
    io = u.dtype
    Bt, Dc, L = u.shape
    N = A.shape[1]
    y = torch.empty_like(u) if out is None else out
    args = [_io(u, io, "u"), _io(delta, io, "delta", (Bt, Dc, L)), _par(A, "A", (Dc, N)),
            _io(B, io, "B", (Bt, N, L)), _io(C, io, "C", (Bt, N, L)),
            _par(D, "D", (Dc,), True), _io(z, io, "z", (Bt, Dc, L), True),
            _par(delta_bias, "delta_bias", (Dc,), True)]
    wp, wn = _workspace("single", io, Bt, Dc, L, N, u.device, workspace)
    if last_state is None:
        _check(_lib.selective_scan_fwd(_dtype_code(u), Bt, Dc, L, N, *args,
                                       int(bool(delta_softplus)), _io(y, io, "out", (Bt, Dc, L)),
                                       wp, wn, _stream(stream)), "selective_scan_fwd")
        return y
    _check(_lib.selective_scan_fwd_ls(_dtype_code(u), Bt, Dc, L, N, *args,
                                      int(bool(delta_softplus)), _io(y, io, "out", (Bt, Dc, L)),
                                      _par(last_state, "last_state", (1, Bt, Dc, N)), wp, wn,
                                      _stream(stream)), "selective_scan_fwd_ls")
    return y


def bimamba_scan_fwd_v1(u, delta, A, A_b, B, C, D=None, z=None, delta_bias=None,
                        delta_softplus=True, out_scale=1.0, out=None, workspace=None,
                        stream=None, last_state=None):
    """BiMamba v1: shared delta/B/C/D/bias, separate A and A_b.  Original order.
    last_state: optional fp32 [2, Bt, Dc, N] (forward, backward branch)."""
    io = u.dtype
    Bt, Dc, L = u.shape
    N = A.shape[1]
    y = torch.empty_like(u) if out is None else out
    args = [_io(u, io, "u"), _io(delta, io, "delta", (Bt, Dc, L)), _par(A, "A", (Dc, N)),
            _par(A_b, "A_b", (Dc, N)), _io(B, io, "B", (Bt, N, L)), _io(C, io, "C", (Bt, N, L)),
            _par(D, "D", (Dc,), True), _io(z, io, "z", (Bt, Dc, L), True),
            _par(delta_bias, "delta_bias", (Dc,), True)]
    wp, wn = _workspace("v1", io, Bt, Dc, L, N, u.device, workspace)
    if last_state is None:
        _check(_lib.bimamba_scan_fwd_v1(_dtype_code(u), Bt, Dc, L, N, *args,
                                        int(bool(delta_softplus)), float(out_scale),
                                        _io(y, io, "out", (Bt, Dc, L)), wp, wn, _stream(stream)),
               "bimamba_scan_fwd_v1")
        return y
    _check(_lib.bimamba_scan_fwd_v1_ls(_dtype_code(u), Bt, Dc, L, N, *args,
                                       int(bool(delta_softplus)), float(out_scale),
                                       _io(y, io, "out", (Bt, Dc, L)),
                                       _par(last_state, "last_state", (2, Bt, Dc, N)), wp, wn,
                                       _stream(stream)), "bimamba_scan_fwd_v1_ls")
    return y


def bimamba_scan_fwd_v2(u, delta, delta_b, A, A_b, B, C, B_b, C_b, D=None, D_b=None, z=None,
                        delta_bias=None, delta_bias_b=None, u_b=None, delta_softplus=True,
                        out_scale=0.5, out=None, workspace=None, stream=None,
                        last_state=None, scan_order=False):
    """BiMamba v2: independent backward set.  Original token order, or with
    scan_order=True the backward set (delta_b, B_b, C_b, u_b) time-reversed.
    last_state: optional fp32 [2, Bt, Dc, N] (forward, backward branch)."""
    io = u.dtype
    Bt, Dc, L = u.shape
    N = A.shape[1]
    y = torch.empty_like(u) if out is None else out
    sh, shn = (Bt, Dc, L), (Bt, N, L)
    args = [_io(u, io, "u"), _io(u_b, io, "u_b", sh, True), _io(delta, io, "delta", sh),
            _io(delta_b, io, "delta_b", sh), _par(A, "A", (Dc, N)), _par(A_b, "A_b", (Dc, N)),
            _io(B, io, "B", shn), _io(C, io, "C", shn), _io(B_b, io, "B_b", shn),
            _io(C_b, io, "C_b", shn), _par(D, "D", (Dc,), True), _par(D_b, "D_b", (Dc,), True),
            _io(z, io, "z", sh, True), _par(delta_bias, "delta_bias", (Dc,), True),
            _par(delta_bias_b, "delta_bias_b", (Dc,), True)]
    wp, wn = _workspace("v2", io, Bt, Dc, L, N, u.device, workspace)
    if scan_order:
        ls = None if last_state is None else _par(last_state, "last_state", (2, Bt, Dc, N))
        _check(_lib.bimamba_scan_fwd_v2_so(_dtype_code(u), Bt, Dc, L, N, *args,
                                           int(bool(delta_softplus)), float(out_scale),
                                           _io(y, io, "out", sh), ls, wp, wn, _stream(stream)),
               "bimamba_scan_fwd_v2_so")
        return y
    if last_state is None:
        _check(_lib.bimamba_scan_fwd_v2(_dtype_code(u), Bt, Dc, L, N, *args,
                                        int(bool(delta_softplus)), float(out_scale),
                                        _io(y, io, "out", sh), wp, wn, _stream(stream)),
               "bimamba_scan_fwd_v2")
        return y
    _check(_lib.bimamba_scan_fwd_v2_ls(_dtype_code(u), Bt, Dc, L, N, *args,
                                       int(bool(delta_softplus)), float(out_scale),
                                       _io(y, io, "out", sh),
                                       _par(last_state, "last_state", (2, Bt, Dc, N)), wp, wn,
                                       _stream(stream)), "bimamba_scan_fwd_v2_ls")
    return y


def ss2d_scan_fwd(x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                  out=None, workspace=None, stream=None, last_state=None):
    """SS2D, K=4.  x, z: [Bt, Dc, H, W]; delta: [Bt, 4, Dc, H*W] and B, C: [Bt, 4, N, H*W]
    in each direction's scan order; A: [4, Dc, N]; D, delta_bias: [4, Dc]."""
    io = x.dtype
    Bt, Dc, H, W = x.shape
    K = 4
    L = H * W
    N = A.shape[2]
    y = torch.empty_like(x) if out is None else out
    args = [_io(x, io, "x"), _io(delta, io, "delta", (Bt, K, Dc, L)), _par(A, "A", (K, Dc, N)),
            _io(B, io, "B", (Bt, K, N, L)), _io(C, io, "C", (Bt, K, N, L)),
            _par(D, "D", (K, Dc), True), _io(z, io, "z", (Bt, Dc, H, W), True),
            _par(delta_bias, "delta_bias", (K, Dc), True)]
    wp, wn = _workspace("ss2d", io, Bt, Dc, L, N, x.device, workspace, K)
    if last_state is None:
        _check(_lib.ss2d_scan_fwd(_dtype_code(x), Bt, Dc, H, W, N, K, *args,
                                  int(bool(delta_softplus)), _io(y, io, "out", (Bt, Dc, H, W)),
                                  wp, wn, _stream(stream)), "ss2d_scan_fwd")
        return y
    _check(_lib.ss2d_scan_fwd_ls(_dtype_code(x), Bt, Dc, H, W, N, K, *args,
                                 int(bool(delta_softplus)), _io(y, io, "out", (Bt, Dc, H, W)),
                                 _par(last_state, "last_state", (4, Bt, Dc, N)), wp, wn,
                                 _stream(stream)), "ss2d_scan_fwd_ls")
    return y


def bimamba_scan_fwd_v2_noalloc(u, delta, delta_b, A, A_b, B, C, B_b, C_b, D=None, D_b=None,
                                z=None, delta_bias=None, delta_bias_b=None, u_b=None,
                                delta_softplus=True, out_scale=0.5, out=None, stream=None):
    """BiMamba v2 through the allocation-free entry point: the library's fixed
    scratch array replaces the workspace, so only `out` (if not given) is
    allocated here, by PyTorch.  Raises SsmError (status 5) when the problem
    needs more scratch than the array holds."""
    io = u.dtype
    Bt, Dc, L = u.shape
    N = A.shape[1]
    y = torch.empty_like(u) if out is None else out
    sh, shn = (Bt, Dc, L), (Bt, N, L)
    args = [_io(u, io, "u"), _io(u_b, io, "u_b", sh, True), _io(delta, io, "delta", sh),
            _io(delta_b, io, "delta_b", sh), _par(A, "A", (Dc, N)), _par(A_b, "A_b", (Dc, N)),
            _io(B, io, "B", shn), _io(C, io, "C", shn), _io(B_b, io, "B_b", shn),
            _io(C_b, io, "C_b", shn), _par(D, "D", (Dc,), True), _par(D_b, "D_b", (Dc,), True),
            _io(z, io, "z", sh, True), _par(delta_bias, "delta_bias", (Dc,), True),
            _par(delta_bias_b, "delta_bias_b", (Dc,), True)]
    _check(_lib.bimamba_scan_fwd_v2_noalloc(_dtype_code(u), Bt, Dc, L, N, *args,
                                            int(bool(delta_softplus)), float(out_scale),
                                            _io(y, io, "out", sh), _stream(stream)),
           "bimamba_scan_fwd_v2_noalloc")
    return y


# ---------------------------------------------------------------- backward
def bwd_workspace_bytes(op: str, dtype: torch.dtype, B: int, D: int, L: int, N: int,
                        K: int = 4, separate_u_b: bool = False) -> int:
    code = _CODES[dtype]
    n = _lib.ssm_bwd_workspace_bytes(OPS[op], code, B, D, L, N, K, int(bool(separate_u_b)))
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid sizes")
    return int(n)


def bwd_context_bytes(op: str, dtype: torch.dtype, B: int, D: int, L: int, N: int) -> int:
    """Bytes of a saved backward context (0: d_state > 16, none is kept)."""
    n = _lib.ssm_bwd_context_bytes(OPS[op], _CODES[dtype], B, D, L, N)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid sizes or operation")
    return int(n)


def set_bwd_context(ctx=None) -> None:
    """Saved backward context for later calls on this thread: a uint8 CUDA
    tensor of at least bwd_context_bytes(...) bytes, or None to stop.  While
    it is set, forward calls (single, v1, v2; d_state <= 16) also store the
    pre-gate output and chunk-start states there, and backward calls on the
    same inputs read them instead of running the forward pass again.  The
    caller keeps the tensor alive and pairs each backward call with the
    forward call that filled the context."""
    if ctx is None:
        _lib.ssm_set_bwd_context(None, 0)
        return
    if not (isinstance(ctx, torch.Tensor) and ctx.is_cuda and ctx.dtype == torch.uint8 and
            ctx.is_contiguous()):
        raise ValueError("the context is a contiguous uint8 CUDA tensor")
    _lib.ssm_set_bwd_context(ctypes.c_void_p(ctx.data_ptr()), ctx.numel())


def _bwd_workspace(op, dtype, B, D, L, N, device, workspace, K=4, separate_u_b=False):
    need = bwd_workspace_bytes(op, dtype, B, D, L, N, K, separate_u_b)
    if need == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    if not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError("workspace must be a CUDA tensor of at least %d bytes" % need)
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def _ptr_or_none(t):
    return None if t is None else t.data_ptr()


def selective_scan_bwd(dout, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                       delta_softplus=True, workspace=None, stream=None):
    """Gradients of sum(dout * selective_scan_fwd(...)).  Returns a dict:
    du, ddelta, dA, dB, dC, and dD / dz / ddelta_bias for the inputs given."""
    io = u.dtype
    Bt, Dc, L = u.shape
    N = A.shape[1]
    sh, shn = (Bt, Dc, L), (Bt, N, L)
    g = {"du": torch.empty_like(u), "ddelta": torch.empty_like(u),
         "dA": torch.empty_like(A), "dB": torch.empty(shn, dtype=io, device=u.device),
         "dC": torch.empty(shn, dtype=io, device=u.device)}
    if D is not None:
        g["dD"] = torch.empty_like(D)
    if z is not None:
        g["dz"] = torch.empty_like(u)
    if delta_bias is not None:
        g["ddelta_bias"] = torch.empty_like(delta_bias)
    args = [_io(u, io, "u"), _io(delta, io, "delta", sh), _par(A, "A", (Dc, N)),
            _io(B, io, "B", shn), _io(C, io, "C", shn), _par(D, "D", (Dc,), True),
            _io(z, io, "z", sh, True), _par(delta_bias, "delta_bias", (Dc,), True)]
    outs = [g["du"], g["ddelta"], g["dA"], g["dB"], g["dC"], g.get("dD"), g.get("dz"),
            g.get("ddelta_bias")]
    wp, wn = _bwd_workspace("single", io, Bt, Dc, L, N, u.device, workspace)
    _check(_lib.selective_scan_bwd(_dtype_code(u), Bt, Dc, L, N, *args,
                                   int(bool(delta_softplus)), _io(dout, io, "dout", sh),
                                   *map(_ptr_or_none, outs), wp, wn, _stream(stream)),
           "selective_scan_bwd")
    return g


def bimamba_scan_bwd_v1(dout, u, delta, A, A_b, B, C, D=None, z=None, delta_bias=None,
                        delta_softplus=True, out_scale=1.0, workspace=None, stream=None):
    """Gradients of sum(dout * bimamba_scan_fwd_v1(...)): du, ddelta, dA, dA_b,
    dB, dC, and dD / dz / ddelta_bias for the inputs given."""
    io = u.dtype
    Bt, Dc, L = u.shape
    N = A.shape[1]
    sh, shn = (Bt, Dc, L), (Bt, N, L)
    g = {"du": torch.empty_like(u), "ddelta": torch.empty_like(u),
         "dA": torch.empty_like(A), "dA_b": torch.empty_like(A_b),
         "dB": torch.empty(shn, dtype=io, device=u.device),
         "dC": torch.empty(shn, dtype=io, device=u.device)}
    if D is not None:
        g["dD"] = torch.empty_like(D)
    if z is not None:
        g["dz"] = torch.empty_like(u)
    if delta_bias is not None:
        g["ddelta_bias"] = torch.empty_like(delta_bias)
    args = [_io(u, io, "u"), _io(delta, io, "delta", sh), _par(A, "A", (Dc, N)),
            _par(A_b, "A_b", (Dc, N)), _io(B, io, "B", shn), _io(C, io, "C", shn),
            _par(D, "D", (Dc,), True), _io(z, io, "z", sh, True),
            _par(delta_bias, "delta_bias", (Dc,), True)]
    outs = [g["du"], g["ddelta"], g["dA"], g["dA_b"], g["dB"], g["dC"], g.get("dD"),
            g.get("dz"), g.get("ddelta_bias")]
    wp, wn = _bwd_workspace("v1", io, Bt, Dc, L, N, u.device, workspace)
    _check(_lib.bimamba_scan_bwd_v1(_dtype_code(u), Bt, Dc, L, N, *args,
                                    int(bool(delta_softplus)), float(out_scale),
                                    _io(dout, io, "dout", sh), *map(_ptr_or_none, outs),
                                    wp, wn, _stream(stream)), "bimamba_scan_bwd_v1")
    return g


def bimamba_scan_bwd_v2(dout, u, delta, delta_b, A, A_b, B, C, B_b, C_b, D=None, D_b=None,
                        z=None, delta_bias=None, delta_bias_b=None, u_b=None,
                        delta_softplus=True, out_scale=0.5, workspace=None, stream=None):
    """Gradients of sum(dout * bimamba_scan_fwd_v2(...)): one per input given
    (du_b only with u_b)."""
    io = u.dtype
    Bt, Dc, L = u.shape
    N = A.shape[1]
    sh, shn = (Bt, Dc, L), (Bt, N, L)
    dev = u.device
    g = {"du": torch.empty_like(u), "ddelta": torch.empty_like(u),
         "ddelta_b": torch.empty_like(u), "dA": torch.empty_like(A),
         "dA_b": torch.empty_like(A_b)}
    for k in ("dB", "dC", "dB_b", "dC_b"):
        g[k] = torch.empty(shn, dtype=io, device=dev)
    if u_b is not None:
        g["du_b"] = torch.empty_like(u)
    if D is not None:
        g["dD"] = torch.empty_like(D)
    if D_b is not None:
        g["dD_b"] = torch.empty_like(D_b)
    if z is not None:
        g["dz"] = torch.empty_like(u)
    if delta_bias is not None:
        g["ddelta_bias"] = torch.empty_like(delta_bias)
    if delta_bias_b is not None:
        g["ddelta_bias_b"] = torch.empty_like(delta_bias_b)
    args = [_io(u, io, "u"), _io(u_b, io, "u_b", sh, True), _io(delta, io, "delta", sh),
            _io(delta_b, io, "delta_b", sh), _par(A, "A", (Dc, N)), _par(A_b, "A_b", (Dc, N)),
            _io(B, io, "B", shn), _io(C, io, "C", shn), _io(B_b, io, "B_b", shn),
            _io(C_b, io, "C_b", shn), _par(D, "D", (Dc,), True), _par(D_b, "D_b", (Dc,), True),
            _io(z, io, "z", sh, True), _par(delta_bias, "delta_bias", (Dc,), True),
            _par(delta_bias_b, "delta_bias_b", (Dc,), True)]
    outs = [g["du"], g.get("du_b"), g["ddelta"], g["ddelta_b"], g["dA"], g["dA_b"], g["dB"],
            g["dC"], g["dB_b"], g["dC_b"], g.get("dD"), g.get("dD_b"), g.get("dz"),
            g.get("ddelta_bias"), g.get("ddelta_bias_b")]
    wp, wn = _bwd_workspace("v2", io, Bt, Dc, L, N, dev, workspace,
                            separate_u_b=u_b is not None)
    _check(_lib.bimamba_scan_bwd_v2(_dtype_code(u), Bt, Dc, L, N, *args,
                                    int(bool(delta_softplus)), float(out_scale),
                                    _io(dout, io, "dout", sh), *map(_ptr_or_none, outs),
                                    wp, wn, _stream(stream)), "bimamba_scan_bwd_v2")
    return g


def ss2d_scan_bwd(dout, x, delta, A, B, C, D=None, z=None, delta_bias=None,
                  delta_softplus=True, workspace=None, stream=None):
    """Gradients of sum(dout * ss2d_scan_fwd(...)): dx, ddelta, dA, dB, dC, and
    dD / dz / ddelta_bias for the inputs given."""
    io = x.dtype
    Bt, Dc, H, W = x.shape
    K = 4
    L = H * W
    N = A.shape[2]
    dev = x.device
    g = {"dx": torch.empty_like(x), "ddelta": torch.empty_like(delta),
         "dA": torch.empty_like(A), "dB": torch.empty_like(B), "dC": torch.empty_like(C)}
    if D is not None:
        g["dD"] = torch.empty_like(D)
    if z is not None:
        g["dz"] = torch.empty_like(x)
    if delta_bias is not None:
        g["ddelta_bias"] = torch.empty_like(delta_bias)
    args = [_io(x, io, "x"), _io(delta, io, "delta", (Bt, K, Dc, L)), _par(A, "A", (K, Dc, N)),
            _io(B, io, "B", (Bt, K, N, L)), _io(C, io, "C", (Bt, K, N, L)),
            _par(D, "D", (K, Dc), True), _io(z, io, "z", (Bt, Dc, H, W), True),
            _par(delta_bias, "delta_bias", (K, Dc), True)]
    outs = [g["dx"], g["ddelta"], g["dA"], g["dB"], g["dC"], g.get("dD"), g.get("dz"),
            g.get("ddelta_bias")]
    wp, wn = _bwd_workspace("ss2d", io, Bt, Dc, L, N, dev, workspace, K)
    _check(_lib.ss2d_scan_bwd(_dtype_code(x), Bt, Dc, H, W, N, K, *args,
                              int(bool(delta_softplus)), _io(dout, io, "dout", (Bt, Dc, H, W)),
                              *map(_ptr_or_none, outs), wp, wn, _stream(stream)),
           "ss2d_scan_bwd")
    return g


# ---------------------------------------------------------------- prologue
def mamba_prologue_fwd(x, conv_w, conv_b, W_x, W_dt, dt_rank, d_state, reverse=False,
                       workspace=None, stream=None):
    """One direction's conv1d + SiLU, x_proj split and dt_proj.  x: [Bt, Dc, L]
    (I/O dtype); conv_w [Dc, K], conv_b [Dc] (or None), W_x [R + 2N, Dc],
    W_dt [Dc, R] fp32.  Returns (u, delta, B, C): [Bt, Dc, L] x2, [Bt, N, L] x2,
    in scan order of the reversed sequence when reverse=True."""
    io = x.dtype
    Bt, Dc, L = x.shape
    R, N = int(dt_rank), int(d_state)
    K = conv_w.shape[1]
    u = torch.empty_like(x)
    delta = torch.empty_like(x)
    Bm = torch.empty((Bt, N, L), dtype=io, device=x.device)
    Cm = torch.empty((Bt, N, L), dtype=io, device=x.device)
    need = int(_lib.ssm_prologue_workspace_bytes(Bt, L, R))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    _check(_lib.mamba_prologue_fwd(_dtype_code(x), Bt, Dc, L, N, R, K, _io(x, io, "x"),
                                   _par(conv_w, "conv_w", (Dc, K)),
                                   _par(conv_b, "conv_b", (Dc,), True),
                                   _par(W_x, "W_x", (R + 2 * N, Dc)),
                                   _par(W_dt, "W_dt", (Dc, R)), int(bool(reverse)),
                                   u.data_ptr(), delta.data_ptr(), Bm.data_ptr(), Cm.data_ptr(),
                                   workspace.data_ptr(),
                                   workspace.numel() * workspace.element_size(),
                                   _stream(stream)), "mamba_prologue_fwd")
    return u, delta, Bm, Cm


def out_proj_fwd(y, W_out, stream=None):
    """The block's output projection: out[b, m, t] = sum_k W_out[m, k] y[b, k, t].
    y: [Bt, Di, L] (I/O dtype, the gated scan output); W_out [Dm, Di] in the
    same dtype.  Returns out [Bt, Dm, L]."""
    io = y.dtype
    Bt, Di, L = y.shape
    if W_out.dim() != 2 or W_out.shape[1] != Di:
        raise ValueError("W_out: expected [Dm, %d], got %s" % (Di, tuple(W_out.shape)))
    Dm = W_out.shape[0]
    out = torch.empty((Bt, Dm, L), dtype=io, device=y.device)
    _check(_lib.out_proj_fwd(_dtype_code(y), Bt, Di, Dm, L, _io(y, io, "y"),
                             _io(W_out, io, "W_out"), out.data_ptr(), _stream(stream)),
           "out_proj_fwd")
    return out


def ss2d_prologue_fwd(x, conv_w, conv_b, W_x, W_dt, dt_rank, d_state, silu_act=True,
                      workspace=None, stream=None):
    """SS2D's conv2d (+ SiLU) and its four directions' x_proj and dt_proj.
    x: [Bt, Dc, H, W] (I/O dtype); conv_w [Dc, Kc, Kc], conv_b [Dc] (or
    None), W_x [4, R + 2N, Dc], W_dt [4, Dc, R] fp32.  Returns (u, delta, B,
    C): u [Bt, Dc, H, W]; delta [Bt, 4, Dc, H*W], B, C [Bt, 4, N, H*W], each
    direction in its own scan order (what ss2d_scan_fwd takes, u as its x)."""
    io = x.dtype
    Bt, Dc, H, W = x.shape
    R, N = int(dt_rank), int(d_state)
    Kc = conv_w.shape[-1]
    L = H * W
    u = torch.empty_like(x)
    delta = torch.empty((Bt, 4, Dc, L), dtype=io, device=x.device)
    Bm = torch.empty((Bt, 4, N, L), dtype=io, device=x.device)
    Cm = torch.empty((Bt, 4, N, L), dtype=io, device=x.device)
    need = int(_lib.ss2d_prologue_workspace_bytes(Bt, H, W, R))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    _check(_lib.ss2d_prologue_fwd(_dtype_code(x), Bt, Dc, H, W, N, R, Kc, _io(x, io, "x"),
                                  _par(conv_w, "conv_w", (Dc, Kc, Kc)),
                                  _par(conv_b, "conv_b", (Dc,), True),
                                  _par(W_x, "W_x", (4, R + 2 * N, Dc)),
                                  _par(W_dt, "W_dt", (4, Dc, R)), int(bool(silu_act)),
                                  u.data_ptr(), delta.data_ptr(), Bm.data_ptr(), Cm.data_ptr(),
                                  workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(),
                                  _stream(stream)), "ss2d_prologue_fwd")
    return u, delta, Bm, Cm
