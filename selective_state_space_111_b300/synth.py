"""Seeded synthetic inputs for the selective-scan operations.

This module serves both the CUDA path and the fp64 oracle: it draws the
tensors, rounds activations to the I/O dtype once, and hands the same values
to both sides.  It holds none of the scan's arithmetic.

Recipe (shapes from the Vision Mamba / VMamba pages' workloads):
  * A[d, n] = -(n + 1) for n = 0..N-1 on every channel: the A_log = log(1..N)
    initialisation ("从Transformer到Mamba" section 2.1, "Vision Mamba实战"
    section 2.1) with A = -exp(A_log).  ``perturb`` scales each entry by
    U(0.75, 1.25) so that swapped-parameter bugs show.
  * Per-channel step sizes: delta_d = exp(U(ln 1e-3, ln 1e-1)) (the dt_min /
    dt_max range, "VMamba的SS2D模块详解" section 4.2); delta_bias_d is the value
    whose softplus is delta_d, i.e. log(expm1(delta_d)).
  * dt ~ N(0, 0.5^2); u (x), z, B, C ~ N(0, 1); D = 1 (``perturb``: U(0.5, 1.5)).
  * Every activation is drawn in fp32 and rounded to the I/O dtype (round to
    nearest even for bf16 and fp16); A, D and delta_bias stay fp32.
Tensors are drawn on the CPU from ``torch.Generator().manual_seed(seed)`` in a
fixed order, so a (spec, seed) pair always gives the same values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

IO_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclass(frozen=True)
class Spec:
    """One workload: operation, I/O dtype and sizes."""

    op: str            # "single" | "v1" | "v2" | "ss2d"
    io: str            # "f32" | "bf16" | "f16"
    B: int
    D: int
    N: int = 16
    L: int = 0         # sequence length (single / v1 / v2)
    H: int = 0         # SS2D map height
    W: int = 0         # SS2D map width
    K: int = 4         # SS2D directions
    out_scale: float = 1.0
    delta_softplus: bool = True
    gate: bool = True
    shared_u: bool = True      # v2: backward branch scans the same u
    a_b_noise: float = 0.0     # v1: A_b = A + N(0, a_b_noise^2)
    perturb: bool = False
    name: str = ""
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def seq_len(self) -> int:
        return self.H * self.W if self.op == "ss2d" else self.L

    @property
    def directions(self) -> int:
        return {"single": 1, "v1": 2, "v2": 2, "ss2d": self.K}[self.op]

    def updates(self) -> int:
        """Element updates: one (b, d, n, t, direction) recurrence step each."""
        return self.directions * self.B * self.D * self.seq_len * self.N

    def backward_bytes(self) -> int:
        """The backward pass's algorithmic bytes: every forward input and the
        output gradient read once, every input's gradient written once (the
        fp32 parameter gradients A, D, bias are ignored)."""
        e = 4 if self.io == "f32" else 2
        BD, L, N = self.B * self.D, self.seq_len, self.N
        z = 1 if self.gate else 0
        if self.op in ("single", "v1"):
            rows, bc = 2 + z, 2          # u, delta (+ z); B, C
        elif self.op == "v2":
            rows, bc = 3 + z + (0 if self.shared_u else 1), 4
        else:
            rows, bc = 1 + z + self.K, 2 * self.K
        return e * (BD * L * (2 * rows + 1) + self.B * L * N * 2 * bc)

    def algorithmic_bytes(self) -> int:
        """Each I/O tensor read once and y written once (A, D, bias ignored)."""
        e = 4 if self.io == "f32" else 2
        BD, L, N = self.B * self.D, self.seq_len, self.N
        z = 1 if self.gate else 0
        if self.op == "single":
            per_row = 3 + z            # u, delta, y (+ z)
            bc = 2                     # B, C
        elif self.op == "v1":
            per_row = 3 + z
            bc = 2
        elif self.op == "v2":
            per_row = 4 + z + (0 if self.shared_u else 1)   # u, delta, delta_b, y
            bc = 4
        else:  # ss2d: x, y (+ z) spatial and K per-direction deltas
            per_row = 2 + z + self.K
            bc = 2 * self.K
        return e * (BD * L * per_row + self.B * N * L * bc)


# The workloads named by the pages: Vim-Ti / Vim-S token sequences (16x16
# patches + cls token) and VMamba's 56x56 stage-1 map.
WORKLOADS = {
    "vim_ti_224_single_f32": Spec("single", "f32", B=1, D=384, L=197),
    "vim_ti_224_bimamba_v2": Spec("v2", "bf16", B=64, D=384, L=197, out_scale=0.5),
    "vim_s_1248_bimamba_v2": Spec("v2", "bf16", B=8, D=768, L=6085, out_scale=0.5),
    "vmamba_56x56_ss2d": Spec("ss2d", "bf16", B=32, D=192, H=56, W=56),
}
for _L in (4096, 16384, 65536, 262144):
    WORKLOADS["bimamba_v1_L%d" % _L] = Spec("v1", "bf16", B=2, D=1536, L=_L,
                                            out_scale=1.0, a_b_noise=0.1)
for _k, _s in list(WORKLOADS.items()):
    WORKLOADS[_k] = Spec(**{**_s.__dict__, "name": _k})


def _normal(g, shape, std, dtype):
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _a_matrix(g, lead, D, N, perturb):
    a = -torch.arange(1, N + 1, dtype=torch.float32).repeat(*lead, D, 1)
    if perturb:
        a = a * (0.75 + 0.5 * torch.rand(a.shape, generator=g))
    return a.contiguous()


def _bias(g, shape):
    # per-channel step size in [1e-3, 1e-1], log-uniform; bias = softplus^-1
    lo, hi = math.log(1e-3), math.log(1e-1)
    d64 = torch.exp(lo + (hi - lo) * torch.rand(*shape, generator=g, dtype=torch.float64))
    return torch.log(torch.expm1(d64)).to(torch.float32)


def _dskip(g, shape, perturb):
    if perturb:
        return (0.5 + torch.rand(*shape, generator=g)).to(torch.float32)
    return torch.ones(*shape, dtype=torch.float32)


def make_inputs(spec: Spec, seed: int) -> dict:
    """Draw every input of ``spec`` on the CPU.  Returns a dict of tensors
    keyed by the C ABI's argument names, plus the scalar arguments."""
    g = torch.Generator().manual_seed(int(seed))
    io = IO_DTYPES[spec.io]
    B, D, N = spec.B, spec.D, spec.N
    out = {"delta_softplus": spec.delta_softplus, "out_scale": spec.out_scale}
    if spec.op in ("single", "v1", "v2"):
        L = spec.L
        out["A"] = _a_matrix(g, (), D, N, spec.perturb)
        out["delta_bias"] = _bias(g, (D,))
        out["D"] = _dskip(g, (D,), spec.perturb)
        out["u"] = _normal(g, (B, D, L), 1.0, io)
        out["delta"] = _normal(g, (B, D, L), 0.5, io)
        out["B"] = _normal(g, (B, N, L), 1.0, io)
        out["C"] = _normal(g, (B, N, L), 1.0, io)
        out["z"] = _normal(g, (B, D, L), 1.0, io) if spec.gate else None
        if spec.op == "v1":
            a_b = _a_matrix(g, (), D, N, spec.perturb)
            if spec.a_b_noise:
                a_b = a_b + spec.a_b_noise * torch.randn(a_b.shape, generator=g)
            out["A_b"] = a_b.contiguous()
        elif spec.op == "v2":
            out["A_b"] = _a_matrix(g, (), D, N, spec.perturb)
            out["delta_bias_b"] = _bias(g, (D,))
            out["D_b"] = _dskip(g, (D,), spec.perturb)
            out["delta_b"] = _normal(g, (B, D, L), 0.5, io)
            out["B_b"] = _normal(g, (B, N, L), 1.0, io)
            out["C_b"] = _normal(g, (B, N, L), 1.0, io)
            out["u_b"] = None if spec.shared_u else _normal(g, (B, D, L), 1.0, io)
    elif spec.op == "ss2d":
        H, W, K = spec.H, spec.W, spec.K
        L = H * W
        out["A"] = _a_matrix(g, (K,), D, N, spec.perturb)
        out["delta_bias"] = _bias(g, (K, D))
        out["D"] = _dskip(g, (K, D), spec.perturb)
        out["x"] = _normal(g, (B, D, H, W), 1.0, io)
        out["delta"] = _normal(g, (B, K, D, L), 0.5, io)
        out["B"] = _normal(g, (B, K, N, L), 1.0, io)
        out["C"] = _normal(g, (B, K, N, L), 1.0, io)
        out["z"] = _normal(g, (B, D, H, W), 1.0, io) if spec.gate else None
    else:
        raise ValueError("unknown op %r" % spec.op)
    return out


def seed_for(name: str, base: int = 20261202) -> int:
    """Stable per-workload seed: base + the workload's index in WORKLOADS."""
    return base + list(WORKLOADS).index(name)
