"""Pins of the oracle's backward pass (CPU).

Every gradient element of every form is compared with a central finite
difference of the oracle's FORWARD pass (fp64, step 1e-6), which shares
nothing with the backward code: a dropped term, a wrong sign, a missing flip
or a transposed operand in the backward changes some element by far more
than the difference's error (~1e-9 here).  The loss is sum(g * out) for a
random incoming gradient g, so each input's gradient is one directional
derivative per element.
"""
import numpy as np
import pytest

import oracle

EPS = 1e-6
RTOL, ATOL = 1e-6, 1e-8


def _fd_check(fwd, inputs, grads, g, names):
    """Central differences of sum(g * fwd(**inputs)) against grads[name] for
    every element of every input in `names` (gradient key 'd' + name)."""
    for name in names:
        x = inputs[name]
        got = grads["d" + name]
        assert got.shape == x.shape, name
        fd = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + EPS
            lp = float((g * fwd(**inputs)).sum())
            x[idx] = old - EPS
            lm = float((g * fwd(**inputs)).sum())
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * EPS)
        np.testing.assert_allclose(got, fd, rtol=RTOL, atol=ATOL, err_msg=name)


def _seq_inputs(rng, B, D, L, N, two_sets=False, with_ub=False):
    """Small well-conditioned inputs: delta near 0.1..1, A negative."""
    t = {
        "u": rng.normal(size=(B, D, L)),
        "delta": rng.normal(size=(B, D, L)) * 0.5,
        "A": -rng.uniform(0.2, 2.0, size=(D, N)),
        "B": rng.normal(size=(B, N, L)),
        "C": rng.normal(size=(B, N, L)),
        "D": rng.normal(size=(D,)),
        "z": rng.normal(size=(B, D, L)),
        "delta_bias": rng.normal(size=(D,)) * 0.2,
    }
    if two_sets:
        t.update({
            "delta_b": rng.normal(size=(B, D, L)) * 0.5,
            "A_b": -rng.uniform(0.2, 2.0, size=(D, N)),
            "B_b": rng.normal(size=(B, N, L)),
            "C_b": rng.normal(size=(B, N, L)),
            "D_b": rng.normal(size=(D,)),
            "delta_bias_b": rng.normal(size=(D,)) * 0.2,
        })
    if with_ub:
        t["u_b"] = rng.normal(size=(B, D, L))
    return t


@pytest.mark.parametrize("softplus", [True, False])
@pytest.mark.parametrize("gated", [True, False])
def test_selective_scan_bwd_matches_finite_differences(softplus, gated):
    rng = np.random.default_rng(11 + 2 * softplus + gated)
    B, D, L, N = 2, 2, 6, 3
    t = _seq_inputs(rng, B, D, L, N)
    if not softplus:
        t["delta"] = np.abs(t["delta"]) + 0.05
        t["delta_bias"] = np.abs(t["delta_bias"])
    if not gated:
        t["z"] = None
    g = rng.normal(size=(B, D, L))

    def fwd(**kw):
        return oracle.selective_scan(delta_softplus=softplus, **kw)

    grads = oracle.selective_scan_bwd(g, delta_softplus=softplus, **t)
    names = ["u", "delta", "A", "B", "C", "D", "delta_bias"] + (["z"] if gated else [])
    _fd_check(fwd, t, grads, g, names)
    assert ("dz" in grads) == gated


def test_selective_scan_bwd_optional_inputs_absent():
    # no skip, no bias: those gradients are not produced; the rest still pin
    rng = np.random.default_rng(5)
    t = _seq_inputs(rng, 1, 2, 5, 2)
    t["D"] = None
    t["delta_bias"] = None
    g = rng.normal(size=(1, 2, 5))
    grads = oracle.selective_scan_bwd(g, **t)
    assert "dD" not in grads and "ddelta_bias" not in grads
    _fd_check(lambda **kw: oracle.selective_scan(**kw), t, grads, g,
              ["u", "delta", "A", "B", "C", "z"])


@pytest.mark.parametrize("with_ub", [False, True])
def test_bimamba_v2_bwd_matches_finite_differences(with_ub):
    rng = np.random.default_rng(21 + with_ub)
    B, D, L, N = 2, 2, 5, 2
    t = _seq_inputs(rng, B, D, L, N, two_sets=True, with_ub=with_ub)
    g = rng.normal(size=(B, D, L))

    def fwd(**kw):
        return oracle.bimamba_v2(out_scale=0.5, **kw)

    grads = oracle.bimamba_v2_bwd(g, out_scale=0.5, **t)
    names = ["u", "delta", "delta_b", "A", "A_b", "B", "C", "B_b", "C_b", "D", "D_b", "z",
             "delta_bias", "delta_bias_b"] + (["u_b"] if with_ub else [])
    _fd_check(fwd, t, grads, g, names)
    assert ("du_b" in grads) == with_ub


def test_bimamba_v1_bwd_matches_finite_differences():
    rng = np.random.default_rng(31)
    B, D, L, N = 2, 2, 5, 3
    t = _seq_inputs(rng, B, D, L, N)
    t["A_b"] = t["A"] + rng.normal(size=t["A"].shape) * 0.1
    g = rng.normal(size=(B, D, L))

    def fwd(**kw):
        return oracle.bimamba_v1(out_scale=1.0, **kw)

    grads = oracle.bimamba_v1_bwd(g, out_scale=1.0, **t)
    _fd_check(fwd, t, grads, g, ["u", "delta", "A", "A_b", "B", "C", "D", "z", "delta_bias"])


@pytest.mark.parametrize("hw", [(2, 3), (3, 2)])
def test_ss2d_bwd_matches_finite_differences(hw):
    H, W = hw
    rng = np.random.default_rng(41 + H)
    B, D, N, K = 1, 2, 2, 4
    L = H * W
    t = {
        "x": rng.normal(size=(B, D, H, W)),
        "delta": rng.normal(size=(B, K, D, L)) * 0.5,
        "A": -rng.uniform(0.2, 2.0, size=(K, D, N)),
        "B": rng.normal(size=(B, K, N, L)),
        "C": rng.normal(size=(B, K, N, L)),
        "D": rng.normal(size=(K, D)),
        "z": rng.normal(size=(B, D, H, W)),
        "delta_bias": rng.normal(size=(K, D)) * 0.2,
    }
    g = rng.normal(size=(B, D, H, W))
    grads = oracle.ss2d_bwd(g, **t)
    _fd_check(lambda **kw: oracle.ss2d(**kw), t, grads, g,
              ["x", "delta", "A", "B", "C", "D", "z", "delta_bias"])


def test_bwd_special_cases():
    # A = 0 and no softplus: y_t = sum_n C_t sum_{s<=t} delta_s B_s u_s + D u_t,
    # so dC_t = g_t * (prefix sum of delta B u), written out with np.cumsum
    rng = np.random.default_rng(3)
    B, D, L, N = 1, 1, 7, 2
    u = rng.normal(size=(B, D, L))
    dl = np.abs(rng.normal(size=(B, D, L))) + 0.1
    Bm = rng.normal(size=(B, N, L))
    Cm = rng.normal(size=(B, N, L))
    g = rng.normal(size=(B, D, L))
    r = oracle.selective_scan_bwd(g, u, dl, np.zeros((D, N)), Bm, Cm, delta_softplus=False)
    pref = np.cumsum(dl[0, 0][None, :] * Bm[0] * u[0, 0][None, :], axis=1)
    np.testing.assert_allclose(r["dC"][0], g[0, 0][None, :] * pref, rtol=1e-12, atol=1e-12)
    # dD = sum over rows and time of g * u (the skip term is linear)
    r = oracle.selective_scan_bwd(g, u, dl, -np.ones((D, N)), Bm, Cm, D=np.ones(D))
    assert abs(r["dD"][0] - float((g * u).sum())) < 1e-12
