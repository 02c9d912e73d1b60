"""Pins for the fp64 oracle (CPU only).

The oracle is checked against things other than itself: the unrolled closed
form (tests/bruteforce.py, no recurrence), a 50-digit mpmath evaluation,
limits with closed forms, algebraic invariants, reductions between the three
operations, and the hand-derived SS2D cross-scan orders in tests/golden/.
"""
import os

import mpmath
import numpy as np
import pytest

import oracle
from bruteforce import closed_form_sequence, silu_gate, softplus

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_single(rng, Bn, Dn, L, N, scale_dt=0.5):
    return dict(
        u=rng.standard_normal((Bn, Dn, L)),
        delta=scale_dt * rng.standard_normal((Bn, Dn, L)),
        A=-rng.uniform(0.3, 4.0, (Dn, N)),
        B=rng.standard_normal((Bn, N, L)),
        C=rng.standard_normal((Bn, N, L)),
        D=rng.uniform(0.5, 1.5, Dn),
        z=rng.standard_normal((Bn, Dn, L)),
        delta_bias=rng.uniform(-3.0, 0.5, Dn),
    )


def brute_single(p, delta_softplus=True, gate=True):
    u, dt, A, B, C = p["u"], p["delta"], p["A"], p["B"], p["C"]
    Bn, Dn, L = u.shape
    y = np.empty_like(u)
    for b in range(Bn):
        for d in range(Dn):
            y[b, d] = closed_form_sequence(u[b, d], dt[b, d], A[d], B[b], C[b],
                                           p["D"][d], p["delta_bias"][d], delta_softplus)
            if gate:
                y[b, d] = silu_gate(y[b, d], p["z"][b, d])
    return y


def rel_err(a, b):
    return np.max(np.abs(a - b) / (1.0 + np.abs(b)))


# ---------------------------------------------------------------- closed form
@pytest.mark.parametrize("L,N", [(1, 1), (2, 3), (7, 16), (24, 16), (13, 5)])
@pytest.mark.parametrize("sp", [True, False])
def test_single_matches_closed_form(L, N, sp):
    rng = np.random.default_rng(100 + L * 7 + N)
    p = rand_single(rng, 2, 3, L, N)
    if not sp:  # keep delta positive without softplus
        p["delta"] = np.abs(p["delta"]) * 0.1
        p["delta_bias"] = np.abs(p["delta_bias"]) * 0.05
    y = oracle.selective_scan(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"],
                              p["z"], p["delta_bias"], delta_softplus=sp)
    assert rel_err(y, brute_single(p, sp)) < 1e-12


def test_single_matches_50_digit_closed_form():
    # rational inputs, evaluated at 50 significant digits
    mpmath.mp.dps = 50
    L, N = 5, 3
    u = [0.5, -1.25, 2.0, 0.75, -0.5]
    dt = [0.125, -0.5, 0.25, 1.0, -1.5]
    A = [-1.0, -2.5, -0.75]
    Bm = [[1.0, -0.5, 0.25, 2.0, 1.5], [0.5, 0.5, -1.0, 0.125, -2.0],
          [-1.5, 1.0, 0.75, -0.25, 0.5]]
    Cm = [[0.25, 1.0, -1.0, 0.5, 2.0], [-0.75, 0.5, 1.25, -1.0, 0.25],
          [1.0, -2.0, 0.5, 0.75, -0.5]]
    Dd, bias = 0.875, -0.375
    z = [0.5, -1.0, 1.5, -0.25, 2.0]

    def sp(x):
        return mpmath.log(1 + mpmath.exp(x))

    delta = [sp(mpmath.mpf(dt[t]) + bias) for t in range(L)]
    ref = []
    for t in range(L):
        tot = mpmath.mpf(0)
        for s in range(t + 1):
            run = sum(delta[s + 1:t + 1], mpmath.mpf(0))
            for n in range(N):
                tot += Cm[n][t] * mpmath.exp(A[n] * run) * delta[s] * Bm[n][s] * u[s]
        v = tot + Dd * u[t]
        ref.append(float(v * z[t] / (1 + mpmath.exp(-z[t]))))
    y = oracle.selective_scan(np.array(u)[None, None], np.array(dt)[None, None],
                              np.array(A)[None], np.array(Bm)[None], np.array(Cm)[None],
                              np.array([Dd]), np.array(z)[None, None], np.array([bias]))
    np.testing.assert_allclose(y[0, 0], ref, rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- limits
def test_delta_zero_gives_skip_only():
    rng = np.random.default_rng(1)
    p = rand_single(rng, 2, 4, 9, 16)
    p["delta"][:] = 0.0
    p["delta_bias"][:] = 0.0
    y = oracle.selective_scan(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"],
                              None, p["delta_bias"], delta_softplus=False)
    assert np.array_equal(y, p["D"][None, :, None] * p["u"])
    yg = oracle.selective_scan(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"],
                               p["z"], p["delta_bias"], delta_softplus=False)
    np.testing.assert_allclose(yg, silu_gate(p["D"][None, :, None] * p["u"], p["z"]),
                               rtol=1e-15, atol=0)


def test_A_zero_is_a_prefix_sum():
    rng = np.random.default_rng(2)
    p = rand_single(rng, 2, 3, 31, 7)
    p["A"][:] = 0.0
    y = oracle.selective_scan(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"],
                              None, p["delta_bias"])
    delta = softplus(p["delta"] + p["delta_bias"][None, :, None])       # [B,D,L]
    inp = delta[:, :, None, :] * p["B"][:, None] * p["u"][:, :, None]  # [B,D,N,L]
    h = np.cumsum(inp, axis=-1)
    ref = np.sum(p["C"][:, None] * h, axis=2) + p["D"][None, :, None] * p["u"]
    assert rel_err(y, ref) < 1e-12


def test_constant_input_geometric_series():
    L, dlt, a, Dd = 40, 0.3, -1.7, 0.25
    ones = np.ones((1, 1, L))
    y = oracle.selective_scan(ones, np.full((1, 1, L), dlt), np.array([[a]]),
                              np.ones((1, 1, L)), np.ones((1, 1, L)), np.array([Dd]),
                              None, np.array([0.0]), delta_softplus=False)
    r = np.exp(dlt * a)
    t = np.arange(L)
    ref = dlt * (1 - r ** (t + 1)) / (1 - r) + Dd
    np.testing.assert_allclose(y[0, 0], ref, rtol=1e-13)


def test_length_one():
    rng = np.random.default_rng(3)
    p = rand_single(rng, 3, 5, 1, 16)
    y = oracle.selective_scan(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"],
                              None, p["delta_bias"])
    delta = softplus(p["delta"] + p["delta_bias"][None, :, None])
    ref = (np.einsum("bnl,bdl->bdl", p["C"] * p["B"], delta * p["u"])
           + p["D"][None, :, None] * p["u"])
    assert rel_err(y, ref) < 1e-13
    # At L = 1 with equal parameter sets, the two branches agree (the one case
    # where the forward output at 0 equals the backward output at L-1).
    yv2 = oracle.bimamba_v2(p["u"], p["delta"], p["delta"], p["A"], p["A"], p["B"],
                            p["C"], p["B"], p["C"], p["D"], p["D"], None,
                            p["delta_bias"], p["delta_bias"], out_scale=0.5)
    assert rel_err(yv2, y) < 1e-15


# ---------------------------------------------------------------- invariants
def test_linear_in_u_before_gate():
    rng = np.random.default_rng(4)
    p = rand_single(rng, 2, 3, 25, 16)
    u2 = rng.standard_normal(p["u"].shape)
    al, be = 1.75, -0.625

    def run(u):
        return oracle.selective_scan(u, p["delta"], p["A"], p["B"], p["C"], p["D"],
                                     None, p["delta_bias"])

    lhs = run(al * p["u"] + be * u2)
    rhs = al * run(p["u"]) + be * run(u2)
    assert rel_err(lhs, rhs) < 1e-12


def rand_v2(rng, Bn, Dn, L, N, shared_u=True):
    f = rand_single(rng, Bn, Dn, L, N)
    b = rand_single(rng, Bn, Dn, L, N)
    return dict(u=f["u"], u_b=None if shared_u else b["u"], delta=f["delta"],
                delta_b=b["delta"], A=f["A"], A_b=b["A"], B=f["B"], C=f["C"],
                B_b=b["B"], C_b=b["C"], D=f["D"], D_b=b["D"], z=f["z"],
                delta_bias=f["delta_bias"], delta_bias_b=b["delta_bias"])


def v2(p, out_scale=0.5, **over):
    q = {**p, **over}
    return oracle.bimamba_v2(q["u"], q["delta"], q["delta_b"], q["A"], q["A_b"],
                             q["B"], q["C"], q["B_b"], q["C_b"], q["D"], q["D_b"],
                             q["z"], q["delta_bias"], q["delta_bias_b"], q["u_b"],
                             out_scale=out_scale)


@pytest.mark.parametrize("shared_u", [True, False])
def test_v2_matches_closed_form_both_branches(shared_u):
    rng = np.random.default_rng(5)
    p = rand_v2(rng, 2, 3, 17, 16, shared_u)
    y = v2(p, out_scale=0.5)
    ub = p["u"] if p["u_b"] is None else p["u_b"]
    ref = np.empty_like(y)
    for b in range(2):
        for d in range(3):
            yf = closed_form_sequence(p["u"][b, d], p["delta"][b, d], p["A"][d], p["B"][b],
                                      p["C"][b], p["D"][d], p["delta_bias"][d])
            yb = closed_form_sequence(ub[b, d][::-1], p["delta_b"][b, d][::-1], p["A_b"][d],
                                      p["B_b"][b][:, ::-1], p["C_b"][b][:, ::-1],
                                      p["D_b"][d], p["delta_bias_b"][d])
            ref[b, d] = silu_gate(0.5 * (yf + yb[::-1]), p["z"][b, d])
    assert rel_err(y, ref) < 1e-12


def test_v2_time_reversal_swaps_branches():
    rng = np.random.default_rng(6)
    p = rand_v2(rng, 2, 3, 23, 16, shared_u=False)
    y = v2(p)
    r = lambda a: None if a is None else a[..., ::-1].copy()
    q = dict(u=r(p["u_b"]), u_b=r(p["u"]), delta=r(p["delta_b"]), delta_b=r(p["delta"]),
             A=p["A_b"], A_b=p["A"], B=r(p["B_b"]), C=r(p["C_b"]), B_b=r(p["B"]),
             C_b=r(p["C"]), D=p["D_b"], D_b=p["D"], z=r(p["z"]),
             delta_bias=p["delta_bias_b"], delta_bias_b=p["delta_bias"])
    assert rel_err(v2(q), y[..., ::-1]) < 1e-13


def test_v2_with_silent_backward_is_scaled_single():
    rng = np.random.default_rng(7)
    p = rand_v2(rng, 2, 3, 19, 16)
    zeros = np.zeros_like(p["C_b"])
    y = v2(p, out_scale=0.5, C_b=zeros, D_b=np.zeros(3))
    ys = oracle.selective_scan(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"],
                               p["z"], p["delta_bias"])
    assert rel_err(y, 0.5 * ys) < 1e-14


def test_v1_equals_v2_with_shared_sets():
    rng = np.random.default_rng(8)
    p = rand_v2(rng, 2, 3, 21, 16)
    y1 = oracle.bimamba_v1(p["u"], p["delta"], p["A"], p["A_b"], p["B"], p["C"], p["D"],
                           p["z"], p["delta_bias"], out_scale=1.0)
    y2 = v2(p, out_scale=1.0, delta_b=p["delta"], B_b=p["B"], C_b=p["C"], D_b=p["D"],
            delta_bias_b=p["delta_bias"])
    assert np.array_equal(y1, y2)


def test_gate_commutes_with_flip():
    # The pages' v2 path gates each branch by its own z (the backward branch
    # runs on xz.flip), then averages; the oracle gates once after the fuse.
    rng = np.random.default_rng(9)
    p = rand_v2(rng, 2, 2, 15, 16)
    y = v2(p, out_scale=0.5)
    yf = oracle.selective_scan(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                               p["delta_bias"])
    f = lambda a: a[..., ::-1].copy()
    yb = oracle.selective_scan(f(p["u"]), f(p["delta_b"]), p["A_b"], f(p["B_b"]),
                               f(p["C_b"]), p["D_b"], f(p["z"]), p["delta_bias_b"])
    assert rel_err(y, 0.5 * (yf + f(yb))) < 1e-13


# ---------------------------------------------------------------- SS2D
def read_golden_orders():
    orders = {}
    with open(os.path.join(GOLDEN, "ss2d_cross_scan_2x3.txt")) as fh:
        for line in fh:
            if line.strip() and not line.startswith("#"):
                k, *idx = map(int, line.split())
                orders[k] = idx
    return orders


def test_cross_scan_orders_match_hand_derived_2x3():
    gold = read_golden_orders()
    for k in range(4):
        assert list(oracle.cross_scan_index(2, 3, k)) == gold[k]


@pytest.mark.parametrize("H,W", [(3, 4), (5, 2), (4, 4)])
def test_cross_scan_orders_match_numpy_views(H, W):
    img = np.arange(H * W).reshape(H, W)
    ref = [img.reshape(-1), img.T.reshape(-1), img.reshape(-1)[::-1], img.T.reshape(-1)[::-1]]
    for k in range(4):
        assert np.array_equal(oracle.cross_scan_index(H, W, k), ref[k])


def rand_ss2d(rng, Bn, Dn, H, W, N):
    L = H * W
    return dict(x=rng.standard_normal((Bn, Dn, H, W)),
                delta=0.5 * rng.standard_normal((Bn, 4, Dn, L)),
                A=-rng.uniform(0.3, 4.0, (4, Dn, N)),
                B=rng.standard_normal((Bn, 4, N, L)), C=rng.standard_normal((Bn, 4, N, L)),
                D=rng.uniform(0.5, 1.5, (4, Dn)), z=rng.standard_normal((Bn, Dn, H, W)),
                delta_bias=rng.uniform(-3.0, 0.5, (4, Dn)))


def ss2d(p, **over):
    q = {**p, **over}
    return oracle.ss2d(q["x"], q["delta"], q["A"], q["B"], q["C"], q["D"], q["z"],
                       q["delta_bias"])


@pytest.mark.parametrize("H,W", [(3, 4), (4, 3), (2, 2)])
def test_ss2d_matches_closed_form(H, W):
    rng = np.random.default_rng(10 + H * W)
    p = rand_ss2d(rng, 2, 2, H, W, 16)
    y = ss2d(p)
    img = np.arange(H * W).reshape(H, W)
    orders = [img.reshape(-1), img.T.reshape(-1), img.reshape(-1)[::-1], img.T.reshape(-1)[::-1]]
    ref = np.zeros((2, 2, H * W))
    for b in range(2):
        for d in range(2):
            xf = p["x"][b, d].reshape(-1)
            for k in range(4):
                yk = closed_form_sequence(xf[orders[k]], p["delta"][b, k, d], p["A"][k, d],
                                          p["B"][b, k], p["C"][b, k], p["D"][k, d],
                                          p["delta_bias"][k, d])
                ref[b, d, orders[k]] += yk
            ref[b, d] = silu_gate(ref[b, d], p["z"][b, d].reshape(-1))
    assert rel_err(y.reshape(2, 2, -1), ref) < 1e-12


def test_ss2d_transpose_symmetry():
    rng = np.random.default_rng(11)
    H, W = 3, 5
    p = rand_ss2d(rng, 2, 3, H, W, 16)
    y = ss2d(p)
    sw = [1, 0, 3, 2]  # transposing the map swaps row-major and column-major scans
    q = dict(x=p["x"].transpose(0, 1, 3, 2).copy(), z=p["z"].transpose(0, 1, 3, 2).copy(),
             delta=p["delta"][:, sw].copy(), A=p["A"][sw].copy(), B=p["B"][:, sw].copy(),
             C=p["C"][:, sw].copy(), D=p["D"][sw].copy(), delta_bias=p["delta_bias"][sw].copy())
    assert rel_err(ss2d(q), y.transpose(0, 1, 3, 2)) < 1e-13
    # identical per-direction parameters (and streams): symmetric without a swap
    same = {k: (np.repeat(v[:, :1], 4, axis=1) if k in ("delta", "B", "C")
                else np.repeat(v[:1], 4, axis=0)) for k, v in p.items()
            if k in ("delta", "B", "C", "A", "D", "delta_bias")}
    p2 = {**p, **same}
    q2 = {**p2, "x": p["x"].transpose(0, 1, 3, 2).copy(), "z": p["z"].transpose(0, 1, 3, 2).copy()}
    assert rel_err(ss2d(q2), ss2d(p2).transpose(0, 1, 3, 2)) < 1e-13


def test_ss2d_row_pair_reduces_to_bimamba_v2():
    rng = np.random.default_rng(12)
    H, W = 4, 5
    p = rand_ss2d(rng, 2, 3, H, W, 16)
    Cz = p["C"].copy()
    Cz[:, 1] = 0.0
    Cz[:, 3] = 0.0
    Dz = p["D"].copy()
    Dz[1] = 0.0
    Dz[3] = 0.0
    y = ss2d(p, C=Cz, D=Dz)
    f = lambda a: a[..., ::-1].copy()  # direction 2 streams are in scan (reversed) order
    yv = oracle.bimamba_v2(p["x"].reshape(2, 3, -1), p["delta"][:, 0], f(p["delta"][:, 2]),
                           p["A"][0], p["A"][2], p["B"][:, 0], p["C"][:, 0], f(p["B"][:, 2]),
                           f(p["C"][:, 2]), p["D"][0], p["D"][2], p["z"].reshape(2, 3, -1),
                           p["delta_bias"][0], p["delta_bias"][2], out_scale=1.0)
    assert rel_err(y.reshape(2, 3, -1), yv) < 1e-13


# ---------------------------------------------------------------- regression
def test_oracle_regression_fixture():
    import json

    with open(os.path.join(GOLDEN, "oracle_regression.json")) as fh:
        fx = json.load(fh)
    import sys

    sys.path.insert(0, GOLDEN)
    from make_golden import compute_cases  # the script that wrote the fixture

    got = compute_cases()
    for name, ref in fx["cases"].items():
        np.testing.assert_allclose(np.array(got[name]), np.array(ref), rtol=1e-13, atol=1e-15,
                                   err_msg=name)
