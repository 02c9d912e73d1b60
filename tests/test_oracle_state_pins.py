"""Pins of the oracle's final states (CPU): every direction's last state
against the unrolled closed form of tests/bruteforce.py, which never runs
the recurrence, on the flipped or cross-scanned sequences built here with
numpy views (independent of the oracle's own copies)."""
import numpy as np
import pytest

import oracle
from bruteforce import closed_form_last_state


def _rand(rng, B, D, L, N):
    return dict(u=rng.normal(size=(B, D, L)), delta=rng.normal(size=(B, D, L)) * 0.5,
                A=-rng.uniform(0.2, 2.0, size=(D, N)), B=rng.normal(size=(B, N, L)),
                C=rng.normal(size=(B, N, L)), delta_bias=rng.normal(size=(D,)) * 0.2)


@pytest.mark.parametrize("sp", [True, False])
def test_single_last_state_matches_closed_form(sp):
    rng = np.random.default_rng(5 + sp)
    p = _rand(rng, 2, 3, 9, 4)
    if not sp:
        p["delta"] = np.abs(p["delta"]) + 0.05
    got = oracle.selective_scan_last_state(p["u"], p["delta"], p["A"], p["B"],
                                           delta_bias=p["delta_bias"], delta_softplus=sp)
    assert got.shape == (1, 2, 3, 4)
    for b in range(2):
        for d in range(3):
            ref = closed_form_last_state(p["u"][b, d], p["delta"][b, d], p["A"][d], p["B"][b],
                                         p["delta_bias"][d], sp)
            np.testing.assert_allclose(got[0, b, d], ref, rtol=1e-12, atol=1e-14)


def test_v2_backward_branch_state_is_the_flipped_sequence_at_position_0():
    rng = np.random.default_rng(9)
    p = _rand(rng, 1, 2, 7, 3)
    q = _rand(rng, 1, 2, 7, 3)              # the backward branch's own set
    got = oracle.bimamba_v2_last_state(p["u"], p["delta"], q["delta"], p["A"], q["A"], p["B"],
                                       p["C"], q["B"], q["C"], delta_bias=p["delta_bias"],
                                       delta_bias_b=q["delta_bias"], u_b=q["u"])
    for d in range(2):
        f = closed_form_last_state(p["u"][0, d], p["delta"][0, d], p["A"][d], p["B"][0],
                                   p["delta_bias"][d])
        bk = closed_form_last_state(q["u"][0, d][::-1], q["delta"][0, d][::-1], q["A"][d],
                                    q["B"][0][:, ::-1], q["delta_bias"][d])
        np.testing.assert_allclose(got[0, 0, d], f, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(got[1, 0, d], bk, rtol=1e-12, atol=1e-14)


def test_ss2d_last_states_match_closed_form_on_numpy_orders():
    rng = np.random.default_rng(13)
    B, D, H, W, N = 1, 2, 2, 3, 2
    L = H * W
    x = rng.normal(size=(B, D, H, W))
    delta = rng.normal(size=(B, 4, D, L)) * 0.5
    A = -rng.uniform(0.2, 2.0, size=(4, D, N))
    Bm = rng.normal(size=(B, 4, N, L))
    bias = rng.normal(size=(4, D)) * 0.2
    got = oracle.ss2d_last_state(x, delta, A, Bm, Bm, delta_bias=bias)
    for d in range(D):
        img = x[0, d]
        seqs = [img.reshape(-1), img.T.reshape(-1), img.reshape(-1)[::-1], img.T.reshape(-1)[::-1]]
        for k in range(4):
            ref = closed_form_last_state(seqs[k], delta[0, k, d], A[k, d], Bm[0, k], bias[k, d])
            np.testing.assert_allclose(got[k, 0, d], ref, rtol=1e-12, atol=1e-14)
