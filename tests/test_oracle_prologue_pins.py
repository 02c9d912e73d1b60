"""Pins of the prologue oracle (CPU): the causal convolution against
numpy's convolve row by row and its impulse response and causality; the
projections against selection and one-hot inputs (a transposed operand or
a wrong split row fails them)."""
import numpy as np
import pytest

from oracle import prologue as pro


@pytest.mark.parametrize("K", [3, 4])
@pytest.mark.parametrize("reverse", [False, True])
def test_conv_matches_numpy_convolve(K, reverse):
    rng = np.random.default_rng(K + 10 * reverse)
    x = rng.normal(size=(2, 3, 11))
    w = rng.normal(size=(3, K))
    b = rng.normal(size=(3,))
    got = pro.causal_conv(x, w, b, reverse)
    for bb in range(2):
        for d in range(3):
            xs = x[bb, d, ::-1] if reverse else x[bb, d]
            # full convolution with the flipped taps, first L outputs: causal
            ref = np.convolve(xs, w[d][::-1])[:11] + b[d]
            np.testing.assert_allclose(got[bb, d], ref, rtol=1e-13, atol=1e-13)


def test_conv_impulse_response_and_causality():
    K, L = 4, 9
    w = np.array([[1.0, 2.0, 3.0, 4.0]])
    x = np.zeros((1, 1, L))
    x[0, 0, 3] = 1.0
    y = pro.causal_conv(x, w)
    # tap k reads position t - (K-1-k): the impulse shows up reversed
    np.testing.assert_array_equal(y[0, 0], [0, 0, 0, 4, 3, 2, 1, 0, 0])
    # nothing before the impulse moves when a later input changes
    x2 = x.copy()
    x2[0, 0, 6] = 5.0
    np.testing.assert_array_equal(pro.causal_conv(x2, w)[0, 0, :6], y[0, 0, :6])


def test_projection_split_with_selection_weights():
    rng = np.random.default_rng(3)
    B, D, L, R, N, K = 1, 6, 5, 2, 2, 3
    x = rng.normal(size=(B, D, L))
    cw = rng.normal(size=(D, K))
    cb = rng.normal(size=(D,))
    # W_x picks channels 5,4 | 0,1 | 2,3 ; W_dt expands dt_low by a one-hot map
    W_x = np.zeros((R + 2 * N, D))
    for row, ch in enumerate([5, 4, 0, 1, 2, 3]):
        W_x[row, ch] = 1.0
    W_dt = np.zeros((D, R))
    W_dt[0, 1] = 1.0
    W_dt[3, 0] = 2.0
    u, dt, Bm, Cm = pro.prologue(x, cw, cb, W_x, W_dt, R, N)
    np.testing.assert_allclose(Bm[0], u[0, [0, 1]], rtol=0, atol=0)
    np.testing.assert_allclose(Cm[0], u[0, [2, 3]], rtol=0, atol=0)
    np.testing.assert_allclose(dt[0, 0], u[0, 4], rtol=0, atol=0)
    np.testing.assert_allclose(dt[0, 3], 2.0 * u[0, 5], rtol=0, atol=0)
    assert not dt[0, [1, 2, 4, 5]].any()


def test_reverse_is_the_prologue_of_the_flipped_input():
    rng = np.random.default_rng(8)
    B, D, L, R, N, K = 2, 4, 7, 2, 3, 4
    x = rng.normal(size=(B, D, L))
    cw, cb = rng.normal(size=(D, K)), rng.normal(size=(D,))
    W_x, W_dt = rng.normal(size=(R + 2 * N, D)), rng.normal(size=(D, R))
    a = pro.prologue(x, cw, cb, W_x, W_dt, R, N, reverse=True)
    b = pro.prologue(x[..., ::-1].copy(), cw, cb, W_x, W_dt, R, N, reverse=False)
    for p, q in zip(a, b):
        np.testing.assert_allclose(p, q, rtol=1e-14, atol=1e-14)
