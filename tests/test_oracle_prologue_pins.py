"""Pins of the prologue oracle (CPU): the causal convolution against
numpy's convolve row by row and its impulse response and causality; the
projections against selection and one-hot inputs (a transposed operand or
a wrong split row fails them).  SS2D: the depthwise conv2d against scipy's
correlate2d and its impulse response; the four directions' sequences
against numpy flatten / transpose / flip; the per-direction projections
with selection weights."""
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


# ---------------------------------------------------------------- SS2D


@pytest.mark.parametrize("Kc,H,W", [(3, 5, 7), (5, 6, 4), (1, 3, 3), (3, 1, 6)])
def test_conv2d_matches_scipy_correlate2d(Kc, H, W):
    from scipy.signal import correlate2d
    rng = np.random.default_rng(Kc * 100 + H * 10 + W)
    x = rng.normal(size=(2, 3, H, W))
    w = rng.normal(size=(3, Kc, Kc))
    b = rng.normal(size=(3,))
    got = pro.depthwise_conv2d(x, w, b)
    for bb in range(2):
        for d in range(3):
            ref = correlate2d(x[bb, d], w[d], mode="same", boundary="fill", fillvalue=0) + b[d]
            np.testing.assert_allclose(got[bb, d], ref, rtol=1e-13, atol=1e-13)


def test_conv2d_impulse_response():
    # a correlation: an impulse at (h0, w0) leaves the kernel rotated by
    # 180 degrees around it
    w = np.arange(1.0, 10.0).reshape(1, 3, 3)
    x = np.zeros((1, 1, 5, 6))
    x[0, 0, 2, 3] = 1.0
    y = pro.depthwise_conv2d(x, w)[0, 0]
    ref = np.zeros((5, 6))
    ref[1:4, 2:5] = w[0, ::-1, ::-1]
    np.testing.assert_array_equal(y, ref)


def _ss2d_weights(rng, D, R, N):
    return (rng.normal(size=(4, R + 2 * N, D)), rng.normal(size=(4, D, R)))


def test_ss2d_directions_are_flatten_transpose_flip():
    # B_k row n selects channel n: B_k must be u's channel n in direction
    # k's order, written independently with numpy
    rng = np.random.default_rng(5)
    Bn, D, H, W, R, N = 2, 4, 3, 5, 2, 3
    x = rng.normal(size=(Bn, D, H, W))
    cw = rng.normal(size=(D, 3, 3))
    W_x = np.zeros((4, R + 2 * N, D))
    for k in range(4):
        for n in range(N):
            W_x[k, R + n, (n + k) % D] = 1.0        # B rows: channel (n + k) mod D
            W_x[k, R + N + n, n] = 2.0              # C rows: twice channel n
    W_dt = rng.normal(size=(4, D, R))
    u, delta, Bm, Cm = pro.ss2d_prologue(x, cw, None, W_x, W_dt, R, N)
    orders = [lambda m: m.reshape(Bn, -1),
              lambda m: m.transpose(0, 2, 1).reshape(Bn, -1),
              lambda m: m.reshape(Bn, -1)[:, ::-1],
              lambda m: m.transpose(0, 2, 1).reshape(Bn, -1)[:, ::-1]]
    for k in range(4):
        for n in range(N):
            np.testing.assert_array_equal(Bm[:, k, n], orders[k](u[:, (n + k) % D]))
            np.testing.assert_array_equal(Cm[:, k, n], 2.0 * orders[k](u[:, n]))


def test_ss2d_dt_projection_per_direction():
    # dt_low rows select channels; W_dt[k] one-hot: delta_k[d] = dt_low
    # row r(d, k), which is channel c(r, k) in direction k's order
    rng = np.random.default_rng(6)
    Bn, D, H, W, R, N = 1, 3, 4, 2, 2, 1
    x = rng.normal(size=(Bn, D, H, W))
    cw = rng.normal(size=(D, 3, 3))
    cb = rng.normal(size=(D,))
    W_x = np.zeros((4, R + 2 * N, D))
    W_dt = np.zeros((4, D, R))
    for k in range(4):
        for r in range(R):
            W_x[k, r, (r + k) % D] = 1.0
        for d in range(D):
            W_dt[k, d, (d + k) % R] = 3.0
    u, delta, _, _ = pro.ss2d_prologue(x, cw, cb, W_x, W_dt, R, N)
    orders = [lambda m: m.reshape(-1), lambda m: m.T.reshape(-1),
              lambda m: m.reshape(-1)[::-1], lambda m: m.T.reshape(-1)[::-1]]
    for k in range(4):
        for d in range(D):
            r = (d + k) % R
            np.testing.assert_array_equal(delta[0, k, d], 3.0 * orders[k](u[0, (r + k) % D]))


def test_ss2d_silu_flag_and_activation():
    rng = np.random.default_rng(7)
    x = rng.normal(size=(1, 2, 3, 4))
    cw = rng.normal(size=(2, 3, 3))
    W_x, W_dt = _ss2d_weights(rng, 2, 1, 2)
    u0, *_ = pro.ss2d_prologue(x, cw, None, W_x, W_dt, 1, 2, silu_act=False)
    u1, *_ = pro.ss2d_prologue(x, cw, None, W_x, W_dt, 1, 2, silu_act=True)
    np.testing.assert_allclose(u0, pro.depthwise_conv2d(x, cw), rtol=0, atol=0)
    np.testing.assert_allclose(u1, u0 / (1.0 + np.exp(-u0)), rtol=1e-15, atol=0)


def test_out_proj_with_selection_weights():
    # W_out rows pick and scale channels (a wrong operand order or a
    # transposed W fails): out[0] = y[2], out[1] = -3 y[0], out[2] = y[1] + y[3]
    rng = np.random.default_rng(11)
    y = rng.normal(size=(2, 4, 7))
    W = np.zeros((3, 4))
    W[0, 2] = 1.0
    W[1, 0] = -3.0
    W[2, 1] = W[2, 3] = 1.0
    out = pro.out_proj(y, W)
    assert out.shape == (2, 3, 7)
    np.testing.assert_array_equal(out[:, 0], y[:, 2])
    np.testing.assert_array_equal(out[:, 1], -3.0 * y[:, 0])
    np.testing.assert_array_equal(out[:, 2], y[:, 1] + y[:, 3])


def test_out_proj_is_position_independent_and_linear():
    # each position is W @ y[:, :, t] (brute force per position) and the
    # map is linear in y
    rng = np.random.default_rng(12)
    y1, y2 = rng.normal(size=(1, 5, 6)), rng.normal(size=(1, 5, 6))
    W = rng.normal(size=(4, 5))
    out = pro.out_proj(y1, W)
    for t in range(6):
        ref = [sum(W[m, k] * y1[0, k, t] for k in range(5)) for m in range(4)]
        np.testing.assert_allclose(out[0, :, t], ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(pro.out_proj(2.0 * y1 + y2, W), 2.0 * out + pro.out_proj(y2, W),
                               rtol=1e-12, atol=1e-12)
