"""Pins of the oracle's causal depth-wise conv + SiLU (CPU): the impulse response is the
filter reversed in time, splitting a sequence and carrying the 3-input state changes
nothing, the decode step is the forward over one token, and the hand-derived gradient
matches central finite differences."""
import numpy as np
import pytest

import oracle


def test_impulse_response_is_the_filter():
    D, T = 3, 9
    w = np.array([[1.0, 2.0, 3.0, 4.0], [0.5, -1.0, 0.25, 2.0], [0.0, 0.0, 0.0, 1.0]])
    x = np.zeros((1, T, D))
    x[0, 2, :] = 1.0  # unit impulse at t = 2
    y, fin = oracle.conv_fwd(x, w)
    # z_t = w[d, 3 - (t - 2)] for t = 2..5, 0 elsewhere; y = z sigmoid(z)
    for t in range(T):
        for d in range(D):
            k = 3 - (t - 2)
            zt = w[d, k] if 0 <= k <= 3 else 0.0
            assert abs(y[0, t, d] - zt / (1 + np.exp(-zt))) < 1e-15
    assert np.array_equal(fin[0], x[0, -3:])


def test_state_carry_and_decode():
    r = np.random.default_rng(5)
    B, T, D, T1 = 2, 11, 8, 5
    x = r.normal(size=(B, T, D))
    w, b = r.normal(size=(D, 4)), r.normal(size=D)
    init = r.normal(size=(B, 3, D))
    y, fin = oracle.conv_fwd(x, w, b, init)
    y1, f1 = oracle.conv_fwd(x[:, :T1], w, b, init)
    y2, f2 = oracle.conv_fwd(x[:, T1:], w, b, f1)
    assert np.allclose(np.concatenate([y1, y2], 1), y, rtol=0, atol=1e-14)
    assert np.array_equal(f2, fin)
    st = init.copy()
    for t in range(T):
        yt, st = oracle.conv_decode_step(st, x[:, t], w, b)
        assert np.allclose(yt, y[:, t], rtol=0, atol=1e-14)
    assert np.array_equal(st, fin)
    # a sequence shorter than the state keeps part of the initial state
    _, f = oracle.conv_fwd(x[:, :1], w, b, init)
    assert np.array_equal(f[:, :2], init[:, 1:]) and np.array_equal(f[:, 2], x[:, 0])


def test_gradient_matches_finite_differences():
    r = np.random.default_rng(6)
    B, T, D = 2, 7, 4
    x, dy = r.normal(size=(B, T, D)), r.normal(size=(B, T, D))
    w, b, init = r.normal(size=(D, 4)), r.normal(size=D), r.normal(size=(B, 3, D))
    dx, dinit, dw, db = oracle.conv_bwd(x, w, dy, b, init)
    loss = lambda x_, w_, b_, i_: np.sum(oracle.conv_fwd(x_, w_, b_, i_)[0] * dy)
    h = 1e-6

    def fd(arr, idx, fn):
        p, m = arr.copy(), arr.copy()
        p[idx] += h
        m[idx] -= h
        return (fn(p) - fn(m)) / (2 * h)
    for idx in [(0, 0, 0), (1, 6, 3), (0, 3, 2)]:
        assert abs(fd(x, idx, lambda a: loss(a, w, b, init)) - dx[idx]) < 1e-7
    for idx in [(0, 0, 0), (1, 2, 3), (1, 1, 1)]:
        assert abs(fd(init, idx, lambda a: loss(x, w, b, a)) - dinit[idx]) < 1e-7
    for idx in [(0, 0), (3, 3), (2, 1)]:
        assert abs(fd(w, idx, lambda a: loss(x, a, b, init)) - dw[idx]) < 1e-7
    for idx in [(0,), (3,)]:
        assert abs(fd(b, idx, lambda a: loss(x, w, a, init)) - db[idx]) < 1e-7
