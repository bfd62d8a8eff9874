"""Pins of the oracle's output epilogue (Head RMSNorm per decay tier, then the SiLU(g) gate),
on the CPU: textbook values of SiLU, unit RMS of the normalised head, invariance to the scale
of o, the tier a head takes its weight from, and central finite differences of the
hand-derived gradient."""
import numpy as np
import pytest

import oracle


def _rand(seed, N, H, C=192):
    r = np.random.default_rng(seed)
    return r.normal(size=(N, H, C)), r.normal(size=(N, H, C))


def test_silu_values():
    # y / (o r w) = SiLU(g): SiLU(0) = 0, SiLU(1) = 1/(1 + e^-1), SiLU(x) -> x for large x
    o = np.ones((1, 1, 4))
    g = np.array([[[0.0, 1.0, 40.0, -40.0]]])
    y, r = oracle.head_norm_gate(o, g, np.ones((1, 4)), 1, 0.0)
    assert r[0, 0] == 1.0
    assert y[0, 0, 0] == 0.0
    assert abs(y[0, 0, 1] - 0.7310585786300049) < 1e-15
    assert abs(y[0, 0, 2] - 40.0) < 1e-12 and abs(y[0, 0, 3]) < 1e-15


def test_normalised_head_has_unit_rms_and_scale_invariance():
    o, _ = _rand(1, 5, 4)
    g = np.full_like(o, 40.0)  # SiLU(40) = 40 to fp64 precision
    y, r = oracle.head_norm_gate(o, g, np.ones((2, 192)), 2, 0.0)
    assert np.allclose(np.sqrt(np.mean((y / 40.0) ** 2, axis=-1)), 1.0, rtol=1e-12)
    y2, _ = oracle.head_norm_gate(7.5 * o, g, np.ones((2, 192)), 2, 0.0)
    assert np.allclose(y, y2, rtol=1e-12)
    # eps enters as mean + eps: a row of zeros stays zero, r = eps^-1/2
    _, r0 = oracle.head_norm_gate(np.zeros((1, 1, 192)), g[:1, :1], np.ones((1, 192)), 1, 0.25)
    assert r0[0, 0] == 2.0


def test_heads_take_their_tiers_weight():
    N, H, T = 3, 6, 3  # tiers of 2 consecutive heads
    o, g = _rand(2, N, H)
    o[:] = o[:, :1]    # every head sees the same row
    g[:] = g[:, :1]
    w = np.arange(1, T + 1, dtype=np.float64)[:, None] * np.ones((T, 192))
    y, _ = oracle.head_norm_gate(o, g, w, T, 1e-6)
    for h in range(H):
        assert np.allclose(y[:, h], (h // 2 + 1) * y[:, 0] / 1.0, rtol=1e-12)


@pytest.mark.parametrize("n_tiers", [1, 2, 4])
def test_gradient_matches_finite_differences(n_tiers):
    N, H, C, eps = 2, 4, 192, 1e-3
    r = np.random.default_rng(3)
    o, g = r.normal(size=(N, H, C)), r.normal(size=(N, H, C))
    w = r.normal(size=(n_tiers, C))
    dy = r.normal(size=(N, H, C))
    d_o, dg, dw = oracle.head_norm_gate_bwd(dy, o, g, w, n_tiers, eps)
    loss = lambda o_, g_, w_: np.sum(oracle.head_norm_gate(o_, g_, w_, n_tiers, eps)[0] * dy)
    h = 1e-6
    for idx in [(0, 0, 0), (1, 3, 191), (0, 2, 77), (1, 1, 5)]:
        for x, d, name in ((o, d_o, "o"), (g, dg, "g")):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = (xp, g, w) if name == "o" else (o, xp, w)
            args_m = (xm, g, w) if name == "o" else (o, xm, w)
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - d[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, d[idx])
    for idx in [(0, 0), (n_tiers - 1, 191), (n_tiers // 2, 100)]:
        wp, wm = w.copy(), w.copy()
        wp[idx] += h
        wm[idx] -= h
        fd = (loss(o, g, wp) - loss(o, g, wm)) / (2 * h)
        assert abs(fd - dw[idx]) <= 1e-6 * max(1.0, abs(fd))


def test_tiers_must_divide_heads():
    o, g = _rand(4, 1, 6)
    with pytest.raises(ValueError):
        oracle.head_norm_gate(o, g, np.ones((4, 192)), 4, 1e-6)
