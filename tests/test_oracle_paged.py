"""Pins of the oracle's state-pool decode (tests run on the CPU): with every page active in
order it is the plain decode step over the whole pool; the order of the active set does not
matter; states it does not name are untouched; one page twice in a call is refused."""
import numpy as np
import pytest

import oracle
import synth


def _case(seed, P=5, PL=3, H=2, n=3, L=2):
    pool = synth.normal(seed, synth.INIT, (P, PL, H, 96, 192), 0.05)
    q = synth.normal(seed, synth.Q, (n, L, H, 96), 96 ** -0.5)
    k = synth.normal(seed, synth.K, (n, L, H, 96))
    v = synth.normal(seed, synth.V, (n, L, H, 192))
    a = synth.aug_balance(seed, (L, H, 96), 0.1)
    return pool, q, k, v, a, oracle.decay_schedule(H)


def test_all_pages_in_order_is_the_plain_step():
    pool, q, k, v, a, g = _case(61, P=3, PL=2, n=3, L=2)
    o, new = oracle.decode_step_paged(pool, [0, 1, 2], 0, q, k, v, g, a)
    o2, st = oracle.decode_step(pool, q, k, v, g, a)
    assert np.array_equal(o, o2) and np.array_equal(new, st)


def test_active_set_order_does_not_matter():
    pool, q, k, v, a, g = _case(62)
    page = np.array([4, 0, 2])
    perm = np.array([2, 0, 1])
    o1, n1 = oracle.decode_step_paged(pool, page, 1, q, k, v, g, a)
    o2, n2 = oracle.decode_step_paged(pool, page[perm], 1, q[perm], k[perm], v[perm], g, a)
    assert np.array_equal(o1[perm], o2) and np.array_equal(n1, n2)


def test_untouched_states_and_one_token_update():
    pool, q, k, v, a, g = _case(63)
    page = [3, 1, 4]
    _, new = oracle.decode_step_paged(pool, page, 1, q, k, v, g, a)
    keep = np.ones(pool.shape[:2], bool)
    keep[np.ix_(page, [1, 2])] = False
    assert np.array_equal(new[keep], pool[keep])
    # a touched state moved by exactly one rank-1 update: S' - lambda S = k v^T
    lam = np.exp(g)
    d = new[3, 1, 0] - lam[0] * pool[3, 1, 0]
    kv = np.outer(k[0, 0, 0].astype(np.float64), v[0, 0, 0].astype(np.float64))
    assert np.allclose(d, kv, rtol=0, atol=1e-12)


def test_duplicate_pages_refused():
    pool, q, k, v, a, g = _case(64)
    with pytest.raises(ValueError):
        oracle.decode_step_paged(pool, [1, 1, 2], 0, q, k, v, g, a)
