"""Pins of the oracle's slice functions (a sequence cut into consecutive slices, as the
sequence-sharded prefill across ranks does), on the CPU: the link of the slices' sums must
reproduce the token recurrence's state at every slice boundary, and the reverse link the
backward's adjoint there; the state sum must equal its closed form.  Planted mistakes in a
copy of the link (one decay step short, slices taken from the wrong end, the boundary
dropped) each fail a pin."""
import numpy as np
import pytest

import synth

LENS = [64, 200, 36]
H = 3


def _seq(T=sum(LENS), seed=71):
    q, k, v = synth.qkv(seed, 2, T, H, bf16=False)
    dO = synth.grad_out(seed, 2, T, H, bf16=False)
    a = synth.aug_balance(seed, (H, 96), 0.1)
    init = synth.init_state(seed, 2, H, 0.05)
    dfin = synth.normal(seed, synth.DFIN, (2, H, 96, 192), 0.05)
    return [np.asarray(x, np.float64) for x in (q, k, v, dO, a, init, dfin)]


def _gamma():
    import oracle
    # half-lives 1, 8, 64: every slice length leaves a visible decay
    return oracle.decay_schedule(H, 1.0, 64.0)


def _boundary_errors(link):
    """Largest relative error of the linked states and adjoints at every slice boundary."""
    import oracle
    q, k, v, dO, a, init, dfin = _seq()
    g = _gamma()
    edges = np.cumsum([0] + LENS)
    U = np.stack([oracle.slice_state_sum(k[:, s:e], v[:, s:e], g)
                  for s, e in zip(edges[:-1], edges[1:])])
    Up = np.stack([oracle.slice_adjoint_sum(q[:, s:e], dO[:, s:e], g)
                   for s, e in zip(edges[:-1], edges[1:])])
    rel = lambda x, y: float(np.abs(x - y).max() / np.sqrt(np.mean(y * y)))
    errs = []
    for r in range(len(LENS)):
        # the state entering slice r = the recurrence's state after the tokens before it
        t = edges[r]
        want = init if t == 0 else oracle.fwd(q[:, :t], k[:, :t], v[:, :t], g, a, init)[1]
        errs.append(rel(link(U, LENS, r, g, init, False), want))
        # the adjoint of the state leaving slice r = the d_init_state of the backward over the
        # tokens after it
        e = edges[r + 1]
        want = dfin if e == edges[-1] else oracle.bwd(q[:, e:], k[:, e:], v[:, e:], g, a,
                                                       dO[:, e:], None, dfin)["d_init_state"]
        errs.append(rel(link(Up, LENS, r, g, dfin, True), want))
    # past the last slice: the whole sequence's final state
    fin = oracle.fwd(q, k, v, g, a, init)[1]
    errs.append(rel(link(U, LENS, len(LENS), g, init, False), fin))
    return max(errs)


def test_link_of_slice_sums_reproduces_the_recurrence_at_every_boundary():
    import oracle
    assert _boundary_errors(oracle.state_link) < 1e-11


def test_slice_sums_equal_their_closed_forms():
    import oracle
    q, k, v, dO, *_ = _seq(T=37)
    g = _gamma()
    lam = np.exp(g)
    T = q.shape[1]
    t = np.arange(T)
    w_fwd = lam[None, :] ** (T - 1 - t)[:, None]  # [T, H]
    w_rev = lam[None, :] ** (t + 1)[:, None]
    U = np.einsum("th,bthi,bthn->bhin", w_fwd, k, v)
    Up = np.einsum("th,bthi,bthn->bhin", w_rev, q, dO)
    rel = lambda x, y: float(np.abs(x - y).max() / np.sqrt(np.mean(y * y)))
    assert rel(oracle.slice_state_sum(k, v, g), U) < 1e-12
    assert rel(oracle.slice_adjoint_sum(q, dO, g), Up) < 1e-12


def _mutant(kind):
    def link(U_all, lens, rank, gamma, boundary=None, reverse=False):
        U = np.asarray(U_all, np.float64)
        lam = np.exp(np.asarray(gamma, np.float64))[None, :, None, None]
        s = np.zeros(U.shape[1:]) if (boundary is None or kind == "boundary_dropped") \
            else np.array(boundary, np.float64)
        order = range(len(lens) - 1, rank, -1) if reverse else range(rank)
        if kind == "wrong_end":
            order = range(rank) if reverse else range(len(lens) - 1, len(lens) - 1 - rank, -1)
        for j in order:
            n = int(lens[j]) - (1 if kind == "one_step_short" else 0)
            s = lam ** n * s + U[j]
        return s
    return link


@pytest.mark.parametrize("kind", ["one_step_short", "wrong_end", "boundary_dropped"])
def test_planted_link_mistakes_fail_the_pin(kind):
    assert _boundary_errors(_mutant(kind)) > 1e-3
