"""Pins of the fp64 oracle to things other than itself.

Each ``pin_*`` takes a loaded oracle library and returns (ok, detail).  They are
used by tests/test_oracle_pins.py on the real oracle and by
tests/test_oracle_mutants.py on copies of it with a planted mistake, to show that
every plausible mistake fails at least one pin.

What pins what (source: "Beyond the KV cache ... Laplace 3B ...", section
"i14 and the Laplace 3B architecture"):
  * pin_decay          -- the decay values printed in "Decay schedule's reach"
                          (lambda_0 = 0.5, lambda_15 ~ 0.9997) and 2^(-1/2048).
  * pin_closed_form    -- brute force o_t = sum_{s<=t} lambda^(t-s) (q_t.k_s) v_s
                          + lambda^(t+1) S_0^T q_t + sigmoid(z_t) v_t (0-based t),
                          and S_T in closed form.
  * pin_aug_zero       -- the article's initialisation a = 0 passes half of the
                          value through: q = 0 gives o = v/2 exactly, and with
                          a = 0 the aug term is exactly v/2.
  * pin_lambda_one     -- lambda = 1, S_0 = 0, a = 0 reduces to the textbook
                          causal (unnormalised) linear attention tril(QK^T)V + v/2.
  * pin_fd             -- central finite differences of the scalar loss for
                          every gradient output of the backward.
  * pin_init_zero      -- init_state = 0 equals no state, bit for bit.
  * pin_state_carry    -- fwd(T1 || T2) = fwd(T2, init = final(T1)).
  * pin_decode         -- one decode step equals token T+1 of the forward
                          (serving matched the reference token for token).
  * pin_chunked        -- an independent fp64 chunked restatement (intra-chunk
                          masked attention + inter-chunk state, section
                          "Challenge 1"), forward and backward, for several chunk
                          sizes, some leaving a shorter last chunk, equals the
                          token recurrence.
  * pin_parts          -- sequences cut into parts that each start from the state
                          and adjoint the linear recurrences give at their
                          boundaries (the decomposition the GPU's long-sequence
                          path uses) equal the token recurrence.
"""
from __future__ import annotations

import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    den = max(np.abs(b).max(), 1e-300)
    return float(np.abs(a - b).max() / den)


def _rand_problem(seed, B, T, H, dk, dv, a_std=0.5, with_init=True, t_max=8.0, lib=None):
    r = _rng(seed)
    q = r.standard_normal((B, T, H, dk)) * dk ** -0.5
    k = r.standard_normal((B, T, H, dk))
    v = r.standard_normal((B, T, H, dv))
    a = r.standard_normal((H, dk)) * a_std
    init = r.standard_normal((B, H, dk, dv)) * 0.3 if with_init else None
    gamma = oracle.decay_schedule(H, 1.0, t_max, lib=lib)
    return q, k, v, gamma, a, init


def _sig(z):
    return 1.0 / (1.0 + np.exp(-z))


# ---------------------------------------------------------------------------
def pin_decay(lib):
    g = json.load(open(os.path.join(GOLDEN, "decay_schedule_printed.json")))
    gam = oracle.decay_schedule(g["H"], g["T_min"], g["T_max"], lib=lib)
    lam = np.exp(gam)
    ok = True
    msgs = []
    # lambda_0 = 0.5 exactly (to 1 ulp) -- printed
    if abs(lam[0] - g["lambda_0"]) > np.spacing(0.5):
        ok = False; msgs.append(f"lambda_0={lam[0]!r}")
    # lambda_15 ~ 0.9997 as printed (4 decimals), and = 2^(-1/2048) to 1 ulp
    if round(float(lam[-1]), g["lambda_15_printed_decimals"]) != g["lambda_15_printed"]:
        ok = False; msgs.append(f"lambda_15={lam[-1]!r}")
    if abs(lam[-1] - 2.0 ** (-1.0 / 2048)) > np.spacing(1.0):
        ok = False; msgs.append("lambda_15 != 2^(-1/2048)")
    # half-lives: lambda_h ^ T_h = 1/2 with T_0 = 1 and T_15 = 2048 tokens
    if abs(lam[0] ** g["lambda_0_half_life_tokens"] - 0.5) > 1e-15:
        ok = False; msgs.append("half-life head 0")
    if abs(lam[-1] ** g["lambda_15_half_life_tokens"] - 0.5) > 1e-12:
        ok = False; msgs.append("half-life head 15")
    # geometric spread: half-life ratios between neighbours are all equal
    hl = -np.log(2.0) / gam
    ratios = hl[1:] / hl[:-1]
    if np.abs(ratios - 2048.0 ** (1 / 15)).max() > 1e-12:
        ok = False; msgs.append("not geometric")
    # two heads: the two ends of the range
    g2 = oracle.decay_schedule(2, 1.0, 2048.0, lib=lib)
    if abs(np.exp(g2[0]) - 0.5) > 1e-16 or abs(np.exp(g2[1]) - 2 ** (-1 / 2048)) > 1e-16:
        ok = False; msgs.append("H=2 ends")
    return ok, "; ".join(msgs)


def closed_form(q, k, v, gamma, a, init):
    """Brute force, straight from the closed form (no recurrence)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    fin = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            lam = np.exp(gamma[h])
            for t in range(T):
                acc = np.zeros(dv)
                for s in range(t + 1):
                    acc += lam ** (t - s) * np.dot(q[b, t, h], k[b, s, h]) * v[b, s, h]
                if init is not None:
                    acc += lam ** (t + 1) * (init[b, h].T @ q[b, t, h])
                z = np.sum(a[h] * q[b, t, h] * k[b, t, h])
                o[b, t, h] = acc + _sig(z) * v[b, t, h]
            S = np.zeros((dk, dv)) if init is None else lam ** T * init[b, h]
            for s in range(T):
                S = S + lam ** (T - 1 - s) * np.outer(k[b, s, h], v[b, s, h])
            fin[b, h] = S
    return o, fin


def pin_closed_form(lib):
    worst = 0.0
    for seed, (B, T, H, dk, dv), init in [(1, (2, 9, 3, 5, 7), True), (2, (1, 6, 16, 96, 192), True),
                                          (3, (2, 7, 2, 4, 4), False)]:
        q, k, v, gamma, a, ini = _rand_problem(seed, B, T, H, dk, dv, with_init=init,
                                               t_max=2048.0 if H == 16 else 8.0, lib=lib)
        o, fin = oracle.fwd(q, k, v, gamma, a, ini, lib=lib)
        o2, fin2 = closed_form(q, k, v, gamma, a, ini)
        worst = max(worst, _rel(o, o2), _rel(fin, fin2))
    return worst < 1e-12, f"max rel {worst:.2e}"


def pin_aug_zero(lib):
    B, T, H, dk, dv = 2, 5, 3, 6, 4
    q, k, v, gamma, a, init = _rand_problem(11, B, T, H, dk, dv, lib=lib)
    # q = 0: the readout vanishes and z = 0, so o = sigmoid(0) v = v/2 exactly
    o, _ = oracle.fwd(np.zeros_like(q), k, v, gamma, a, init, lib=lib)
    ok1 = np.array_equal(o, 0.5 * v)
    # a = 0: o minus the closed-form readout is exactly half of v (up to rounding)
    o, _ = oracle.fwd(q, k, v, gamma, np.zeros_like(a), init, lib=lib)
    ro, _ = closed_form(q, k, v, gamma, np.zeros_like(a), init)
    ok2 = _rel(o - (ro - 0.5 * v), 0.5 * v) < 1e-12
    return ok1 and ok2, f"q=0 exact: {ok1}, a=0 half skip: {ok2}"


def pin_lambda_one(lib):
    B, T, H, dk, dv = 2, 11, 3, 5, 6
    q, k, v, _, a, _ = _rand_problem(12, B, T, H, dk, dv, lib=lib)
    gamma = np.zeros(H)
    o, _ = oracle.fwd(q, k, v, gamma, np.zeros_like(a), None, lib=lib)
    worst = 0.0
    for b in range(B):
        for h in range(H):
            Q, K, V = q[b, :, h], k[b, :, h], v[b, :, h]
            ref = np.tril(Q @ K.T) @ V + 0.5 * V      # causal linear attention + v/2
            worst = max(worst, _rel(o[b, :, h], ref))
    return worst < 1e-12, f"max rel {worst:.2e}"


def _loss(lib, q, k, v, gamma, a, init, dO, dfin):
    o, fin = oracle.fwd(q, k, v, gamma, a, init, nthreads=1, lib=lib)
    return float(np.sum(o * dO) + np.sum(fin * dfin))


def pin_fd(lib):
    B, T, H, dk, dv = 2, 5, 3, 4, 3
    q, k, v, gamma, a, init = _rand_problem(13, B, T, H, dk, dv, lib=lib)
    r = _rng(14)
    dO = r.standard_normal((B, T, H, dv))
    dfin = r.standard_normal((B, H, dk, dv))
    g = oracle.bwd(q, k, v, gamma, a, dO, init, dfin, lib=lib)
    args = dict(q=q, k=k, v=v, a=a, init=init)
    names = dict(q="dq", k="dk", v="dv", a="d_a", init="d_init_state")
    eps = 1e-5
    worst = 0.0
    for name, gname in names.items():
        x = args[name]
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            x0 = x[idx]
            x[idx] = x0 + eps
            lp = _loss(lib, q, k, v, gamma, a, init, dO, dfin)
            x[idx] = x0 - eps
            lm = _loss(lib, q, k, v, gamma, a, init, dO, dfin)
            x[idx] = x0
            num[idx] = (lp - lm) / (2 * eps)
        worst = max(worst, _rel(g[gname], num))
    # and without dS_final / init (the NULL paths)
    g0 = oracle.bwd(q, k, v, gamma, a, dO, None, None, lib=lib)
    num = np.zeros_like(q)
    for idx in np.ndindex(q.shape):
        x0 = q[idx]
        q[idx] = x0 + eps
        lp = _loss(lib, q, k, v, gamma, a, None, dO, np.zeros_like(dfin))
        q[idx] = x0 - eps
        lm = _loss(lib, q, k, v, gamma, a, None, dO, np.zeros_like(dfin))
        q[idx] = x0
        num[idx] = (lp - lm) / (2 * eps)
    worst = max(worst, _rel(g0["dq"], num))
    return worst < 1e-7, f"max rel {worst:.2e}"


def pin_init_zero(lib):
    B, T, H, dk, dv = 2, 6, 3, 5, 4
    q, k, v, gamma, a, _ = _rand_problem(15, B, T, H, dk, dv, lib=lib)
    o1, f1 = oracle.fwd(q, k, v, gamma, a, None, lib=lib)
    o2, f2 = oracle.fwd(q, k, v, gamma, a, np.zeros((B, H, dk, dv)), lib=lib)
    dO = _rng(16).standard_normal((B, T, H, dv))
    g1 = oracle.bwd(q, k, v, gamma, a, dO, None, None, lib=lib)
    g2 = oracle.bwd(q, k, v, gamma, a, dO, np.zeros((B, H, dk, dv)), np.zeros((B, H, dk, dv)),
                    lib=lib)
    ok = np.array_equal(o1, o2) and np.array_equal(f1, f2) and all(
        np.array_equal(g1[n], g2[n]) for n in g1)
    return ok, "bit-exact" if ok else "differs"


def pin_state_carry(lib):
    B, T, H, dk, dv = 2, 12, 3, 5, 4
    q, k, v, gamma, a, init = _rand_problem(17, B, T, H, dk, dv, lib=lib)
    o, fin = oracle.fwd(q, k, v, gamma, a, init, lib=lib)
    T1 = 5
    o1, f1 = oracle.fwd(q[:, :T1], k[:, :T1], v[:, :T1], gamma, a, init, lib=lib)
    o2, f2 = oracle.fwd(q[:, T1:], k[:, T1:], v[:, T1:], gamma, a, f1, lib=lib)
    ok = np.array_equal(np.concatenate([o1, o2], 1), o) and np.array_equal(f2, fin)
    return ok, "bit-exact" if ok else "differs"


def pin_decode(lib):
    N, L, H, dk, dv, T = 3, 4, 3, 5, 6, 4
    r = _rng(18)
    gamma = oracle.decay_schedule(H, 1.0, 8.0, lib=lib)
    a = r.standard_normal((L, H, dk)) * 0.5
    state = r.standard_normal((N, L, H, dk, dv))
    q = r.standard_normal((N, L, H, dk))
    k = r.standard_normal((N, L, H, dk))
    v = r.standard_normal((N, L, H, dv))
    o, st = oracle.decode_step(state, q, k, v, gamma, a, lib=lib)
    worst = 0.0
    for n in range(N):
        for l in range(L):
            # forward over T warm tokens then the decode token, per layer
            wq = r.standard_normal((1, T, H, dk))
            wk = r.standard_normal((1, T, H, dk))
            wv = r.standard_normal((1, T, H, dv))
            _, s0 = oracle.fwd(wq, wk, wv, gamma, a[l], None, lib=lib)
            od, sd = oracle.decode_step(s0[:, None], q[n:n + 1, l:l + 1], k[n:n + 1, l:l + 1],
                                        v[n:n + 1, l:l + 1], gamma, a[l:l + 1], lib=lib)
            of, sf = oracle.fwd(np.concatenate([wq, q[n:n + 1, l][:, None]], 1),
                                np.concatenate([wk, k[n:n + 1, l][:, None]], 1),
                                np.concatenate([wv, v[n:n + 1, l][:, None]], 1), gamma, a[l], None,
                                lib=lib)
            worst = max(worst, _rel(od[0, 0], of[0, -1]), _rel(sd[0, 0], sf[0]))
            # the pooled call agrees with the per-state call for the same state
            o1, s1 = oracle.fwd(q[n:n + 1, l][:, None], k[n:n + 1, l][:, None],
                                v[n:n + 1, l][:, None], gamma, a[l], state[n:n + 1, l], lib=lib)
            worst = max(worst, _rel(o[n, l], o1[0, 0]), _rel(st[n, l], s1[0]))
    return worst < 1e-14, f"max rel {worst:.2e}"


# ---------------------------------------------------------------------------
# Independent chunked restatement (test only): intra-chunk masked attention plus
# the inter-chunk state, and the chunked backward with a reverse state-adjoint
# scan.  A chunk of L tokens (the last one may be shorter than C) uses
# D_ij = lambda^(i-j) for i >= j, Lq = lambda^(i+1), Lk = lambda^(L-1-j), and
# advances the state by lambda^L.

def _chunk_consts(lam, L):
    i = np.arange(L)
    D = np.where(i[:, None] >= i[None, :], lam ** (i[:, None] - i[None, :]), 0.0)
    return D, lam ** (i + 1), lam ** (L - 1 - i)


def chunked_fwd(q, k, v, gamma, a, init, C):
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    fin = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            lam = np.exp(gamma[h])
            S = np.zeros((dk, dv)) if init is None else init[b, h].copy()
            for c0 in range(0, T, C):
                L = min(C, T - c0)
                D, Lq, Lk = _chunk_consts(lam, L)
                sl = slice(c0, c0 + L)
                Q, K, V = q[b, sl, h], k[b, sl, h], v[b, sl, h]
                P = (Q @ K.T) * D
                sg = _sig(np.sum(Q * a[h] * K, 1))
                o[b, sl, h] = P @ V + (Lq[:, None] * Q) @ S + sg[:, None] * V
                S = lam ** L * S + (Lk[:, None] * K).T @ V
            fin[b, h] = S
    return o, fin


def chunked_bwd(q, k, v, gamma, a, init, dO, dfin, C):
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dq, dk_, dv_ = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    da = np.zeros((H, dk))
    dinit = np.zeros((B, H, dk, dv))
    starts = list(range(0, T, C))
    for b in range(B):
        for h in range(H):
            lam = np.exp(gamma[h])
            S = np.zeros((dk, dv)) if init is None else init[b, h].copy()
            states = []
            for c0 in starts:
                L = min(C, T - c0)
                _, _, Lk = _chunk_consts(lam, L)
                sl = slice(c0, c0 + L)
                states.append(S)
                S = lam ** L * S + (Lk[:, None] * k[b, sl, h]).T @ v[b, sl, h]
            dS = np.zeros((dk, dv)) if dfin is None else dfin[b, h].copy()
            for c, c0 in reversed(list(enumerate(starts))):
                L = min(C, T - c0)
                D, Lq, Lk = _chunk_consts(lam, L)
                sl = slice(c0, c0 + L)
                Q, K, V, G = q[b, sl, h], k[b, sl, h], v[b, sl, h], dO[b, sl, h]
                Sm = states[c]
                P = (Q @ K.T) * D
                dP = (G @ V.T) * D
                sg = _sig(np.sum(Q * a[h] * K, 1))
                r = sg * (1 - sg) * np.sum(G * V, 1)
                dq[b, sl, h] = dP @ K + Lq[:, None] * (G @ Sm.T) + r[:, None] * (a[h] * K)
                dk_[b, sl, h] = dP.T @ Q + Lk[:, None] * (V @ dS.T) + r[:, None] * (a[h] * Q)
                dv_[b, sl, h] = P.T @ G + Lk[:, None] * (K @ dS) + sg[:, None] * G
                da[h] += np.sum(r[:, None] * Q * K, 0)
                dS = lam ** L * dS + Q.T @ (Lq[:, None] * G)
            dinit[b, h] = dS
    return dict(dq=dq, dk=dk_, dv=dv_, d_a=da, d_init_state=dinit)


# Cut into parts (test only): a sequence of nc chunks cut into p consecutive chunk ranges
# (part j: chunks [j*nc/p, (j+1)*nc/p)), each run from its own starting state and adjoint,
# which follow from the linear recurrences
#   S entering part j+1 = lambda^(L_j) S entering part j + sum_{t in j} lambda^(e_j - t) k_t v_t^T
#   dS leaving part j-1 = lambda^(L_j) dS leaving part j + sum_{t in j} lambda^(t - s_j + 1) q_t dO_t^T
# (s_j, e_j: first and last token of part j, L_j its tokens).
def parts_fwd_bwd(q, k, v, gamma, a, init, dO, dfin, C, p):
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    nc = -(-T // C)
    bounds = [min((j * nc // p) * C, T) for j in range(p + 1)]
    S_in = np.zeros((p, B, H, dk, dv))
    dS_out = np.zeros((p, B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            lam = np.exp(gamma[h])
            S_in[0, b, h] = 0.0 if init is None else init[b, h]
            for j in range(p - 1):
                s, e = bounds[j], bounds[j + 1]
                w = lam ** (e - 1 - np.arange(s, e))
                U = (w[:, None] * k[b, s:e, h]).T @ v[b, s:e, h]
                S_in[j + 1, b, h] = lam ** (e - s) * S_in[j, b, h] + U
            dS_out[p - 1, b, h] = 0.0 if dfin is None else dfin[b, h]
            for j in range(p - 1, 0, -1):
                s, e = bounds[j], bounds[j + 1]
                w = lam ** (np.arange(s, e) - s + 1)
                U = (w[:, None] * q[b, s:e, h]).T @ dO[b, s:e, h]
                dS_out[j - 1, b, h] = lam ** (e - s) * dS_out[j, b, h] + U
    o = np.zeros((B, T, H, dv))
    g = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
             d_a=np.zeros((H, dk)), d_init_state=None)
    fin = None
    for j in range(p):
        s, e = bounds[j], bounds[j + 1]
        cut = lambda x: x[:, s:e]
        oj, fin = chunked_fwd(cut(q), cut(k), cut(v), gamma, a, S_in[j], C)
        o[:, s:e] = oj
        gj = chunked_bwd(cut(q), cut(k), cut(v), gamma, a, S_in[j], cut(dO), dS_out[j], C)
        for n in ("dq", "dk", "dv"):
            g[n][:, s:e] = gj[n]
        g["d_a"] += gj["d_a"]
        if j == 0:
            g["d_init_state"] = gj["d_init_state"]
    return o, fin, g


def pin_chunked(lib):
    B, T, H, dk, dv = 2, 32, 4, 6, 5
    q, k, v, gamma, a, init = _rand_problem(19, B, T, H, dk, dv, t_max=64.0, lib=lib)
    r = _rng(20)
    dO = r.standard_normal((B, T, H, dv))
    dfin = r.standard_normal((B, H, dk, dv))
    o, fin = oracle.fwd(q, k, v, gamma, a, init, lib=lib)
    g = oracle.bwd(q, k, v, gamma, a, dO, init, dfin, lib=lib)
    worst = 0.0
    # C = 5 and 12 leave a shorter last chunk (32 = 6*5 + 2 = 2*12 + 8)
    for C in (1, 4, 5, 12, 16, 32):
        oc, fc = chunked_fwd(q, k, v, gamma, a, init, C)
        gc = chunked_bwd(q, k, v, gamma, a, init, dO, dfin, C)
        worst = max(worst, _rel(oc, o), _rel(fc, fin), *[_rel(gc[n], g[n]) for n in g])
    return worst < 1e-11, f"max rel {worst:.2e}"


def pin_parts(lib):
    """Pairs cut into parts, each run from the state and adjoint the linear recurrences give at
    its boundary, equal the token recurrence (forward, every gradient, d_init and the final
    state); parts of unequal length and a ragged last chunk included."""
    B, T, H, dk, dv = 2, 45, 3, 6, 5
    q, k, v, gamma, a, init = _rand_problem(21, B, T, H, dk, dv, t_max=32.0, lib=lib)
    r = _rng(22)
    dO = r.standard_normal((B, T, H, dv))
    dfin = r.standard_normal((B, H, dk, dv))
    o, fin = oracle.fwd(q, k, v, gamma, a, init, lib=lib)
    g = oracle.bwd(q, k, v, gamma, a, dO, init, dfin, lib=lib)
    worst = 0.0
    for C, p in ((4, 2), (4, 3), (4, 12), (8, 5), (16, 3)):  # 45 tokens: 12, 6 or 3 chunks
        if p > -(-T // C):
            continue
        op, fp, gp = parts_fwd_bwd(q, k, v, gamma, a, init, dO, dfin, C, p)
        worst = max(worst, _rel(op, o), _rel(fp, fin), *[_rel(gp[n], g[n]) for n in g])
    return worst < 1e-11, f"max rel {worst:.2e}"


ALL_PINS = dict(decay=pin_decay, closed_form=pin_closed_form, aug_zero=pin_aug_zero,
                lambda_one=pin_lambda_one, fd=pin_fd, init_zero=pin_init_zero,
                state_carry=pin_state_carry, decode=pin_decode, chunked=pin_chunked,
                parts=pin_parts)
