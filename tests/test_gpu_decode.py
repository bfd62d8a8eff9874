"""GPU parity of gla_decode_step against the fp64 oracle (bar: 1e-4 of the output RMS)."""
import numpy as np
import pytest

import synth
from _util import TOL_DECODE, rel_err, oracle_decays

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU test without a CUDA device"
    import gated_linear_attention_chunked_gb300 as gla
    from gated_linear_attention_chunked_gb300 import _build
    _build.build()
    gla.load()
    return gla, torch


def _t(torch, x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()


@pytest.mark.parametrize("N,L,H", [(1, 1, 1), (5, 3, 16), (7, 2, 5)])
def test_decode_small(env, N, L, H):
    import oracle
    gla, torch = env
    rng = np.random.default_rng(N * 100 + L * 10 + H)
    st = (rng.standard_normal((N, L, H, 96, 192)) * 0.5).astype(np.float32)
    q, k, v = synth.decode_token(9, N, L, H)
    a = synth.aug_balance(9, (L, H, 96), 0.3)
    gam = oracle_decays(H)[0]
    gam64 = oracle_decays(H)[1]
    st_d = _t(torch, st)
    o = gla.decode_step(st_d, _t(torch, q), _t(torch, k), _t(torch, v), gam.cuda(), _t(torch, a))
    o_ref, st_ref = oracle.decode_step(st, q, k, v, gam64, a)
    eo, es = rel_err(o.cpu().numpy(), o_ref), rel_err(st_d.cpu().numpy(), st_ref)
    print(f"decode N={N} L={L} H={H}: o {eo:.2e} state {es:.2e}")
    assert eo <= TOL_DECODE and es <= TOL_DECODE
    assert gla.get_device_error() == 0


def test_decode_consecutive_steps_carry_the_state(env):
    import oracle
    gla, torch = env
    N, L, H = 3, 2, 16
    q1, k1, v1 = synth.decode_token(5, N, L, H, step=0)
    q2, k2, v2 = synth.decode_token(5, N, L, H, step=1)
    a = synth.aug_balance(5, (L, H, 96), 0.02)
    gam = oracle_decays(H)[0]
    gam64 = oracle_decays(H)[1]
    st = np.zeros((N, L, H, 96, 192), np.float32)
    st_d = _t(torch, st)
    gla.decode_step(st_d, _t(torch, q1), _t(torch, k1), _t(torch, v1), gam.cuda(), _t(torch, a))
    o2 = gla.decode_step(st_d, _t(torch, q2), _t(torch, k2), _t(torch, v2), gam.cuda(), _t(torch, a))
    _, s1 = oracle.decode_step(st, q1, k1, v1, gam64, a)
    o2r, s2 = oracle.decode_step(s1, q2, k2, v2, gam64, a)
    assert rel_err(o2.cpu().numpy(), o2r) <= TOL_DECODE
    assert rel_err(st_d.cpu().numpy(), s2) <= TOL_DECODE


def warm_state(gam64, a, seqs, L, H, cfg):
    """Oracle recurrence over the workload's warm-up tokens, from a zero state, for the
    given sequences; rounded to fp32 (the state both sides start from)."""
    import oracle
    out = np.empty((len(seqs), L, H, 96, 192), np.float32)
    for n, s in enumerate(seqs):
        wq, wk, wv = synth.decode_warm_tokens(cfg["seed"], s, cfg["warm_tokens"], L, H)
        st = np.zeros((1, L, H, 96, 192))
        for t in range(cfg["warm_tokens"]):
            _, st = oracle.decode_step(st, wq[t][None], wk[t][None], wv[t][None], gam64, a)
        out[n] = st[0]
    return out


def test_decode_full_serving_pool(env):
    """The serving workload: 1,280 sequences x 24 layers x 16 heads of 96x192 fp32 states
    (36.2 GB) resident in HBM, one new token per sequence, launched as the benchmark does.
    Every 64th sequence (all layers and heads) is checked against the oracle after 1 and
    after 100 consecutive steps, each step with a new token for those sequences; every output
    is checked finite."""
    import oracle
    gla, torch = env
    cfg = synth.DECODE
    N, L, H = cfg["N"], cfg["L"], cfg["H"]
    seqs = list(range(0, N, 64))
    gam = oracle_decays(H)[0]
    gam64 = oracle_decays(H)[1]
    a = synth.aug_balance(cfg["seed"], (L, H, 96), cfg["a_std"])
    st0 = warm_state(gam64, a, seqs, L, H, cfg)
    pool = torch.empty((N, L, H, 96, 192), dtype=torch.float32, device="cuda")
    pool.normal_(0.0, 2.0)  # unchecked sequences: arbitrary states of a similar size
    for n, s in enumerate(seqs):
        pool[s].copy_(torch.from_numpy(st0[n]))
    q, k, v = synth.decode_token(cfg["seed"], N, L, H)
    qd, kd, vd, ad = (torch.from_numpy(x).cuda() for x in (q, k, v, a))
    o = torch.empty((N, L, H, 192), dtype=torch.float32, device="cuda")
    gla.decode_step(pool, qd, kd, vd, gam.cuda(), ad, out=o)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(o).all())
    sub = seqs
    o_ref, st_ref = oracle.decode_step(st0, q[sub], k[sub], v[sub], gam64, a)
    eo = rel_err(o[sub].cpu().numpy(), o_ref)
    es = rel_err(pool[sub].cpu().numpy(), st_ref)
    print(f"decode pool step 1: o {eo:.2e} state {es:.2e}")
    assert eo <= TOL_DECODE and es <= TOL_DECODE
    # steps 2..100: a new token per step for the checked sequences (its own seeded stream per
    # step), so their states move in 100 directions; the unchecked ones repeat their token
    idx = torch.tensor(sub, device="cuda")
    for s in range(1, 100):
        qs, ks, vs = synth.decode_token(cfg["seed"], len(sub), L, H, step=s)
        for dst, src in ((qd, qs), (kd, ks), (vd, vs)):
            dst.index_copy_(0, idx, torch.from_numpy(src).cuda())
        gla.decode_step(pool, qd, kd, vd, gam.cuda(), ad, out=o)
        o_ref, st_ref = oracle.decode_step(st_ref, qs, ks, vs, gam64, a)
    torch.cuda.synchronize()
    eo = rel_err(o[sub].cpu().numpy(), o_ref)
    es = rel_err(pool[sub].cpu().numpy(), st_ref)
    print(f"decode pool step 100: o {eo:.2e} state {es:.2e}")
    assert eo <= TOL_DECODE and es <= TOL_DECODE
    assert bool(torch.isfinite(o).all())
    assert gla.get_device_error() == 0
    del pool
    torch.cuda.empty_cache()
