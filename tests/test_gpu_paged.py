"""GPU parity of the state-pool calls (one fixed page of recurrent state per sequence):
gla_decode_step_paged and gla_chunk_fwd_paged against the fp64 oracle.  States of pages
and layers a call does not name must come back bit-identical."""
import numpy as np
import pytest

import synth
from _util import TOL_CHUNK, TOL_DECODE, rel_err, to_dev, oracle_decays

pytestmark = pytest.mark.gpu

GLA_ERR_RANGE = 6


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU test without a CUDA device"
    import gated_linear_attention_chunked_gb300 as gla
    from gated_linear_attention_chunked_gb300 import _build
    _build.build()
    gla.load()
    return gla, torch


def _pool(seed, P, PL, H, std=0.05):
    return synth.normal(seed, synth.INIT, (P, PL, H, 96, 192), std).astype(np.float32)


def _decode_inputs(seed, n, L, H):
    q = synth.normal(seed, synth.Q, (n, L, H, 96), 96 ** -0.5).astype(np.float32)
    k = synth.normal(seed, synth.K, (n, L, H, 96), 1.0).astype(np.float32)
    v = synth.normal(seed, synth.V, (n, L, H, 192), 1.0).astype(np.float32)
    a = synth.aug_balance(seed, (L, H, 96), 0.1)
    return q, k, v, a


def test_decode_paged_matches_oracle(env):
    import oracle
    gla, torch = env
    P, PL, H, L, layer0 = 9, 3, 4, 2, 1
    page = np.array([7, 2, 0, 5, 3], np.int32)  # any order, no padding
    pool = _pool(51, P, PL, H)
    q, k, v, a = _decode_inputs(51, len(page), L, H)
    gam = oracle_decays(H)[0]
    gam64 = gam.numpy().astype(np.float64)
    pool_d = to_dev(pool, torch.float32)
    o = gla.decode_step_paged(pool_d, to_dev(page, torch.int32), to_dev(q, torch.float32),
                              to_dev(k, torch.float32), to_dev(v, torch.float32), gam.cuda(),
                              to_dev(a, torch.float32), layer0=layer0)
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    o_ref, pool_ref = oracle.decode_step_paged(pool, page, layer0, q, k, v, gam64, a)
    new = pool_d.cpu().numpy()
    eo = rel_err(o.cpu().numpy(), o_ref)
    es = rel_err(new[page, layer0:layer0 + L], pool_ref[page, layer0:layer0 + L])
    print(f"decode paged: o {eo:.2e} states {es:.2e}")
    assert eo <= TOL_DECODE and es <= TOL_DECODE
    touched = np.zeros((P, PL), bool)
    touched[np.ix_(page, np.arange(layer0, layer0 + L))] = True
    assert np.array_equal(new[~touched], pool[~touched])


def test_decode_paged_bad_page_touches_nothing(env):
    """A page index outside the pool is caught by the kernel's own check: the device error
    word reads GLA_ERR_RANGE, that sequence's states and output are left alone, the other
    sequences of the call are updated."""
    import oracle
    gla, torch = env
    P, PL, H, L = 4, 1, 2, 1
    page = np.array([2, 99], np.int32)
    pool = _pool(52, P, PL, H)
    q, k, v, a = _decode_inputs(52, 2, L, H)
    gam = oracle_decays(H)[0]
    pool_d = to_dev(pool, torch.float32)
    o = torch.full((2, L, H, 192), float("nan"), device="cuda")
    gla.decode_step_paged(pool_d, to_dev(page, torch.int32), to_dev(q, torch.float32),
                          to_dev(k, torch.float32), to_dev(v, torch.float32), gam.cuda(),
                          to_dev(a, torch.float32), out=o)
    torch.cuda.synchronize()
    assert gla.get_device_error() == GLA_ERR_RANGE
    assert gla.get_device_error() == 0  # read and cleared
    oc, new = o.cpu().numpy(), pool_d.cpu().numpy()
    assert np.all(np.isnan(oc[1]))
    o_ref, pool_ref = oracle.decode_step_paged(pool, page[:1], 0, q[:1], k[:1], v[:1],
                                               gam.numpy().astype(np.float64), a)
    assert rel_err(oc[:1], o_ref) <= TOL_DECODE
    assert rel_err(new[2], pool_ref[2]) <= TOL_DECODE
    assert np.array_equal(new[[0, 1, 3]], pool[[0, 1, 3]])


@pytest.mark.parametrize("B,T,H,P,PL,layer,from_pool,seed", [
    (3, 384, 4, 6, 2, 1, True, 53),    # serial scan, initial states from the pool
    (2, 256, 3, 4, 3, 0, False, 54),   # starting from zero: the pages' contents are ignored
    (1, 4096, 2, 4, 1, 0, True, 55),   # few long sequences: pairs cut into parts
    (2, 300, 3, 4, 2, 1, True, 56),    # ragged last chunk
])
def test_chunk_fwd_paged(env, B, T, H, P, PL, layer, from_pool, seed):
    import oracle
    gla, torch = env
    rng = np.random.default_rng(seed)
    page = rng.permutation(P)[:B].astype(np.int32)
    pool = _pool(seed, P, PL, H)
    q, k, v = synth.qkv(seed, B, T, H)
    a = synth.aug_balance(seed, (H, 96), 0.1)
    gam = oracle_decays(H)[0]
    gam64 = gam.numpy().astype(np.float64)
    pool_d = to_dev(pool, torch.float32)
    o = gla.chunk_fwd_paged(to_dev(q, torch.bfloat16), to_dev(k, torch.bfloat16),
                            to_dev(v, torch.bfloat16), gam.cuda(), to_dev(a, torch.float32),
                            pool_d, to_dev(page, torch.int32), layer, init_from_pool=from_pool)
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    init = pool[page, layer] if from_pool else None
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a, init)
    new = pool_d.cpu().numpy()
    eo, ef = rel_err(o.cpu().numpy(), o_ref), rel_err(new[page, layer], fin_ref)
    print(f"fwd paged B={B} T={T} H={H}: o {eo:.2e} final {ef:.2e}")
    assert eo <= TOL_CHUNK and ef <= TOL_CHUNK
    touched = np.zeros((P, PL), bool)
    touched[page, layer] = True
    assert np.array_equal(new[~touched], pool[~touched])


def test_prefill_then_decode_matches_one_forward(env):
    """Prefill T tokens into a page, then one paged decode step with token T: the decode
    output and the page equal the oracle forward over T + 1 tokens (its last output and its
    final state) -- the prefill/decode consistency of the serving path."""
    import oracle
    gla, torch = env
    T, H, P = 256, 4, 3
    q, k, v = synth.qkv(56, 1, T + 1, H)
    a = synth.aug_balance(56, (H, 96), 0.1)
    gam = oracle_decays(H)[0]
    gam64 = gam.numpy().astype(np.float64)
    pool_d = torch.zeros((P, 1, H, 96, 192), device="cuda")
    page = to_dev(np.array([1], np.int32), torch.int32)
    gla.chunk_fwd_paged(to_dev(q[:, :T], torch.bfloat16), to_dev(k[:, :T], torch.bfloat16),
                        to_dev(v[:, :T], torch.bfloat16), gam.cuda(), to_dev(a, torch.float32),
                        pool_d, page, 0, init_from_pool=False)
    o = gla.decode_step_paged(pool_d, page, to_dev(q[:, T:T + 1], torch.float32),
                              to_dev(k[:, T:T + 1], torch.float32),
                              to_dev(v[:, T:T + 1], torch.float32), gam.cuda(),
                              to_dev(a[None], torch.float32))
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a)
    eo = rel_err(o.cpu().numpy()[0, 0], o_ref[0, T])
    ef = rel_err(pool_d.cpu().numpy()[1, 0], fin_ref[0])
    print(f"prefill {T} + decode 1: o {eo:.2e} state {ef:.2e}")
    assert eo <= TOL_CHUNK and ef <= TOL_CHUNK
    assert torch.count_nonzero(pool_d[[0, 2]]).item() == 0
