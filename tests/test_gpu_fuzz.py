"""A randomized parity sweep with a fixed seed (the same cases every run): the chunked forward
and backward against the fp64 oracle over shapes (any T, few or many (b, h) pairs), input
types, forced part counts, both orders of the segment passes, initial state and final-state
adjoint present or absent, and the forward's saved activations (gate and state copies) handed
to the backward or not; then the forward with the fused output epilogue and the prefill into a
state pool over the same kinds of layouts.  It looks for interactions the targeted tests leave
out; the bar is the usual 2e-2 of each output's RMS.  Wide cases (160-176 pairs, short T) put
at least a wave of whole pairs beside the cut ones, so the passes run beside them and a
sum-pass CTA can take several parts in turn."""
import numpy as np
import pytest

import synth
from _util import TOL_CHUNK, rel_err, to_dev, oracle_decays

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "d_a", "d_init_state")


def _cases(n=24, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        wide = i % 4 == 3
        B = int(rng.integers(10, 12)) if wide else int(rng.integers(1, 4))
        H = 16 if wide else int(rng.choice([1, 2, 3, 5, 16]))
        T = int(rng.integers(129, 400)) if wide else int(rng.integers(1, 900))
        dtype = str(rng.choice(["bf16", "fp16", "fp32"]))
        parts = int(rng.choice([0, 1, 2, 3, 5]))
        overlap = bool(rng.integers(0, 2))
        with_init = bool(rng.integers(0, 2))
        with_dfin = bool(rng.integers(0, 2))
        saved = bool(rng.integers(0, 2))
        out.append((i, B, T, H, dtype, parts, overlap, with_init, with_dfin, saved))
    return out


CASES = _cases()


def _id(c):
    i, B, T, H, dtype, parts, overlap, wi, wd, saved = c
    return (f"{i}-B{B}T{T}H{H}-{dtype}-p{parts}{'-ov' if overlap else ''}"
            f"{'-init' if wi else ''}{'-dfin' if wd else ''}{'-saved' if saved else ''}")


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU test without a CUDA device"
    import gated_linear_attention_chunked_gb300 as gla
    from gated_linear_attention_chunked_gb300 import _build
    _build.build()
    gla.load()
    yield gla, torch
    gla.set_split_parts(0)
    gla.set_pass_overlap(True)


@pytest.mark.parametrize("case", CASES, ids=[_id(c) for c in CASES])
def test_random_case_matches_oracle(env, case):
    import oracle
    gla, torch = env
    i, B, T, H, dtype, parts, overlap, with_init, with_dfin, saved = case
    seed = 900 + i
    q, k, v = synth.qkv(seed, B, T, H, bf16=(dtype == "bf16"))
    dO = synth.grad_out(seed, B, T, H, bf16=(dtype == "bf16"))
    if dtype == "fp16":
        q, k, v, dO = (x.astype(np.float16).astype(np.float32) for x in (q, k, v, dO))
    a = synth.aug_balance(seed, (H, 96), 0.1)
    init = synth.init_state(seed, B, H, 0.05) if with_init else None
    dfin = synth.normal(seed, synth.DFIN, (B, H, 96, 192), 0.05) if with_dfin else None
    td = dict(bf16=torch.bfloat16, fp16=torch.float16, fp32=torch.float32)[dtype]
    gam32, gam64 = oracle_decays(H)
    gla.set_split_parts(parts)
    gla.set_pass_overlap(overlap)
    try:
        qd, kd, vd, gd = (to_dev(x, td) for x in (q, k, v, dO))
        ad = to_dev(a, torch.float32)
        idd = to_dev(init, torch.float32) if init is not None else None
        fd = to_dev(dfin, torch.float32) if dfin is not None else None
        gam = gam32.cuda()
        gate = sv = None
        if saved:
            gate = torch.empty(B, H, T, device="cuda")
            sv = torch.empty(gla.chunk_saved_states_size(B, T, H), dtype=torch.uint8,
                             device="cuda")
        o, fin = gla.chunk_fwd(qd, kd, vd, gam, ad, idd, gate=gate, saved_states=sv)
        g = gla.chunk_bwd(qd, kd, vd, gam, ad, gd, idd, fd, gate=gate, saved_states=sv)
        torch.cuda.synchronize()
        assert gla.get_device_error() == 0
        o, fin = o.cpu().numpy(), fin.cpu().numpy()
        g = [x.cpu().numpy() for x in g]
    finally:
        gla.set_split_parts(0)
        gla.set_pass_overlap(True)
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a, init)
    ref = oracle.bwd(q, k, v, gam64, a, dO, init, dfin)
    errs = dict(o=rel_err(o, o_ref), final=rel_err(fin, fin_ref))
    errs.update({n: rel_err(x, ref[n]) for n, x in zip(NAMES, g)})
    print(_id(case) + ": " + " ".join(f"{n} {e:.2e}" for n, e in errs.items()))
    assert all(e <= TOL_CHUNK for e in errs.values()), errs


def _fwd_cases(n=12, seed=2027):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        wide = i % 4 == 3
        B = int(rng.integers(10, 12)) if wide else int(rng.integers(1, 4))
        H = 16 if wide else int(rng.choice([2, 4, 8, 16]))
        T = int(rng.integers(129, 400)) if wide else int(rng.integers(1, 900))
        parts = int(rng.choice([0, 1, 2, 3, 5]))
        overlap = bool(rng.integers(0, 2))
        extra = int(rng.integers(0, 2))  # gated: o written too; paged: start from the pool
        out.append((i, B, T, H, parts, overlap, extra))
    return out


FWD_CASES = _fwd_cases()


def _fwd_id(c):
    i, B, T, H, parts, overlap, extra = c
    return f"{i}-B{B}T{T}H{H}-p{parts}{'-ov' if overlap else ''}{'-x' if extra else ''}"


@pytest.mark.parametrize("case", FWD_CASES, ids=[_fwd_id(c) for c in FWD_CASES])
def test_random_gated_forward_matches_oracle(env, case):
    """The forward with the output epilogue fused in (bf16 inputs, an initial state, the
    heads in H/2 decay tiers): y, rstd and the final state against the oracle's forward
    followed by its epilogue; o too when it is written."""
    import oracle
    gla, torch = env
    i, B, T, H, parts, overlap, want_o = case
    seed, n_tiers = 950 + i, max(1, H // 2)
    q, k, v = synth.qkv(seed, B, T, H)
    a = synth.aug_balance(seed, (H, 96), 0.1)
    init = synth.init_state(seed, B, H, 0.05)
    g = synth.round_bf16(synth.normal(seed, synth.DO, (B, T, H, 192), 1.5))
    w = 1.0 + synth.normal(seed, synth.A, (n_tiers, 192), 0.2)
    gam32, gam64 = oracle_decays(H)
    gla.set_split_parts(parts)
    gla.set_pass_overlap(overlap)
    try:
        qd, kd, vd, gd = (to_dev(x, torch.bfloat16) for x in (q, k, v, g))
        ad, idd, wd = (to_dev(x, torch.float32) for x in (a, init, w))
        y, rstd, o, fin = gla.chunk_fwd_gated(qd, kd, vd, gam32.cuda(), ad, gd, wd, n_tiers,
                                              1e-6, idd, want_o=bool(want_o))
        torch.cuda.synchronize()
        assert gla.get_device_error() == 0
    finally:
        gla.set_split_parts(0)
        gla.set_pass_overlap(True)
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a, init)
    y_ref, r_ref = oracle.head_norm_gate(o_ref.reshape(B * T, H, 192), g.reshape(B * T, H, 192),
                                         w, n_tiers, 1e-6)
    errs = dict(y=rel_err(y.cpu().numpy().reshape(B * T, H, 192), y_ref),
                rstd=rel_err(rstd.cpu().numpy().reshape(B * T, H), r_ref),
                final=rel_err(fin.cpu().numpy(), fin_ref))
    if want_o:
        errs["o"] = rel_err(o.cpu().numpy(), o_ref)
    print(_fwd_id(case) + ": " + " ".join(f"{n} {e:.2e}" for n, e in errs.items()))
    assert all(e <= TOL_CHUNK for e in errs.values()), errs


@pytest.mark.parametrize("case", FWD_CASES, ids=[_fwd_id(c) for c in FWD_CASES])
def test_random_paged_forward_matches_oracle(env, case):
    """Prefill into a state pool (bf16 inputs; a permutation of pages, layer 1 of 2): o and
    the pages written against the oracle's forward from the pages' states (or zero); every
    other page and layer untouched."""
    import oracle
    gla, torch = env
    i, B, T, H, parts, overlap, from_pool = case
    seed, P, PL, layer = 970 + i, B + 3, 2, 1
    rng = np.random.default_rng(seed)
    page = rng.permutation(P)[:B].astype(np.int32)
    pool = synth.normal(seed, synth.INIT, (P, PL, H, 96, 192), 0.05)
    q, k, v = synth.qkv(seed, B, T, H)
    a = synth.aug_balance(seed, (H, 96), 0.1)
    gam32, gam64 = oracle_decays(H)
    gla.set_split_parts(parts)
    gla.set_pass_overlap(overlap)
    try:
        pool_d = to_dev(pool, torch.float32)
        o = gla.chunk_fwd_paged(to_dev(q, torch.bfloat16), to_dev(k, torch.bfloat16),
                                to_dev(v, torch.bfloat16), gam32.cuda(), to_dev(a, torch.float32),
                                pool_d, to_dev(page, torch.int32), layer,
                                init_from_pool=bool(from_pool))
        torch.cuda.synchronize()
        assert gla.get_device_error() == 0
    finally:
        gla.set_split_parts(0)
        gla.set_pass_overlap(True)
    init = pool[page, layer] if from_pool else None
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a, init)
    new = pool_d.cpu().numpy()
    errs = dict(o=rel_err(o.cpu().numpy(), o_ref), final=rel_err(new[page, layer], fin_ref))
    print(_fwd_id(case) + ": " + " ".join(f"{n} {e:.2e}" for n, e in errs.items()))
    assert all(e <= TOL_CHUNK for e in errs.values()), errs
    touched = np.zeros((P, PL), bool)
    touched[page, layer] = True
    assert np.array_equal(new[~touched], pool[~touched])
