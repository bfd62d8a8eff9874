"""A randomized parity sweep with a fixed seed (the same cases every run): the chunked forward
and backward against the fp64 oracle over shapes (any T, few or many (b, h) pairs), input
types, forced part counts, both orders of the segment passes, initial state and final-state
adjoint present or absent, and the forward's saved activations (gate and state copies) handed
to the backward or not.  It looks for interactions the targeted tests leave out; the bar is
the usual 2e-2 of each output's RMS.  Wide cases (160-176 pairs, short T) put at least a wave
of whole pairs beside the cut ones, so the passes run beside them and a sum-pass CTA can take
several parts in turn."""
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
