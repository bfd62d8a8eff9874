"""GPU parity of the chunked calls when (b, h) pairs are cut into chunk ranges run as separate
CTAs (each part starting from the state, or the adjoint, that the segment passes computed at
its boundary).  The cut is forced with gla_set_split_parts so that small shapes exercise it;
every case is checked against the fp64 oracle (bar 2e-2 of each output's RMS) and against the
same call with nothing cut."""
import numpy as np
import pytest

import synth
from _util import TOL_CHUNK, rel_err, to_dev, oracle_decays

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "d_a", "d_init_state")


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


def n_sm(torch):
    return torch.cuda.get_device_properties(0).multi_processor_count


CASES = [
    # B, T, H, forced parts, input dtype, seed
    (1, 512, 2, 4, "bf16", 61),     # every pair cut into 4 parts of one chunk
    (2, 700, 3, 3, "bf16", 62),     # ragged T: the last part ends in a 60-token chunk
    (1, 1000, 2, 5, "fp16", 63),    # 8 chunks in 5 unequal parts (1-2 chunks), ragged
    (1, 384, 2, 2, "fp32", 64),     # fp32 inputs: the passes read the fp16 copies
    (3, 300, 16, 3, "bf16", 65),    # all 16 decay tiers, a 44-token last chunk
]


def _inputs(seed, B, T, H, dtype):
    q, k, v = synth.qkv(seed, B, T, H, bf16=(dtype == "bf16"))
    dO = synth.grad_out(seed, B, T, H, bf16=(dtype == "bf16"))
    if dtype == "fp16":
        q, k, v, dO = (x.astype(np.float16).astype(np.float32) for x in (q, k, v, dO))
    a = synth.aug_balance(seed, (H, 96), 0.1)
    init = synth.init_state(seed, B, H, 0.05)
    dfin = synth.normal(seed, synth.DFIN, (B, H, 96, 192), 0.05)
    return q, k, v, dO, a, init, dfin


def _run(env, parts, q, k, v, dO, a, init, dfin, H, dtype):
    gla, torch = env
    td = dict(bf16=torch.bfloat16, fp16=torch.float16, fp32=torch.float32)[dtype]
    gla.set_split_parts(parts)
    try:
        gam = oracle_decays(H)[0].cuda()
        qd, kd, vd, gd = (to_dev(x, td) for x in (q, k, v, dO))
        ad, idd, fd = (to_dev(x, torch.float32) for x in (a, init, dfin))
        o, fin = gla.chunk_fwd(qd, kd, vd, gam, ad, idd)
        g = gla.chunk_bwd(qd, kd, vd, gam, ad, gd, idd, fd)
        torch.cuda.synchronize()
        assert gla.get_device_error() == 0
    finally:
        gla.set_split_parts(0)
    return o.cpu().numpy(), fin.cpu().numpy(), [x.cpu().numpy() for x in g]


@pytest.mark.parametrize("B,T,H,parts,dtype,seed", CASES)
def test_cut_pairs_match_oracle_and_uncut(env, B, T, H, parts, dtype, seed):
    import oracle
    gla, torch = env
    wf, pf = gla.split_plan(B, T, H, False, n_sm(torch))
    nc = -(-T // 128)
    # with parts forced, the calls cut every pair (B*H < SMs) into min(parts, nc) parts
    gla.set_split_parts(parts)
    try:
        assert gla.split_plan(B, T, H, False, n_sm(torch)) == (0, min(parts, nc))
        assert gla.split_plan(B, T, H, True, n_sm(torch)) == (0, min(parts, nc))
    finally:
        gla.set_split_parts(0)
    q, k, v, dO, a, init, dfin = _inputs(seed, B, T, H, dtype)
    o, fin, g = _run(env, parts, q, k, v, dO, a, init, dfin, H, dtype)
    o1, fin1, g1 = _run(env, 1, q, k, v, dO, a, init, dfin, H, dtype)
    gam64 = oracle_decays(H)[1]
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a, init)
    ref = oracle.bwd(q, k, v, gam64, a, dO, init, dfin)
    errs = dict(o=rel_err(o, o_ref), final=rel_err(fin, fin_ref))
    errs.update({n: rel_err(x, ref[n]) for n, x in zip(NAMES, g)})
    uncut = dict(o=rel_err(o, o1), final=rel_err(fin, fin1))
    uncut.update({n: rel_err(x, y) for n, x, y in zip(NAMES, g, g1)})
    print(f"cut B={B} T={T} H={H} parts={parts} {dtype}: " +
          " ".join(f"{n} {e:.2e}" for n, e in errs.items()) +
          " | vs uncut " + " ".join(f"{n} {e:.1e}" for n, e in uncut.items()))
    assert all(e <= TOL_CHUNK for e in errs.values()), errs
    assert all(e <= TOL_CHUNK for e in uncut.values()), uncut


def test_whole_and_cut_pairs_in_one_launch(env):
    """B*H = 160 pairs on a 152-SM device: 152 run whole and the last 8 are cut (forward);
    the backward's 480 role CTAs leave 24 for a fourth wave, so 8 pairs are cut there too."""
    import oracle
    gla, torch = env
    B, T, H, seed = 10, 256, 16, 66
    if n_sm(torch) != 152:
        pytest.skip("the layout of this case assumes 152 SMs")
    gla.set_split_parts(2)
    try:
        assert gla.split_plan(B, T, H, False, 152) == (152, 2)
        assert gla.split_plan(B, T, H, True, 152) == (152, 2)
    finally:
        gla.set_split_parts(0)
    q, k, v, dO, a, init, dfin = _inputs(seed, B, T, H, "bf16")
    o, fin, g = _run(env, 2, q, k, v, dO, a, init, dfin, H, "bf16")
    gam64 = oracle_decays(H)[1]
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a, init)
    ref = oracle.bwd(q, k, v, gam64, a, dO, init, dfin)
    errs = dict(o=rel_err(o, o_ref), final=rel_err(fin, fin_ref))
    errs.update({n: rel_err(x, ref[n]) for n, x in zip(NAMES, g)})
    # the cut pairs are the last 8: (b, h) = (9, 8..15)
    errs["o_cut"] = rel_err(o[9, :, 8:], o_ref[9, :, 8:])
    errs["dq_cut"] = rel_err(g[0][9, :, 8:], ref["dq"][9, :, 8:])
    print("whole+cut B=10 T=256 H=16: " + " ".join(f"{n} {e:.2e}" for n, e in errs.items()))
    assert all(e <= TOL_CHUNK for e in errs.values()), errs


def test_cut_pairs_paged_and_gated(env):
    """The cut applies to the pool-addressed prefill (initial state from the pool, final state
    back to it) and to the forward with the fused output epilogue."""
    import oracle
    gla, torch = env
    B, T, H, P, PL, layer, seed = 2, 600, 3, 5, 2, 1, 67
    rng = np.random.default_rng(seed)
    page = rng.permutation(P)[:B].astype(np.int32)
    pool = synth.normal(seed, synth.INIT, (P, PL, H, 96, 192), 0.05).astype(np.float32)
    q, k, v = synth.qkv(seed, B, T, H)
    a = synth.aug_balance(seed, (H, 96), 0.1)
    gam = oracle_decays(H)[0]
    gam64 = gam.numpy().astype(np.float64)
    g_in = synth.round_bf16(synth.normal(seed, synth.DO, (B, T, H, 192), 1.5))
    w = 1.0 + synth.normal(seed, synth.A, (1, 192), 0.2)
    gla.set_split_parts(4)
    try:
        pool_d = to_dev(pool, torch.float32)
        qd, kd, vd = (to_dev(x, torch.bfloat16) for x in (q, k, v))
        o = gla.chunk_fwd_paged(qd, kd, vd, gam.cuda(), to_dev(a, torch.float32), pool_d,
                                to_dev(page, torch.int32), layer, init_from_pool=True)
        init = pool[page, layer]
        y, rstd, o2, fin2 = gla.chunk_fwd_gated(qd, kd, vd, gam.cuda(), to_dev(a, torch.float32),
                                                to_dev(g_in, torch.bfloat16),
                                                to_dev(w, torch.float32), 1, 1e-6,
                                                to_dev(init, torch.float32), want_o=True)
        torch.cuda.synchronize()
        assert gla.get_device_error() == 0
    finally:
        gla.set_split_parts(0)
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a, init)
    new = pool_d.cpu().numpy()
    y_ref, _ = oracle.head_norm_gate(o_ref.reshape(B * T, H, 192), g_in.reshape(B * T, H, 192),
                                     w, 1, 1e-6)
    errs = dict(o=rel_err(o.cpu().numpy(), o_ref), pool_final=rel_err(new[page, layer], fin_ref),
                gated_y=rel_err(y.cpu().numpy().reshape(B * T, H, 192), y_ref),
                gated_o=rel_err(o2.cpu().numpy(), o_ref), gated_final=rel_err(fin2.cpu().numpy(), fin_ref))
    print("cut paged/gated: " + " ".join(f"{n} {e:.2e}" for n, e in errs.items()))
    assert all(e <= TOL_CHUNK for e in errs.values()), errs
    touched = np.zeros((P, PL), bool)
    touched[page, layer] = True
    assert np.array_equal(new[~touched], pool[~touched])


def test_pass_overlap_matches_serial_order(env):
    """With a full wave of whole pairs the segment passes run beside them (the chunked kernel a
    programmatic dependent of the passes, its parts waiting for them); with
    gla_set_pass_overlap(0) the passes run first.  The kernels and their arithmetic are the
    same, so every output is bit-identical between the two orders -- plain and training path
    (saved gate and state copies), the forward with the fused output epilogue and the
    prefill into a state pool.  B = 13 leaves 56 forward pairs for a last wave: beside the
    whole pairs their 56 sums run on 51 CTAs, so some CTAs of the sum pass take two parts in a
    row, against one part per CTA in the serial order."""
    gla, torch = env
    B, T, H, seed = 13, 256, 16, 68
    if n_sm(torch) != 152:
        pytest.skip("the layout of this case assumes 152 SMs")
    q, k, v, dO, a, init, dfin = _inputs(seed, B, T, H, "bf16")
    gam = oracle_decays(H)[0].cuda()
    qd, kd, vd, gd = (to_dev(x, torch.bfloat16) for x in (q, k, v, dO))
    ad, idd, fd = (to_dev(x, torch.float32) for x in (a, init, dfin))
    g_in = to_dev(synth.normal(seed, synth.DO, (B, T, H, 192), 1.5), torch.bfloat16)
    w_n = to_dev(1.0 + synth.normal(seed, synth.A, (4, 192), 0.2), torch.float32)
    P = B + 3  # a pool of 16 pages of 2 layers; sequence b uses page[b]
    pool = to_dev(synth.normal(seed, synth.INIT, (P, 2, H, 96, 192), 0.05), torch.float32)
    page = to_dev(np.random.default_rng(seed).permutation(P)[:B].astype(np.int32), torch.int32)

    def run(overlap):
        gla.set_pass_overlap(overlap)
        gla.set_split_parts(2)
        try:
            out = []
            o, fin = gla.chunk_fwd(qd, kd, vd, gam, ad, idd)
            out += [o, fin, *gla.chunk_bwd(qd, kd, vd, gam, ad, gd, idd, fd)]
            gate = torch.empty(B, H, T, device="cuda")
            saved = torch.empty(gla.chunk_saved_states_size(B, T, H), dtype=torch.uint8,
                                device="cuda")
            o2, fin2 = gla.chunk_fwd(qd, kd, vd, gam, ad, idd, gate=gate, saved_states=saved)
            out += [o2, fin2, gate,
                    *gla.chunk_bwd(qd, kd, vd, gam, ad, gd, idd, fd, gate=gate,
                                   saved_states=saved)]
            y, rstd, o3, fin3 = gla.chunk_fwd_gated(qd, kd, vd, gam, ad, g_in, w_n, 4, 1e-6, idd,
                                                    want_o=True)
            pool_d = pool.clone()
            o4 = gla.chunk_fwd_paged(qd, kd, vd, gam, ad, pool_d, page, 1, init_from_pool=True)
            out += [y, rstd, o3, fin3, o4, pool_d]
            torch.cuda.synchronize()
            assert gla.get_device_error() == 0
            return [x.cpu().numpy() for x in out]
        finally:
            gla.set_split_parts(0)
            gla.set_pass_overlap(True)

    on, off = run(True), run(False)
    names = ["o", "final", *NAMES, "o_saved", "final_saved", "gate",
             *(n + "_saved" for n in NAMES), "gated_y", "gated_rstd", "gated_o", "gated_final",
             "paged_o", "paged_pool"]
    diff = [n for n, x, y in zip(names, on, off) if not np.array_equal(x, y)]
    assert not diff, f"outputs differ between the launch orders: {diff}"
