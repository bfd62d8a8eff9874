"""GPU parity of the sequence-sharded calls (a long sequence cut into consecutive slices, one
per rank): the slice sums and the link against the fp64 oracle, and the whole sharded forward
and backward -- two ranks as two threads on this one GPU, their states passed through the same
exchange code multi-GPU runs use -- against the oracle over the whole sequence."""
import threading

import numpy as np
import pytest

import synth
from _util import TOL_CHUNK, oracle_decays, rel_err, to_dev

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


@pytest.mark.parametrize("B,T,H,dtype,seed", [
    (2, 128, 3, "bf16", 81),    # one chunk
    (1, 77, 2, "bf16", 82),     # one partial chunk
    (2, 300, 16, "bf16", 83),   # ragged last chunk, all decay tiers
    (1, 1, 4, "fp16", 84),      # a single token
    (2, 4000, 5, "fp16", 85),   # many chunks, ragged
    (10, 256, 16, "bf16", 86),  # 160 pairs, not fewer than the SMs: one CTA per pair (fewer
                                # pairs split each sum into three 64-column CTAs)
])
def test_slice_sums_match_oracle(env, B, T, H, dtype, seed):
    import oracle
    gla, torch = env
    td = torch.bfloat16 if dtype == "bf16" else torch.float16
    q, k, v = synth.qkv(seed, B, T, H, bf16=dtype == "bf16")
    dO = synth.grad_out(seed, B, T, H, bf16=dtype == "bf16")
    if dtype == "fp16":
        q, k, v, dO = (x.astype(np.float16).astype(np.float32) for x in (q, k, v, dO))
    gam, gam64 = oracle_decays(H)
    U = gla.chunk_state_sum(to_dev(k, td), to_dev(v, td), gam.cuda())
    Up = gla.chunk_adjoint_sum(to_dev(q, td), to_dev(dO, td), gam.cuda())
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    eu = rel_err(U.cpu().numpy(), oracle.slice_state_sum(k, v, gam64))
    ep = rel_err(Up.cpu().numpy(), oracle.slice_adjoint_sum(q, dO, gam64))
    print(f"slice sums B={B} T={T} H={H} {dtype}: U {eu:.2e} U' {ep:.2e}")
    assert eu <= TOL_CHUNK and ep <= TOL_CHUNK


@pytest.mark.parametrize("reverse", [False, True])
def test_state_link_matches_oracle(env, reverse):
    import oracle
    gla, torch = env
    lens, B, H = [300, 128, 4096, 1, 77], 2, 16
    U = synth.normal(86, synth.INIT, (len(lens), B, H, 96, 192), 0.3)
    bnd = synth.normal(86, synth.DFIN, (B, H, 96, 192), 0.1)
    gam, gam64 = oracle_decays(H)
    Ud, bd = to_dev(U, torch.float32), to_dev(bnd, torch.float32)
    for r in range(len(lens)):
        for b in (bd, None):
            out = gla.state_link(Ud, lens, r, gam.cuda(), b, reverse=reverse)
            ref = oracle.state_link(U, lens, r, gam64, None if b is None else bnd, reverse)
            # (the link is fp32 arithmetic on fp32 inputs)
            assert rel_err(out.cpu().numpy(), ref) <= 1e-5, (r, b is None)
    assert gla.get_device_error() == 0


def _sharded(env, q, k, v, dO, a, init, dfin, lens, H):
    """Both ranks' forward and backward, as threads sharing this GPU; returns per-rank
    results."""
    gla, torch = env
    from gated_linear_attention_chunked_gb300 import seqshard
    shared = seqshard.ThreadExchange(len(lens))
    gam = oracle_decays(H)[0].cuda()
    res, errors = {}, []
    edges = np.cumsum([0] + lens)

    def body(r):
        try:
            sl = slice(edges[r], edges[r + 1])
            qd, kd, vd, gd = (to_dev(np.ascontiguousarray(x[:, sl]), torch.bfloat16)
                              for x in (q, k, v, dO))
            ad, idd, fd = (to_dev(x, torch.float32) for x in (a, init, dfin))
            ex = shared.view(r)
            gate = torch.empty((q.shape[0], H, lens[r]), dtype=torch.float32, device="cuda")
            o, s_out, s_in = seqshard.chunk_fwd_sharded(qd, kd, vd, gam, ad, idd, exchange=ex,
                                                        gate=gate)
            dq, dk, dv, d_aug, d_in = seqshard.chunk_bwd_sharded(qd, kd, vd, gam, ad, gd, s_in, fd,
                                                                 exchange=ex, gate=gate)
            torch.cuda.synchronize()
            res[r] = {n: x.cpu().numpy() for n, x in dict(o=o, s_out=s_out, dq=dq, dk=dk, dv=dv,
                                                           d_aug=d_aug, d_in=d_in).items()}
        except BaseException as e:  # surfaced by the caller
            errors.append(e)
            shared._barrier.abort()

    threads = [threading.Thread(target=body, args=(r,)) for r in range(len(lens))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=600)
    assert not errors, errors
    assert gla.get_device_error() == 0
    return res


@pytest.mark.parametrize("lens,seed", [([4196, 3996], 87), ([128, 300], 88)])
def test_two_ranks_on_one_gpu_match_the_whole_sequence(env, lens, seed):
    """Two slices of unequal length (the first ends inside a chunk), a nonzero initial state
    and final-state adjoint: the pieces the ranks return equal the oracle's forward and
    backward over the whole sequence (every output, the final state, d_init_state on rank 0,
    d_aug summed over the ranks)."""
    import oracle
    gla, torch = env
    B, H, T = 2, 16, sum(lens)
    q, k, v = synth.qkv(seed, B, T, H)
    dO = synth.grad_out(seed, B, T, H)
    a = synth.aug_balance(seed, (H, 96), 0.02)
    init = synth.init_state(seed, B, H, 0.01)
    dfin = synth.normal(seed, synth.DFIN, (B, H, 96, 192), 0.05)
    res = _sharded(env, q, k, v, dO, a, init, dfin, lens, H)
    gam64 = oracle_decays(H)[1]
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a, init)
    ref = oracle.bwd(q, k, v, gam64, a, dO, init, dfin)
    cat = lambda n: np.concatenate([res[r][n] for r in range(len(lens))], axis=1)
    errs = dict(o=rel_err(cat("o"), o_ref), final=rel_err(res[len(lens) - 1]["s_out"], fin_ref),
                dq=rel_err(cat("dq"), ref["dq"]), dk=rel_err(cat("dk"), ref["dk"]),
                dv=rel_err(cat("dv"), ref["dv"]), d_init=rel_err(res[0]["d_in"], ref["d_init_state"]))
    for r in range(len(lens)):
        errs[f"d_aug{r}"] = rel_err(res[r]["d_aug"], ref["d_a"])
    # the first and last 4096 outputs on their own (the long-prefill check)
    n = min(4096, T)
    errs["o_first"] = rel_err(cat("o")[:, :n], o_ref[:, :n])
    errs["o_last"] = rel_err(cat("o")[:, -n:], o_ref[:, -n:])
    print(f"sharded lens={lens}: " + " ".join(f"{k_} {e:.1e}" for k_, e in errs.items()))
    for name, e in errs.items():
        assert e <= TOL_CHUNK, f"{name}: {e:.3e}"
