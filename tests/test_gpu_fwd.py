"""GPU parity of gla_chunk_fwd against the fp64 oracle (bar: 2e-2 of the output RMS)."""
import numpy as np
import pytest

import synth
from _util import TOL_CHUNK, as_dtype_values, rel_err, to_dev, oracle_decays

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


TDT = {"bf16": "bfloat16", "fp16": "float16", "fp32": "float32"}


def run_fwd(env, q, k, v, a, init, H, dtype):
    import oracle
    gla, torch = env
    td = getattr(torch, TDT[dtype])
    q, k, v = (as_dtype_values(x, dtype) for x in (q, k, v))
    gam = oracle_decays(H)[0]
    gam64 = oracle_decays(H)[1]
    init_d = None if init is None else to_dev(init, torch.float32)
    o, fin = gla.chunk_fwd(to_dev(q, td), to_dev(k, td), to_dev(v, td), gam.cuda(),
                           to_dev(a, torch.float32), init_d)
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    return o.cpu().numpy(), fin.cpu().numpy(), (q, k, v, gam64)


CASES = [
    # B, T, H, dtype, init std, a std, seed
    (1, 128, 1, "bf16", 0.0, 0.1, 11),     # one chunk, one head
    (2, 384, 5, "bf16", 0.05, 0.1, 12),    # odd head count, 3 chunks, initial state
    (1, 256, 2, "fp16", 0.05, 0.1, 13),
    (1, 256, 2, "fp32", 0.0, 0.1, 0),      # the tiny fp32 workload shape
    (3, 640, 16, "bf16", 0.02, 0.02, 14),  # all 16 decay tiers, 5 chunks
    # ragged: the last chunk holds T mod 128 tokens (zero rows past T, its own decay powers)
    (2, 1, 3, "bf16", 0.05, 0.1, 15),      # a single token per sequence
    (2, 77, 3, "bf16", 0.05, 0.1, 16),     # one partial chunk
    (2, 200, 16, "bf16", 0.05, 0.02, 17),  # a full chunk and 72 tokens, all decay tiers
    (1, 300, 2, "fp32", 0.05, 0.1, 18),    # fp32 inputs
    (3, 511, 5, "fp16", 0.02, 0.1, 19),    # four chunks, the last one 127 tokens
]


@pytest.mark.parametrize("B,T,H,dtype,init_std,a_std,seed", CASES)
def test_fwd_small(env, B, T, H, dtype, init_std, a_std, seed):
    import oracle
    q, k, v = synth.qkv(seed, B, T, H, bf16=False)
    a = synth.aug_balance(seed, (H, 96), a_std)
    init = synth.init_state(seed, B, H, init_std) if init_std > 0 else None
    o, fin, (q, k, v, gam64) = run_fwd(env, q, k, v, a, init, H, dtype)
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a, init)
    eo, ef = rel_err(o, o_ref), rel_err(fin, fin_ref)
    print(f"fwd B={B} T={T} H={H} {dtype}: o {eo:.2e} final {ef:.2e}")
    assert eo <= TOL_CHUNK and ef <= TOL_CHUNK


def test_fwd_tiny_fp32_workload(env):
    import oracle
    x = synth.chunk_inputs("tiny_fp32")
    c = x["cfg"]
    o, fin, (q, k, v, gam64) = run_fwd(env, x["q"], x["k"], x["v"], x["a"], None, c["H"], "fp32")
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, x["a"])
    eo, ef = rel_err(o, o_ref), rel_err(fin, fin_ref)
    print(f"fwd tiny fp32: o {eo:.2e} final {ef:.2e}")
    assert eo <= TOL_CHUNK and ef <= TOL_CHUNK


@pytest.mark.parametrize("name", ["layer_fwd", "layer_fwd_aug"])
def test_fwd_layer_workload(env, name):
    """One training-shape layer, B=8, T=2048, H=16, bf16; a = 0 and a ~ N(0, 0.02)."""
    import oracle
    x = synth.chunk_inputs(name)
    c = x["cfg"]
    o, fin, (q, k, v, gam64) = run_fwd(env, x["q"], x["k"], x["v"], x["a"], None, c["H"], "bf16")
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, x["a"])
    eo, ef = rel_err(o, o_ref), rel_err(fin, fin_ref)
    print(f"fwd {name}: o {eo:.2e} final {ef:.2e}")
    assert eo <= TOL_CHUNK and ef <= TOL_CHUNK


def test_fwd_zero_init_equals_no_init(env):
    gla, torch = env
    B, T, H = 2, 256, 3
    q, k, v = synth.qkv(21, B, T, H)
    a = synth.aug_balance(21, (H, 96), 0.1)
    o1, f1, _ = run_fwd(env, q, k, v, a, None, H, "bf16")
    o2, f2, _ = run_fwd(env, q, k, v, a, np.zeros((B, H, 96, 192), np.float32), H, "bf16")
    assert np.array_equal(o1, o2) and np.array_equal(f1, f2)


def test_fwd_state_carry(env):
    """fwd over T tokens equals fwd over the second part started from the first part's
    final state (the chunk boundary is a multiple of 128)."""
    B, T, H, T1 = 2, 512, 4, 256
    q, k, v = synth.qkv(22, B, T, H)
    a = synth.aug_balance(22, (H, 96), 0.1)
    o, fin, _ = run_fwd(env, q, k, v, a, None, H, "bf16")
    o1, f1, _ = run_fwd(env, q[:, :T1], k[:, :T1], v[:, :T1], a, None, H, "bf16")
    o2, f2, _ = run_fwd(env, q[:, T1:], k[:, T1:], v[:, T1:], a, f1, H, "bf16")
    assert rel_err(np.concatenate([o1, o2], 1), o) <= 1e-6
    assert rel_err(f2, fin) <= 1e-6


def test_fwd_long_prefill_workload(env):
    """Long-context prefill: B=2, T=131072, H=16, bf16, initial state ~ N(0, 0.01).
    Checked on the first and last 4,096 outputs and on the full final state."""
    import oracle
    x = synth.chunk_inputs("long_prefill")
    c = x["cfg"]
    o, fin, (q, k, v, gam64) = run_fwd(env, x["q"], x["k"], x["v"], x["a"], x["init_state"],
                                       c["H"], "bf16")
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, x["a"], x["init_state"])
    n = 4096
    e_first = rel_err(o[:, :n], o_ref[:, :n])
    e_last = rel_err(o[:, -n:], o_ref[:, -n:])
    ef = rel_err(fin, fin_ref)
    print(f"fwd long: first {e_first:.2e} last {e_last:.2e} final {ef:.2e}")
    assert e_first <= TOL_CHUNK and e_last <= TOL_CHUNK and ef <= TOL_CHUNK
    assert np.all(np.isfinite(o))


@pytest.mark.parametrize("B,T,H,seed", [(1, 4096, 2, 31), (1, 8192, 3, 32)])
def test_fwd_segmented_path(env, B, T, H, seed):
    """Few long sequences have their pairs cut into parts (the state sums of the parts in
    parallel, their recurrence, then every part as its own CTA).  The call must match the
    oracle, initial and final state included, and one chain per pair, which the same call
    runs when it is given no workspace."""
    import oracle
    gla, torch = env
    assert gla.chunk_fwd_workspace_size(B, T, H, gla.GLA_BF16) > 0, "pairs not cut"
    q, k, v = synth.qkv(seed, B, T, H)
    a = synth.aug_balance(seed, (H, 96), 0.1)
    init = synth.init_state(seed, B, H, 0.05)
    o, fin, (q, k, v, gam64) = run_fwd(env, q, k, v, a, init, H, "bf16")
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a, init)
    eo, ef = rel_err(o, o_ref), rel_err(fin, fin_ref)
    # one chain per pair: same call through the C ABI without a workspace
    lib = gla.load()
    qd, kd, vd = (to_dev(x, torch.bfloat16) for x in (q, k, v))
    gam = oracle_decays(H)[0].cuda()
    ad, idd = to_dev(a, torch.float32), to_dev(init, torch.float32)
    o2 = torch.empty((B, T, H, 192), dtype=torch.float32, device="cuda")
    f2 = torch.empty((B, H, 96, 192), dtype=torch.float32, device="cuda")
    rc = lib.gla_chunk_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), gla.GLA_BF16,
                           gam.data_ptr(), ad.data_ptr(), idd.data_ptr(), o2.data_ptr(),
                           f2.data_ptr(), None, None, 0, None, 0, B, T, H, 96, 192,
                           torch.cuda.current_stream().cuda_stream)
    assert rc == 0, gla.status_string(rc)
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    es = rel_err(o, o2.cpu().numpy())
    print(f"fwd cut B={B} T={T} H={H}: o {eo:.2e} final {ef:.2e} vs uncut {es:.2e}")
    assert eo <= TOL_CHUNK and ef <= TOL_CHUNK
    assert rel_err(o2.cpu().numpy(), o_ref) <= TOL_CHUNK
    assert rel_err(f2.cpu().numpy(), fin_ref) <= TOL_CHUNK


@pytest.mark.parametrize("B,T,H,n_tiers,want_o,seed", [
    (2, 384, 4, 2, True, 41),      # serial scan, o written too
    (1, 4096, 2, 1, False, 42),    # pairs cut into parts, y only
    (8, 2048, 16, 4, True, 43),    # one training-shape layer
    (2, 200, 4, 2, True, 44),      # ragged last chunk: y, rstd and o stop at T
])
def test_fwd_gated(env, B, T, H, n_tiers, want_o, seed):
    """The forward with the output epilogue fused in: y (Head RMSNorm per tier, SiLU(g) gate)
    and rstd against the oracle's forward followed by its epilogue; o, when written, is the
    plain forward's output bit for bit, and y equals the standalone epilogue applied to it."""
    import oracle
    gla, torch = env
    q, k, v = synth.qkv(seed, B, T, H)
    a = synth.aug_balance(seed, (H, 96), 0.1)
    init = synth.init_state(seed, B, H, 0.05)
    g = synth.round_bf16(synth.normal(seed, synth.DO, (B, T, H, 192), 1.5))
    w = 1.0 + synth.normal(seed, synth.A, (n_tiers, 192), 0.2)
    qd, kd, vd, gd = (to_dev(x, torch.bfloat16) for x in (q, k, v, g))
    gam = oracle_decays(H)[0].cuda()
    ad, idd, wd = (to_dev(x, torch.float32) for x in (a, init, w))
    y, rstd, o, fin = gla.chunk_fwd_gated(qd, kd, vd, gam, ad, gd, wd, n_tiers, 1e-6, idd,
                                          want_o=want_o)
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    gam64 = oracle_decays(H)[1]
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a, init)
    y_ref, r_ref = oracle.head_norm_gate(o_ref.reshape(B * T, H, 192), g.reshape(B * T, H, 192),
                                         w, n_tiers, 1e-6)
    ey = rel_err(y.cpu().numpy().reshape(B * T, H, 192), y_ref)
    er = rel_err(rstd.cpu().numpy().reshape(B * T, H), r_ref)
    ef = rel_err(fin.cpu().numpy(), fin_ref)
    print(f"fwd gated B={B} T={T} H={H} tiers={n_tiers}: y {ey:.2e} rstd {er:.2e} final {ef:.2e}")
    assert ey <= TOL_CHUNK and er <= TOL_CHUNK and ef <= TOL_CHUNK
    if want_o:
        o_plain, _ = gla.chunk_fwd(qd, kd, vd, gam, ad, idd)
        y2, _ = gla.head_norm_gate(o_plain, gd, wd, n_tiers, 1e-6)
        torch.cuda.synchronize()
        assert torch.equal(o, o_plain)
        assert rel_err(y.cpu().numpy(), y2.cpu().numpy()) <= 1e-5


def test_fwd_ragged_writes_nothing_past_t(env):
    """With T = 200 the last chunk's rows 72..127 are padding: o and the final state match the
    oracle, and the output buffer's elements right after the last sequence stay untouched."""
    import oracle
    gla, torch = env
    B, T, H, seed = 2, 200, 3, 19
    q, k, v = synth.qkv(seed, B, T, H)
    a = synth.aug_balance(seed, (H, 96), 0.1)
    init = synth.init_state(seed, B, H, 0.05)
    n = B * T * H * 192
    big = torch.full((n + 64 * H * 192,), float("nan"), dtype=torch.float32, device="cuda")
    o = big[:n].view(B, T, H, 192)
    fin = torch.empty((B, H, 96, 192), dtype=torch.float32, device="cuda")
    gam = oracle_decays(H)[0]
    gla.chunk_fwd(to_dev(q, torch.bfloat16), to_dev(k, torch.bfloat16), to_dev(v, torch.bfloat16),
                  gam.cuda(), to_dev(a, torch.float32), to_dev(init, torch.float32), out=o,
                  final_state=fin)
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    o_ref, fin_ref = oracle.fwd(q, k, v, gam.numpy().astype(np.float64), a, init)
    eo, ef = rel_err(o.cpu().numpy(), o_ref), rel_err(fin.cpu().numpy(), fin_ref)
    print(f"fwd ragged T={T}: o {eo:.2e} final {ef:.2e}")
    assert eo <= TOL_CHUNK and ef <= TOL_CHUNK
    assert torch.isnan(big[n:]).all()
