"""The C ABI without a GPU: the library loads, exports every declared symbol, and rejects
bad arguments with its documented status codes before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import gated_linear_attention_chunked_gb300 as gla
from gated_linear_attention_chunked_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return gla.load()


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "gla.h")).read()
    return sorted(set(re.findall(r"GLA_API\s+[\w\s\*]+?\b(gla_\w+)\s*\(", txt)))


def test_header_declares_the_calls():
    names = declared_symbols()
    for n in ("gla_chunk_fwd", "gla_chunk_bwd", "gla_decode_step", "gla_decay_schedule",
              "gla_get_device_error", "gla_status_string", "gla_decode_step_paged",
              "gla_chunk_fwd_paged"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(gla.lib_path())
    for n in declared_symbols():
        assert hasattr(raw, n), f"{n} not exported"


def test_status_strings(lib):
    for code in gla.STATUS:
        assert gla.status_string(code)
    assert gla.status_string(0) == "ok"


def test_decay_schedule_matches_oracle(lib):
    import oracle
    for H, tmin, tmax in [(16, 1.0, 2048.0), (2, 1.0, 2048.0), (1, 4.0, 4.0), (7, 2.0, 300.0)]:
        g = gla.decay_schedule(H, tmin, tmax).numpy()
        ref = oracle.decay_schedule(H, tmin, tmax)
        # same fp64 formula on both sides, rounded once to fp32
        assert np.array_equal(g, ref.astype(np.float32))
    g = gla.decay_schedule(16).numpy().astype(np.float64)
    assert np.exp(g[0]) == pytest.approx(0.5, rel=1e-7)
    assert np.exp(g[15]) == pytest.approx(2 ** (-1 / 2048), rel=1e-7)


def test_decay_schedule_rejects(lib):
    out = (ctypes.c_float * 4)()
    assert lib.gla_decay_schedule(0, 1.0, 2.0, ctypes.addressof(out)) == 1
    assert lib.gla_decay_schedule(4, 0.0, 2.0, ctypes.addressof(out)) == 1
    assert lib.gla_decay_schedule(4, 1.0, 2.0, None) == 1


A16 = 0x1000  # a 16-byte aligned fake address; never dereferenced by the checks below


def fwd(lib, q=A16, k=A16, v=A16, dt=0, ld=A16, a=A16, init=None, o=A16, fin=None, gate=None,
        ws=None, wsb=0, B=1, T=128, H=1, dk=96, dv=192):
    return lib.gla_chunk_fwd(q, k, v, dt, ld, a, init, o, fin, gate, None, 0, ws, wsb, B, T, H,
                             dk, dv, None)


def test_chunk_fwd_argument_checks(lib):
    assert fwd(lib, dk=64) == 2                      # unsupported head size
    assert fwd(lib, dv=128) == 2
    assert fwd(lib, T=200, q=A16 + 8) == 3           # any T: the sizes pass, the next check fails
    assert fwd(lib, B=1 << 20, T=1 << 12) == 2       # 2^32 tokens: beyond the index range
    assert fwd(lib, dt=7) == 2                       # unknown dtype
    assert fwd(lib, B=0) == 1 and fwd(lib, T=0) == 1 and fwd(lib, H=-1) == 1
    assert fwd(lib, q=None) == 1 and fwd(lib, o=None) == 1 and fwd(lib, a=None) == 1
    assert fwd(lib, q=A16 + 8) == 3                  # misaligned
    assert fwd(lib, init=A16 + 4) == 3
    assert fwd(lib, gate=A16 + 2) == 3               # the saved gate: 4-byte aligned fp32
    # fp32 inputs need a workspace for their fp16 copies
    assert gla.chunk_fwd_workspace_size(1, 128, 1, gla.GLA_FP32) > 0
    assert gla.chunk_fwd_workspace_size(1, 128, 1, gla.GLA_BF16) == 0
    assert fwd(lib, dt=1) == 7
    need = gla.chunk_fwd_workspace_size(1, 128, 1, gla.GLA_FP32)
    assert fwd(lib, dt=1, ws=A16, wsb=need - 1) == 7
    assert fwd(lib, dt=1, ws=A16 + 16, wsb=need) == 3  # workspace must be 256-aligned


def test_chunk_bwd_argument_checks(lib):
    def bwd(dO=A16, dq=A16, dk_=64, T=128, d_aug=A16, gate=None):
        return lib.gla_chunk_bwd(A16, A16, A16, 0, A16, A16, None, dO, None, gate, None, 0, dq,
                                 A16, A16,
                                 d_aug, None, None, 0, 1, T, 1, dk_, 192, None)
    assert bwd() == 2
    assert bwd(dk_=96, T=100, dq=A16 + 2) == 3         # any T: the sizes pass
    assert bwd(dk_=96, dO=None) == 1
    assert bwd(dk_=96, d_aug=None) == 1
    assert bwd(dk_=96, gate=A16 + 1) == 3
    assert bwd(dk_=96, dq=A16 + 2) == 3


def test_decode_argument_checks(lib):
    def dec(st=A16, N=1, L=1, H=1, dk=96, dv=192, o=A16):
        return lib.gla_decode_step(st, A16, A16, A16, A16, A16, o, N, L, H, dk, dv, None)
    assert dec(N=0) == 1 and dec(L=0) == 1
    assert dec(dk=64) == 2 and dec(dv=96) == 2
    assert dec(st=None) == 1 and dec(o=None) == 1
    assert dec(st=A16 + 4) == 3


def test_binding_refuses_host_tensors(lib):
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 128, 1, 96, dtype=torch.bfloat16)
    v = torch.zeros(1, 128, 1, 192, dtype=torch.bfloat16)
    with pytest.raises((ValueError, RuntimeError, AssertionError)):
        gla.chunk_fwd(q, q, v, torch.zeros(1), torch.zeros(1, 96))


def test_paged_argument_checks(lib):
    def dec(n=2, P=4, PL=3, l0=0, L=2, H=2, dk=96, pool=A16, page=A16, q=A16):
        return lib.gla_decode_step_paged(pool, page, n, P, PL, l0, q, A16, A16, A16, A16, A16,
                                         L, H, dk, 192, None)
    assert dec(n=0) == 0                   # empty active set: nothing to do
    assert dec(l0=2, L=2) == 1             # layers beyond the page
    assert dec(P=0) == 1 and dec(PL=0) == 1 and dec(n=-1) == 1 and dec(H=0) == 1
    assert dec(dk=64) == 2
    assert dec(page=None) == 1 and dec(pool=None) == 1
    assert dec(q=A16 + 4) == 3

    def fwdp(layer=0, PL=2, P=3, page=A16, pool=A16, T=128):
        return lib.gla_chunk_fwd_paged(A16, A16, A16, 0, A16, A16, pool, page, P, PL, layer, 1,
                                       A16, None, 0, 1, T, 1, 96, 192, None)
    assert fwdp(layer=2) == 1 and fwdp(layer=-1) == 1 and fwdp(P=0) == 1
    assert fwdp(page=None) == 1 and fwdp(pool=None) == 1
    assert fwdp(page=A16 + 4) == 3
    assert fwdp(T=100, page=A16 + 4) == 3


def test_head_norm_argument_checks(lib):
    def fwdn(n_tiers=4, H=16, dv=192, eps=1e-6, gdt=0, o=A16, y=A16, N=3):
        return lib.gla_head_norm_gate_fwd(o, A16, gdt, A16, n_tiers, eps, y, None, N, H, dv, None)
    assert fwdn(n_tiers=3) == 1          # tiers must divide the heads
    assert fwdn(n_tiers=0) == 1 and fwdn(H=0) == 1 and fwdn(N=-1) == 1
    assert fwdn(eps=-1.0) == 1
    assert fwdn(dv=96) == 2 and fwdn(gdt=2) == 2   # fp16 gate not offered
    assert fwdn(o=None) == 1 and fwdn(y=None) == 1
    assert fwdn(o=A16 + 8) == 3
    assert lib.gla_head_norm_gate_bwd_workspace_size(0, 16, 192) == 0
    assert lib.gla_head_norm_gate_bwd(A16, A16, A16, 0, A16, 4, 1e-6, A16, A16, A16, None, 0,
                                      3, 16, 192, None) in (7, 4)  # needs a workspace


def test_conv_argument_checks(lib):
    def cf(B=1, T=8, D=16, dt=0, x=A16, w=A16, y=A16, init=None):
        return lib.gla_conv_fwd(x, dt, w, None, init, y, None, B, T, D, None)
    assert cf(D=6) == 2 and cf(dt=2) == 2
    assert cf(B=0) == 1 and cf(T=0) == 1 and cf(D=0) == 1
    assert cf(x=None) == 1 and cf(w=None) == 1 and cf(y=None) == 1
    assert cf(x=A16 + 8) == 3 and cf(init=A16 + 4) == 3
    assert lib.gla_conv_bwd_workspace_size(1, 8, 16) > 0
    assert lib.gla_conv_bwd(A16, 0, A16, None, None, A16, A16, None, A16, None, None, 0, 1, 8, 16,
                            None) == 7
    assert lib.gla_conv_decode_step(A16, A16, A16, None, A16, 0, 16, None) == 0
    assert lib.gla_conv_decode_step(A16, A16, A16, None, A16, 2, 6, None) == 2


def test_split_plan_query(lib):
    """The layout of (b, h) pairs over CTAs: a host function, no device needed."""
    def plan(B, T, H, bwd, n_sm=152):
        w, p = ctypes.c_int(), ctypes.c_int()
        rc = lib.gla_chunk_split_plan(B, T, H, bwd, n_sm, ctypes.byref(w), ctypes.byref(p))
        assert rc == 0
        return w.value, p.value
    assert lib.gla_set_split_parts(0) == 0
    # T = 2048 (16 chunks), B = 32: the forward's last wave is 56 of 152 CTAs full.  Its pairs
    # are cut in two whether the segment passes run beside the whole pairs (the default: they
    # cost only their share of the SMs) or before them: with two parts the sum pass is the only
    # extra launch.  The backward's 1536 CTAs leave 16 for an eleventh wave: its 6 pairs are cut
    # (>= 4 chunks a part) either way.
    assert plan(32, 2048, 16, 0) == (456, 2)
    try:
        assert lib.gla_set_pass_overlap(0) == 0
        assert plan(32, 2048, 16, 0) == (456, 2)
        w, p = plan(32, 2048, 16, 1)
        assert w == 506 and 2 <= p <= 4
    finally:
        assert lib.gla_set_pass_overlap(1) == 0
    w, p = plan(32, 2048, 16, 1)
    assert w == 506 and 2 <= p <= 4
    # a last wave more than half full is not worth cutting
    assert plan(24, 2048, 16, 0) == (384, 1) and plan(24, 2048, 16, 1) == (384, 1)
    # backward, three CTAs per pair: 192 = one wave + 40 CTAs -> the last 14 pairs cut
    w, p = plan(4, 8192, 16, 1)
    assert w == 50 and 2 <= p <= 4
    # a multiple of the SM count: nothing to cut; one chunk: nothing to cut
    assert plan(19, 2048, 8, 0) == (152, 1)
    assert plan(4, 100, 3, 0) == (12, 1)
    # few long sequences: every pair is cut, into at most 32 parts
    w, p = plan(2, 131072, 16, 0)
    assert w == 0 and 2 <= p <= 32
    w, p = plan(2, 131072, 16, 1)
    assert w == 0 and 2 <= p <= 32
    # the backward reading the forward's state copies sums its segment passes in one direction
    # only, so the cheaper passes let it cut the long pairs into more parts
    w2, p2 = plan(2, 131072, 16, 2)
    assert w2 == 0 and p <= p2 <= 32
    # forced: 1 never cuts, p >= 2 cuts the considered pairs into min(p, chunks) parts (the
    # pairs of the partial last wave: 56 of 512 forward, 6 of 512 backward)
    try:
        assert lib.gla_set_split_parts(1) == 0
        assert plan(32, 2048, 16, 0) == (512, 1) and plan(2, 131072, 16, 1) == (32, 1)
        assert lib.gla_set_split_parts(5) == 0
        assert plan(32, 2048, 16, 0) == (456, 5) and plan(32, 2048, 16, 1) == (506, 5)
        assert plan(1, 300, 2, 1) == (0, 3)          # 3 chunks: at most 3 parts
        assert lib.gla_set_split_parts(-1) == 1
    finally:
        lib.gla_set_split_parts(0)
    w, p = ctypes.c_int(), ctypes.c_int()
    assert lib.gla_chunk_split_plan(0, 128, 1, 0, 152, ctypes.byref(w), ctypes.byref(p)) == 1
    assert lib.gla_chunk_split_plan(1, 128, 1, 0, 0, ctypes.byref(w), ctypes.byref(p)) == 1
    assert lib.gla_chunk_split_plan(1, 128, 1, 0, 152, None, ctypes.byref(p)) == 1


def test_split_plan_invariants(lib):
    """For random shapes and SM counts: whole_pairs <= B*H; 1 <= parts <= min(32, chunks)
    (min(p, chunks) when forced); nothing cut means every pair whole; the cut pairs are those of
    the partial last wave (all pairs when one wave holds every CTA); automatic cuts keep at
    least 4 chunks per part."""
    rng = np.random.default_rng(5)
    w, p = ctypes.c_int(), ctypes.c_int()
    try:
        for trial in range(400):
            B, H = int(rng.integers(1, 65)), int(rng.integers(1, 33))
            T = int(rng.integers(1, 40000))
            n_sm = int(rng.choice([1, 7, 100, 132, 152, 160]))
            bwd = int(rng.integers(0, 3))  # 2: the backward reading saved state copies
            force = int(rng.choice([0, 0, 0, 1, 2, 5, 40]))
            assert lib.gla_set_split_parts(force) == 0
            assert lib.gla_chunk_split_plan(B, T, H, bwd, n_sm, ctypes.byref(w), ctypes.byref(p)) == 0
            whole, parts = w.value, p.value
            BH, nc, roles = B * H, -(-T // 128), 3 if bwd else 1
            assert 0 <= whole <= BH and 1 <= parts
            if parts == 1:
                assert whole == BH
                continue
            assert parts <= min(force if force >= 2 else 32, nc)
            if force == 0:
                assert nc // parts >= 4
            if force >= 2:
                assert parts == min(force, nc)
            cut = BH - whole
            if roles * BH <= n_sm:
                assert cut == BH
            else:
                rem = (roles * BH) % n_sm
                assert rem and cut == -(-rem // roles)
    finally:
        lib.gla_set_split_parts(0)


def test_binding_checks_the_gate_shape():
    """The saved gate is head-major [B,H,T]; the binding refuses any other shape before it
    touches a device (so this runs on the CPU)."""
    import torch
    B, T, H = 2, 256, 3
    q = torch.zeros(B, T, H, 96, dtype=torch.bfloat16)
    v = torch.zeros(B, T, H, 192, dtype=torch.bfloat16)
    lg, a = torch.zeros(H), torch.zeros(H, 96)
    with pytest.raises(ValueError, match=r"gate must be \[B,H,T\]"):
        gla.chunk_fwd(q, q, v, lg, a, gate=torch.zeros(B, T, H))
    with pytest.raises(ValueError, match=r"gate must be \[B,H,T\]"):
        gla.chunk_bwd(q, q, v, lg, a, v, gate=torch.zeros(B, T, H))


def test_binding_argument_lists_match_the_header():
    """Every entry point the binding declares takes as many arguments as include/gla.h gives
    it (a parameter added to one and not the other would shift every argument after it)."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = open(os.path.join(root, "include", "gla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    decls = dict(re.findall(r"GLA_API\s+[\w\s\*]+?\b(gla_\w+)\s*\(([^)]*)\)\s*;", src))
    lib = gla.load()
    checked = 0
    for name, params in decls.items():
        argtypes = getattr(lib, name).argtypes
        if argtypes is None:  # not declared by the binding (called only from C)
            continue
        n = 0 if params.strip() in ("", "void") else params.count(",") + 1
        assert len(argtypes) == n, f"{name}: header {n} parameters, binding {len(argtypes)}"
        checked += 1
    assert checked >= 15, checked


def test_header_compiles_as_plain_c(tmp_path):
    """include/gla.h is a C header (plain pointers, sizes, enums, no C++ or torch types): a C99
    translation unit that includes it and references every entry point compiles."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda_inc = "/usr/local/cuda/include"
    if not gcc or not os.path.isdir(cuda_inc):
        pytest.skip("needs gcc and the CUDA headers")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    hdr = open(os.path.join(root, "include", "gla.h")).read()
    names = sorted(set(re.findall(r"GLA_API\s+[\w\s\*]+?\b(gla_\w+)\s*\(", hdr)))
    src = tmp_path / "use_header.c"
    src.write_text('#include "gla.h"\nvoid* table[] = {\n' +
                   "".join(f"  (void*){n},\n" for n in names) + "};\nint main(void) { return 0; }\n")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror=implicit-function-declaration",
                        "-fsyntax-only", "-I", os.path.join(root, "include"), "-I", cuda_inc,
                        str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert len(names) >= 20, names


def test_slice_call_argument_checks(lib):
    def ssum(k=A16, v=A16, dt=0, ld=A16, U=A16, B=1, T=128, H=1, dk=96, dv=192):
        return lib.gla_chunk_state_sum(k, v, dt, ld, U, B, T, H, dk, dv, None)

    def asum(q=A16, dO=A16, dt=0, ld=A16, U=A16, B=1, T=128, H=1, dk=96, dv=192):
        return lib.gla_chunk_adjoint_sum(q, dO, dt, ld, U, B, T, H, dk, dv, None)

    for f in (ssum, asum):
        assert f(dk=64) == 2 and f(dv=96) == 2
        assert f(dt=1) == 2                         # fp32 inputs: no workspace for fp16 copies
        assert f(B=0) == 1 and f(T=0) == 1 and f(H=0) == 1
        assert f(U=None) == 1 and f(ld=None) == 1
        assert f(U=A16 + 4) == 3 and f(T=77, ld=A16 + 8) == 3  # any T: the next check fails
    lens = (ctypes.c_int * 3)(5, 7, 9)
    bad_lens = (ctypes.c_int * 3)(5, 0, 9)

    def link(U=A16, L=lens, n=3, r=1, rev=0, ld=A16, bnd=None, out=A16, B=1, H=1, dk=96, dv=192):
        return lib.gla_state_link(U, None if L is None else ctypes.addressof(L), n, r, rev, ld,
                                  bnd, out, B, H, dk, dv, None)

    assert link(r=3) == 1 and link(r=-1) == 1 and link(n=0, r=0) == 1
    assert link(L=bad_lens) == 1 and link(L=None) == 1 and link(out=None) == 1
    assert link(n=257, r=0) == 2 and link(dk=64) == 2 and link(B=65536, H=2) == 2
    assert link(bnd=A16 + 4) == 3 and link(U=A16 + 8) == 3


def test_sharded_binding_keeps_the_library_in_the_product_path():
    """seqshard's default ops are the library's calls (no CPU arithmetic in the product path)."""
    import inspect

    from gated_linear_attention_chunked_gb300 import seqshard
    src = inspect.getsource(seqshard)
    assert "oracle" not in src and "numpy" not in src
    ops = seqshard.KernelOps()
    for name in ("state_sum", "adjoint_sum", "link", "fwd", "bwd"):
        assert callable(getattr(ops, name))
