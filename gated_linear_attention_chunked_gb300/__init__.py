"""GB300 (sm_103a) Simple GLA mixer: Python binding of libgla.

Argument marshalling only: every step of the method runs in the CUDA kernels behind the
C ABI in include/gla.h.  PyTorch supplies device memory and the current CUDA stream.
There is no CPU fallback: if libgla.so is missing or the tensors are not on a CUDA device,
the calls raise.

Functions (same names as the C ABI, without the ``gla_`` prefix):
  decay_schedule(H, t_min, t_max)                     -> float32 [H] (host) log-decays
  chunk_fwd(q, k, v, log_decay, aug_balance, ...)     -> (o, final_state)
  chunk_bwd(q, k, v, log_decay, aug_balance, dO, ...) -> (dq, dk, dv, d_aug, d_init_state)
  decode_step(state, q, k, v, log_decay, aug_balance) -> o  (state updated in place)
  chunk_state_sum, chunk_adjoint_sum, state_link     (a sequence cut into slices across ranks;
                                                      seqshard.py runs the exchange)
  get_device_error(), set_wait_timeout_ns(ns), status_string(code)
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

GLA_BF16, GLA_FP32, GLA_FP16 = 0, 1, 2
STATUS = {0: "GLA_OK", 1: "GLA_ERR_INVALID_ARG", 2: "GLA_ERR_UNSUPPORTED",
          3: "GLA_ERR_ALIGNMENT", 4: "GLA_ERR_CUDA", 5: "GLA_ERR_TIMEOUT", 6: "GLA_ERR_RANGE",
          7: "GLA_ERR_WORKSPACE", 8: "GLA_ERR_LAYOUT"}
DK, DV, CHUNK = 96, 192, 128

_lib = None
_lock = threading.Lock()
_P = ctypes.c_void_p
_I = ctypes.c_int
_S = ctypes.c_size_t


class GlaError(RuntimeError):
    def __init__(self, call: str, code: int):
        self.code = code
        super().__init__(f"{call}: {STATUS.get(code, code)} ({status_string(code)})")


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libgla.so (built by ``_build.build()`` / ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or lib_path()
            if not os.path.exists(p):
                raise RuntimeError(f"libgla.so not built ({p}); run __graft_entry__.build()")
            lib = ctypes.CDLL(p)
            lib.gla_status_string.argtypes = [_I]
            lib.gla_status_string.restype = ctypes.c_char_p
            lib.gla_get_device_error.argtypes = []
            lib.gla_get_device_error.restype = _I
            lib.gla_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
            lib.gla_set_wait_timeout_ns.restype = _I
            lib.gla_decay_schedule.argtypes = [_I, ctypes.c_double, ctypes.c_double, _P]
            lib.gla_decay_schedule.restype = _I
            lib.gla_chunk_fwd_workspace_size.argtypes = [_I] * 6
            lib.gla_chunk_fwd_workspace_size.restype = _S
            lib.gla_chunk_fwd.argtypes = ([_P, _P, _P, _I] + [_P] * 6 + [_P, _S, _P, _S] +
                                          [_I] * 5 + [_P])
            lib.gla_chunk_fwd.restype = _I
            lib.gla_chunk_bwd_workspace_size.argtypes = [_I] * 6
            lib.gla_chunk_bwd_workspace_size.restype = _S
            lib.gla_chunk_bwd.argtypes = ([_P] * 3 + [_I] + [_P] * 7 + [_S] + [_P] * 6 + [_S] +
                                          [_I] * 5 + [_P])
            lib.gla_chunk_saved_states_size.argtypes = [_I] * 3
            lib.gla_chunk_saved_states_size.restype = _S
            lib.gla_chunk_bwd.restype = _I
            lib.gla_decode_step.argtypes = [_P] * 7 + [_I] * 5 + [_P]
            lib.gla_wait_probe.argtypes = [_P]
            lib.gla_wait_probe.restype = _I
            lib.gla_decode_step_paged.argtypes = [_P, _P] + [_I] * 4 + [_P] * 6 + [_I] * 4 + [_P]
            lib.gla_decode_step_paged.restype = _I
            lib.gla_chunk_fwd_paged.argtypes = ([_P] * 3 + [_I] + [_P] * 4 + [_I] * 4 + [_P] * 2 +
                                                [_S] + [_I] * 5 + [_P])
            lib.gla_chunk_fwd_paged.restype = _I
            _L = ctypes.c_longlong
            _F = ctypes.c_float
            lib.gla_head_norm_gate_fwd.argtypes = [_P, _P, _I, _P, _I, _F, _P, _P, _L, _I, _I, _P]
            lib.gla_head_norm_gate_fwd.restype = _I
            lib.gla_head_norm_gate_bwd_workspace_size.argtypes = [_L, _I, _I]
            lib.gla_head_norm_gate_bwd_workspace_size.restype = _S
            lib.gla_head_norm_gate_bwd.argtypes = ([_P] * 3 + [_I, _P, _I, _F] + [_P] * 4 + [_S] +
                                                   [_L, _I, _I, _P])
            lib.gla_head_norm_gate_bwd.restype = _I
            lib.gla_chunk_fwd_gated.argtypes = ([_P] * 3 + [_I] + [_P] * 5 + [_I, _F] + [_P] * 5 +
                                                [_S] + [_I] * 5 + [_P])
            lib.gla_chunk_fwd_gated.restype = _I
            lib.gla_conv_fwd.argtypes = [_P, _I] + [_P] * 5 + [_I] * 3 + [_P]
            lib.gla_conv_fwd.restype = _I
            lib.gla_conv_bwd_workspace_size.argtypes = [_I] * 3
            lib.gla_conv_bwd_workspace_size.restype = _S
            lib.gla_conv_bwd.argtypes = [_P, _I] + [_P] * 9 + [_S] + [_I] * 3 + [_P]
            lib.gla_conv_bwd.restype = _I
            lib.gla_conv_decode_step.argtypes = [_P] * 5 + [_L, _I, _P]
            lib.gla_conv_decode_step.restype = _I
            lib.gla_decode_step.restype = _I
            lib.gla_chunk_split_plan.argtypes = [_I] * 5 + [_P, _P]
            lib.gla_chunk_split_plan.restype = _I
            lib.gla_set_split_parts.argtypes = [_I]
            lib.gla_set_split_parts.restype = _I
            lib.gla_set_pass_overlap.argtypes = [_I]
            lib.gla_set_pass_overlap.restype = _I
            lib.gla_set_stall_step.argtypes = [_I]
            lib.gla_set_stall_step.restype = _I
            lib.gla_chunk_state_sum.argtypes = [_P, _P, _I, _P, _P] + [_I] * 5 + [_P]
            lib.gla_chunk_state_sum.restype = _I
            lib.gla_chunk_adjoint_sum.argtypes = [_P, _P, _I, _P, _P] + [_I] * 5 + [_P]
            lib.gla_chunk_adjoint_sum.restype = _I
            lib.gla_state_link.argtypes = [_P, _P, _I, _I, _I, _P, _P, _P] + [_I] * 4 + [_P]
            lib.gla_state_link.restype = _I
            lib.gla_chunk_bwd_noalloc.argtypes = [_P] * 3 + [_I] + [_P] * 11 + [_I] * 5 + [_P]
            lib.gla_chunk_bwd_noalloc.restype = _I
            if path is not None:
                return lib
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().gla_status_string(int(code)).decode()


def _check(call: str, rc: int):
    if rc != 0:
        raise GlaError(call, rc)


# --------------------------------------------------------------------------- marshalling
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    m = {torch.bfloat16: GLA_BF16, torch.float32: GLA_FP32, torch.float16: GLA_FP16}
    if t.dtype not in m:
        raise TypeError(f"unsupported input dtype {t.dtype}")
    return m[t.dtype]


def _dev(t, name, dtype=None):
    """Pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def decay_schedule(H: int, t_min: float = 1.0, t_max: float = 2048.0):
    """Host float32 tensor [H] of log-decays gamma_h = -ln2 / T_h (gla_decay_schedule)."""
    torch = _torch()
    out = torch.empty(H, dtype=torch.float32)
    _check("gla_decay_schedule", load().gla_decay_schedule(H, t_min, t_max, out.data_ptr()))
    return out


def chunk_fwd_workspace_size(B, T, H, in_dtype) -> int:
    return load().gla_chunk_fwd_workspace_size(B, T, H, DK, DV, in_dtype)


def chunk_bwd_workspace_size(B, T, H, in_dtype) -> int:
    return load().gla_chunk_bwd_workspace_size(B, T, H, DK, DV, in_dtype)


def _workspace(nbytes, device, workspace):
    torch = _torch()
    if nbytes == 0:
        return None
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def chunk_saved_states_size(B, T, H) -> int:
    """Bytes of the state copies a forward saves for the backward (gla_chunk_saved_states_size)."""
    return load().gla_chunk_saved_states_size(B, T, H)


def _saved(t, nbytes, name):
    if t is None:
        return None, 0
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name} holds {have} bytes, {nbytes} needed")
    return _dev(t, name), have


def chunk_fwd(q, k, v, log_decay, aug_balance, init_state=None, *, want_final_state=True,
              out=None, final_state=None, gate=None, saved_states=None, workspace=None,
              stream=None):
    """Chunked forward (gla_chunk_fwd).  q,k [B,T,H,96], v [B,T,H,192] (bf16/fp16/fp32);
    log_decay [H], aug_balance [H,96], init_state [B,H,96,192] fp32 (optional); gate: an
    fp32 [B,H,T] tensor that receives sigmoid(q.(a*k)) for chunk_bwd (optional);
    saved_states: a uint8 device tensor of chunk_saved_states_size(B, T, H) bytes that receives
    the chunks' state copies for chunk_bwd (optional).
    Returns (o fp32 [B,T,H,192], final_state fp32 [B,H,96,192] or None)."""
    torch = _torch()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    code = _dtype_code(q)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=torch.float32, device=q.device)
    if final_state is None and want_final_state:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    if gate is not None and tuple(gate.shape) != (B, H, T):
        raise ValueError(f"gate must be [B,H,T] = {(B, H, T)}, got {tuple(gate.shape)}")
    ws = _workspace(load().gla_chunk_fwd_workspace_size(B, T, H, dk, dv, code), q.device, workspace)
    sp, sb = _saved(saved_states, chunk_saved_states_size(B, T, H), "saved_states")
    rc = load().gla_chunk_fwd(
        _dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype), code,
        _dev(log_decay, "log_decay", torch.float32), _dev(aug_balance, "aug_balance", torch.float32),
        _dev(init_state, "init_state", torch.float32), _dev(out, "o", torch.float32),
        _dev(final_state, "final_state", torch.float32), _dev(gate, "gate", torch.float32),
        sp, sb, _dev(ws, "workspace"), 0 if ws is None else ws.numel() * ws.element_size(), B, T,
        H, dk, dv, _stream(stream))
    _check("gla_chunk_fwd", rc)
    return out, final_state


def chunk_fwd_gated(q, k, v, log_decay, aug_balance, g, norm_weight, n_tiers, eps=1e-6,
                    init_state=None, *, want_o=False, want_rstd=True, want_final_state=True,
                    workspace=None, stream=None):
    """Chunked forward with the output epilogue fused in (gla_chunk_fwd_gated): g [B,T,H,192]
    bf16, norm_weight [n_tiers,192].  Returns (y, rstd or None, o or None, final or None)."""
    torch = _torch()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    code = _dtype_code(q)
    f = torch.float32
    y = torch.empty((B, T, H, dv), dtype=f, device=q.device)
    rstd = torch.empty((B, T, H), dtype=f, device=q.device) if want_rstd else None
    o = torch.empty((B, T, H, dv), dtype=f, device=q.device) if want_o else None
    fin = torch.empty((B, H, dk, dv), dtype=f, device=q.device) if want_final_state else None
    ws = _workspace(load().gla_chunk_fwd_workspace_size(B, T, H, dk, dv, code), q.device, workspace)
    rc = load().gla_chunk_fwd_gated(
        _dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype), code,
        _dev(log_decay, "log_decay", f), _dev(aug_balance, "aug_balance", f),
        _dev(init_state, "init_state", f), _dev(g, "g", torch.bfloat16),
        _dev(norm_weight, "norm_weight", f), n_tiers, eps, _dev(y, "y", f), _dev(rstd, "rstd", f),
        _dev(o, "o", f), _dev(fin, "final_state", f), _dev(ws, "workspace"),
        0 if ws is None else ws.numel() * ws.element_size(), B, T, H, dk, dv, _stream(stream))
    _check("gla_chunk_fwd_gated", rc)
    return y, rstd, o, fin


def chunk_bwd(q, k, v, log_decay, aug_balance, dO, init_state=None, d_final_state=None, *,
              gate=None, saved_states=None, want_d_init_state=True, workspace=None, stream=None):
    """Chunked backward (gla_chunk_bwd).  gate: the fp32 [B,H,T] sigmoid(q.(a*k)) that
    chunk_fwd saved (optional; recomputed if None); saved_states: the state copies chunk_fwd
    saved for the same inputs (optional).  Returns (dq, dk, dv, d_aug, d_init_state), fp32."""
    torch = _torch()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    code = _dtype_code(q)
    f32 = dict(dtype=torch.float32, device=q.device)
    dq = torch.empty((B, T, H, dk), **f32)
    dk_ = torch.empty((B, T, H, dk), **f32)
    dv_ = torch.empty((B, T, H, dv), **f32)
    d_aug = torch.empty((H, dk), **f32)
    dinit = torch.empty((B, H, dk, dv), **f32) if want_d_init_state else None
    if gate is not None and tuple(gate.shape) != (B, H, T):
        raise ValueError(f"gate must be [B,H,T] = {(B, H, T)}, got {tuple(gate.shape)}")
    ws = _workspace(load().gla_chunk_bwd_workspace_size(B, T, H, dk, dv, code), q.device, workspace)
    sp, sb = _saved(saved_states, chunk_saved_states_size(B, T, H), "saved_states")
    rc = load().gla_chunk_bwd(
        _dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype), code,
        _dev(log_decay, "log_decay", torch.float32), _dev(aug_balance, "aug_balance", torch.float32),
        _dev(init_state, "init_state", torch.float32), _dev(dO, "dO", q.dtype),
        _dev(d_final_state, "d_final_state", torch.float32), _dev(gate, "gate", torch.float32),
        sp, sb, _dev(dq, "dq"), _dev(dk_, "dk"),
        _dev(dv_, "dv"), _dev(d_aug, "d_aug"), _dev(dinit, "d_init_state"), _dev(ws, "workspace"),
        0 if ws is None else ws.numel() * ws.element_size(), B, T, H, dk, dv, _stream(stream))
    _check("gla_chunk_bwd", rc)
    return dq, dk_, dv_, d_aug, dinit


def decode_step(state, q, k, v, log_decay, aug_balance, *, out=None, stream=None):
    """One decode token (gla_decode_step).  state [N,L,H,96,192] fp32 is updated in place;
    q,k [N,L,H,96], v [N,L,H,192] fp32; aug_balance [L,H,96].  Returns o [N,L,H,192]."""
    torch = _torch()
    N, L, H, dk, dv = state.shape
    if out is None:
        out = torch.empty((N, L, H, dv), dtype=torch.float32, device=state.device)
    f = torch.float32
    rc = load().gla_decode_step(
        _dev(state, "state", f), _dev(q, "q", f), _dev(k, "k", f), _dev(v, "v", f),
        _dev(log_decay, "log_decay", f), _dev(aug_balance, "aug_balance", f), _dev(out, "o", f),
        N, L, H, dk, dv, _stream(stream))
    _check("gla_decode_step", rc)
    return out


def _pages(page, n):
    torch = _torch()
    if page.dtype != torch.int32 or page.dim() != 1 or page.numel() != n:
        raise ValueError(f"page must be a 1-D int32 tensor of {n} entries")
    return _dev(page, "page")


def decode_step_paged(pool, page, q, k, v, log_decay, aug_balance, *, layer0=0, out=None,
                      stream=None):
    """Decode step over a state pool (gla_decode_step_paged).  pool [P, pool_layers, H, 96, 192]
    fp32 is updated in place for pages page[n] (int32 [n_active]) and layers layer0..layer0+L-1;
    q,k [n_active,L,H,96], v [n_active,L,H,192]; aug_balance [L,H,96].  Returns o."""
    torch = _torch()
    P, PL, H, dk, dv = pool.shape
    n, L = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty((n, L, H, dv), dtype=torch.float32, device=pool.device)
    f = torch.float32
    rc = load().gla_decode_step_paged(
        _dev(pool, "pool", f), _pages(page, n), n, P, PL, layer0, _dev(q, "q", f),
        _dev(k, "k", f), _dev(v, "v", f), _dev(log_decay, "log_decay", f),
        _dev(aug_balance, "aug_balance", f), _dev(out, "o", f), L, H, dk, dv, _stream(stream))
    _check("gla_decode_step_paged", rc)
    return out


def chunk_fwd_paged(q, k, v, log_decay, aug_balance, pool, page, layer, *, init_from_pool=True,
                    out=None, workspace=None, stream=None):
    """Chunked prefill into a state pool (gla_chunk_fwd_paged): sequence b starts from layer
    `layer` of page[b] (or zero) and its final state is written back there.  Returns o."""
    torch = _torch()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    P, PL = pool.shape[0], pool.shape[1]
    code = _dtype_code(q)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=torch.float32, device=q.device)
    ws = _workspace(load().gla_chunk_fwd_workspace_size(B, T, H, dk, dv, code), q.device, workspace)
    f = torch.float32
    rc = load().gla_chunk_fwd_paged(
        _dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype), code,
        _dev(log_decay, "log_decay", f), _dev(aug_balance, "aug_balance", f),
        _dev(pool, "pool", f), _pages(page, B), P, PL, layer, 1 if init_from_pool else 0,
        _dev(out, "o", f), _dev(ws, "workspace"), 0 if ws is None else ws.numel() * ws.element_size(),
        B, T, H, dk, dv, _stream(stream))
    _check("gla_chunk_fwd_paged", rc)
    return out


def _gate_code(g):
    torch = _torch()
    m = {torch.bfloat16: GLA_BF16, torch.float32: GLA_FP32}
    if g.dtype not in m:
        raise TypeError(f"g must be bf16 or fp32, got {g.dtype}")
    return m[g.dtype]


def head_norm_gate_bwd_workspace_size(n_tokens, H) -> int:
    return load().gla_head_norm_gate_bwd_workspace_size(n_tokens, H, DV)


def head_norm_gate(o, g, weight, n_tiers, eps=1e-6, *, want_rstd=False, out=None, stream=None):
    """Head RMSNorm per decay tier, then the SiLU(g) gate (gla_head_norm_gate_fwd).
    o [..., H, 192] fp32, g the same shape (bf16 or fp32), weight [n_tiers, 192] fp32.
    Returns (y fp32, rstd fp32 [..., H] or None)."""
    torch = _torch()
    H, dv = o.shape[-2], o.shape[-1]
    n_tok = o.numel() // (H * dv)
    if g.shape != o.shape:
        raise ValueError("g must have the shape of o")
    if out is None:
        out = torch.empty_like(o)
    rstd = torch.empty(o.shape[:-1], dtype=torch.float32, device=o.device) if want_rstd else None
    f = torch.float32
    rc = load().gla_head_norm_gate_fwd(
        _dev(o, "o", f), _dev(g, "g"), _gate_code(g), _dev(weight, "weight", f), n_tiers, eps,
        _dev(out, "y", f), _dev(rstd, "rstd", f), n_tok, H, dv, _stream(stream))
    _check("gla_head_norm_gate_fwd", rc)
    return out, rstd


def head_norm_gate_bwd(dy, o, g, weight, n_tiers, eps=1e-6, *, workspace=None, stream=None):
    """Gradient of the output epilogue (gla_head_norm_gate_bwd): returns (d_o, dg, d_weight),
    fp32."""
    torch = _torch()
    H, dv = o.shape[-2], o.shape[-1]
    n_tok = o.numel() // (H * dv)
    d_o = torch.empty_like(o)
    dg = torch.empty(o.shape, dtype=torch.float32, device=o.device)
    d_w = torch.empty((n_tiers, dv), dtype=torch.float32, device=o.device)
    ws = _workspace(load().gla_head_norm_gate_bwd_workspace_size(n_tok, H, dv), o.device,
                    workspace)
    f = torch.float32
    rc = load().gla_head_norm_gate_bwd(
        _dev(dy, "dy", f), _dev(o, "o", f), _dev(g, "g"), _gate_code(g), _dev(weight, "weight", f),
        n_tiers, eps, _dev(d_o, "d_o", f), _dev(dg, "dg", f), _dev(d_w, "d_weight", f),
        _dev(ws, "workspace"), 0 if ws is None else ws.numel() * ws.element_size(), n_tok, H, dv,
        _stream(stream))
    _check("gla_head_norm_gate_bwd", rc)
    return d_o, dg, d_w


def _x_code(x):
    torch = _torch()
    m = {torch.bfloat16: GLA_BF16, torch.float32: GLA_FP32}
    if x.dtype not in m:
        raise TypeError(f"x must be bf16 or fp32, got {x.dtype}")
    return m[x.dtype]


def conv_fwd(x, weight, bias=None, init_state=None, *, want_final_state=True, out=None,
             stream=None):
    """Causal depth-wise Conv1d (width 4) + SiLU (gla_conv_fwd).  x [B,T,D] bf16/fp32,
    weight [D,4], bias [D], init_state [B,3,D].  Returns (y fp32, final_state or None)."""
    torch = _torch()
    B, T, D = x.shape
    f = torch.float32
    y = out if out is not None else torch.empty((B, T, D), dtype=f, device=x.device)
    fin = torch.empty((B, 3, D), dtype=f, device=x.device) if want_final_state else None
    rc = load().gla_conv_fwd(_dev(x, "x"), _x_code(x), _dev(weight, "weight", f),
                             _dev(bias, "bias", f), _dev(init_state, "init_state", f),
                             _dev(y, "y", f), _dev(fin, "final_state", f), B, T, D, _stream(stream))
    _check("gla_conv_fwd", rc)
    return y, fin


def conv_bwd(x, weight, dy, bias=None, init_state=None, *, want_d_init_state=True,
             workspace=None, stream=None):
    """Gradient of conv_fwd (gla_conv_bwd): returns (dx, d_init_state or None, d_weight,
    d_bias), fp32."""
    torch = _torch()
    B, T, D = x.shape
    f = torch.float32
    dx = torch.empty((B, T, D), dtype=f, device=x.device)
    dinit = torch.empty((B, 3, D), dtype=f, device=x.device) if want_d_init_state else None
    dw = torch.empty((D, 4), dtype=f, device=x.device)
    db = torch.empty((D,), dtype=f, device=x.device)
    ws = _workspace(load().gla_conv_bwd_workspace_size(B, T, D), x.device, workspace)
    rc = load().gla_conv_bwd(_dev(x, "x"), _x_code(x), _dev(weight, "weight", f),
                             _dev(bias, "bias", f), _dev(init_state, "init_state", f),
                             _dev(dy, "dy", f), _dev(dx, "dx", f), _dev(dinit, "d_init_state", f),
                             _dev(dw, "d_weight", f), _dev(db, "d_bias", f), _dev(ws, "workspace"),
                             ws.numel() * ws.element_size(), B, T, D, _stream(stream))
    _check("gla_conv_bwd", rc)
    return dx, dinit, dw, db


def conv_decode_step(state, x, weight, bias=None, *, out=None, stream=None):
    """One decode token of the conv (gla_conv_decode_step): state [..., 3, D] fp32 updated in
    place, x [..., D] fp32.  Returns y [..., D]."""
    torch = _torch()
    D = x.shape[-1]
    n = x.numel() // D
    f = torch.float32
    y = out if out is not None else torch.empty_like(x)
    rc = load().gla_conv_decode_step(_dev(state, "state", f), _dev(x, "x", f),
                                     _dev(weight, "weight", f), _dev(bias, "bias", f),
                                     _dev(y, "y", f), n, D, _stream(stream))
    _check("gla_conv_decode_step", rc)
    return y


def chunk_state_sum(k, v, log_decay, *, out=None, stream=None):
    """gla_chunk_state_sum: U[b,h] = sum_t lambda_h^(T-1-t) k_t v_t^T over the T tokens given
    (k [B,T,H,96], v [B,T,H,192], bf16 or fp16).  Returns U fp32 [B,H,96,192]."""
    torch = _torch()
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    f = torch.float32
    if out is None:
        out = torch.empty((B, H, dk, dv), dtype=f, device=k.device)
    rc = load().gla_chunk_state_sum(_dev(k, "k"), _dev(v, "v", k.dtype), _dtype_code(k),
                                    _dev(log_decay, "log_decay", f), _dev(out, "U", f), B, T, H,
                                    dk, dv, _stream(stream))
    _check("gla_chunk_state_sum", rc)
    return out


def chunk_adjoint_sum(q, dO, log_decay, *, out=None, stream=None):
    """gla_chunk_adjoint_sum: U'[b,h] = sum_t lambda_h^(t+1) q_t dO_t^T (q [B,T,H,96], dO
    [B,T,H,192], bf16 or fp16).  Returns U' fp32 [B,H,96,192]."""
    torch = _torch()
    B, T, H, dk = q.shape
    dv = dO.shape[-1]
    f = torch.float32
    if out is None:
        out = torch.empty((B, H, dk, dv), dtype=f, device=q.device)
    rc = load().gla_chunk_adjoint_sum(_dev(q, "q"), _dev(dO, "dO", q.dtype), _dtype_code(q),
                                      _dev(log_decay, "log_decay", f), _dev(out, "U", f), B, T,
                                      H, dk, dv, _stream(stream))
    _check("gla_chunk_adjoint_sum", rc)
    return out


def state_link(U_all, lens, slice_index, log_decay, boundary=None, *, reverse=False, out=None,
               stream=None):
    """gla_state_link: the state entering slice `slice_index` (reverse=False; boundary = the
    initial state) or the adjoint of the state leaving it (reverse=True; boundary =
    d_final_state) of a sequence cut into slices of `lens` tokens, from every slice's sums
    U_all fp32 [n_slices,B,H,96,192].  Returns fp32 [B,H,96,192]."""
    torch = _torch()
    n, B, H, dk, dv = U_all.shape
    lens = [int(x) for x in lens]
    if len(lens) != n:
        raise ValueError(f"lens must have {n} entries")
    f = torch.float32
    if out is None:
        out = torch.empty((B, H, dk, dv), dtype=f, device=U_all.device)
    host_lens = (ctypes.c_int * n)(*lens)
    rc = load().gla_state_link(_dev(U_all, "U_all", f), ctypes.addressof(host_lens), n,
                               int(slice_index), 1 if reverse else 0,
                               _dev(log_decay, "log_decay", f), _dev(boundary, "boundary", f),
                               _dev(out, "out", f), B, H, dk, dv, _stream(stream))
    _check("gla_state_link", rc)
    return out


def get_device_error() -> int:
    """Read and clear the device error word (synchronises the device).  0 = none."""
    return load().gla_get_device_error()


def wait_probe(stream=None) -> None:
    """Launch the failure-path diagnostic (gla_wait_probe): a wait that nothing completes,
    given up after the configured limit; get_device_error() then reads GLA_ERR_TIMEOUT."""
    _check("gla_wait_probe", load().gla_wait_probe(_stream(stream)))


def set_wait_timeout_ns(ns: int) -> None:
    _check("gla_set_wait_timeout_ns", load().gla_set_wait_timeout_ns(int(ns)))


def set_stall_step(step: int) -> None:
    """gla_set_stall_step: the chunk kernels' MMA issuer stalls at chunk step `step` (its
    bounded wait then gives up: the give-up path's diagnostic); -1 turns it off."""
    _check("gla_set_stall_step", load().gla_set_stall_step(int(step)))


def split_plan(B: int, T: int, H: int, backward: int, n_sm: int) -> tuple[int, int]:
    """(whole_pairs, parts) of gla_chunk_split_plan: pairs whole_pairs.. are cut into parts.
    backward: 0 (False) the forward, 1 (True) the backward, 2 the backward reading the
    forward's saved state copies."""
    w, p = ctypes.c_int(), ctypes.c_int()
    _check("gla_chunk_split_plan", load().gla_chunk_split_plan(
        int(B), int(T), int(H), int(backward), int(n_sm), ctypes.byref(w), ctypes.byref(p)))
    return w.value, p.value


def set_split_parts(parts: int) -> None:
    """gla_set_split_parts: 0 automatic, 1 never cut, p >= 2 cut into p parts."""
    _check("gla_set_split_parts", load().gla_set_split_parts(int(parts)))


def set_pass_overlap(on: bool) -> None:
    """gla_set_pass_overlap: segment passes beside the whole pairs (True, the default) or
    before them on the caller's stream (False)."""
    _check("gla_set_pass_overlap", load().gla_set_pass_overlap(1 if on else 0))
