"""fp64 CPU oracle for the Simple GLA mixer -- TEST INFRASTRUCTURE ONLY.

The plain, slow, obviously-correct reference that the CUDA path is checked
against.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg may import it; the product package never does, and it shares no
code with the CUDA library.

The mixer's arithmetic lives in ``gla_oracle.c`` (token-by-token recurrence,
hand-derived backward, decode step, decay schedule); this module compiles it with
gcc, loads it with ctypes and converts numpy arrays to contiguous float64.  The
state-pool decode is that decode step on gathered pages, and the output epilogue
(Head RMSNorm per decay tier, SiLU gate) is written out below in fp64 numpy.

Source: "Beyond the KV cache: Training and serving i14's Laplace 3B linear
attention model on AWS Trainium2 with native PyTorch", section "i14 and the
Laplace 3B architecture" ("GLA mixer", "Decay schedule", "Decay schedule's
reach") and section "Challenge 3" (backward through the sequential updates).

Pins (tests/test_oracle_*.py): brute-force closed form, central finite
differences, the printed decay values, the a=0 half value skip, the lambda=1
reduction to causal linear attention, state-carry and init-zero invariants,
decode/forward consistency and an independent chunked restatement; the slice sums and
their link (a sequence cut into slices) against the forward's state and the backward's
adjoint at every slice boundary; the gate
(the activation the forward saves) against the forward's own first-token value
skip and the a=0 half value.  Every function here is pinned; none is "parity
unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_L = ctypes.c_long


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle into a shared library with gcc (IEEE fp64, no fast-math)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        os.makedirs(os.path.dirname(out), exist_ok=True)
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", src, "-o", tmp, "-lm"])
        os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` selects another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    lib.oracle_decay_schedule.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double, _D]
    lib.oracle_decay_schedule.restype = None
    lib.oracle_fwd.argtypes = [_D] * 8 + [_L] * 5 + [ctypes.c_int]
    lib.oracle_fwd.restype = ctypes.c_int
    lib.oracle_bwd.argtypes = [_D] * 13 + [_L] * 5 + [ctypes.c_int]
    lib.oracle_bwd.restype = ctypes.c_int
    lib.oracle_decode_step.argtypes = [_D] * 7 + [_L] * 5 + [ctypes.c_int]
    lib.oracle_decode_step.restype = ctypes.c_int
    return lib


def _c(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _p(x):
    return None if x is None else x.ctypes.data_as(_D)


def decay_schedule(H: int, t_min: float = 1.0, t_max: float = 2048.0, lib=None) -> np.ndarray:
    """gamma_h = ln(lambda_h), half-lives geometric from t_min to t_max (float64 [H])."""
    lib = lib or load()
    g = np.empty(H, np.float64)
    lib.oracle_decay_schedule(int(H), float(t_min), float(t_max), _p(g))
    return g


def fwd(q, k, v, gamma, a, init_state=None, nthreads: int = 0, lib=None):
    """Token-by-token forward.  q,k [B,T,H,dk]; v [B,T,H,dv]; returns (o, final_state)."""
    lib = lib or load()
    q, k, v, gamma, a = map(_c, (q, k, v, gamma, a))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    init = None if init_state is None else _c(init_state)
    o = np.empty((B, T, H, dv), np.float64)
    fin = np.empty((B, H, dk, dv), np.float64)
    rc = lib.oracle_fwd(_p(q), _p(k), _p(v), _p(gamma), _p(a), _p(init), _p(o), _p(fin),
                        B, T, H, dk, dv, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_fwd: bad sizes")
    return o, fin


def gate(q, k, a):
    """The self-augmentation gate sigmoid(z_t), z_t = sum_c a_hc q_tc k_tc ("GLA mixer":
    the value skip weighted by the sigmoid of q against the balanced k), in fp64 numpy.
    q, k [B,T,H,dk]; a [H,dk]; returns [B,T,H] -- what the forward saves for the backward."""
    q, k, a = (np.asarray(x, np.float64) for x in (q, k, a))
    z = np.einsum("bthc,hc,bthc->bth", q, a, k)
    return 1.0 / (1.0 + np.exp(-z))


def bwd(q, k, v, gamma, a, dO, init_state=None, d_final_state=None, nthreads: int = 0, lib=None):
    """Hand-derived backward.  Returns dict dq, dk, dv, d_a [H,dk], d_init_state [B,H,dk,dv]."""
    lib = lib or load()
    q, k, v, gamma, a, dO = map(_c, (q, k, v, gamma, a, dO))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    init = None if init_state is None else _c(init_state)
    dfin = None if d_final_state is None else _c(d_final_state)
    out = dict(dq=np.empty_like(q), dk=np.empty_like(k), dv=np.empty_like(v),
               d_a=np.empty((H, dk), np.float64), d_init_state=np.empty((B, H, dk, dv), np.float64))
    rc = lib.oracle_bwd(_p(q), _p(k), _p(v), _p(gamma), _p(a), _p(init), _p(dO), _p(dfin),
                        _p(out["dq"]), _p(out["dk"]), _p(out["dv"]), _p(out["d_a"]),
                        _p(out["d_init_state"]), B, T, H, dk, dv, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_bwd: bad sizes")
    return out


# --------------------------------------------------------------------------- slices of a sequence
# A long sequence cut into consecutive slices (long-context prefill across ranks): the state
# recurrence S_t = lambda S_{t-1} + k_t v_t^T ("GLA mixer") and its adjoint are linear, so a
# slice acts on the state entering it through lambda^len and one summed term.  Each function
# is the definition written out with the token recurrence above (section "Challenge 1": the
# state carried across chunks; section "Challenge 3": the backward through the updates).

def slice_state_sum(k, v, gamma, lib=None):
    """U[b,h] = sum_t lambda_h^(T-1-t) k_t v_t^T: the state the recurrence reaches from a zero
    state over these tokens (the forward's final state with q = 0, a = 0).  [B,H,dk,dv]."""
    k = np.asarray(k, np.float64)
    z = np.zeros_like(k)
    return fwd(z, k, v, gamma, np.zeros(k.shape[2:]), lib=lib)[1]


def slice_adjoint_sum(q, dO, gamma, lib=None):
    """U'[b,h] = sum_t lambda_h^(t+1) q_t dO_t^T: the adjoint of the state entering these
    tokens when nothing flows in from after them (the backward's d_init_state with a zero
    d_final_state; k and v do not enter it).  [B,H,dk,dv]."""
    q, dO = np.asarray(q, np.float64), np.asarray(dO, np.float64)
    return bwd(q, np.zeros_like(q), np.zeros_like(dO), gamma, np.zeros(q.shape[2:]), dO,
               lib=lib)["d_init_state"]


def state_link(U_all, lens, rank, gamma, boundary=None, reverse=False):
    """The state entering slice `rank` (forward: S_0 = boundary, S_{j+1} = lambda^len_j S_j +
    U_j) or the adjoint of the state leaving it (reverse: A_{n-1} = boundary, A_{j-1} =
    lambda^len_j A_j + U'_j), slices of `lens` tokens, U_all [n,B,H,dk,dv]."""
    U = np.asarray(U_all, np.float64)
    lam = np.exp(np.asarray(gamma, np.float64))[None, :, None, None]  # per head
    s = np.zeros(U.shape[1:]) if boundary is None else np.array(boundary, np.float64)
    order = range(len(lens) - 1, rank, -1) if reverse else range(rank)
    for j in order:
        s = lam ** int(lens[j]) * s + U[j]
    return s


def decode_step(state, q, k, v, gamma, a, nthreads: int = 0, lib=None):
    """One decode token.  state [N,L,H,dk,dv]; q,k [N,L,H,dk]; v [N,L,H,dv]; a [L,H,dk].
    Returns (o [N,L,H,dv], new_state); the input array is not modified."""
    lib = lib or load()
    st = np.array(state, dtype=np.float64, order="C", copy=True)
    q, k, v, gamma, a = map(_c, (q, k, v, gamma, a))
    N, L, H, dk, dv = st.shape
    o = np.empty((N, L, H, dv), np.float64)
    rc = lib.oracle_decode_step(_p(st), _p(q), _p(k), _p(v), _p(gamma), _p(a), _p(o),
                                N, L, H, dk, dv, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_decode_step: bad sizes")
    return o, st


def decode_step_paged(pool, page, layer0, q, k, v, gamma, a, nthreads: int = 0, lib=None):
    """Decode step over a state pool with one page per sequence (the serving pool of section
    "Inference optimization on Trainium2").  pool [P, pool_layers, H, dk, dv]; active sequence
    n updates the states of page[n], layers layer0 .. layer0+L-1, and every other state is
    left as it is.  It is decode_step on the gathered states, scattered back.
    Returns (o [n_active, L, H, dv], new_pool); the input array is not modified."""
    page = np.asarray(page, dtype=np.int64)
    L = np.asarray(q).shape[1]
    if len(set(page.tolist())) != len(page):
        raise ValueError("pages of one call must be distinct")
    new = np.array(pool, dtype=np.float64, order="C", copy=True)
    o, st = decode_step(new[page, layer0:layer0 + L], q, k, v, gamma, a, nthreads, lib)
    new[page, layer0:layer0 + L] = st
    return o, new


# --------------------------------------------------------------------------- output epilogue
# Head RMSNorm shared within each decay tier, then the SiLU(g) gate (section "i14 and the
# Laplace 3B architecture", "GLA mixer" and "Decay schedule's reach").  Plain fp64 numpy, the
# definition written out: tier(h) = h // (H // n_tiers).

def _tiers(H, n_tiers):
    if n_tiers <= 0 or H % n_tiers:
        raise ValueError("n_tiers must divide H")
    return np.arange(H) // (H // n_tiers)


def head_norm_gate(o, g, weight, n_tiers, eps):
    """y[t,h,c] = o[t,h,c] r[t,h] weight[tier(h),c] SiLU(g[t,h,c]) with
    r = 1/sqrt(mean_c o^2 + eps).  o, g [N,H,C]; weight [n_tiers,C].  Returns (y, r)."""
    o, g, w = (np.asarray(x, np.float64) for x in (o, g, weight))
    tier = _tiers(o.shape[1], n_tiers)
    r = 1.0 / np.sqrt(np.mean(o * o, axis=-1) + eps)
    silu = g / (1.0 + np.exp(-g))
    return o * r[..., None] * w[tier][None] * silu, r


def head_norm_gate_bwd(dy, o, g, weight, n_tiers, eps):
    """Gradient of sum(y * dy) (hand-derived): returns (d_o, dg, d_weight)."""
    dy, o, g, w = (np.asarray(x, np.float64) for x in (dy, o, g, weight))
    H, C = o.shape[1], o.shape[2]
    tier = _tiers(H, n_tiers)
    r = (1.0 / np.sqrt(np.mean(o * o, axis=-1) + eps))[..., None]
    n = o * r
    sg = 1.0 / (1.0 + np.exp(-g))
    s = g * sg
    wt = w[tier][None]
    dg = dy * n * wt * sg * (1.0 + g * (1.0 - sg))
    dn = dy * s * wt
    d_o = r * (dn - n * np.mean(dn * n, axis=-1, keepdims=True))
    per_head = np.sum(dy * s * n, axis=0)  # [H, C]
    d_w = np.zeros((n_tiers, C))
    for h in range(H):
        d_w[tier[h]] += per_head[h]
    return d_o, dg, d_w


# --------------------------------------------------------------------------- causal conv
# Depth-wise causal Conv1d of width 4 + SiLU with its 3-input state (section "i14 and the
# Laplace 3B architecture", "Normalization and convolution").  Plain fp64 numpy, the
# definition written out: x_{-3..-1} is the state carried in.

def conv_fwd(x, weight, bias=None, init_state=None):
    """y_t[d] = SiLU(sum_{j=0..3} weight[d,j] x_{t-3+j}[d] + bias[d]).  x [B,T,D], weight
    [D,4], bias [D], init_state [B,3,D] (x_{-3..-1}; zeros if None).  Returns (y,
    final_state = x_{T-3..T-1})."""
    x, w = np.asarray(x, np.float64), np.asarray(weight, np.float64)
    B, T, D = x.shape
    prev = np.zeros((B, 3, D)) if init_state is None else np.asarray(init_state, np.float64)
    xe = np.concatenate([prev, x], axis=1)  # xe[:, t + 3] = x_t
    z = np.zeros((B, T, D)) if bias is None else np.broadcast_to(np.asarray(bias, np.float64),
                                                                  (B, T, D)).copy()
    for j in range(4):
        z += w[:, j] * xe[:, j:j + T]
    return z / (1.0 + np.exp(-z)), xe[:, T:T + 3].copy()


def conv_bwd(x, weight, dy, bias=None, init_state=None):
    """Gradient of sum(y * dy) (hand-derived): returns (dx, d_init_state, d_weight, d_bias)."""
    x, w, dy = (np.asarray(a, np.float64) for a in (x, weight, dy))
    B, T, D = x.shape
    prev = np.zeros((B, 3, D)) if init_state is None else np.asarray(init_state, np.float64)
    xe = np.concatenate([prev, x], axis=1)
    z = np.zeros((B, T, D)) if bias is None else np.broadcast_to(np.asarray(bias, np.float64),
                                                                  (B, T, D)).copy()
    for j in range(4):
        z += w[:, j] * xe[:, j:j + T]
    sg = 1.0 / (1.0 + np.exp(-z))
    dz = dy * sg * (1.0 + z * (1.0 - sg))
    dxe = np.zeros((B, T + 3, D))
    dw = np.zeros((D, 4))
    for j in range(4):
        dxe[:, j:j + T] += w[:, j] * dz
        dw[:, j] = np.sum(dz * xe[:, j:j + T], axis=(0, 1))
    return dxe[:, 3:], dxe[:, :3], dw, np.sum(dz, axis=(0, 1))


def conv_decode_step(state, x, weight, bias=None):
    """One token: the forward with T = 1 from the 3-input state.  state [N,3,D], x [N,D].
    Returns (y [N,D], new_state)."""
    y, fin = conv_fwd(np.asarray(x, np.float64)[:, None], weight, bias, state)
    return y[:, 0], fin
