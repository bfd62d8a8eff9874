"""A long sequence cut into consecutive slices across ranks (seqshard.py): the ordering of the
slice sums, the exchange and the linked states, checked on the CPU.

The ranks are two gloo processes (and, separately, three threads) whose kernels are replaced
by the fp64 oracle (`OracleOps`): each rank holds one slice of a seeded sequence (slices of
unequal, ragged lengths, a nonzero initial state and final-state adjoint), and the pieces
they return must equal the oracle's forward and backward over the whole sequence.  A wrong
slice order, a link taken in the wrong direction or a sum weighted from the wrong end fails
these checks.  The same code path with the library's kernels runs on the GPU in
tests/test_gpu_seqshard.py."""
import multiprocessing as mp
import os
import socket
import sys
import threading

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
H, SEED = 3, 61
LENS2 = [173, 127]
LENS3 = [64, 200, 37]


def _inputs(T):
    import synth
    B = 2
    q, k, v = synth.qkv(SEED, B, T, H, bf16=False)
    dO = synth.grad_out(SEED, B, T, H, bf16=False)
    a = synth.aug_balance(SEED, (H, 96), 0.1)
    init = synth.init_state(SEED, B, H, 0.05)
    dfin = synth.normal(SEED, synth.DFIN, (B, H, 96, 192), 0.05)
    return q, k, v, dO, a, init, dfin


class OracleOps:
    """The kernels' results from the fp64 oracle, on torch CPU float64 tensors."""

    @staticmethod
    def _n(x):
        return None if x is None else x.numpy()

    @staticmethod
    def _t(x):
        import torch
        return torch.from_numpy(np.ascontiguousarray(x, np.float64))

    def state_sum(self, k, v, g):
        import oracle
        return self._t(oracle.slice_state_sum(self._n(k), self._n(v), self._n(g)))

    def adjoint_sum(self, q, dO, g):
        import oracle
        return self._t(oracle.slice_adjoint_sum(self._n(q), self._n(dO), self._n(g)))

    def link(self, U_all, lens, rank, g, boundary, reverse):
        import oracle
        return self._t(oracle.state_link(self._n(U_all), lens, rank, self._n(g),
                                         self._n(boundary), reverse))

    def fwd(self, q, k, v, g, a, init, gate):
        import oracle
        o, fin = oracle.fwd(self._n(q), self._n(k), self._n(v), self._n(g), self._n(a),
                            self._n(init))
        return self._t(o), self._t(fin)

    def bwd(self, q, k, v, g, a, dO, init, dfin, gate):
        import oracle
        r = oracle.bwd(self._n(q), self._n(k), self._n(v), self._n(g), self._n(a), self._n(dO),
                       self._n(init), self._n(dfin))
        return tuple(self._t(r[n]) for n in ("dq", "dk", "dv", "d_a", "d_init_state"))


def _run_rank(exchange, lens, out):
    """One rank's forward and backward over its slice; results into out[rank]."""
    import torch

    import oracle
    from gated_linear_attention_chunked_gb300 import seqshard
    r = exchange.rank
    q, k, v, dO, a, init, dfin = _inputs(sum(lens))
    t0 = sum(lens[:r])
    sl = slice(t0, t0 + lens[r])
    T = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float64))
    g = T(oracle.decay_schedule(H).astype(np.float32))
    ops = OracleOps()
    o, s_out, s_in = seqshard.chunk_fwd_sharded(T(q[:, sl]), T(k[:, sl]), T(v[:, sl]), g, T(a),
                                                T(init), exchange=exchange, ops=ops)
    dq, dk, dv, d_aug, d_in = seqshard.chunk_bwd_sharded(
        T(q[:, sl]), T(k[:, sl]), T(v[:, sl]), g, T(a), T(dO[:, sl]), s_in, T(dfin),
        exchange=exchange, ops=ops)
    out[r] = dict(o=o.numpy(), s_out=s_out.numpy(), dq=dq.numpy(), dk=dk.numpy(),
                  dv=dv.numpy(), d_aug=d_aug.numpy(), d_in=d_in.numpy())


def _check_against_whole_sequence(res, lens):
    import oracle
    q, k, v, dO, a, init, dfin = _inputs(sum(lens))
    g = oracle.decay_schedule(H).astype(np.float32).astype(np.float64)
    o_ref, fin_ref = oracle.fwd(q, k, v, g, a, init)
    ref = oracle.bwd(q, k, v, g, a, dO, init, dfin)
    R = len(lens)
    cat = lambda name: np.concatenate([res[r][name] for r in range(R)], axis=1)
    rel = lambda x, y: float(np.abs(x - y).max() / np.sqrt(np.mean(y * y)))
    errs = dict(o=rel(cat("o"), o_ref), final=rel(res[R - 1]["s_out"], fin_ref),
                dq=rel(cat("dq"), ref["dq"]), dk=rel(cat("dk"), ref["dk"]),
                dv=rel(cat("dv"), ref["dv"]), d_init=rel(res[0]["d_in"], ref["d_init_state"]))
    for r in range(R):
        errs[f"d_aug{r}"] = rel(res[r]["d_aug"], ref["d_a"])
    for name, e in errs.items():
        assert e < 1e-9, f"{name}: {e:.3e}"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gloo_worker(rank, world, port, lens, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist

    from gated_linear_attention_chunked_gb300 import seqshard
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out = {}
        _run_rank(seqshard.TorchDistExchange(), lens, out)
        queue.put((rank, out[rank]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_match_the_whole_sequence():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gloo_worker, args=(r, 2, port, LENS2, queue)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        r, d = queue.get(timeout=300)
        res[r] = d
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    _check_against_whole_sequence(res, LENS2)


def test_three_thread_ranks_match_the_whole_sequence():
    from gated_linear_attention_chunked_gb300 import seqshard
    shared = seqshard.ThreadExchange(len(LENS3))
    res, errors = {}, []

    def body(r):
        try:
            _run_rank(shared.view(r), LENS3, res)
        except BaseException as e:  # surfaced below
            errors.append(e)
            shared._barrier.abort()

    threads = [threading.Thread(target=body, args=(r,)) for r in range(len(LENS3))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    _check_against_whole_sequence(res, LENS3)


@pytest.mark.parametrize("mistake", ["sums_reversed", "lengths_reversed"])
def test_a_wrong_slice_order_is_caught(mistake):
    """The check above is not vacuous: an exchange that hands the ranks the slices' sums, or
    their lengths, in reversed order (the plausible mistake of linking from the wrong end)
    changes the result enough to fail it."""
    from gated_linear_attention_chunked_gb300 import seqshard
    lens = LENS3
    shared = seqshard.ThreadExchange(len(lens))
    res = {}

    class Mistaken:
        def __init__(self, view):
            self.v, self.rank, self.world = view, view.rank, view.world

        def all_gather(self, t):
            g = self.v.all_gather(t)
            return g.flip(0) if mistake == "sums_reversed" and g.dim() > 2 else g

        def all_gather_int(self, x, device=None):
            n = self.v.all_gather_int(x)
            return n[::-1] if mistake == "lengths_reversed" else n

        def all_reduce_sum(self, t):
            return self.v.all_reduce_sum(t)

    threads = [threading.Thread(target=_run_rank, args=(Mistaken(shared.view(r)), lens, res))
               for r in range(len(lens))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert len(res) == len(lens)
    with pytest.raises(AssertionError):
        _check_against_whole_sequence(res, lens)
