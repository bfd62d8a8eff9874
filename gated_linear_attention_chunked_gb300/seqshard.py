"""Long-context prefill (and its backward) with the sequence cut into consecutive slices, one
slice per rank.

Method.  Section "Challenge 1" of "Beyond the KV cache: Training and serving i14's Laplace 3B
linear attention model on AWS Trainium2 with native PyTorch" carries one fixed-size state from
chunk to chunk, and section "Inference optimization on Trainium2" keeps that state the same
size however long the prompt.  The recurrence S_t = lambda S_{t-1} + k_t v_t^T ("GLA mixer")
is linear, so slice j (len_j tokens) maps the state entering it to the state leaving it as

    S_{j+1} = lambda^(len_j) S_j + U_j,        U_j = sum_{t in j} lambda^(e_j - t) k_t v_t^T

and, for the backward ("Challenge 3"), the adjoint A_j of the state leaving slice j obeys

    A_{j-1} = lambda^(len_j) A_j + U'_j,       U'_j = sum_{t in j} lambda^(t - s_j + 1) q_t dO_t^T.

One rank holds slice r.  Forward: it computes U_r (gla_chunk_state_sum), the ranks all-gather
the U's (the one exchange, B*H*96*192 fp32 per rank), each rank links the state entering its
slice (gla_state_link) and runs the chunked forward on its slice from that state.  Backward:
the same with U'_r (gla_chunk_adjoint_sum) in reverse order, then the chunked backward of the
slice from its entering state and leaving adjoint; d_aug is summed over the ranks.  Every
arithmetic step runs in the library's kernels; this module only orders the calls and the
exchange.

The exchange is an object with `rank`, `world`, `all_gather(tensor) -> [world, ...]`,
`all_gather_int(int) -> list[int]` and `all_reduce_sum(tensor)`: `TorchDistExchange` for one
process per GPU (NCCL through torch.distributed, or gloo), `ThreadExchange` for ranks that are
threads of one process.  `ops` (the kernels) can be replaced for tests of the ordering logic on
a machine without a GPU.
"""
from __future__ import annotations

import threading


class TorchDistExchange:
    """The exchange over a torch.distributed process group (NCCL for GPUs)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def all_gather(self, t):
        import torch
        t = t.contiguous()
        parts = [torch.empty_like(t) for _ in range(self.world)]
        self.dist.all_gather(parts, t, group=self.group)
        return torch.stack(parts)

    def all_gather_int(self, x: int, device) -> list[int]:
        import torch
        t = torch.tensor([int(x)], dtype=torch.int64, device=device)
        return [int(v) for v in self.all_gather(t).view(-1).tolist()]

    def all_reduce_sum(self, t):
        self.dist.all_reduce(t, op=self.dist.ReduceOp.SUM, group=self.group)
        return t


class ThreadExchange:
    """The exchange between ranks that are threads of one process (e.g. one thread per GPU).
    `ThreadExchange(world).view(r)` is rank r's handle.  Each rank's tensor is complete on its
    device before the others read it (its stream is synchronised at the exchange)."""

    def __init__(self, world: int):
        self.world = world
        self._barrier = threading.Barrier(world)
        self._slots = [None] * world

    def view(self, rank: int) -> "_ThreadRank":
        return _ThreadRank(self, rank)


class _ThreadRank:
    def __init__(self, shared: ThreadExchange, rank: int):
        self.shared = shared
        self.rank = rank
        self.world = shared.world

    def _swap(self, value):
        s = self.shared
        s._slots[self.rank] = value
        s._barrier.wait()
        got = list(s._slots)
        s._barrier.wait()  # every rank has read the slots before they are reused
        return got

    def all_gather(self, t):
        import torch
        if t.is_cuda:
            torch.cuda.current_stream(t.device).synchronize()
        return torch.stack([x.to(t.device) for x in self._swap(t)])

    def all_gather_int(self, x: int, device=None) -> list[int]:
        return [int(v) for v in self._swap(int(x))]

    def all_reduce_sum(self, t):
        total = self.all_gather(t).sum(dim=0)
        t.copy_(total)
        return t


class KernelOps:
    """The library's calls (the default `ops`)."""

    def state_sum(self, k, v, log_decay):
        from . import chunk_state_sum
        return chunk_state_sum(k, v, log_decay)

    def adjoint_sum(self, q, dO, log_decay):
        from . import chunk_adjoint_sum
        return chunk_adjoint_sum(q, dO, log_decay)

    def link(self, U_all, lens, rank, log_decay, boundary, reverse):
        from . import state_link
        return state_link(U_all, lens, rank, log_decay, boundary, reverse=reverse)

    def fwd(self, q, k, v, log_decay, aug, init, gate):
        from . import chunk_fwd
        return chunk_fwd(q, k, v, log_decay, aug, init, gate=gate)

    def bwd(self, q, k, v, log_decay, aug, dO, init, dfin, gate):
        from . import chunk_bwd
        return chunk_bwd(q, k, v, log_decay, aug, dO, init, dfin, gate=gate)


def chunk_fwd_sharded(q, k, v, log_decay, aug_balance, init_state=None, *, exchange, gate=None,
                      ops=None):
    """Chunked forward of this rank's slice of a sequence cut into consecutive slices, one
    per rank in rank order.  q, k [B,T_r,H,96], v [B,T_r,H,192] hold this rank's T_r tokens
    (slices may differ in length); init_state [B,H,96,192] is the sequence's initial state,
    the same on every rank (or None).  Returns (o of the slice, the state leaving the slice --
    the sequence's final state on the last rank --, the state entering the slice, which
    chunk_bwd_sharded takes)."""
    ops = ops or KernelOps()
    T_r = q.shape[1]
    lens = exchange.all_gather_int(T_r, q.device)
    U = ops.state_sum(k, v, log_decay)
    U_all = exchange.all_gather(U)
    s_in = ops.link(U_all, lens, exchange.rank, log_decay, init_state, False)
    o, s_out = ops.fwd(q, k, v, log_decay, aug_balance, s_in, gate)
    return o, s_out, s_in


def chunk_bwd_sharded(q, k, v, log_decay, aug_balance, dO, state_in, d_final_state=None, *,
                      exchange, gate=None, ops=None):
    """Backward of chunk_fwd_sharded for this rank's slice.  state_in: the state entering the
    slice (chunk_fwd_sharded's third result); d_final_state [B,H,96,192]: the adjoint of the
    sequence's final state, the same on every rank (or None).  Returns (dq, dk, dv of the
    slice, d_aug summed over all ranks, the adjoint of the state entering the slice -- the
    sequence's d_init_state on rank 0)."""
    ops = ops or KernelOps()
    T_r = q.shape[1]
    lens = exchange.all_gather_int(T_r, q.device)
    Up = ops.adjoint_sum(q, dO, log_decay)
    Up_all = exchange.all_gather(Up)
    a_out = ops.link(Up_all, lens, exchange.rank, log_decay, d_final_state, True)
    dq, dk, dv, d_aug, d_in = ops.bwd(q, k, v, log_decay, aug_balance, dO, state_in, a_out, gate)
    d_aug = exchange.all_reduce_sum(d_aug)
    return dq, dk, dv, d_aug, d_in
