"""Ring schedule over the ranks of a process group ("bpt.py", _ring_attention_fwd and
_ring_attention_bwd).

Rank i keeps query block i.  The key / value blocks travel around the ring one hop per
step towards rank i + 1 (the ppermute with pairs (i, (i + 1) mod n)), so at step t rank i
holds key / value block (i - t) mod n and folds it into its own state with a caller-given
step function.  In the backward the dK / dV accumulators travel with their K / V block;
after n hops every block and its gradient are back on the rank that owns them.

Each hop is a pair of point-to-point messages per tensor whose completion is awaited with a
bound: a block that never arrives (a dropped message, a rank that died) raises RingTimeout
on the receiving rank instead of leaving it waiting.

The single-GPU library runs the same schedule as a sweep of launches over one device's
memory (ring_size in the descriptor); this module is the host side of the multi-rank form,
the per-block computation being the caller's.
"""
from __future__ import annotations

import datetime
from typing import Callable, Sequence

import torch
import torch.distributed as dist


class RingTimeout(RuntimeError):
    """A block of the ring did not arrive within the bound."""


def exchange(tensors: Sequence[torch.Tensor], *, group=None,
             timeout: datetime.timedelta = datetime.timedelta(seconds=30)) -> list:
    """One hop: send every tensor to rank i + 1, receive the same shapes from rank i - 1.
    Message t of a hop carries tag t, so the tensors cannot be confused.

    The hop's sends and receives are posted together as one batch
    (``batch_isend_irecv``): with NCCL that is one group of point-to-point operations, so
    no rank's send waits behind a receive its peer queued after its own send (two ranks,
    where the next and the previous rank are the same peer, would otherwise deadlock).
    A timeout only ends the host's wait; with NCCL the queued transfer may still be pending
    on the device, so a rank that sees RingTimeout must not launch further work on that
    process group."""
    n = dist.get_world_size(group)
    i = dist.get_rank(group)
    dst, src = (i + 1) % n, (i - 1) % n
    if n == 1:
        return list(tensors)
    out = [torch.empty_like(t) for t in tensors]
    ops = [dist.P2POp(dist.isend, t.contiguous(), dst, group=group, tag=tag) for tag, t in enumerate(tensors)]
    ops += [dist.P2POp(dist.irecv, r, src, group=group, tag=tag) for tag, r in enumerate(out)]
    for w in dist.batch_isend_irecv(ops):
        try:
            w.wait(timeout)
        except RuntimeError as e:
            raise RingTimeout(f"rank {i}: the hop (block to rank {dst}, block from rank {src}) did not "
                              f"complete within {timeout.total_seconds():g} s") from e
    return out


def ring_forward(q, k, v, step: Callable, *, group=None,
                 timeout: datetime.timedelta = datetime.timedelta(seconds=30), hop: Callable = exchange):
    """Forward sweep.  step(q, k, v, state, i, j) -> state folds key / value block j into
    query block i's state (None before the first step) and is called once per step, j in
    ring order i, i - 1, ...; returns the final state.  K and V make n hops, ending home."""
    n = dist.get_world_size(group)
    i = dist.get_rank(group)
    state = None
    for t in range(n):
        state = step(q, k, v, state, i, (i - t) % n)
        k, v = hop([k, v], group=group, timeout=timeout)
    return state


def ring_backward(q, k, v, do, step: Callable, *, group=None,
                  timeout: datetime.timedelta = datetime.timedelta(seconds=30), hop: Callable = exchange):
    """Backward sweep.  step(q, k, v, do, dq, dk, dv, i, j) -> (dq, dk, dv) adds the
    contributions of the pair (query block i, key / value block j): dq belongs to this rank
    (None before the first step), dk and dv to block j and travel with it.  Returns this
    rank's dq and, after n hops, the dk, dv of its own key / value block."""
    n = dist.get_world_size(group)
    i = dist.get_rank(group)
    dq = None
    dk = torch.zeros_like(k, dtype=torch.float64 if k.dtype == torch.float64 else torch.float32)
    dv = torch.zeros_like(v, dtype=dk.dtype)
    for t in range(n):
        dq, dk, dv = step(q, k, v, do, dq, dk, dv, i, (i - t) % n)
        k, v, dk, dv = hop([k, v, dk, dv], group=group, timeout=timeout)
    return dq, dk, dv
