"""The multi-rank ring schedule (ring_attention_gb300.ring) on CPU ranks over gloo.

Each rank holds one query block and one key / value block of a small causal GQA problem;
the blocks travel around the ring as bpt.py's _ring_attention_fwd / _ring_attention_bwd
move them.  The per-block arithmetic below is test code (the online-softmax fold and the
block-pair gradients, in float64); the reference is the oracle's one-shot attention.
The failure tests drop a message or stop a rank: the waiting rank must raise RingTimeout
within its bound instead of hanging.  No GPU is involved.
"""
import datetime
import multiprocessing as mp
import os
import socket
import time

import numpy as np
import pytest

B, S, HQ, HKV, D = 1, 12, 2, 1, 3
SCALE = 0.8
SEED = 311


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    rng = np.random.default_rng(SEED)
    q = rng.standard_normal((B, S, HQ, D))
    k = rng.standard_normal((B, S, HKV, D))
    v = rng.standard_normal((B, S, HKV, D))
    do = rng.standard_normal((B, S, HQ, D))
    return q, k, v, do


def _scores(qb, kb, i, j, blk):
    """s * Q_i K_j^T per q head with the causal rule by global position: [HQ, blk, blk]."""
    g = HQ // HKV
    z = np.stack([SCALE * qb[0, :, h] @ kb[0, :, h // g].T for h in range(HQ)])
    qpos = i * blk + np.arange(blk)[:, None]
    kpos = j * blk + np.arange(blk)[None, :]
    return np.where(kpos <= qpos, z, -np.inf)


def _fwd_step(qb, kb, vb, state, i, j, blk, order):
    """bpt.py scan_kv_block: fold block j into (m, l, acc) of query block i."""
    order.append(j)
    qn, kn, vn = qb.numpy(), kb.numpy(), vb.numpy()
    if state is None:
        state = (np.full((HQ, blk), -np.inf), np.zeros((HQ, blk)), np.zeros((blk, HQ, D)))
    m, l, acc = state
    z = _scores(qn, kn, i, j, blk)
    mn = np.maximum(m, z.max(axis=2))
    safe = np.where(np.isfinite(mn), mn, 0.0)
    c = np.where(np.isfinite(m), np.exp(m - safe), 0.0)
    p = np.exp(z - safe[:, :, None])
    g = HQ // HKV
    pv = np.stack([p[h] @ vn[0, :, h // g] for h in range(HQ)], axis=1)   # [blk, HQ, D]
    return (mn, l * c + p.sum(axis=2), acc * c.T[:, :, None] + pv)


def _bwd_step(qb, kb, vb, dob, dq, dk, dv, i, j, blk, lse, Dr):
    """Contributions of the pair (query block i, key block j) to dq_i, dk_j, dv_j."""
    import torch
    qn, kn, vn, don = qb.numpy(), kb.numpy(), vb.numpy(), dob.numpy()
    g = HQ // HKV
    z = _scores(qn, kn, i, j, blk)
    p = np.where(np.isfinite(z), np.exp(z - lse[:, :, None]), 0.0)            # [HQ, blk, blk]
    dp = np.stack([don[0, :, h] @ vn[0, :, h // g].T for h in range(HQ)])
    ds = p * (dp - Dr[:, :, None])
    dq = np.zeros((1, blk, HQ, D)) if dq is None else dq
    dkn, dvn = dk.numpy().copy(), dv.numpy().copy()
    for h in range(HQ):
        dq[0, :, h] += SCALE * ds[h] @ kn[0, :, h // g]
        dkn[0, :, h // g] += SCALE * ds[h].T @ qn[0, :, h]
        dvn[0, :, h // g] += p[h].T @ don[0, :, h]
    return dq, torch.from_numpy(dkn), torch.from_numpy(dvn)


def _rank_ring(rank, world, port, out):
    import torch
    import torch.distributed as dist
    from ring_attention_gb300 import ring
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    try:
        blk = S // world
        q, k, v, do = _inputs()
        sl = slice(rank * blk, (rank + 1) * blk)
        tq, tk, tv, tdo = (torch.from_numpy(np.ascontiguousarray(x[:, sl])) for x in (q, k, v, do))
        order = []
        m, l, acc = ring.ring_forward(tq, tk, tv, lambda a, b_, c, st, i, j: _fwd_step(a, b_, c, st, i, j, blk, order),
                                      timeout=datetime.timedelta(seconds=20))
        o = np.where(l.T[:, :, None] > 0, acc / np.where(l > 0, l, 1.0).T[:, :, None], 0.0)
        lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), np.inf)
        Dr = np.einsum("shd,shd->hs", tdo.numpy()[0], o)
        dq, dk, dv = ring.ring_backward(
            tq, tk, tv, tdo,
            lambda a, b_, c, d_, dq_, dk_, dv_, i, j: _bwd_step(a, b_, c, d_, dq_, dk_, dv_, i, j, blk, lse, Dr),
            timeout=datetime.timedelta(seconds=20))
        out.put((rank, order, o, dq, dk.numpy(), dv.numpy()))
    finally:
        dist.destroy_process_group()


def _run(target, world, extra=()):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, out) + tuple(extra)) for r in range(world)]
    for p in procs:
        p.start()
    got = []
    try:
        for _ in procs:
            got.append(out.get(timeout=120))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    return got, [p.exitcode for p in procs]


@pytest.mark.parametrize("world", [2, 3])
def test_ring_blocks_travel_and_match_one_shot(ora, world):
    got, codes = _run(_rank_ring, world)
    assert codes == [0] * world
    q, k, v, do = _inputs()
    rq, rk, rv, ro, _, _ = ora.attention_bwd(q, k, v, do, causal=True, scale=SCALE)
    blk = S // world
    for rank, order, o, dq, dk, dv in got:
        # ring order: block (i - t) mod n at step t
        assert order == [(rank - t) % world for t in range(world)]
        sl = slice(rank * blk, (rank + 1) * blk)
        np.testing.assert_allclose(o, ro[0, sl], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dq[0], rq[0, sl], rtol=1e-11, atol=1e-12)
        # dK / dV travelled with their blocks and came home
        np.testing.assert_allclose(dk[0], rk[0, sl], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dv[0], rv[0, sl], rtol=1e-11, atol=1e-12)


def _rank_fault(rank, world, port, out, fault):
    import torch
    import torch.distributed as dist
    from ring_attention_gb300 import ring
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))

    def dropping_hop(tensors, *, group=None, timeout=None):
        # receives like the real hop, sends nothing: its messages are lost
        src = (rank - 1) % world
        got = [torch.empty_like(t) for t in tensors]
        for w in [dist.irecv(r, src, tag=tag) for tag, r in enumerate(got)]:
            w.wait(timeout)
        return got

    def step(a, b_, c, st, i, j):
        if fault == "dies" and rank == 1:
            raise SystemExit(3)   # this rank stops before its first hop
        return st

    t0 = time.perf_counter()
    kind = "finished"
    try:
        hop = dropping_hop if (fault == "drop" and rank == 0) else ring.exchange
        x = torch.zeros(2, 3)
        ring.ring_forward(x, x.clone(), x.clone(), step, timeout=datetime.timedelta(seconds=2), hop=hop)
    except ring.RingTimeout:
        kind = "RingTimeout"
    except SystemExit:
        kind = "stopped"
    except RuntimeError:
        kind = "RuntimeError"
    out.put((rank, kind, time.perf_counter() - t0))
    out.close()
    out.join_thread()
    os._exit(0)   # no teardown handshake with a peer that may be gone


@pytest.mark.parametrize("fault", ["drop", "dies"])
def test_lost_message_or_rank_times_out(fault):
    got, codes = _run(_rank_fault, 2, (fault,))
    res = {r: (kind, dt) for r, kind, dt in got}
    assert codes == [0, 0]
    # the rank waiting for the block that never comes gives up within its bound
    waiting = 1 if fault == "drop" else 0
    kind, dt = res[waiting]
    assert kind == "RingTimeout" and dt < 15.0
    if fault == "dies":
        assert res[1][0] == "stopped"
