"""GPU parity on the five workloads of the hot path, at their full sizes.

Inputs follow the seeded recipe (ring_attention_gb300.inputs); the same bits
go to the oracle.  The long-context ring workload (S = 131072) is too large
for a full float64 run, so it is checked on sampled query rows (O, m, l, dQ)
and sampled keys (dK, dV) at full size, and in full at S = 16384 with the
same ring geometry and the padding scaled.
"""
import numpy as np
import pytest
import torch

from ring_attention_gb300 import inputs as W
from tests.gpu_util import (BF16_GRAD_REL_L2, BF16_O_MAX_ABS, FP32_MAX_ABS, check_stats, dev, host,
                            max_abs, rel_l2)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bpa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_attention_gb300 import build
    build.build()
    from ring_attention_gb300 import bpa as mod
    return mod


def _kw(w, bias_t=None):
    return dict(causal=w.causal, window=w.window, bias=bias_t, query_chunk=w.query_chunk,
                key_chunk=w.key_chunk, ring_size=w.ring_size)


def _run(bpa, w, q, k, v, do, bias):
    tq, tk, tv = dev(q), dev(k), dev(v)
    tb = dev(bias) if bias is not None else None
    o, m, l = bpa.bpa_fwd(tq, tk, tv, **_kw(w, tb))
    grads = None
    if do is not None:
        grads = bpa.bpa_bwd(tq, tk, tv, o, dev(do), m, l, **_kw(w, tb))
    torch.cuda.synchronize()
    return o, m, l, grads


def test_tiny_fp32_workload(bpa, ora):
    w = W.TINY_F32
    q, k, v, do, bias = W.make_inputs(w)
    o, m, l, (dq, dk, dv) = _run(bpa, w, q, k, v, do, bias)
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, causal=True)
    for got, ref in ((o, ro), (dq, rq), (dk, rk), (dv, rv)):
        assert max_abs(host(got), ref) <= FP32_MAX_ABS
    check_stats(m, l, rm, rl)


@pytest.mark.parametrize("w", [W.GQA_CAUSAL, W.GQA_SWA], ids=lambda w: w.name)
def test_gqa_workloads_full(bpa, ora, w):
    q, k, v, do, bias = W.make_inputs(w)
    o, m, l, (dq, dk, dv) = _run(bpa, w, q, k, v, do, bias)
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, causal=w.causal, window=w.window)
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)
    assert rel_l2(host(dq), rq) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dk), rk) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dv), rv) <= BF16_GRAD_REL_L2


def test_ring_workload_reduced_length(bpa, ora):
    # same ring geometry (8 super-blocks, chunks 512/1024 -> scaled), padding scaled to S
    w = W.RING_LONG
    S = 16384
    q, k, v, do, bias = W.make_inputs(w, S=S, Hq=8, Hkv=2)
    from dataclasses import replace
    wr = replace(w, S=S, Hq=8, Hkv=2, query_chunk=256, key_chunk=512)
    o, m, l, (dq, dk, dv) = _run(bpa, wr, q, k, v, do, bias)
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, causal=True, bias=bias)
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)
    assert rel_l2(host(dq), rq) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dk), rk) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dv), rv) <= BF16_GRAD_REL_L2


@pytest.mark.slow
def test_ring_workload_full_size_sampled(bpa, ora):
    w = W.RING_LONG
    q, k, v, do, bias = W.make_inputs(w)
    o, m, l, (dq, dk, dv) = _run(bpa, w, q, k, v, do, bias)
    S, blk = w.S, w.S // w.ring_size
    rng = np.random.default_rng(123)
    # rows: super-block edges, the padded tail, the first rows, and random rows
    qs = {0, 1, 127, 128, S - 1, S - 4096, S - 4097}
    for j in range(1, w.ring_size):
        qs |= {j * blk - 1, j * blk, j * blk + 1}
    qs |= set(rng.integers(0, S, 200).tolist())
    rows = [(0, int(rng.integers(0, w.Hq)), qq) for qq in sorted(qs)]
    ro, rm, rl, rdq = ora.rows(q, k, v, do, rows, causal=True, bias=bias)
    ho, hdq = o.cpu(), dq.cpu()
    go = np.stack([ho[b, s, h].float().numpy() for b, h, s in rows])
    gdq = np.stack([hdq[b, s, h].float().numpy() for b, h, s in rows])
    assert max_abs(go, ro) <= BF16_O_MAX_ABS
    gm = np.array([m[b, h, s].item() for b, h, s in rows])
    gl = np.array([l[b, h, s].item() for b, h, s in rows])
    assert np.max(np.abs(gm - rm) / (1 + np.abs(rm))) <= 1e-3
    assert np.max(np.abs(gl - rl) / np.abs(rl)) <= 1e-3
    assert rel_l2(gdq, rdq) <= BF16_GRAD_REL_L2
    # keys just before the padding: every row >= key attends to them
    g = 3
    keys = sorted({S - 8192, S - 8191, S - 6000, S - 4097} | set(rng.integers(S - 8192, S - 4096, 12).tolist()))
    rdk, rdv = ora.keys(q, k, v, do, 0, g, keys, causal=True, bias=bias)
    gdk = dk[0, keys, g].float().cpu().numpy()
    gdv = dv[0, keys, g].float().cpu().numpy()
    assert rel_l2(gdk, rdk) <= BF16_GRAD_REL_L2
    assert rel_l2(gdv, rdv) <= BF16_GRAD_REL_L2
    # padded keys carry no weight: their gradients vanish
    assert float(dk[0, S - 4096:].abs().max()) == 0.0 and float(dv[0, S - 4096:].abs().max()) == 0.0


def test_block_selected_workload_full(bpa, ora):
    w = W.BLOCK_SEL
    q, k, v, _, _ = W.make_inputs(w)
    tq, tk, tv = dev(q), dev(k), dev(v)
    idx = bpa.bpa_select_blocks(tq, tk, block_size=w.sel_block, top_n=w.top_n)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, causal=True, block_idx=idx, sel_block=w.sel_block, top_n=w.top_n,
                          local_window=w.local_window)
    torch.cuda.synchronize()
    ridx = ora.select_blocks(q, k, block_size=w.sel_block, top_n=w.top_n)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    ro, rm, rl = ora.attention_fwd(q, k, v, causal=True, block_idx=ridx, sel_block=w.sel_block,
                                   top_n=w.top_n, local_window=w.local_window)
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)


def test_block_selected_workload_backward_reduced(bpa, ora):
    # the block-selected workload's recipe (dO drawn after Q, K, V from the same
    # generator) at S = 2048: selection, forward and the backward through the gather
    from dataclasses import replace
    w = replace(W.BLOCK_SEL, backward=True)
    q, k, v, do, _ = W.make_inputs(w, B=1, S=2048)
    tq, tk, tv = dev(q), dev(k), dev(v)
    idx = bpa.bpa_select_blocks(tq, tk, block_size=w.sel_block, top_n=w.top_n)
    kw = dict(causal=True, sel_block=w.sel_block, top_n=w.top_n, local_window=w.local_window)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, block_idx=idx, **kw)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, dev(do), m, l, block_idx=idx, **kw)
    torch.cuda.synchronize()
    ridx = ora.select_blocks(q, k, block_size=w.sel_block, top_n=w.top_n)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, block_idx=ridx, **kw)
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)
    assert rel_l2(host(dq), rq) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dk), rk) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dv), rv) <= BF16_GRAD_REL_L2


def test_block_selected_joint_workload_reduced(bpa, ora):
    # the joint view (one head of 512 channels) of the block-selected workload's numbers
    # at S = 2048: selection on the 512-channel block sums, forward and backward
    w = W.BLOCK_SEL_JOINT
    q, k, v, do, _ = W.make_inputs(w, B=1, S=2048)
    tq, tk, tv = dev(q), dev(k), dev(v)
    idx = bpa.bpa_select_blocks(tq, tk, block_size=w.sel_block, top_n=w.top_n)
    kw = dict(causal=True, sel_block=w.sel_block, top_n=w.top_n, local_window=w.local_window)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, block_idx=idx, **kw)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, dev(do), m, l, block_idx=idx, **kw)
    torch.cuda.synchronize()
    ridx = ora.select_blocks(q, k, block_size=w.sel_block, top_n=w.top_n)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, block_idx=ridx, **kw)
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)
    assert rel_l2(host(dq), rq) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dk), rk) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dv), rv) <= BF16_GRAD_REL_L2


def test_varlen_workload_reduced(bpa, ora):
    # the variable-length workload's recipe and lengths with fewer heads (GQA ratio 4)
    w = W.VARLEN_CAUSAL
    q, k, v, do, _ = W.make_inputs(w, Hq=8, Hkv=2)
    lq = list(w.seqlens_q)
    tl = torch.tensor(lq, dtype=torch.int32, device="cuda")
    tq, tk, tv = dev(q), dev(k), dev(v)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, causal=True, seqlens_q=tl)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, dev(do), m, l, causal=True, seqlens_q=tl)
    torch.cuda.synchronize()
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, causal=True, seqlens_q=lq)
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)
    assert rel_l2(host(dq), rq) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dk), rk) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dv), rv) <= BF16_GRAD_REL_L2


def test_mla_workload_reduced(bpa, ora):
    # the separate-value-head-dim workload (d_qk 128, d_v 64, causal) on a reduced
    # sequence and head count with the same recipe and GQA ratio 16
    w = W.MLA_CAUSAL
    q, k, v, do, bias = W.make_inputs(w, B=1, S=1024, Hq=16, Hkv=1)
    assert v.shape[-1] == 64 and do.shape[-1] == 64
    from dataclasses import replace
    o, m, l, (dq, dk, dv) = _run(bpa, replace(w, B=1, S=1024, Hq=16, Hkv=1), q, k, v, do, bias)
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, causal=True)
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)
    assert rel_l2(host(dq), rq) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dk), rk) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dv), rv) <= BF16_GRAD_REL_L2


@pytest.mark.slow
def test_mla_workload_full_size_sampled(bpa, ora):
    # full size (B 2, S 4096, Hq 128, Hkv 8, d_qk 128, d_v 64, causal): sampled query rows
    # (O, m, l, dQ) and sampled keys (dK, dV) against the oracle
    w = W.MLA_CAUSAL
    q, k, v, do, bias = W.make_inputs(w)
    o, m, l, (dq, dk, dv) = _run(bpa, w, q, k, v, do, bias)
    assert tuple(o.shape) == (w.B, w.S, w.Hq, 64) and tuple(dv.shape) == (w.B, w.S, w.Hkv, 64)
    rng = np.random.default_rng(2027)
    qs = sorted({0, 1, 127, 128, 129, w.S - 1} | set(rng.integers(0, w.S, 60).tolist()))
    rows = [(int(rng.integers(0, w.B)), int(rng.integers(0, w.Hq)), qq) for qq in qs]
    ro, rm, rl, rdq = ora.rows(q, k, v, do, rows, causal=True)
    ho, hdq = o.cpu(), dq.cpu()
    go = np.stack([ho[b, s, h].float().numpy() for b, h, s in rows])
    gdq = np.stack([hdq[b, s, h].float().numpy() for b, h, s in rows])
    assert max_abs(go, ro) <= BF16_O_MAX_ABS
    gm = np.array([m[b, h, s].item() for b, h, s in rows])
    gl = np.array([l[b, h, s].item() for b, h, s in rows])
    assert np.max(np.abs(gm - rm) / (1 + np.abs(rm))) <= 1e-3
    assert np.max(np.abs(gl - rl) / np.abs(rl)) <= 1e-3
    assert rel_l2(gdq, rdq) <= BF16_GRAD_REL_L2
    keys = sorted({0, 1, 127, 128, w.S - 1} | set(rng.integers(0, w.S, 20).tolist()))
    b, g = 1, 5
    rdk, rdv = ora.keys(q, k, v, do, b, g, keys, causal=True)
    assert rel_l2(dk[b, keys, g].float().cpu().numpy(), rdk) <= BF16_GRAD_REL_L2
    assert rel_l2(dv[b, keys, g].float().cpu().numpy(), rdv) <= BF16_GRAD_REL_L2
