"""GPU parity of libbpa against the float64 oracle on small seeded problems.

Every call goes through the C ABI (ring_attention_gb300.bpa is ctypes
marshalling only).  Sizes span several 128-row tiles and ragged tails, and
the mask / bias / GQA / head-dim combinations the method has.
"""
import numpy as np
import pytest
import torch

from ring_attention_gb300.inputs import draw
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


SHAPES = [  # B, S, Hq, Hkv, d
    (1, 1, 1, 1, 64),
    (1, 17, 2, 1, 128),
    (2, 128, 4, 2, 64),
    (1, 129, 4, 4, 128),
    (2, 300, 8, 2, 128),
    (1, 640, 16, 4, 64),
]
MASKS = [
    dict(causal=True, window=(-1, -1)),
    dict(causal=False, window=(-1, -1)),
    dict(causal=True, window=(7, 0)),
    dict(causal=False, window=(64, 64)),
    dict(causal=False, window=(0, 0)),
    dict(causal=True, window=(130, 0)),
]


def _mask_id(m):
    return f"c{int(m['causal'])}_w{m['window'][0]}_{m['window'][1]}"


def _inputs(shape, seed, dtype="bf16", backward=True):
    B, S, Hq, Hkv, d = shape
    shapes = [(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, d)] + ([(B, S, Hq, d)] if backward else [])
    return draw(shapes, seed, dtype)


def _bias(kind, B, Hq, S, seed):
    rng = np.random.default_rng(seed)
    if kind == "none":
        return None
    if kind == "keys":
        return rng.standard_normal((1, 1, 1, S)).astype(np.float32)
    return rng.standard_normal((B, Hq, S, S)).astype(np.float32)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mask", MASKS, ids=_mask_id)
@pytest.mark.parametrize("bias_kind", ["none", "keys"])
def test_forward_bf16(bpa, ora, shape, mask, bias_kind):
    B, S, Hq, Hkv, d = shape
    q, k, v = _inputs(shape, 11 + S, backward=False)
    bias = _bias(bias_kind, B, Hq, S, 5)
    o, m, l = bpa.bpa_fwd(dev(q), dev(k), dev(v), bias=None if bias is None else dev(bias), **mask)
    torch.cuda.synchronize()
    oo, om, ol = ora.attention_fwd(q, k, v, bias=bias, **mask)
    assert max_abs(host(o), oo) <= BF16_O_MAX_ABS
    check_stats(m, l, om, ol)


def test_forward_full_bias_and_strided_views(bpa, ora):
    # q, k, v as views into one packed [B, S, Hq + 2 Hkv, d] tensor; a full [B, Hq, S, S] bias
    B, S, Hq, Hkv, d = 2, 200, 4, 2, 128
    (packed,) = draw([(B, S, Hq + 2 * Hkv, d)], 77, "bf16")
    bias = _bias("full", B, Hq, S, 78)
    t = dev(packed)
    q, k, v = t[:, :, :Hq], t[:, :, Hq:Hq + Hkv], t[:, :, Hq + Hkv:]
    o, m, l = bpa.bpa_fwd(q, k, v, causal=True, bias=dev(bias))
    torch.cuda.synchronize()
    oo, om, ol = ora.attention_fwd(np.ascontiguousarray(packed[:, :, :Hq]),
                                   np.ascontiguousarray(packed[:, :, Hq:Hq + Hkv]),
                                   np.ascontiguousarray(packed[:, :, Hq + Hkv:]), causal=True, bias=bias)
    assert max_abs(host(o), oo) <= BF16_O_MAX_ABS
    check_stats(m, l, om, ol)


@pytest.mark.parametrize("shape", SHAPES[1:], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mask", [MASKS[0], MASKS[2], MASKS[3]], ids=_mask_id)
def test_backward_bf16(bpa, ora, shape, mask):
    B, S, Hq, Hkv, d = shape
    q, k, v, do = _inputs(shape, 21 + S)
    bias = _bias("keys", B, Hq, S, 6)
    tq, tk, tv, tdo, tb = dev(q), dev(k), dev(v), dev(do), dev(bias)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, bias=tb, **mask)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, bias=tb, **mask)
    torch.cuda.synchronize()
    rq, rk, rv, *_ = ora.attention_bwd(q, k, v, do, bias=bias, **mask)
    assert rel_l2(host(dq), rq) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dk), rk) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dv), rv) <= BF16_GRAD_REL_L2


BAND_CASES = [  # (B, S, Hq, Hkv, d), mask: windows of at most one tile, grouped heads
    ((1, 1024, 32, 2, 128), dict(causal=True, window=(128, 0))),
    ((2, 1000, 8, 4, 128), dict(causal=True, window=(128, 0))),
    ((1, 700, 4, 2, 64), dict(causal=True, window=(7, 0))),
    ((2, 300, 4, 1, 128), dict(causal=False, window=(0, 0))),
    ((1, 520, 6, 3, 128), dict(causal=False, window=(64, 0))),
    ((1, 640, 4, 2, 64), dict(causal=False, window=(0, 100))),
    ((1, 130, 2, 1, 128), dict(causal=True, window=(128, 0))),
]


@pytest.mark.parametrize("case", BAND_CASES, ids=lambda c: "x".join(map(str, c[0])) + "_" + _mask_id(c[1]))
def test_band_forward(bpa, ora, case):
    # narrow windows with grouped heads take the band kernel (key / value tiles resident
    # while the group's heads pass, static per-CTA shares): several CTAs share one group,
    # groups straddle CTAs, ragged tails
    shape, mask = case
    B, S, Hq, Hkv, d = shape
    q, k, v = _inputs(shape, 81 + S, backward=False)
    o, m, l = bpa.bpa_fwd(dev(q), dev(k), dev(v), **mask)
    torch.cuda.synchronize()
    oo, om, ol = ora.attention_fwd(q, k, v, **mask)
    assert max_abs(host(o), oo) <= BF16_O_MAX_ABS
    check_stats(m, l, om, ol)


BAND_BWD_CASES = [  # (B, S, Hq, Hkv), mask: every 64-row query tile seen by at most two key tiles
    ((1, 1024, 32, 2), dict(causal=True, window=(128, 0))),
    ((2, 1000, 8, 4), dict(causal=True, window=(128, 0))),
    ((1, 700, 4, 4), dict(causal=True, window=(7, 0))),
    ((2, 300, 4, 1), dict(causal=False, window=(0, 0))),
    ((1, 520, 6, 3), dict(causal=False, window=(64, 0))),
    ((1, 640, 4, 2), dict(causal=False, window=(0, 60))),
    ((1, 130, 2, 1), dict(causal=True, window=(128, 0))),
]


@pytest.mark.parametrize("case", BAND_BWD_CASES, ids=lambda c: "x".join(map(str, c[0])) + "_" + _mask_id(c[1]))
@pytest.mark.parametrize("bias_kind", ["none", "keys"])
def test_band_backward(bpa, ora, case, bias_kind):
    # narrow windows: dQ is added in bf16 pairs straight into dq (at most two key tiles
    # contribute to any element, so the result does not depend on their order)
    (B, S, Hq, Hkv), mask = case
    d = 128
    q, k, v, do = _inputs((B, S, Hq, Hkv, d), 91 + S)
    bias = _bias(bias_kind, B, Hq, S, 92)
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    tb = None if bias is None else dev(bias)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, bias=tb, **mask)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, bias=tb, **mask)
    dq2, dk2, dv2 = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, bias=tb, **mask)
    torch.cuda.synchronize()
    rq, rk, rv, *_ = ora.attention_bwd(q, k, v, do, bias=bias, **mask)
    assert rel_l2(host(dq), rq) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dk), rk) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dv), rv) <= BF16_GRAD_REL_L2
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


SPLIT_CASES = [  # (B, S, Hq, Hkv, d), mask: groups of eight or more q heads split over two CTAs
    ((1, 300, 16, 2, 128), dict(causal=True, window=(-1, -1))),
    ((2, 257, 8, 1, 128), dict(causal=True, window=(100, 0))),    # the band backward
    ((1, 600, 8, 1, 128), dict(causal=True, window=(300, 0))),
    ((1, 384, 16, 1, 128), dict(causal=False, window=(-1, -1))),
]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=lambda c: "x".join(map(str, c[0])) + "_" + _mask_id(c[1]))
@pytest.mark.parametrize("deterministic", [False, True])
def test_backward_head_split(bpa, ora, case, deterministic):
    # a kv head with at least eight q heads: two CTAs per key tile take half the heads each and
    # add their dK, dV halves in bf16 pairs into the zeroed dk, dv (two contributions, so the
    # result is repeatable); a strided dk / dv view keeps the single-CTA path
    shape, mask = case
    q, k, v, do = _inputs(shape, 97 + shape[1])
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, **mask)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, deterministic=deterministic, **mask)
    dq2, dk2, dv2 = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, deterministic=deterministic, **mask)
    # k, v (and so dk, dv) as views with a row stride of 2 d: not contiguous, no split
    big_k = torch.zeros(shape[0], shape[1], shape[3], 2 * shape[4], dtype=tk.dtype, device=tk.device)
    big_v = torch.zeros_like(big_k)
    big_k[..., :shape[4]] = tk
    big_v[..., :shape[4]] = tv
    _, dk3, dv3 = bpa.bpa_bwd(tq, big_k[..., :shape[4]], big_v[..., :shape[4]], o, tdo, m, l,
                              deterministic=deterministic, **mask)
    torch.cuda.synchronize()
    rq, rk, rv, *_ = ora.attention_bwd(q, k, v, do, **mask)
    assert rel_l2(host(dq), rq) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dk), rk) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dv), rv) <= BF16_GRAD_REL_L2
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    if deterministic:
        assert torch.equal(dq, dq2)
    assert rel_l2(host(dk3), rk) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dv3), rv) <= BF16_GRAD_REL_L2


def _general_bias(kind, B, Hq, S, seed):
    # bpt.py's bias takes each dim as 1 (broadcast) or full: a bias that depends on the
    # query position ([B, Hq, S, S] or a per-row [B, 1, S, 1]) reaches the backward
    # kernels' query-dependent branch
    rng = np.random.default_rng(seed)
    shape = {"full": (B, Hq, S, S), "rows": (B, 1, S, 1)}[kind]
    return rng.standard_normal(shape).astype(np.float32)


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("mask", [MASKS[0], MASKS[3]], ids=_mask_id)
@pytest.mark.parametrize("bias_kind", ["full", "rows"])
def test_backward_general_bias_bf16(bpa, ora, d, mask, bias_kind):
    B, S, Hq, Hkv = 2, 300, 4, 2
    q, k, v, do = _inputs((B, S, Hq, Hkv, d), 51 + d)
    bias = _general_bias(bias_kind, B, Hq, S, 52)
    tq, tk, tv, tdo, tb = dev(q), dev(k), dev(v), dev(do), dev(bias)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, bias=tb, **mask)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, bias=tb, **mask)
    torch.cuda.synchronize()
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, bias=bias, **mask)
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)
    assert rel_l2(host(dq), rq) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dk), rk) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dv), rv) <= BF16_GRAD_REL_L2


@pytest.mark.parametrize("mask", [MASKS[0], MASKS[3]], ids=_mask_id)
@pytest.mark.parametrize("bias_kind", ["full", "rows"])
def test_backward_general_bias_fp32(bpa, ora, mask, bias_kind):
    B, S, Hq, Hkv, d = 2, 300, 4, 2, 64
    q, k, v, do = _inputs((B, S, Hq, Hkv, d), 53, dtype="f32")
    bias = _general_bias(bias_kind, B, Hq, S, 54)
    tq, tk, tv, tdo, tb = dev(q), dev(k), dev(v), dev(do), dev(bias)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, bias=tb, **mask)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, bias=tb, **mask)
    torch.cuda.synchronize()
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, bias=bias, **mask)
    assert max_abs(host(o), ro) <= FP32_MAX_ABS
    assert max_abs(host(dq), rq) <= FP32_MAX_ABS
    assert max_abs(host(dk), rk) <= FP32_MAX_ABS
    assert max_abs(host(dv), rv) <= FP32_MAX_ABS
    check_stats(m, l, rm, rl)


@pytest.mark.parametrize("mask", [MASKS[0], MASKS[3], MASKS[4]], ids=_mask_id)
def test_fp32_forward_backward(bpa, ora, mask):
    shape = (2, 150, 4, 2, 64)
    q, k, v, do = _inputs(shape, 31, dtype="f32")
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, **mask)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, **mask)
    torch.cuda.synchronize()
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, **mask)
    assert max_abs(host(o), ro) <= FP32_MAX_ABS
    assert max_abs(host(dq), rq) <= FP32_MAX_ABS
    assert max_abs(host(dk), rk) <= FP32_MAX_ABS
    assert max_abs(host(dv), rv) <= FP32_MAX_ABS
    check_stats(m, l, rm, rl)


@pytest.mark.parametrize("ring", [2, 4, 8])
def test_ring_forward_equals_one_shot(bpa, ora, ring):
    B, S, Hq, Hkv, d = 1, 1024, 4, 2, 128
    q, k, v = _inputs((B, S, Hq, Hkv, d), 41, backward=False)
    bias = np.zeros((1, 1, 1, S), np.float32)
    bias[..., -32:] = -1e9
    o, m, l = bpa.bpa_fwd(dev(q), dev(k), dev(v), causal=True, bias=dev(bias), ring_size=ring,
                          query_chunk=S // ring // 2, key_chunk=S // ring)
    torch.cuda.synchronize()
    oo, om, ol = ora.attention_fwd(q, k, v, causal=True, bias=bias)
    assert max_abs(host(o), oo) <= BF16_O_MAX_ABS
    check_stats(m, l, om, ol)


def test_ring_sweep_resumes_from_carry(bpa):
    B, S, Hq, Hkv, d = 1, 1024, 4, 2, 64
    q, k, v = (dev(x) for x in _inputs((B, S, Hq, Hkv, d), 42, backward=False))
    full = bpa.bpa_fwd(q, k, v, causal=True, ring_size=8)
    D = bpa.make_desc(q, k, v, causal=True, ring_size=8)
    ws = bpa.workspace(bpa.bpa_workspace_size(bpa.BPA_OP_FWD, D), q.device)
    o = torch.empty_like(q)
    m = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    l = torch.empty_like(m)
    for steps in ((0, 3), (3, 5), (5, 8)):
        bpa.bpa_fwd(q, k, v, causal=True, ring_size=8, ring_steps=steps, o=o, m=m, l=l, workspace_buf=ws)
    torch.cuda.synchronize()
    bpa.bpa_check(ws)
    assert torch.equal(o, full[0]) and torch.equal(m, full[1]) and torch.equal(l, full[2])


@pytest.mark.parametrize("ring", [2, 4])
def test_ring_backward(bpa, ora, ring):
    B, S, Hq, Hkv, d = 1, 512, 4, 2, 128
    q, k, v, do = _inputs((B, S, Hq, Hkv, d), 43)
    bias = np.zeros((1, 1, 1, S), np.float32)
    bias[..., -16:] = -1e9
    tq, tk, tv, tdo, tb = dev(q), dev(k), dev(v), dev(do), dev(bias)
    kw = dict(causal=True, bias=tb, ring_size=ring)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, **kw)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, **kw)
    torch.cuda.synchronize()
    rq, rk, rv, *_ = ora.attention_bwd(q, k, v, do, causal=True, bias=bias)
    assert rel_l2(host(dq), rq) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dk), rk) <= BF16_GRAD_REL_L2
    assert rel_l2(host(dv), rv) <= BF16_GRAD_REL_L2


@pytest.mark.parametrize("dims", [(1, 256, 2, 16, 4, 3), (2, 1024, 4, 64, 32, 8), (1, 96, 1, 8, 32, 64)])
def test_select_blocks_bit_exact(bpa, ora, dims):
    B, S, H, d, bs, n = dims
    q, k = draw([(B, S, H, d), (B, S, H, d)], 51 + S, "bf16")
    idx = bpa.bpa_select_blocks(dev(q), dev(k), block_size=bs, top_n=n)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), ora.select_blocks(q, k, block_size=bs, top_n=n))


@pytest.mark.parametrize("dims", [(1, 512, 2, 24, 64, 4, "bf16"),    # blocks of 64 rows: the column kernel
                                  (1, 256, 3, 7, 16, 3, "bf16"),     # odd head dim: one channel per thread
                                  (2, 512, 2, 40, 32, 5, "f32")])    # float32 inputs
def test_select_blocks_bit_exact_sum_paths(bpa, ora, dims):
    B, S, H, d, bs, n, dt = dims
    q, k = draw([(B, S, H, d), (B, S, H, d)], 53 + d, dt)
    idx = bpa.bpa_select_blocks(dev(q), dev(k), block_size=bs, top_n=n)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), ora.select_blocks(q, k, block_size=bs, top_n=n))


def test_select_blocks_nan_scores(bpa, ora):
    # a NaN in a key block (every score against it NaN) and one in a query block (all its
    # scores NaN): NaN ranks below every number, and no kernel access leaves its buffers
    B, S, H, d, bs, n = 1, 512, 2, 16, 16, 4
    q, k = draw([(B, S, H, d), (B, S, H, d)], 57, "f32")
    k[0, 3 * bs + 2, 0, 5] = np.nan
    q[0, 9 * bs, 1, 1] = np.nan
    q[0, 0, 0, 0] = np.nan       # block 0 of warp 0 (no candidates: all -1)
    idx = bpa.bpa_select_blocks(dev(q), dev(k), block_size=bs, top_n=n)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), ora.select_blocks(q, k, block_size=bs, top_n=n))


def test_select_blocks_near_ties(bpa, ora):
    # scores that differ far below float32 resolution (2^-30 against a magnitude of ~16):
    # the float32 pre-filter keeps them all, the float64 contract scores decide; plus exact
    # ties among them (lower block first) and random blocks the filter drops
    B, S, H, d, bs, n = 1, 1024, 2, 16, 8, 6
    rng = np.random.default_rng(58)
    q = np.zeros((B, S, H, d), np.float32)
    k = rng.standard_normal((B, S, H, d)).astype(np.float32) * 0.01
    u = rng.standard_normal(d).astype(np.float32)
    for i in range(S // bs):
        q[0, i * bs, :, :] = u
        if i % 3 == 0:   # a third of the key blocks nearly tie with each other
            k[0, i * bs:(i + 1) * bs, :, :] = 0.0
            k[0, i * bs, :, :] = u
            k[0, i * bs + 1, :, 0] = np.float32(((i * 7) % 11) * 2.0 ** -30)
    idx = bpa.bpa_select_blocks(dev(q), dev(k), block_size=bs, top_n=n)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), ora.select_blocks(q, k, block_size=bs, top_n=n))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_select_blocks_sum_rounding(bpa, ora, dtype):
    # block sums whose float64 additions in row order round (2^60 + 2 - 2^60 = 0, not 2) or
    # are exact only just inside the range the kernel sums with integers (a span of 42 bits
    # between the largest and smallest last bit for bfloat16 over 8 rows, 26 for float32)
    # and just outside it; the ranking depends on every one of these sums
    B, S, H, d, bs, n = 1, 256, 1, 16, 8, 4
    big_in, small_in = (2.0 ** 42, 1.0 + 2.0 ** -7) if dtype == "bf16" else (2.0 ** 26, 1.0 + 2.0 ** -23)
    q = np.zeros((B, S, H, d), np.float32)
    k = np.zeros((B, S, H, d), np.float32)
    q[0, ::bs, 0, 0] = 1.0
    for j in range(S // bs):
        r = j * bs
        cls = j % 4
        if cls == 0:     # rounds away: the contract sum is 0 (the exact sum, 2, would rank first)
            k[0, r:r + 3, 0, 0] = (2.0 ** 60, 2.0, -(2.0 ** 60))
        elif cls == 1:   # integer path at its widest span: big + small - big = small exactly
            k[0, r:r + 3, 0, 0] = (big_in, small_in, -big_in)
        elif cls == 2:
            k[0, r + 5, 0, 0] = 1.0
        else:            # one bit wider: the float64 additions (exact here as well)
            k[0, r:r + 3, 0, 0] = (2 * big_in, small_in, -2 * big_in)
        k[0, r + 7, 0, 1 + j % (d - 1)] = 0.25   # a second channel the query does not weigh
    if dtype == "bf16":
        q = (q.view(np.uint32) >> 16).astype(np.uint16)
        k = (k.view(np.uint32) >> 16).astype(np.uint16)
    idx = bpa.bpa_select_blocks(dev(q), dev(k), block_size=bs, top_n=n)
    torch.cuda.synchronize()
    ref = ora.select_blocks(q, k, block_size=bs, top_n=n)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)
    # the float64 additions in row order rank the boundary classes first (ties: lower block)
    # and the rounded-away class last
    assert ref[0, 0, -1].tolist() == [1, 3, 5, 7]


def test_select_blocks_ties(bpa, ora):
    # block sums with many exactly equal scores: ties must keep the lower block
    B, S, H, d, bs = 1, 256, 1, 8, 8
    q = np.zeros((B, S, H, d), np.float32)
    k = np.zeros((B, S, H, d), np.float32)
    q[0, ::bs, 0, :] = 1.0
    for j in range(S // bs):
        k[0, j * bs, 0, :] = float(j % 3)
    idx = bpa.bpa_select_blocks(dev(q), dev(k), block_size=bs, top_n=5)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), ora.select_blocks(q, k, block_size=bs, top_n=5))


def test_block_selected_attention(bpa, ora):
    B, S, H, d, bs, n = 2, 512, 2, 64, 32, 4
    q, k, v = draw([(B, S, H, d)] * 3, 61, "bf16")
    tq, tk, tv = dev(q), dev(k), dev(v)
    idx = bpa.bpa_select_blocks(tq, tk, block_size=bs, top_n=n)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, causal=True, block_idx=idx, sel_block=bs, top_n=n, local_window=32)
    torch.cuda.synchronize()
    ridx = ora.select_blocks(q, k, block_size=bs, top_n=n)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    oo, om, ol = ora.attention_fwd(q, k, v, causal=True, block_idx=ridx, sel_block=bs, top_n=n,
                                   local_window=32)
    assert max_abs(host(o), oo) <= BF16_O_MAX_ABS
    check_stats(m, l, om, ol)


def _planted_selection(B, H, S, bs, n, seed):
    """Valid block indices without running a selection: per query block up to n distinct
    strictly earlier blocks, ascending, padded with -1 (the layout bpa_select_blocks writes)."""
    rng = np.random.default_rng(seed)
    idx = np.full((B, H, S // bs, n), -1, dtype=np.int32)
    for b in range(B):
        for h in range(H):
            for i in range(S // bs):
                pick = np.sort(rng.permutation(i)[:rng.integers(0, n + 1)])
                idx[b, h, i, :len(pick)] = pick
    return idx


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_block_selected_backward(bpa, ora, dtype):
    # gradients through the gathered attention with the selection held fixed
    B, S, H, d, bs, n = 2, 512, 2, 64, 32, 4
    q, k, v, do = draw([(B, S, H, d)] * 4, 62, dtype)
    tq, tk, tv = dev(q), dev(k), dev(v)
    idx = bpa.bpa_select_blocks(tq, tk, block_size=bs, top_n=n)
    kw = dict(causal=True, sel_block=bs, top_n=n, local_window=32)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, block_idx=idx, **kw)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, dev(do), m, l, block_idx=idx, **kw)
    torch.cuda.synchronize()
    ridx = ora.select_blocks(q, k, block_size=bs, top_n=n)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, block_idx=ridx, **kw)
    check_stats(m, l, rm, rl)
    if dtype == "f32":
        for got, ref in ((o, ro), (dq, rq), (dk, rk), (dv, rv)):
            assert max_abs(host(got), ref) <= FP32_MAX_ABS
    else:
        for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
            assert rel_l2(host(got), ref) <= BF16_GRAD_REL_L2


@pytest.mark.parametrize("geom", [(336, 16, 3, 20), (320, 32, 8, 0), (320, 64, 2, 100)],
                         ids=lambda g: "S%d_bs%d_n%d_w%d" % g)
def test_block_selected_backward_planted(bpa, ora, geom):
    # GQA, a per-key bias, a separate value head dim, a sequence that ends inside a
    # chunk of 32 rows (S = 336), local windows narrower and wider than a block (and
    # none), and query blocks that select nothing
    S, bs, n, lw = geom
    B, Hq, Hkv, d, dv = 1, 4, 2, 64, 32
    q, k, v, do = draw([(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, dv), (B, S, Hq, dv)], 63 + bs, "bf16")
    bias = _bias("keys", B, Hq, S, 7)
    idx = _planted_selection(B, Hq, S, bs, n, 64 + bs)
    kw = dict(causal=True, sel_block=bs, top_n=n, local_window=lw)
    tq, tk, tv, tb, ti = dev(q), dev(k), dev(v), dev(bias), torch.from_numpy(idx).cuda()
    o, m, l = bpa.bpa_fwd(tq, tk, tv, bias=tb, block_idx=ti, **kw)
    dq, dk, dvv = bpa.bpa_bwd(tq, tk, tv, o, dev(do), m, l, bias=tb, block_idx=ti, **kw)
    torch.cuda.synchronize()
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, bias=bias, block_idx=idx, **kw)
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)
    for got, ref in ((dq, rq), (dk, rk), (dvv, rv)):
        assert rel_l2(host(got), ref) <= BF16_GRAD_REL_L2


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_block_index_contract_is_checked_on_the_device(bpa, ora, dtype):
    # entries that are not -1 or an earlier block (its own block, a later block inside the
    # tensor, a block past the end, a negative value) are ignored by the kernels and
    # recorded as a device-side check failure; the index array is only read, so no access
    # goes outside a buffer even without the check
    B, H, S, bs, n, lw, d = 1, 2, 256, 32, 4, 32, 64
    q, k, v, do = draw([(B, S, H, d), (B, S, H, d), (B, S, H, d), (B, S, H, d)], 96, dtype)
    idx = _planted_selection(B, H, S, bs, n, 97)
    bad = idx.copy()
    bad[0, 0, 3, n - 1] = 3            # its own block
    bad[0, 1, 2, n - 1] = 6            # a later block, inside the tensor
    bad[0, 1, 5, n - 1] = S // bs + 5  # past the last block
    bad[0, 0, 7, n - 1] = -7
    clean = np.where((bad == -1) | ((bad >= 0) & (bad < np.arange(S // bs)[None, None, :, None])), bad, -1)
    kw = dict(causal=True, sel_block=bs, top_n=n, local_window=lw)
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    D = bpa.make_desc(tq, tk, tv, block_idx=torch.from_numpy(bad).cuda(), **kw)
    wsf = bpa.workspace(bpa.bpa_workspace_size(bpa.BPA_OP_FWD, D), tq.device)
    wsb = bpa.workspace(bpa.bpa_workspace_size(bpa.BPA_OP_BWD, D), tq.device)
    ti = torch.from_numpy(bad).cuda()
    o, m, l = bpa.bpa_fwd(tq, tk, tv, block_idx=ti, workspace_buf=wsf, **kw)
    dq, dk, dvv = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, block_idx=ti, workspace_buf=wsb, **kw)
    torch.cuda.synchronize()
    for ws in (wsf, wsb):
        with pytest.raises(bpa.BpaError) as err:
            bpa.bpa_check(ws)
        assert err.value.status == bpa.BPA_ERR_DEVICE_CHECK
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, block_idx=clean, **kw)
    if dtype == "f32":
        for got, ref in ((o, ro), (dq, rq), (dk, rk), (dvv, rv)):
            assert max_abs(host(got), ref) <= FP32_MAX_ABS
    else:
        assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
        for got, ref in ((dq, rq), (dk, rk), (dvv, rv)):
            assert rel_l2(host(got), ref) <= BF16_GRAD_REL_L2
    # a valid selection on the same workspaces clears the status
    tc = torch.from_numpy(clean).cuda()
    o, m, l = bpa.bpa_fwd(tq, tk, tv, block_idx=tc, workspace_buf=wsf, **kw)
    bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, block_idx=tc, workspace_buf=wsb, **kw)
    torch.cuda.synchronize()
    bpa.bpa_check(wsf)
    bpa.bpa_check(wsb)


@pytest.mark.parametrize("lw", [0, 20, 64])
def test_block_selected_backward_gathered(bpa, ora, lw):
    # the shapes the gathered kernels take (bf16, d = d_v = 64, 32-row blocks, no bias):
    # GQA, planted selections with -1 padding and blocks shared by many query blocks,
    # local windows of none, part of a block and two blocks
    B, S, Hq, Hkv, d, bs, n = 2, 384, 4, 2, 64, 32, 5
    q, k, v, do = draw([(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, d), (B, S, Hq, d)], 65 + lw, "bf16")
    idx = _planted_selection(B, Hq, S, bs, n, 66 + lw)
    kw = dict(causal=True, sel_block=bs, top_n=n, local_window=lw)
    tq, tk, tv, ti = dev(q), dev(k), dev(v), torch.from_numpy(idx).cuda()
    o, m, l = bpa.bpa_fwd(tq, tk, tv, block_idx=ti, **kw)
    dq, dk, dvv = bpa.bpa_bwd(tq, tk, tv, o, dev(do), m, l, block_idx=ti, **kw)
    torch.cuda.synchronize()
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, block_idx=idx, **kw)
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)
    for got, ref in ((dq, rq), (dk, rk), (dvv, rv)):
        assert rel_l2(host(got), ref) <= BF16_GRAD_REL_L2
    # rows with no allowed key (first query block without a local window) have zero dQ
    if lw == 0:
        assert float(dq[:, :bs].abs().max()) == 0.0


@pytest.mark.parametrize("d", [128, 256, 512])
def test_block_selected_wide_heads(bpa, ora, d):
    # the joint view: the channels of all heads read as fewer, wider heads (512 = H d),
    # selection on the wide block sums, forward and backward on the channel-split gather
    B, S, C = 1, 512, 512
    H, bs, n = C // d, 32, 6
    q, k, v, do = (x.reshape(B, S, H, d) for x in draw([(B, S, 8, 64)] * 4, 67, "bf16"))
    tq, tk, tv = dev(q), dev(k), dev(v)
    idx = bpa.bpa_select_blocks(tq, tk, block_size=bs, top_n=n)
    kw = dict(causal=True, sel_block=bs, top_n=n, local_window=32)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, block_idx=idx, **kw)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, dev(do), m, l, block_idx=idx, **kw)
    torch.cuda.synchronize()
    ridx = ora.select_blocks(q, k, block_size=bs, top_n=n)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, block_idx=ridx, **kw)
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert rel_l2(host(got), ref) <= BF16_GRAD_REL_L2


def test_block_selected_wide_heads_gqa_planted(bpa, ora):
    # channel-split gather with GQA (4 q heads on 2 kv heads of 128 channels), planted
    # selections and a local window of part of a block
    B, S, Hq, Hkv, d, bs, n, lw = 2, 256, 4, 2, 128, 32, 4, 20
    q, k, v, do = draw([(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, d), (B, S, Hq, d)], 68, "bf16")
    idx = _planted_selection(B, Hq, S, bs, n, 69)
    kw = dict(causal=True, sel_block=bs, top_n=n, local_window=lw)
    tq, tk, tv, ti = dev(q), dev(k), dev(v), torch.from_numpy(idx).cuda()
    o, m, l = bpa.bpa_fwd(tq, tk, tv, block_idx=ti, **kw)
    dq, dk, dvv = bpa.bpa_bwd(tq, tk, tv, o, dev(do), m, l, block_idx=ti, **kw)
    torch.cuda.synchronize()
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, block_idx=idx, **kw)
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)
    for got, ref in ((dq, rq), (dk, rk), (dvv, rv)):
        assert rel_l2(host(got), ref) <= BF16_GRAD_REL_L2


def test_fp32_head_dim_512(bpa, ora):
    # the CUDA-core kernels with 16 channels per lane
    B, S, Hq, Hkv, d = 1, 70, 2, 1, 512
    q, k, v, do = draw([(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, d), (B, S, Hq, d)], 70, "f32")
    tq, tk, tv = dev(q), dev(k), dev(v)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, causal=True)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, dev(do), m, l, causal=True)
    torch.cuda.synchronize()
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, causal=True)
    check_stats(m, l, rm, rl)
    for got, ref in ((o, ro), (dq, rq), (dk, rk), (dv, rv)):
        assert max_abs(host(got), ref) <= FP32_MAX_ABS


VARLEN = [   # (query lengths, key lengths or None, bottom-right)
    ([300, 129, 1, 0], None, False),
    ([300, 77, 256, 5], [300, 200, 129, 0], False),
    ([64, 129, 300, 2], [300, 131, 257, 300], True),
    ([300, 200, 17, 128], [150, 128, 3, 300], True),
]


@pytest.mark.parametrize("case", VARLEN, ids=["same", "topleft", "bottomright", "bottomright_short_keys"])
@pytest.mark.parametrize("mask", [MASKS[0], MASKS[1], MASKS[2], MASKS[3]], ids=_mask_id)
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 64)], ids=["bf16_d128", "bf16_d64", "f32"])
def test_variable_lengths(bpa, ora, case, mask, dtype, d):
    # padded batches: per-entry query / key lengths crossing tile boundaries, empty
    # entries, both diagonal alignments; the padding holds random finite numbers
    lq, lk, br = case
    B, S, Hq, Hkv = 4, 300, 4, 2
    q, k, v, do = draw([(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, d), (B, S, Hq, d)], 81 + d, dtype)
    tlq = torch.tensor(lq, dtype=torch.int32, device="cuda")
    tlk = None if lk is None else torch.tensor(lk, dtype=torch.int32, device="cuda")
    kw = dict(seqlens_q=tlq, seqlens_kv=tlk, bottom_right=br, **mask)
    tq, tk, tv = dev(q), dev(k), dev(v)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, **kw)
    dq, dk, dvv = bpa.bpa_bwd(tq, tk, tv, o, dev(do), m, l, **kw)
    torch.cuda.synchronize()
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, seqlens_q=lq, seqlens_kv=lk, bottom_right=br, **mask)
    check_stats(m, l, rm, rl)
    if dtype == "f32":
        for got, ref in ((o, ro), (dq, rq), (dk, rk), (dvv, rv)):
            assert max_abs(host(got), ref) <= FP32_MAX_ABS
    else:
        assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
        for got, ref in ((dq, rq), (dk, rk), (dvv, rv)):
            assert rel_l2(host(got), ref) <= BF16_GRAD_REL_L2
    # padding rows are exactly zero
    lkk = lq if lk is None else lk
    for b in range(B):
        assert float(o[b, lq[b]:].abs().max() if lq[b] < S else 0) == 0.0
        assert float(dq[b, lq[b]:].abs().max() if lq[b] < S else 0) == 0.0
        assert float(dk[b, lkk[b]:].abs().max() if lkk[b] < S else 0) == 0.0
        assert float(dvv[b, lkk[b]:].abs().max() if lkk[b] < S else 0) == 0.0


@pytest.mark.parametrize("path", ["tc_d128", "tc_d64_swa", "f32", "gather", "varlen"])
def test_sink_attention(bpa, ora, path):
    # sink logits per q head (a "learnable" set, one of them 0 as in off_by_one) on the
    # tensor-core, CUDA-core and gathered forwards, and the sink gradient
    B, S, Hq, Hkv = 2, 300, 4, 2
    d = 128 if path == "tc_d128" else 64
    dtype = "f32" if path == "f32" else "bf16"
    q, k, v, do = draw([(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, d), (B, S, Hq, d)], 90 + d, dtype)
    sink = np.array([0.0, 1.5, -2.0, 4.0])
    kw, okw = dict(causal=True), dict(causal=True)
    if path == "tc_d64_swa":
        kw["window"] = okw["window"] = (40, 0)
    if path == "gather":   # block-selected, d = 64: rows of the first block see no key
        q, k, v, do = (np.ascontiguousarray(x[:, :288]) for x in (q, k, v, do))
        idx = _planted_selection(B, Hq, 288, 32, 3, 92)
        kw.update(block_idx=torch.from_numpy(idx).cuda(), sel_block=32, top_n=3, local_window=0)
        okw.update(block_idx=idx, sel_block=32, top_n=3, local_window=0)
    if path == "varlen":
        lens = [300, 131]
        kw["seqlens_q"] = torch.tensor(lens, dtype=torch.int32, device="cuda")
        okw["seqlens_q"] = lens
    tsink = torch.tensor(sink, dtype=torch.float32, device="cuda")
    tds = torch.zeros(Hq, dtype=torch.float32, device="cuda")
    tq, tk, tv = dev(q), dev(k), dev(v)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, sink=tsink, **kw)
    dq, dk, dvv = bpa.bpa_bwd(tq, tk, tv, o, dev(do), m, l, sink=tsink, dsink=tds, **kw)
    torch.cuda.synchronize()
    rq, rk, rv, ro, rm, rl, rds = ora.attention_bwd(q, k, v, do, sink=sink, want_dsink=True, **okw)
    check_stats(m, l, rm, rl)
    if dtype == "f32":
        for got, ref in ((o, ro), (dq, rq), (dk, rk), (dvv, rv)):
            assert max_abs(host(got), ref) <= FP32_MAX_ABS
        assert rel_l2(host(tds), rds) <= 1e-5
    else:
        assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
        for got, ref in ((dq, rq), (dk, rk), (dvv, rv)):
            assert rel_l2(host(got), ref) <= BF16_GRAD_REL_L2
        assert rel_l2(host(tds), rds) <= BF16_GRAD_REL_L2


@pytest.mark.parametrize("case", ["causal", "swa_gqa4", "varlen", "f32", "block_selected"])
def test_deterministic_backward(bpa, ora, case):
    # the determinism knob: two backward calls give bit-identical gradients, and they match
    # the oracle like the default mode
    B, S, Hq, Hkv, d = 2, 300, 8, 2, 128
    dtype, kw, okw = "bf16", dict(causal=True), dict(causal=True)
    if case == "swa_gqa4":
        kw["window"] = okw["window"] = (70, 0)
    if case == "f32":
        dtype, d = "f32", 64
    if case == "block_selected":
        S, Hkv, d = 256, 8, 64
        idx = _planted_selection(B, Hq, S, 32, 3, 93)
        kw.update(block_idx=torch.from_numpy(idx).cuda(), sel_block=32, top_n=3, local_window=32)
        okw.update(block_idx=idx, sel_block=32, top_n=3, local_window=32)
    if case == "varlen":
        kw["seqlens_q"] = torch.tensor([300, 170], dtype=torch.int32, device="cuda")
        okw["seqlens_q"] = [300, 170]
    q, k, v, do = draw([(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, d), (B, S, Hq, d)], 94 + d, dtype)
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, **kw)
    g1 = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, deterministic=True, **kw)
    g2 = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, deterministic=True, **kw)
    torch.cuda.synchronize()
    for x, y in zip(g1, g2):
        assert torch.equal(x, y)
    rq, rk, rv, *_ = ora.attention_bwd(q, k, v, do, **okw)
    for got, ref in zip(g1, (rq, rk, rv)):
        if dtype == "f32":
            assert max_abs(host(got), ref) <= FP32_MAX_ABS
        else:
            assert rel_l2(host(got), ref) <= BF16_GRAD_REL_L2


def test_bounded_wait_reports_timeout(bpa):
    ws = bpa.workspace(256, "cuda")
    bpa.bpa_debug_wait_timeout(ws, 200_000_000)   # 0.2 s
    torch.cuda.synchronize()
    with pytest.raises(bpa.BpaError) as e:
        bpa.bpa_check(ws)
    assert e.value.status == bpa.BPA_ERR_TIMEOUT
    # the context is still usable afterwards
    x = torch.ones(4, device="cuda")
    assert float((x + 1).sum()) == 8.0


def test_status_clean_after_normal_call(bpa):
    q, k, v = (dev(x) for x in _inputs((1, 256, 2, 2, 128), 71, backward=False))
    D = bpa.make_desc(q, k, v, causal=True)
    ws = bpa.workspace(bpa.bpa_workspace_size(bpa.BPA_OP_FWD, D), q.device)
    bpa.bpa_fwd(q, k, v, causal=True, workspace_buf=ws)
    torch.cuda.synchronize()
    bpa.bpa_check(ws)


# ---- separate value head dim (q, k with d channels; v, o, dO with dv) ----------------------
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dims", [(128, 64), (64, 128), (96, 32)], ids=lambda d: f"d{d[0]}_dv{d[1]}")
@pytest.mark.parametrize("mask", [dict(causal=True, window=(-1, -1)), dict(causal=False, window=(40, 9))],
                         ids=_mask_id)
def test_separate_value_head_dim(bpa, ora, dtype, dims, mask):
    d, dv = dims
    B, S, Hq, Hkv = 2, 150, 4, 2
    q, k, v, do = draw([(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, dv), (B, S, Hq, dv)], 71 + d + dv, dtype)
    tq, tk, tv = dev(q), dev(k), dev(v)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, **mask)
    assert tuple(o.shape) == (B, S, Hq, dv)
    dq, dk, dvv = bpa.bpa_bwd(tq, tk, tv, o, dev(do), m, l, **mask)
    torch.cuda.synchronize()
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, **mask)
    check_stats(m, l, rm, rl)
    if dtype == "f32":
        for got, ref in ((o, ro), (dq, rq), (dk, rk), (dvv, rv)):
            assert max_abs(host(got), ref) <= FP32_MAX_ABS
    else:
        assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
        for got, ref in ((dq, rq), (dk, rk), (dvv, rv)):
            assert rel_l2(host(got), ref) <= BF16_GRAD_REL_L2


def test_output_strides_differ_from_query_strides(bpa, ora):
    # o and dO as views into a wider [B, S, Hq, 2 dv] buffer: their strides are their own
    B, S, Hq, Hkv, d, dv = 1, 130, 4, 2, 128, 64
    q, k, v, do = draw([(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, dv), (B, S, Hq, dv)], 83, "bf16")
    tq, tk, tv = dev(q), dev(k), dev(v)
    obuf = torch.zeros((B, S, Hq, 2 * dv), dtype=torch.bfloat16, device="cuda")
    o = obuf[..., dv:]
    dobuf = torch.zeros((B, S, Hq, 2 * dv), dtype=torch.bfloat16, device="cuda")
    dobuf[..., dv:] = dev(do)
    tdo = dobuf[..., dv:]
    _, m, l = bpa.bpa_fwd(tq, tk, tv, o=o, causal=True)
    dq, dk, dvv = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, causal=True)
    torch.cuda.synchronize()
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, causal=True)
    assert float(obuf[..., :dv].abs().max()) == 0.0      # nothing written outside the view
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)
    for got, ref in ((dq, rq), (dk, rk), (dvv, rv)):
        assert rel_l2(host(got), ref) <= BF16_GRAD_REL_L2
