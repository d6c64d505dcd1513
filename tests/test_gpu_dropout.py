"""GPU parity of attention dropout (bpt.py: each score entry is dropped with probability p
and leaves the softmax; no 1/(1-p) factor) against the float64 oracle.

The decisions are integers (a Philox4x32-10 draw compared with round(p * 2^32)), so the
kernels' kept / dropped entries must equal the oracle's bit for bit.  They are read back
through the outputs with inputs that expose P: with Q = 0 every kept entry of a row has the
same weight 1 / (kept keys), so one-hot V rows put each key's decision into its own output
channel (forward), and one-hot dO rows put each query's decision into its own dV channel
(backward).  Beside that, O, m, l and the gradients must match the oracle's attention with
the same dropout at the usual tolerances on every path: tensor-core (d 128, d 64, separate
value head dim, ring sweep), CUDA-core fp32 and the gathered block-selected kernels.
"""
import numpy as np
import pytest
import torch

from ring_attention_gb300.inputs import draw, to_bf16_bits
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


def _bf16(x):
    return to_bf16_bits(np.ascontiguousarray(x, dtype=np.float32))


def _oracle_keep(ora, B, H, S, p, seed):
    return np.stack([np.stack([ora.dropout_keep(S, b, h, dropout_p=p, dropout_seed=seed) for h in range(H)])
                     for b in range(B)]).astype(bool)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("p,seed", [(0.3, 7), (0.75, 2 ** 40 + 12345)])
def test_forward_decisions_equal_the_oracle(bpa, ora, dtype, p, seed):
    # S = 256 keys in two 128-key tiles; V row k = (1 + k // 128) * e_(k % 128): output
    # channel c of row q carries keep(q, c) + 2 keep(q, c + 128), scaled by 1 / l
    B, S, H, d = 2, 256, 3, 128
    q = np.zeros((B, S, H, d), np.float32)
    k = np.zeros((B, S, H, d), np.float32)
    v = np.zeros((B, S, H, d), np.float32)
    for kk in range(S):
        v[:, kk, :, kk % 128] = 1.0 + kk // 128
    enc = (lambda x: x) if dtype == "f32" else _bf16
    o, m, l = bpa.bpa_fwd(dev(enc(q)), dev(enc(k)), dev(enc(v)), dropout_p=p, dropout_seed=seed)
    torch.cuda.synchronize()
    code = np.rint(host(o) * np.transpose(host(l), (0, 2, 1))[..., None]).astype(int)   # [B, S, H, 128]
    keep = _oracle_keep(ora, B, H, S, p, seed)                                           # [B, H, q, k]
    want = keep[..., :128].astype(int) + 2 * keep[..., 128:].astype(int)
    np.testing.assert_array_equal(np.transpose(code, (0, 2, 1, 3)), want)
    np.testing.assert_array_equal(host(l), keep.sum(-1))


@pytest.mark.parametrize("p,seed", [(0.3, 11), (0.6, 3 * 2 ** 33 + 5)])
def test_backward_decisions_equal_the_oracle(bpa, ora, p, seed):
    # Q = 0 and dO row q = e_q: dV[k, c] = P[c, k] = keep(c, k) / l_c, so the backward's
    # recomputed decisions show in dV (one kv head per q head)
    B, S, H, d = 2, 128, 2, 128
    q = np.zeros((B, S, H, d), np.float32)
    k = draw([(B, S, H, d)], 61, "f32")[0]
    v = draw([(B, S, H, d)], 62, "f32")[0]
    do = np.zeros((B, S, H, d), np.float32)
    for qq in range(S):
        do[:, qq, :, qq] = 1.0
    tq, tk, tv, tdo = dev(_bf16(q)), dev(_bf16(k)), dev(_bf16(v)), dev(_bf16(do))
    o, m, l = bpa.bpa_fwd(tq, tk, tv, dropout_p=p, dropout_seed=seed)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, dropout_p=p, dropout_seed=seed)
    torch.cuda.synchronize()
    keep = _oracle_keep(ora, B, H, S, p, seed)          # [B, H, q, k]
    got = host(dv) > 0                                   # [B, k, H, c = q]
    np.testing.assert_array_equal(np.transpose(got, (0, 2, 3, 1)), keep)


def _check_fwd_bwd(bpa, ora, q, k, v, do, tol, **kw):
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, **kw)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, **kw)
    torch.cuda.synchronize()
    okw = {key: val for key, val in kw.items() if key not in ("ring_size",)}
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, **okw)
    if tol == "f32":
        for a, b in ((o, ro), (dq, rq), (dk, rk), (dv, rv)):
            assert max_abs(host(a), b) <= FP32_MAX_ABS
    else:
        assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
        assert rel_l2(host(dq), rq) <= BF16_GRAD_REL_L2
        assert rel_l2(host(dk), rk) <= BF16_GRAD_REL_L2
        assert rel_l2(host(dv), rv) <= BF16_GRAD_REL_L2
    check_stats(m, l, rm, rl)


MASKS = [dict(causal=True, window=(-1, -1)), dict(causal=False, window=(-1, -1)),
         dict(causal=False, window=(64, 64)), dict(causal=True, window=(130, 0))]


@pytest.mark.parametrize("shape", [(2, 300, 4, 2, 128), (1, 640, 8, 2, 64), (1, 200, 2, 1, 128)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mask", MASKS, ids=lambda m: f"c{int(m['causal'])}_w{m['window'][0]}_{m['window'][1]}")
def test_tensor_core_dropout_matches_oracle(bpa, ora, shape, mask):
    B, S, Hq, Hkv, d = shape
    q, k, v, do = draw([(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, d), (B, S, Hq, d)], 70 + S, "bf16")
    _check_fwd_bwd(bpa, ora, q, k, v, do, "bf16", dropout_p=0.2, dropout_seed=99 + S, **mask)


def test_tensor_core_dropout_with_bias_and_value_head_dim(bpa, ora):
    B, S, Hq, Hkv, d, dvh = 2, 256, 4, 2, 128, 64
    q, k, v, do = draw([(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, dvh), (B, S, Hq, dvh)], 71, "bf16")
    bias = np.random.default_rng(72).standard_normal((1, 1, 1, S)).astype(np.float32)
    tq, tk, tv, tdo, tb = dev(q), dev(k), dev(v), dev(do), dev(bias)
    kw = dict(causal=True, dropout_p=0.35, dropout_seed=5)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, bias=tb, **kw)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, bias=tb, **kw)
    torch.cuda.synchronize()
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, bias=bias, **kw)
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)
    for a, b in ((dq, rq), (dk, rk), (dv, rv)):
        assert rel_l2(host(a), b) <= BF16_GRAD_REL_L2


def test_ring_sweep_dropout_matches_oracle(bpa, ora):
    # the draws use global positions, so the ring's visiting order does not matter
    B, S, Hq, Hkv, d = 1, 1024, 4, 2, 128
    q, k, v, do = draw([(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, d), (B, S, Hq, d)], 73, "bf16")
    _check_fwd_bwd(bpa, ora, q, k, v, do, "bf16", causal=True, ring_size=4, dropout_p=0.1, dropout_seed=17)


@pytest.mark.parametrize("mask", MASKS[:3], ids=lambda m: f"c{int(m['causal'])}_w{m['window'][0]}_{m['window'][1]}")
def test_fp32_dropout_matches_oracle(bpa, ora, mask):
    B, S, Hq, Hkv, d = 2, 150, 4, 2, 64
    q, k, v, do = draw([(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, d), (B, S, Hq, d)], 74, "f32")
    _check_fwd_bwd(bpa, ora, q, k, v, do, "f32", dropout_p=0.25, dropout_seed=2024, **mask)


@pytest.mark.parametrize("d", [64, 128])
def test_block_selected_dropout_matches_oracle(bpa, ora, d):
    B, S, H, bs, n, lw = 2, 512, 2, 32, 4, 32
    q, k, v, do = draw([(B, S, H, d), (B, S, H, d), (B, S, H, d), (B, S, H, d)], 75 + d, "bf16")
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    idx = bpa.bpa_select_blocks(tq, tk, block_size=bs, top_n=n)
    torch.cuda.synchronize()
    ridx = ora.select_blocks(q, k, block_size=bs, top_n=n)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    kw = dict(causal=True, sel_block=bs, top_n=n, local_window=lw, dropout_p=0.3, dropout_seed=8)
    o, m, l = bpa.bpa_fwd(tq, tk, tv, block_idx=idx, **kw)
    dq, dk, dv = bpa.bpa_bwd(tq, tk, tv, o, tdo, m, l, block_idx=idx, **kw)
    torch.cuda.synchronize()
    rq, rk, rv, ro, rm, rl = ora.attention_bwd(q, k, v, do, block_idx=ridx, **kw)
    assert max_abs(host(o), ro) <= BF16_O_MAX_ABS
    check_stats(m, l, rm, rl)
    for a, b in ((dq, rq), (dk, rk), (dv, rv)):
        assert rel_l2(host(a), b) <= BF16_GRAD_REL_L2


def test_dropout_zero_is_plain_attention(bpa):
    B, S, Hq, Hkv, d = 1, 256, 4, 2, 128
    q, k, v = (dev(x) for x in draw([(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, d)], 76, "bf16"))
    o0, m0, l0 = bpa.bpa_fwd(q, k, v, causal=True)
    o1, m1, l1 = bpa.bpa_fwd(q, k, v, causal=True, dropout_p=0.0, dropout_seed=1234)
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(m0, m1) and torch.equal(l0, l1)
