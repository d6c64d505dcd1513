"""Pins of the float64 oracle against things other than itself.

Every check here runs on the CPU.  The oracle (plain C) is compared with
  * hand-derived closed forms (tests/golden/closed_form.json),
  * an independent per-query brute-force loop written below in Python,
  * a library softmax (scipy) in the unmasked single-query case,
  * invariants that the attention definition implies,
  * central finite differences of L = <dO, O> for the gradients,
  * its own literal blockwise / ring carry, which must equal the one-shot
    result for every chunking (the pages' own self-test claim: bpt.py,
    __main__ compares blockwise_attn with a materialised reference).
A plausible slip in the oracle (a dropped bias term, a wrong sign in the
backward, a transposed GQA head map, an off-by-one window bound) fails at
least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special

from ring_attention_gb300.inputs import bf16_bits_to_f32, to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# independent brute force (pure Python loops; tiny sizes only)
# --------------------------------------------------------------------------
def _is_allowed(i, j, causal, window, sel=None, sel_block=None, local_window=None):
    left, right = window
    if causal and j > i:
        return False
    if left >= 0 and j < i - left:
        return False
    if right >= 0 and j > i + right:
        return False
    if sel is not None:
        local = (i - local_window < j <= i)
        chosen = (j // sel_block) in {int(t) for t in sel if t >= 0}
        if not (local or chosen):
            return False
    return True


def brute_force(q, k, v, causal=False, window=(-1, -1), scale=None, bias=None,
                block_idx=None, sel_block=32, local_window=32):
    B, S, Hq, d = q.shape
    Hkv, dv = k.shape[2], v.shape[3]
    group = Hq // Hkv
    scale = d ** -0.5 if scale is None else scale
    full_bias = None if bias is None else np.broadcast_to(np.asarray(bias, np.float64), (B, Hq, S, S))
    o = np.zeros((B, S, Hq, dv))
    m = np.full((B, Hq, S), -np.inf)
    l = np.zeros((B, Hq, S))
    for b in range(B):
        for h in range(Hq):
            kvh = h // group
            for i in range(S):
                sel = None if block_idx is None else block_idx[b, h, i // sel_block]
                keys = [j for j in range(S)
                        if _is_allowed(i, j, causal, window, sel, sel_block, local_window)]
                if not keys:
                    continue
                z = []
                for j in keys:
                    s = 0.0
                    for c in range(d):
                        s += float(q[b, i, h, c]) * float(k[b, j, kvh, c])
                    z.append(scale * s + (0.0 if full_bias is None else float(full_bias[b, h, i, j])))
                zmax = max(z)
                w = [math.exp(t - zmax) for t in z]
                tot = math.fsum(w)
                for wj, j in zip(w, keys):
                    o[b, i, h] += (wj / tot) * v[b, j, kvh].astype(np.float64)
                m[b, h, i] = zmax
                l[b, h, i] = tot
    return o, m, l


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


MASKS = [
    dict(causal=False, window=(-1, -1)),
    dict(causal=True, window=(-1, -1)),
    dict(causal=False, window=(0, 0)),
    dict(causal=True, window=(3, 0)),
    dict(causal=False, window=(2, 2)),
    dict(causal=False, window=(-1, 1)),
    dict(causal=False, window=(1, -1)),
]


@pytest.mark.parametrize("mask", MASKS, ids=lambda m: f"c{int(m['causal'])}w{m['window'][0]}_{m['window'][1]}")
@pytest.mark.parametrize("heads", [(1, 1), (4, 2), (4, 1)])
@pytest.mark.parametrize("bias_kind", ["none", "keys", "full", "rows"])
def test_fwd_matches_brute_force(ora, mask, heads, bias_kind):
    Hq, Hkv = heads
    B, S, d, dv = 2, 9, 5, 3
    q, k, v = rnd((B, S, Hq, d), 1), rnd((B, S, Hkv, d), 2), rnd((B, S, Hkv, dv), 3)
    bias = {"none": None,
            "keys": rnd((1, 1, 1, S), 4),
            "full": rnd((B, Hq, S, S), 5),
            "rows": rnd((B, 1, S, 1), 6)}[bias_kind]
    o, m, l = ora.attention_fwd(q, k, v, bias=bias, scale=0.7, **mask)
    bo, bm, bl = brute_force(q, k, v, bias=bias, scale=0.7, **mask)
    np.testing.assert_allclose(o, bo, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(np.isinf(m), np.isinf(bm))
    fin = np.isfinite(bm)
    np.testing.assert_allclose(m[fin], bm[fin], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l, bl, rtol=1e-12, atol=1e-13)


def test_default_scale_is_inverse_sqrt_d(ora):
    q, k, v = rnd((1, 6, 2, 16), 7), rnd((1, 6, 2, 16), 8), rnd((1, 6, 2, 16), 9)
    o, _, _ = ora.attention_fwd(q, k, v, causal=True)
    bo, _, _ = brute_force(q, k, v, causal=True, scale=0.25)
    np.testing.assert_allclose(o, bo, rtol=1e-12, atol=1e-13)


def test_row_with_no_allowed_key_is_zero(ora):
    # window (-1, -1) with causal off but right bound -1 is unbounded; use a
    # left window that excludes everything before q and causal + right=-1 ...
    # the simplest empty row: block-selected mode with local_window 0 and no
    # selected block.
    B, S, H, d = 1, 8, 1, 4
    q, k, v = rnd((B, S, H, d), 1), rnd((B, S, H, d), 2), rnd((B, S, H, d), 3)
    idx = np.full((B, H, S // 4, 2), -1, dtype=np.int32)
    o, m, l = ora.attention_fwd(q, k, v, causal=True, block_idx=idx, sel_block=4, top_n=2,
                                local_window=0)
    assert np.all(o == 0) and np.all(np.isneginf(m)) and np.all(l == 0)
    dq, dk, dv, *_ = ora.attention_bwd(q, k, v, rnd((B, S, H, d), 4), causal=True, block_idx=idx,
                                       sel_block=4, top_n=2, local_window=0)
    assert not dq.any() and not dk.any() and not dv.any()


def test_single_query_is_textbook_softmax(ora):
    # one query, no mask: O = softmax(s q.K^T) V (scipy's softmax)
    S, d = 11, 6
    k, v = rnd((1, S, 1, d), 11), rnd((1, S, 1, d), 12)
    q = np.zeros((1, S, 1, d))
    q[0, 0, 0] = rnd((d,), 13)
    o, m, l = ora.attention_fwd(q, k, v, scale=0.5)
    z = 0.5 * (k[0, :, 0] @ q[0, 0, 0])
    p = scipy.special.softmax(z)
    np.testing.assert_allclose(o[0, 0, 0], p @ v[0, :, 0], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(m[0, 0, 0], z.max(), rtol=1e-14)
    np.testing.assert_allclose(l[0, 0, 0], np.exp(z - z.max()).sum(), rtol=1e-13)


def _golden():
    with open(os.path.join(GOLDEN, "closed_form.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: c["name"])
def test_closed_form_fixture(ora, case):
    a = lambda x: None if x is None else np.array(x, dtype=np.float64)
    o, m, l = ora.attention_fwd(a(case["q"]), a(case["k"]), a(case["v"]), scale=case["scale"],
                                causal=case["causal"], window=tuple(case["window"]),
                                bias=a(case["bias"]))
    np.testing.assert_allclose(o, a(case["o"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(m, a(case["m"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(l, a(case["l"]), rtol=0, atol=1e-15)


def test_closed_form_gradient_fixture(ora):
    c = _golden()["grad_case"]
    a = lambda x: np.array(x, dtype=np.float64)
    dq, dk, dv, *_ = ora.attention_bwd(a(c["q"]), a(c["k"]), a(c["v"]), a(c["dout"]),
                                       scale=c["scale"], causal=c["causal"])
    np.testing.assert_allclose(dq, a(c["dq"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk, a(c["dk"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv, a(c["dv"]), rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# the blockwise carry equals the one-shot softmax, for every chunking
# --------------------------------------------------------------------------
@pytest.mark.parametrize("ring", [1, 2, 4])
@pytest.mark.parametrize("mask", [dict(causal=True, window=(-1, -1)),
                                  dict(causal=False, window=(-1, -1)),
                                  dict(causal=True, window=(5, 0)),
                                  dict(causal=False, window=(3, 6))],
                         ids=["causal", "full", "swa5", "win3_6"])
def test_blockwise_carry_equals_one_shot(ora, ring, mask):
    B, S, Hq, Hkv, d = 1, 16, 4, 2, 4
    q, k, v = rnd((B, S, Hq, d), 21), rnd((B, S, Hkv, d), 22), rnd((B, S, Hkv, d), 23)
    bias = rnd((1, 1, 1, S), 24)
    ref = ora.attention_fwd(q, k, v, bias=bias, **mask)
    blk = S // ring
    chunks = [c for c in range(1, blk + 1) if blk % c == 0]
    for qc, kc in itertools.product(chunks, chunks):
        got = ora.blockwise_fwd(q, k, v, query_chunk=qc, key_chunk=kc, ring_size=ring, bias=bias,
                                **mask)
        for g, r in zip(got, ref):
            np.testing.assert_allclose(g, r, rtol=1e-12, atol=1e-12, err_msg=f"qc={qc} kc={kc}")


def test_blockwise_padding_bias_tail(ora):
    # the long-context recipe at toy size: bias -1e9 on the last keys, ring of 4
    B, S, Hq, Hkv, d = 1, 32, 4, 2, 8
    q, k, v = rnd((B, S, Hq, d), 31), rnd((B, S, Hkv, d), 32), rnd((B, S, Hkv, d), 33)
    bias = np.zeros((1, 1, 1, S))
    bias[..., -4:] = -1e9
    ref = ora.attention_fwd(q, k, v, causal=True, bias=bias)
    got = ora.blockwise_fwd(q, k, v, query_chunk=2, key_chunk=4, ring_size=4, causal=True,
                            bias=bias)
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, r, rtol=1e-12, atol=1e-12)
    # padded keys carry exactly zero weight for rows that also see real keys
    o2, _, _ = ora.attention_fwd(q[:, :S - 4], k[:, :S - 4], v[:, :S - 4], causal=True)
    np.testing.assert_allclose(ref[0][:, :S - 4], o2, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# invariants of the definition
# --------------------------------------------------------------------------
def test_constant_value_rows(ora):
    B, S, Hq, Hkv, d = 2, 12, 4, 2, 6
    q, k = rnd((B, S, Hq, d), 41), rnd((B, S, Hkv, d), 42)
    c = rnd((B, 1, Hkv, d), 43)
    v = np.broadcast_to(c, (B, S, Hkv, d)).copy()
    o, _, _ = ora.attention_fwd(q, k, v, causal=True, window=(4, 0), bias=rnd((B, Hq, S, S), 44))
    exp = np.repeat(np.broadcast_to(c, (B, S, Hkv, d)), Hq // Hkv, axis=2)
    np.testing.assert_allclose(o, exp, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("window", [(3, 0), (2, 2), (-1, -1)])
def test_uniform_scores_give_window_mean(ora, window):
    B, S, Hq, Hkv, d = 1, 10, 2, 1, 3
    q = np.zeros((B, S, Hq, d))
    k, v = rnd((B, S, Hkv, d), 51), rnd((B, S, Hkv, d), 52)
    o, _, l = ora.attention_fwd(q, k, v, causal=window[1] == 0, window=window)
    for i in range(S):
        lo = 0 if window[0] < 0 else max(0, i - window[0])
        hi = S - 1 if window[1] < 0 else min(S - 1, i + window[1])
        if window[1] == 0:
            hi = min(hi, i)
        mean = v[0, lo:hi + 1, 0].mean(axis=0)
        for h in range(Hq):
            np.testing.assert_allclose(o[0, i, h], mean, rtol=1e-12, atol=1e-13)
            assert l[0, h, i] == pytest.approx(hi - lo + 1, rel=1e-15)


def test_window_00_is_identity_and_gradients(ora):
    B, S, Hq, Hkv, d = 2, 7, 4, 2, 5
    q, k, v, do = (rnd((B, S, Hq, d), 61), rnd((B, S, Hkv, d), 62), rnd((B, S, Hkv, d), 63),
                   rnd((B, S, Hq, d), 64))
    o, _, l = ora.attention_fwd(q, k, v, window=(0, 0))
    np.testing.assert_allclose(o, np.repeat(v, 2, axis=2), rtol=0, atol=1e-15)
    assert np.all(l == 1.0)
    dq, dk, dv, *_ = ora.attention_bwd(q, k, v, do, window=(0, 0))
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
    np.testing.assert_allclose(dv, do.reshape(B, S, Hkv, 2, d).sum(axis=3), rtol=1e-14, atol=1e-14)


def test_key_gradients_sum_to_zero(ora):
    # sum_k P = 1  =>  each row of dS sums to 0  =>  sum_k dK_k = 0 per kv head
    B, S, Hq, Hkv, d = 2, 13, 4, 2, 6
    q, k, v, do = (rnd((B, S, Hq, d), 71), rnd((B, S, Hkv, d), 72), rnd((B, S, Hkv, d), 73),
                   rnd((B, S, Hq, d), 74))
    for mask in MASKS:
        _, dk, _, *_ = ora.attention_bwd(q, k, v, do, bias=rnd((1, Hq, S, S), 75), **mask)
        np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)


def test_shift_invariances(ora):
    B, S, Hq, Hkv, d = 1, 11, 2, 2, 4
    q, k, v = rnd((B, S, Hq, d), 81), rnd((B, S, Hkv, d), 82), rnd((B, S, Hkv, d), 83)
    base = ora.attention_fwd(q, k, v, causal=True, window=(5, 0))[0]
    shifted_k = ora.attention_fwd(q, k + rnd((1, 1, Hkv, d), 84), v, causal=True, window=(5, 0))[0]
    np.testing.assert_allclose(shifted_k, base, rtol=1e-12, atol=1e-12)
    row_bias = np.broadcast_to(rnd((B, Hq, S, 1), 85), (B, Hq, S, S))
    biased = ora.attention_fwd(q, k, v, causal=True, window=(5, 0), bias=row_bias)[0]
    np.testing.assert_allclose(biased, base, rtol=1e-12, atol=1e-12)


def test_gqa_equals_repeated_heads(ora):
    # GQA reads kv head h // (Hq/Hkv): same as repeating each kv head G times
    B, S, Hq, Hkv, d = 1, 9, 6, 2, 4
    q, k, v, do = (rnd((B, S, Hq, d), 91), rnd((B, S, Hkv, d), 92), rnd((B, S, Hkv, d), 93),
                   rnd((B, S, Hq, d), 94))
    rk, rv = np.repeat(k, 3, axis=2), np.repeat(v, 3, axis=2)
    a = ora.attention_bwd(q, k, v, do, causal=True)
    r = ora.attention_bwd(q, rk, rv, do, causal=True)
    np.testing.assert_allclose(a[0], r[0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(a[1], r[1].reshape(B, S, Hkv, 3, d).sum(3), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(a[2], r[2].reshape(B, S, Hkv, 3, d).sum(3), rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# gradients: central finite differences of L = <dO, O>
# --------------------------------------------------------------------------
@pytest.mark.parametrize("cfg", [
    dict(causal=True, window=(-1, -1), bias=False),
    dict(causal=True, window=(3, 0), bias=True),
    dict(causal=False, window=(2, 1), bias=True),
    dict(causal=False, window=(-1, -1), bias=False),
], ids=["causal", "swa3_bias", "win2_1_bias", "full"])
def test_gradients_match_finite_differences(ora, cfg):
    B, S, Hq, Hkv, d, dv = 1, 8, 4, 2, 3, 2
    q, k, v, do = (rnd((B, S, Hq, d), 101), rnd((B, S, Hkv, d), 102), rnd((B, S, Hkv, dv), 103),
                   rnd((B, S, Hq, dv), 104))
    bias = rnd((B, Hq, S, S), 105) if cfg["bias"] else None
    kw = dict(causal=cfg["causal"], window=cfg["window"], bias=bias, scale=0.8)
    dq, dk, dvv, *_ = ora.attention_bwd(q, k, v, do, **kw)
    h = 1e-6

    def loss(qq, kk, vv):
        return float((ora.attention_fwd(qq, kk, vv, **kw)[0] * do).sum())

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dvv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(fd - g).max() / max(np.abs(g).max(), 1e-30)
        assert err < 1e-6, f"d{name}: relative error {err}"


def test_block_selected_gradients_match_finite_differences(ora):
    """Backward of block-selected attention (AnnAttention, faiss_block_attention, trained
    through): the selection is discrete and held fixed, so the gradients are those of
    attention under the union mask.  Checked against central differences of <dO, O>
    with O from the brute-force loop above, not from the oracle's forward."""
    B, S, Hq, Hkv, d, dv, bs, n, W = 1, 16, 2, 1, 3, 2, 4, 2, 3
    q, k, v, do = (rnd((B, S, Hq, d), 151), rnd((B, S, Hkv, d), 152), rnd((B, S, Hkv, dv), 153),
                   rnd((B, S, Hq, dv), 154))
    # per query block: earlier blocks, -1 padding, and the block just before the query's
    # (which overlaps the local window: union, counted once)
    idx = np.array([[[[-1, -1], [0, -1], [0, 1], [2, 0]],
                     [[-1, -1], [-1, -1], [1, -1], [1, 2]]]], dtype=np.int32)
    kw = dict(causal=True, block_idx=idx, sel_block=bs, local_window=W, scale=0.7)
    dq, dk, dvv, *_ = ora.attention_bwd(q, k, v, do, top_n=n, **kw)
    h = 1e-6

    def loss(qq, kk, vv):
        return float((brute_force(qq, kk, vv, **kw)[0] * do).sum())

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dvv)):
        fd = np.zeros_like(x)
        for ix in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[ix] += h
            xm[ix] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd[ix] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(fd - g).max() / max(np.abs(g).max(), 1e-30)
        assert err < 1e-6, f"d{name}: relative error {err}"
    # keys of block 3 are selected by no query and lie in no local window but their own
    # block's: their gradients come from block 3's queries alone
    assert np.abs(dk[0, 12:]).max() > 0


# --------------------------------------------------------------------------
# variable lengths (TransformerEngine page, section 1: SequenceDescriptor)
# --------------------------------------------------------------------------
def varlen_via_brute(q, k, v, lq, lk, bottom_right, causal, window, scale):
    """Each batch entry rebuilt as an ordinary problem on one position axis: key j at
    position j + shift, query i at i + off + shift (off = Lk - Lq when the queries are the
    last Lq positions of the key sequence, else 0); positions that hold no key get a
    -1e300 bias so they carry no weight.  Rows whose best score is that bias have no real
    key (O = 0, m = -inf, l = 0).  Returns (o, m, l) in the padded layout."""
    B, S, Hq, d = q.shape
    Hkv, dv = k.shape[2], v.shape[3]
    o = np.zeros((B, S, Hq, dv))
    m = np.full((B, Hq, S), -np.inf)
    l = np.zeros((B, Hq, S))
    for b in range(B):
        nq, nk = int(lq[b]), int(lk[b])
        if nq == 0:
            continue
        off = nk - nq if bottom_right else 0
        shift = max(0, -off)
        n = max(nk, nq + off) + shift
        qe = np.zeros((1, n, Hq, d))
        ke = np.zeros((1, n, Hkv, d))
        ve = np.zeros((1, n, Hkv, dv))
        qe[0, off + shift:off + shift + nq] = q[b, :nq]
        ke[0, shift:shift + nk] = k[b, :nk]
        ve[0, shift:shift + nk] = v[b, :nk]
        bias = np.full((1, 1, 1, n), -1e300)
        bias[..., shift:shift + nk] = 0.0
        eo, em, el = brute_force(qe, ke, ve, causal=causal, window=window, scale=scale, bias=bias)
        rows = slice(off + shift, off + shift + nq)
        real = em[0, :, rows] > -1e200            # [Hq, nq]
        o[b, :nq] = np.where(real.T[..., None], eo[0, rows], 0.0)
        m[b, :, :nq] = np.where(real, em[0, :, rows], -np.inf)
        l[b, :, :nq] = np.where(real, el[0, :, rows], 0.0)
    return o, m, l


VARLEN_CASES = [   # (query lengths, key lengths or None (the query lengths), bottom-right)
    ([12, 7, 5, 0], None, False),
    ([12, 7, 5, 3], [12, 9, 3, 6], False),
    ([12, 4, 5, 1], [12, 9, 11, 6], True),
    ([9, 12, 2, 7], [5, 6, 12, 0], True),
]


@pytest.mark.parametrize("case", VARLEN_CASES, ids=["same", "topleft", "bottomright", "bottomright_short_keys"])
@pytest.mark.parametrize("mask", [dict(causal=True, window=(-1, -1)), dict(causal=False, window=(-1, -1)),
                                  dict(causal=True, window=(3, 0)), dict(causal=False, window=(2, 1))],
                         ids=["causal", "full", "swa3", "win2_1"])
def test_varlen_matches_rebuilt_problems(ora, case, mask):
    lq, lk, br = case
    B, S, Hq, Hkv, d, dv = 4, 12, 4, 2, 3, 2
    q, k, v = rnd((B, S, Hq, d), 161), rnd((B, S, Hkv, d), 162), rnd((B, S, Hkv, dv), 163)
    kw = dict(scale=0.7, **mask)
    o, m, l = ora.attention_fwd(q, k, v, seqlens_q=lq, seqlens_kv=lk, bottom_right=br, **kw)
    bo, bm, bl = varlen_via_brute(q, k, v, lq, lq if lk is None else lk, br, **kw)
    np.testing.assert_allclose(o, bo, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(np.isfinite(m), np.isfinite(bm))
    fin = np.isfinite(bm)
    np.testing.assert_allclose(m[fin], bm[fin], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l, bl, rtol=1e-12, atol=1e-13)


def test_varlen_padding_is_inert(ora):
    # padded positions take part in nothing: changing them changes no output, their own
    # outputs and gradients are exactly zero
    B, S, Hq, Hkv, d = 3, 10, 2, 1, 4
    lq, lk = [10, 6, 3], [10, 8, 2]
    q, k, v, do = (rnd((B, S, Hq, d), 171), rnd((B, S, Hkv, d), 172), rnd((B, S, Hkv, d), 173),
                   rnd((B, S, Hq, d), 174))
    kw = dict(causal=True, seqlens_q=lq, seqlens_kv=lk, bottom_right=True)
    r1 = ora.attention_bwd(q, k, v, do, **kw)
    q2, k2, v2, do2 = q.copy(), k.copy(), v.copy(), do.copy()
    for b in range(B):
        q2[b, lq[b]:] = 50.0
        do2[b, lq[b]:] = -7.0
        k2[b, lk[b]:] = 30.0
        v2[b, lk[b]:] = 1e6
    r2 = ora.attention_bwd(q2, k2, v2, do2, **kw)
    for x, y in zip(r1, r2):
        np.testing.assert_array_equal(x, y)
    dq, dk, dvv, o, m, l = r1
    for b in range(B):
        assert not dq[b, lq[b]:].any() and not o[b, lq[b]:].any()
        assert np.all(np.isneginf(m[b, :, lq[b]:])) and not l[b, :, lq[b]:].any()
        assert not dk[b, lk[b]:].any() and not dvv[b, lk[b]:].any()
    # the sampled-key evaluation agrees, padded keys included (no causal rule, so that
    # nothing but the length keeps them out)
    kw = dict(causal=False, seqlens_q=lq, seqlens_kv=lk)
    dq, dk, dvv, *_ = ora.attention_bwd(q, k, v, do, **kw)
    sk, sv = ora.keys(q, k, v, do, 1, 0, [0, 5, 7, 8, 9], **kw)
    np.testing.assert_allclose(sk, dk[1, [0, 5, 7, 8, 9], 0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(sv, dvv[1, [0, 5, 7, 8, 9], 0], rtol=1e-12, atol=1e-14)
    assert not sk[3:].any() and not sv[3:].any() and sk[:3].any()


def test_varlen_gradients_match_finite_differences(ora):
    B, S, Hq, Hkv, d, dv = 2, 6, 2, 1, 2, 2
    lq, lk = [6, 3], [4, 5]
    q, k, v, do = (rnd((B, S, Hq, d), 181), rnd((B, S, Hkv, d), 182), rnd((B, S, Hkv, dv), 183),
                   rnd((B, S, Hq, dv), 184))
    kw = dict(causal=True, window=(2, 0), scale=0.9)
    dq, dk, dvv, *_ = ora.attention_bwd(q, k, v, do, seqlens_q=lq, seqlens_kv=lk, bottom_right=True, **kw)
    h = 1e-6

    def loss(qq, kk, vv):
        return float((varlen_via_brute(qq, kk, vv, lq, lk, True, **kw)[0] * do).sum())

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dvv)):
        fd = np.zeros_like(x)
        for ix in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[ix] += h
            xm[ix] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd[ix] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(fd - g).max() / max(np.abs(g).max(), 1e-30)
        assert err < 1e-6, f"d{name}: relative error {err}"


# --------------------------------------------------------------------------
# sink attention (TransformerEngine page, "Other attention knobs": softmax_type
# off_by_one / learnable): an extra logit per head with no value vector
# --------------------------------------------------------------------------
def sink_via_brute(q, k, v, sink, causal, scale):
    """The sink as one more key: position 0 of a one-longer sequence holds a zero key
    whose per-head bias is the sink logit and a zero value; query i sits at position
    i + 1, so under the causal rule it still sees the sink and its own keys 0..i."""
    B, S, Hq, d = q.shape
    Hkv, dv = k.shape[2], v.shape[3]
    qe = np.concatenate([np.zeros((B, 1, Hq, d)), q], axis=1)
    ke = np.concatenate([np.zeros((B, 1, Hkv, d)), k], axis=1)
    ve = np.concatenate([np.zeros((B, 1, Hkv, dv)), v], axis=1)
    bias = np.zeros((1, Hq, 1, S + 1))
    bias[0, :, 0, 0] = sink
    o, m, l = brute_force(qe, ke, ve, causal=causal, scale=scale, bias=bias)
    return o[:, 1:], m[:, :, 1:], l[:, :, 1:]


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
@pytest.mark.parametrize("kind", ["off_by_one", "learnable"])
def test_sink_equals_extra_key(ora, causal, kind):
    B, S, Hq, Hkv, d, dv = 2, 9, 4, 2, 3, 2
    q, k, v = rnd((B, S, Hq, d), 191), rnd((B, S, Hkv, d), 192), rnd((B, S, Hkv, dv), 193)
    sink = np.zeros(Hq) if kind == "off_by_one" else np.array([0.7, -2.0, 3.5, -0.1])
    o, m, l = ora.attention_fwd(q, k, v, causal=causal, scale=0.8, sink=sink)
    bo, bm, bl = sink_via_brute(q, k, v, sink, causal, 0.8)
    np.testing.assert_allclose(o, bo, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(m, bm, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l, bl, rtol=1e-12, atol=1e-13)


def test_sink_rows_without_keys_and_padding(ora):
    # a row with no allowed key keeps only the sink: O = 0, m = sink, l = 1; padding rows
    # of a shorter sequence take part in nothing (m = -inf, l = 0)
    B, S, H, d = 2, 8, 2, 4
    q, k, v = rnd((B, S, H, d), 194), rnd((B, S, H, d), 195), rnd((B, S, H, d), 196)
    idx = np.full((B, H, S // 4, 2), -1, dtype=np.int32)
    sink = np.array([0.25, -1.5])
    o, m, l = ora.attention_fwd(q, k, v, causal=True, block_idx=idx, sel_block=4, top_n=2,
                                local_window=0, sink=sink)
    assert not o.any() and np.array_equal(l, np.ones_like(l))
    np.testing.assert_array_equal(m, np.broadcast_to(sink[None, :, None], m.shape))
    o, m, l = ora.attention_fwd(q, k, v, causal=True, seqlens_q=[8, 5], sink=sink)
    assert np.all(np.isneginf(m[1, :, 5:])) and not l[1, :, 5:].any() and not o[1, 5:].any()
    assert np.all(np.isfinite(m[:, :, :5]))


def test_sink_gradients_match_finite_differences(ora):
    B, S, Hq, Hkv, d, dv = 1, 6, 2, 1, 3, 2
    q, k, v, do = (rnd((B, S, Hq, d), 197), rnd((B, S, Hkv, d), 198), rnd((B, S, Hkv, dv), 199),
                   rnd((B, S, Hq, dv), 200))
    sink = np.array([0.4, -0.9])
    dq, dk, dvv, o, m, l, dsink = ora.attention_bwd(q, k, v, do, causal=True, scale=0.6, sink=sink,
                                                    want_dsink=True)
    h = 1e-6

    def loss(qq, kk, vv, ss):
        return float((sink_via_brute(qq, kk, vv, ss, True, 0.6)[0] * do).sum())

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dvv), ("sink", sink, dsink)):
        fd = np.zeros_like(x)
        for ix in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[ix] += h
            xm[ix] -= h
            ap = {"q": (xp, k, v, sink), "k": (q, xp, v, sink), "v": (q, k, xp, sink), "sink": (q, k, v, xp)}[name]
            am = {"q": (xm, k, v, sink), "k": (q, xm, v, sink), "v": (q, k, xm, sink), "sink": (q, k, v, xm)}[name]
            fd[ix] = (loss(*ap) - loss(*am)) / (2 * h)
        err = np.abs(fd - g).max() / max(np.abs(g).max(), 1e-30)
        assert err < 1e-6, f"d{name}: relative error {err}"


# --------------------------------------------------------------------------
# attention dropout (bpt.py: a Bernoulli(p) mask over (batch, head, q, k); the dropped
# entries leave the softmax) with the draws of a counter-based generator
# --------------------------------------------------------------------------
def brute_masked(q, k, v, keep, causal, scale):
    """Brute force with the dropped entries given a -1e300 bias; rows whose best score is
    that bias keep no real key (O = 0, m = -inf, l = 0).  keep: [B, Hq, S, S]."""
    bias = np.where(keep.astype(bool), 0.0, -1e300)
    o, m, l = brute_force(q, k, v, causal=causal, scale=scale, bias=bias)
    real = m > -1e200
    o = np.where(np.transpose(real, (0, 2, 1))[..., None], o, 0.0)
    return o, np.where(real, m, -np.inf), np.where(real, l, 0.0)


def _keep_all(B, Hq, S, p, seed, ora):
    return np.stack([np.stack([ora.dropout_keep(S, b, h, dropout_p=p, dropout_seed=seed) for h in range(Hq)])
                     for b in range(B)])


@pytest.mark.parametrize("p", [0.1, 0.5])
def test_dropout_draws_are_bernoulli(ora, p):
    S, n = 512, 512 * 512
    masks = [ora.dropout_keep(S, b, h, dropout_p=p, dropout_seed=1234) for b, h in ((0, 0), (0, 1), (3, 0))]
    for keep in masks:
        drop = 1.0 - keep.astype(np.float64)
        sigma = (p * (1 - p) / n) ** 0.5
        assert abs(drop.mean() - p) < 5 * sigma
        # no correlation between neighbouring keys (in and across the groups of four that
        # share one generator call), neighbouring rows
        for a, b in ((drop[:, :-1], drop[:, 1:]), (drop[:, :-4], drop[:, 4:]), (drop[:-1], drop[1:])):
            c = np.corrcoef(a.ravel(), b.ravel())[0, 1]
            assert abs(c) < 5 / a.size ** 0.5
    # heads and batch entries draw different masks; the seed decides, repeatably
    assert (masks[0] != masks[1]).mean() > 0.5 * 2 * p * (1 - p)
    assert (masks[0] != masks[2]).mean() > 0.5 * 2 * p * (1 - p)
    assert np.array_equal(masks[0], ora.dropout_keep(S, 0, 0, dropout_p=p, dropout_seed=1234))
    assert not np.array_equal(masks[0], ora.dropout_keep(S, 0, 0, dropout_p=p, dropout_seed=1235))
    assert ora.dropout_keep(64, 0, 0, dropout_p=0.0, dropout_seed=7).all()


def test_philox_known_answers(ora):
    # the generator's published known-answer vectors (SC 2011 paper's Random123
    # distribution): a wrong round constant, Weyl increment or word order fails these even
    # though the map would stay a bijection with good statistics
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.json")) as f:
        kat = json.load(f)
    for vec in kat["vectors"]:
        ctr = [int(x, 16) for x in vec["counter"]]
        key = tuple(int(x, 16) for x in vec["key"])
        got = [int(x) for x in ora.philox4x32_10(ctr, key)]
        assert got == [int(x, 16) for x in vec["expected"]], vec


def test_philox_is_a_bijection_of_the_counter(ora):
    # distinct counters give distinct outputs for one key (each round permutes the counter
    # space), and changing the key changes every word
    rng = np.random.default_rng(208)
    ctrs = {tuple(int(x) for x in c) for c in rng.integers(0, 2 ** 32, (4096, 4), dtype=np.uint64)}
    ctrs |= {(i, 0, 0, 0) for i in range(256)} | {(0, 0, i, 0) for i in range(256)}
    outs = {tuple(ora.philox4x32_10(c, (17, 29)).tolist()) for c in ctrs}
    assert len(outs) == len(ctrs)
    a = ora.philox4x32_10([1, 2, 3, 4], (17, 29))
    b = ora.philox4x32_10([1, 2, 3, 4], (18, 29))
    assert np.all(a != b)


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_dropout_is_the_fixed_mask(ora, causal):
    B, S, Hq, Hkv, d, dv = 2, 24, 4, 2, 3, 2
    q, k, v = rnd((B, S, Hq, d), 201), rnd((B, S, Hkv, d), 202), rnd((B, S, Hkv, dv), 203)
    p, seed = 0.4, 99
    o, m, l = ora.attention_fwd(q, k, v, causal=causal, scale=0.7, dropout_p=p, dropout_seed=seed)
    bo, bm, bl = brute_masked(q, k, v, _keep_all(B, Hq, S, p, seed, ora), causal, 0.7)
    np.testing.assert_allclose(o, bo, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(np.isfinite(m), np.isfinite(bm))
    np.testing.assert_allclose(l, bl, rtol=1e-12, atol=1e-13)
    # p = 0 is plain attention
    o0, _, _ = ora.attention_fwd(q, k, v, causal=causal, scale=0.7, dropout_p=0.0, dropout_seed=seed)
    po, _, _ = ora.attention_fwd(q, k, v, causal=causal, scale=0.7)
    np.testing.assert_array_equal(o0, po)


def test_dropout_gradients_match_finite_differences(ora):
    B, S, Hq, Hkv, d, dv = 1, 8, 2, 1, 2, 2
    q, k, v, do = (rnd((B, S, Hq, d), 204), rnd((B, S, Hkv, d), 205), rnd((B, S, Hkv, dv), 206),
                   rnd((B, S, Hq, dv), 207))
    p, seed = 0.3, 5
    dq, dk, dvv, *_ = ora.attention_bwd(q, k, v, do, causal=True, scale=0.9, dropout_p=p, dropout_seed=seed)
    keep = _keep_all(B, Hq, S, p, seed, ora)
    h = 1e-6

    def loss(qq, kk, vv):
        return float((brute_masked(qq, kk, vv, keep, True, 0.9)[0] * do).sum())

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dvv)):
        fd = np.zeros_like(x)
        for ix in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[ix] += h
            xm[ix] -= h
            ap = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            am = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd[ix] = (loss(*ap) - loss(*am)) / (2 * h)
        err = np.abs(fd - g).max() / max(np.abs(g).max(), 1e-30)
        assert err < 1e-6, f"d{name}: relative error {err}"


# --------------------------------------------------------------------------
# sampled rows / keys agree with the full evaluation
# --------------------------------------------------------------------------
def test_sampled_rows_and_keys_match_full(ora):
    B, S, Hq, Hkv, d = 2, 20, 4, 2, 5
    q, k, v, do = (rnd((B, S, Hq, d), 111), rnd((B, S, Hkv, d), 112), rnd((B, S, Hkv, d), 113),
                   rnd((B, S, Hq, d), 114))
    bias = rnd((1, 1, 1, S), 115)
    dq, dk, dv, o, m, l = ora.attention_bwd(q, k, v, do, causal=True, bias=bias)
    rows = [(0, 0, 0), (1, 3, 19), (0, 2, 7), (1, 1, 12)]
    ro, rm, rl, rdq = ora.rows(q, k, v, do, rows, causal=True, bias=bias)
    for t, (b, h, s) in enumerate(rows):
        np.testing.assert_allclose(ro[t], o[b, s, h], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(rdq[t], dq[b, s, h], rtol=1e-12, atol=1e-13)
        assert rm[t] == pytest.approx(m[b, h, s], rel=1e-14)
        assert rl[t] == pytest.approx(l[b, h, s], rel=1e-13)
    keys = [0, 5, 19, 11]
    kdk, kdv = ora.keys(q, k, v, do, 1, 1, keys, causal=True, bias=bias)
    np.testing.assert_allclose(kdk, dk[1, keys, 1], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(kdv, dv[1, keys, 1], rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# block selection (AnnAttention, select_block) and block-selected attention
# --------------------------------------------------------------------------
def brute_select(q, k, block_size, top_n):
    B, S, H, d = q.shape
    nblk = S // block_size
    out = np.full((B, H, nblk, top_n), -1, dtype=np.int32)
    for b in range(B):
        for h in range(H):
            qs, ks = [], []
            for i in range(nblk):
                sq, sk = [0.0] * d, [0.0] * d
                for r in range(block_size):
                    for c in range(d):
                        sq[c] += float(q[b, i * block_size + r, h, c])
                        sk[c] += float(k[b, i * block_size + r, h, c])
                qs.append(sq)
                ks.append(sk)
            for i in range(nblk):
                scored = []
                for j in range(i):
                    s = 0.0
                    for c in range(d):
                        s += qs[i][c] * ks[j][c]
                    # a NaN score ranks below every number, NaNs in block order
                    scored.append((1, 0.0, j) if s != s else (0, -s, j))
                best = sorted(e[-1] for e in sorted(scored)[:top_n])
                out[b, h, i, :len(best)] = best
    return out


@pytest.mark.parametrize("dtype", ["f64", "bf16"])
def test_select_matches_full_sort(ora, dtype):
    B, S, H, d, bs, n = 2, 64, 2, 8, 4, 3
    q, k = rnd((B, S, H, d), 121), rnd((B, S, H, d), 122)
    if dtype == "bf16":
        qb, kb = to_bf16_bits(q.astype(np.float32)), to_bf16_bits(k.astype(np.float32))
        got = ora.select_blocks(qb, kb, block_size=bs, top_n=n)
        exp = brute_select(bf16_bits_to_f32(qb), bf16_bits_to_f32(kb), bs, n)
    else:
        got = ora.select_blocks(q, k, block_size=bs, top_n=n)
        exp = brute_select(q, k, bs, n)
    np.testing.assert_array_equal(got, exp)


def _planted(alpha, bs, d):
    # first row of every query block = u, of key block j = alpha_j * u; others 0
    nblk = len(alpha)
    u = np.array([1.0, 2.0, -1.0, 0.5][:d])
    q = np.zeros((1, nblk * bs, 1, d))
    k = np.zeros((1, nblk * bs, 1, d))
    for j in range(nblk):
        q[0, j * bs, 0] = u
        k[0, j * bs, 0] = alpha[j] * u
    return q, k


def test_select_planted_ranking(ora):
    alpha = [3.0, -1.0, 7.0, 2.0, 5.0, 0.5, 6.0, 4.0, 1.0, -2.0]
    q, k = _planted(alpha, 4, 4)
    got = ora.select_blocks(q, k, block_size=4, top_n=3)[0, 0]
    for i in range(len(alpha)):
        ranked = sorted(range(i), key=lambda j: -alpha[j])[:3]
        exp = sorted(ranked) + [-1] * (3 - len(ranked))
        assert list(got[i]) == exp, f"block {i}"


def test_select_ties_keep_lower_block(ora):
    alpha = [5.0, 3.0, 5.0, 3.0, 5.0, 1.0, 3.0, 0.0]
    q, k = _planted(alpha, 2, 4)
    got = ora.select_blocks(q, k, block_size=2, top_n=2)[0, 0]
    assert list(got[5]) == [0, 2]          # three 5s tie: blocks 0 and 2 win
    assert list(got[7]) == [0, 2]
    got4 = ora.select_blocks(q, k, block_size=2, top_n=4)[0, 0]
    assert list(got4[7]) == [0, 1, 2, 4]   # 5, 5, 5 then the lowest of the 3s


def test_select_fewer_candidates_than_top_n(ora):
    q, k = rnd((1, 24, 1, 4), 131), rnd((1, 24, 1, 4), 132)
    got = ora.select_blocks(q, k, block_size=4, top_n=8)[0, 0]
    for i in range(6):
        assert list(got[i]) == list(range(i)) + [-1] * (8 - i)


def test_select_nan_scores_rank_last(ora):
    # a NaN in one key block makes every score against that block NaN, a NaN in one query
    # block every score of that block: those rank below every number, in block order
    B, S, H, d, bs, n = 1, 48, 2, 4, 4, 3
    q, k = rnd((B, S, H, d), 133), rnd((B, S, H, d), 134)
    k[0, 2 * bs + 1, 0, 2] = np.nan     # key block 2 of head 0
    q[0, 7 * bs, 1, 0] = np.nan         # query block 7 of head 1
    got = ora.select_blocks(q, k, block_size=bs, top_n=n)
    np.testing.assert_array_equal(got, brute_select(q, k, bs, n))
    assert 2 not in got[0, 0, 3 + n:].ravel()     # blocks with n finite candidates skip it
    assert list(got[0, 1, 7]) == [0, 1, 2]        # all NaN: the lowest blocks


def test_block_selected_attention_matches_brute_force(ora):
    B, S, H, d, bs, n, W = 1, 32, 2, 4, 4, 2, 4
    q, k, v = rnd((B, S, H, d), 141), rnd((B, S, H, d), 142), rnd((B, S, H, d), 143)
    idx = ora.select_blocks(q, k, block_size=bs, top_n=n)
    o, m, l = ora.attention_fwd(q, k, v, causal=True, block_idx=idx, sel_block=bs, top_n=n,
                                local_window=W)
    bo, bm, bl = brute_force(q, k, v, causal=True, block_idx=idx, sel_block=bs, local_window=W)
    np.testing.assert_allclose(o, bo, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l, bl, rtol=1e-12, atol=1e-13)
    # the union counts a key once: a selected block that overlaps the local
    # window must not double its weight (block i-1 is usually both)
    assert np.all(l <= W + n * bs)


# --------------------------------------------------------------------------
# the seeded input encoding
# --------------------------------------------------------------------------
def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -7 + 2 ** -9, -2.5,
                  1.0 + 2 ** -8 + 2 ** -20], dtype=np.float32)
    got = bf16_bits_to_f32(to_bf16_bits(x))
    exp = np.array([1.0, 1.0, 1.0 + 2 ** -6, 1.0 + 2 ** -7, -2.5, 1.0 + 2 ** -7], dtype=np.float32)
    np.testing.assert_array_equal(got, exp)
