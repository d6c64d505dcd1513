"""The Python binding's argument marshalling, on the CPU: make_desc fills the descriptor
from tensor shapes and strides and touches no data, so host tensors serve; the library's
own checks (bpa_workspace_size) then accept or refuse the descriptor without a device."""
import ctypes

import pytest
import torch


@pytest.fixture(scope="module")
def bpa():
    from ring_attention_gb300 import build
    build.build()
    from ring_attention_gb300 import bpa as mod
    return mod


def _qkv(B=2, S=64, Hq=4, Hkv=2, d=32, dv=None, dtype=torch.bfloat16):
    dv = d if dv is None else dv
    return (torch.zeros(B, S, Hq, d, dtype=dtype), torch.zeros(B, S, Hkv, d, dtype=dtype),
            torch.zeros(B, S, Hkv, dv, dtype=dtype))


def test_descriptor_fields_from_tensors(bpa):
    q, k, v = _qkv(dv=16)
    o = torch.zeros(2, 64, 4, 16, dtype=torch.bfloat16)
    D = bpa.make_desc(q, k, v, o=o, causal=True, window=(5, 0), scale=0.25, ring_size=2, query_chunk=32,
                      key_chunk=16, deterministic=True, bottom_right=True)
    assert (D.B, D.S, D.Hq, D.Hkv, D.d, D.dv) == (2, 64, 4, 2, 32, 16)
    assert D.struct_size == ctypes.sizeof(bpa.bpa_attn_desc)
    assert tuple(D.q_strides) == q.stride()[:3] and tuple(D.k_strides) == k.stride()[:3]
    assert tuple(D.o_strides) == o.stride()[:3]
    assert (D.causal, D.window_left, D.window_right, D.ring_size) == (1, 5, 0, 2)
    assert D.scale == pytest.approx(0.25) and D.deterministic == 1 and D.bottom_right == 1
    assert D.q == q.data_ptr() and D.v == v.data_ptr()
    # a strided view: the descriptor carries its strides
    big = torch.zeros(2, 64, 8, 32, dtype=torch.bfloat16)
    D = bpa.make_desc(big[:, :, ::2], k, torch.zeros(2, 64, 2, 32, dtype=torch.bfloat16))
    assert tuple(D.q_strides) == big[:, :, ::2].stride()[:3]


def test_bias_broadcast_dims_get_stride_zero(bpa):
    q, k, v = _qkv()
    bias = torch.zeros(1, 1, 1, 64)
    D = bpa.make_desc(q, k, v, bias=bias)
    assert tuple(D.bias_strides) == (0, 0, 0, 1)
    full = torch.zeros(2, 4, 64, 64)
    D = bpa.make_desc(q, k, v, bias=full)
    assert tuple(D.bias_strides) == full.stride()


@pytest.mark.parametrize("bad", [
    dict(bias=torch.zeros(1, 1, 1, 64, dtype=torch.float64)),
    dict(bias=torch.zeros(64, 64)),
    dict(block_idx=torch.zeros(2, 4, 2, 8, dtype=torch.int64)),
    dict(seqlens_q=torch.zeros(2, dtype=torch.int64)),
    dict(seqlens_q=torch.zeros(3, dtype=torch.int32)),
    dict(seqlens_kv=torch.zeros(4, dtype=torch.int32)[::2]),
    dict(sink=torch.zeros(3)),
    dict(dsink=torch.zeros(4, dtype=torch.float64)),
    dict(o=torch.zeros(2, 64, 4, 8, dtype=torch.bfloat16)),
], ids=["bias_f64", "bias_2d", "block_idx_i64", "lens_i64", "lens_len", "lens_strided", "sink_len",
        "dsink_f64", "o_head_dim"])
def test_bad_arguments_are_refused_before_the_library(bpa, bad):
    q, k, v = _qkv()
    with pytest.raises(ValueError):
        bpa.make_desc(q, k, v, **bad)


def test_head_dim_must_be_contiguous(bpa):
    q, k, v = _qkv()
    with pytest.raises(ValueError):
        bpa.make_desc(q.transpose(2, 3), k, v)


def test_library_checks_the_marshalled_descriptor(bpa):
    q, k, v = _qkv()
    ok = bpa.make_desc(q, k, v, causal=True)
    assert bpa.bpa_workspace_size(bpa.BPA_OP_FWD, ok) >= 256
    # a ring that does not divide S, sequence lengths with a ring: refused by the library
    assert bpa.bpa_workspace_size(bpa.BPA_OP_FWD, bpa.make_desc(q, k, v, ring_size=3)) == 0
    lens = torch.tensor([64, 10], dtype=torch.int32)
    assert bpa.bpa_workspace_size(bpa.BPA_OP_FWD, bpa.make_desc(q, k, v, seqlens_q=lens, ring_size=2)) == 0
    # deterministic backward: one dQ slice per 128 keys (S = 64: one)
    base = bpa.bpa_workspace_size(bpa.BPA_OP_BWD, ok)
    det = bpa.bpa_workspace_size(bpa.BPA_OP_BWD, bpa.make_desc(q, k, v, causal=True, deterministic=True))
    assert det == base


def test_dropout_threshold_and_seed(bpa):
    from oracle import oracle
    q, k, v = _qkv()
    for p in (0.0, 0.1, 0.5, 0.999999999999):
        D = bpa.make_desc(q, k, v, dropout_p=p, dropout_seed=2 ** 64 + 7)
        # the same integer decision rule as the oracle's: round(p * 2^32), capped
        assert D.dropout_threshold == oracle.dropout_threshold(p)
        assert D.dropout_seed == 7 and D.dropout_reserved == 0
    with pytest.raises(ValueError):
        bpa.make_desc(q, k, v, dropout_p=1.0)
