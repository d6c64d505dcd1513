"""Host-side helpers of the seeded inputs: the entry count the throughput figures
divide by agrees with the oracle's own mask (with q = k = 0 every allowed key has
weight 1, so the row sums l count the allowed keys)."""
import json
import os
from dataclasses import replace

import numpy as np
import pytest

from ring_attention_gb300 import inputs as W


@pytest.mark.parametrize("w", [
    W.Workload("t_causal", B=2, S=40, Hq=2, Hkv=1, d=4, causal=True),
    W.Workload("t_swa", B=1, S=40, Hq=3, Hkv=1, d=4, causal=True, window=(5, 0)),
    W.Workload("t_win", B=1, S=40, Hq=1, Hkv=1, d=4, window=(3, 7)),
    W.Workload("t_varlen", B=3, S=40, Hq=2, Hkv=2, d=4, causal=True, seqlens_q=(40, 17, 0)),
    W.Workload("t_varlen_br", B=3, S=40, Hq=2, Hkv=1, d=4, causal=True, window=(6, 0),
               seqlens_q=(9, 40, 3), seqlens_kv=(30, 12, 0), bottom_right=True),
], ids=lambda w: w.name)
def test_unmasked_entries_counts_allowed_pairs(ora, w):
    z = np.zeros((w.B, w.S, w.Hq, w.d))
    zk = np.zeros((w.B, w.S, w.Hkv, w.d))
    _, _, l = ora.attention_fwd(z, zk, zk, causal=w.causal, window=w.window,
                                seqlens_q=list(w.seqlens_q) or None,
                                seqlens_kv=list(w.seqlens_kv) or None, bottom_right=w.bottom_right)
    assert W.unmasked_entries(w) == int(round(l.sum()))


def test_named_workload_counts():
    assert W.unmasked_entries(W.GQA_CAUSAL) == 2 * 32 * 4096 * 4097 // 2
    full = replace(W.VARLEN_CAUSAL, seqlens_q=())
    assert W.unmasked_entries(W.VARLEN_CAUSAL) < W.unmasked_entries(full)
    lens = W.VARLEN_CAUSAL.seqlens_q
    assert W.unmasked_entries(W.VARLEN_CAUSAL) == 32 * sum(n * (n + 1) // 2 for n in lens)


def test_mla_workload_matches_the_printed_shapes():
    # the page prints the MLA run's output and gradient shapes; the workload that stands in
    # for it must produce exactly those (o: [B, S, Hq, dv]; dq, dk, dv: q's, k's, v's shapes)
    with open(os.path.join(os.path.dirname(__file__), "golden", "mla_shapes.json")) as f:
        g = json.load(f)
    w = W.MLA_CAUSAL
    assert (w.d, w.d_v, w.seed) == (g["qk_head_dim"], g["v_head_dim"], g["seed"])
    assert [w.B, w.S, w.Hq, w.d_v] == g["output_shape"]
    assert [[w.B, w.S, w.Hq, w.d], [w.B, w.S, w.Hkv, w.d], [w.B, w.S, w.Hkv, w.d_v]] == g["grad_shapes"]
    q, k, v, do, _ = W.make_inputs(w, S=8)
    assert q.shape[-1] == 128 and k.shape[-1] == 128 and v.shape[-1] == 64 and do.shape[-1] == 64


def test_code_digest_ignores_comments_only(tmp_path):
    # the traffic figures stay tied to the kernel's code: comment edits keep the digest,
    # any change of code changes it
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    a = tmp_path / "a.cu"
    a.write_text("// head\nint f(int x) { /* twice */ return 2 * x; }\n")
    b = tmp_path / "b.cu"
    b.write_text("// another head\n\nint f(int x) {\n    return 2 * x;   // doubled\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) { return 3 * x; }\n")
    assert bench.code_digest(str(a)) == bench.code_digest(str(b)) != bench.code_digest(str(c))
