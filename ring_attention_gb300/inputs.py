"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module holds no attention arithmetic: it only draws numbers and encodes
them.  Recipe (the pages draw with JAX ``PRNGKey(seed)``, which is not
available here): ``numpy.random.default_rng(seed).standard_normal(shape,
dtype=float32)`` drawn in the order Q, K, V, dO, then rounded to bfloat16
with round-to-nearest-even (the fp32 workload keeps the float32 draws).

bfloat16 tensors travel as ``uint16`` bit patterns so that exactly the same
bits reach the CPU oracle and the GPU.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass(frozen=True)
class Workload:
    """One attention problem: sizes, masks and the seed of its inputs."""
    name: str
    B: int
    S: int
    Hq: int
    Hkv: int
    d: int
    dtype: str = "bf16"          # "bf16" or "f32"
    causal: bool = False
    window: tuple = (-1, -1)     # inclusive (left, right); -1 = unbounded
    query_chunk: int = 128
    key_chunk: int = 128
    ring_size: int = 1
    pad_tail: int = 0            # bias [B,1,1,S]: -1e9 on the last pad_tail keys
    seed: int = 0
    sel_block: int = 0           # >0: top-n block-selected attention
    top_n: int = 0
    local_window: int = 0
    backward: bool = True
    dv: int = 0                  # head dim of v and dO; 0 = d
    seqlens_q: tuple = ()        # per batch entry: valid queries (empty: all S)
    seqlens_kv: tuple = ()       # valid keys (empty: the query lengths)
    bottom_right: bool = False   # causal / window diagonal at k = q + Lk - Lq
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def d_v(self) -> int:
        return self.dv or self.d


# The five workloads of the hot path, named by what they are.
TINY_F32 = Workload("tiny_fp32_gqa_causal_S256", B=1, S=256, Hq=4, Hkv=2, d=64, dtype="f32",
                    causal=True, query_chunk=64, key_chunk=64, seed=0)
GQA_CAUSAL = Workload("gqa_causal_B2_S4096_Hq32_Hkv8_d128", B=2, S=4096, Hq=32, Hkv=8, d=128,
                      causal=True, query_chunk=128, key_chunk=128, seed=1)
GQA_SWA = Workload("gqa_swa128_B2_S4096_Hq128_Hkv8_d128", B=2, S=4096, Hq=128, Hkv=8, d=128,
                   causal=True, window=(128, 0), seed=2026)
RING_LONG = Workload("ring8_causal_padbias_B1_S131072_Hq32_Hkv8_d128", B=1, S=131072, Hq=32,
                     Hkv=8, d=128, causal=True, query_chunk=512, key_chunk=1024, ring_size=8,
                     pad_tail=4096, seed=3)
BLOCK_SEL = Workload("blocksel_top8_B4_S8192_H8_d64", B=4, S=8192, Hq=8, Hkv=8, d=64,
                     causal=True, seed=4, sel_block=32, top_n=8, local_window=32, backward=False)

# Beyond the five: separate value head dim (q, k with 128 channels, v and the output with
# 64), the DeepSeek-style MLA shapes of the TransformerEngine page (section 4), causal.
MLA_CAUSAL = Workload("mla_causal_B2_S4096_Hq128_Hkv8_dqk128_dv64", B=2, S=4096, Hq=128, Hkv=8, d=128,
                      dv=64, causal=True, seed=2027)

# The joint view of the block-selected workload ("AnnAttention", faiss_block_attention
# flattens the heads into one embedding): the same numbers as BLOCK_SEL (one generator,
# the same seed and C order) read as one head of 8 x 64 = 512 channels, with backward.
BLOCK_SEL_JOINT = Workload("blocksel_joint_top8_B4_S8192_H1_d512", B=4, S=8192, Hq=1, Hkv=1, d=512,
                           causal=True, seed=4, sel_block=32, top_n=8, local_window=32)

# Variable-length (padded) batch of the GQA causal shape: eight sequences of mixed
# lengths in [B, 4096, H, d] tensors (the TransformerEngine page's sequence descriptor
# with padding), lengths chosen to straddle tile boundaries.
VARLEN_CAUSAL = Workload("varlen_gqa_causal_B8_S4096_Hq32_Hkv8_d128", B=8, S=4096, Hq=32, Hkv=8, d=128,
                         causal=True, seed=2028,
                         seqlens_q=(4096, 3511, 2987, 2048, 1536, 1023, 700, 129))

WORKLOADS = {w.name: w for w in (TINY_F32, GQA_CAUSAL, GQA_SWA, RING_LONG, BLOCK_SEL)}
EXTRA_WORKLOADS = {w.name: w for w in (MLA_CAUSAL, BLOCK_SEL_JOINT, VARLEN_CAUSAL)}


def draw(shape_list, seed: int, dtype: str):
    """Draw N(0,1) tensors in order from one seeded generator.

    Returns float32 arrays for dtype "f32", bfloat16 bit patterns otherwise."""
    rng = np.random.default_rng(seed)
    out = []
    for shape in shape_list:
        x = rng.standard_normal(shape, dtype=np.float32)
        out.append(x if dtype == "f32" else to_bf16_bits(x))
    return out


def make_inputs(w: Workload, *, S: int | None = None, B: int | None = None,
                Hq: int | None = None, Hkv: int | None = None):
    """q, k, v, dout (dout is None without a backward) and the bias (or None).

    Sizes may be overridden to draw a reduced case of the same recipe; the
    padding tail of the bias then scales with S."""
    B = w.B if B is None else B
    S = w.S if S is None else S
    Hq = w.Hq if Hq is None else Hq
    Hkv = w.Hkv if Hkv is None else Hkv
    shapes = [(B, S, Hq, w.d), (B, S, Hkv, w.d), (B, S, Hkv, w.d_v)]
    if w.backward:
        shapes.append((B, S, Hq, w.d_v))
    ts = draw(shapes, w.seed, w.dtype)
    q, k, v = ts[:3]
    dout = ts[3] if w.backward else None
    bias = None
    if w.pad_tail:
        tail = w.pad_tail * S // w.S
        bias = np.zeros((B, 1, 1, S), dtype=np.float32)
        bias[..., S - tail:] = -1e9
    return q, k, v, dout, bias


def unmasked_entries(w: Workload, S: int | None = None) -> int:
    """Number of (query, key) pairs the lengths and the causal / window mask allow,
    summed over the batch, times Hq.

    Counts positions only (a key with a -1e9 padding bias still counts)."""
    S = w.S if S is None else S
    total = 0
    for b in range(w.B):
        lq = w.seqlens_q[b] if w.seqlens_q else S
        lk = w.seqlens_kv[b] if w.seqlens_kv else lq
        off = lk - lq if w.bottom_right else 0
        c = np.arange(lq, dtype=np.int64) + off
        lo = np.zeros(lq, dtype=np.int64)
        hi = np.full(lq, lk - 1, dtype=np.int64)
        if w.causal:
            hi = np.minimum(hi, c)
        wl, wr = w.window
        if wr >= 0:
            hi = np.minimum(hi, c + wr)
        if wl >= 0:
            lo = np.maximum(lo, c - wl)
        total += int(np.maximum(hi - lo + 1, 0).sum())
    return total * w.Hq
