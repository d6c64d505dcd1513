"""Float64 CPU oracle for blockwise exact attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this module.  The CUDA
library never calls it, and it shares no code with the CUDA path: this file
only marshals numpy arrays into ``oracle.c`` (plain C, float64), which holds
all of the arithmetic and documents the definitions it follows.

Inputs are contiguous BSHD arrays: ``q [B,S,Hq,d]``, ``k [B,S,Hkv,d]``,
``v [B,S,Hkv,dv]``, ``dout [B,S,Hq,dv]``.  They may be float64, float32, or
bfloat16 bit patterns held in ``uint16`` arrays; the C side widens every
element exactly to double.  Outputs are float64; ``m`` and ``l`` are
``[B,Hq,S]`` in natural-log units of ``z = scale * q.k + bias``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_F64, _F32, _BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP, no FMA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


class _Desc(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("S", ctypes.c_int32), ("Hq", ctypes.c_int32),
        ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32), ("dv", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("causal", ctypes.c_int32), ("window_left", ctypes.c_int32),
        ("window_right", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
        ("bias", ctypes.c_void_p), ("bias_strides", ctypes.c_int64 * 4),
        ("block_idx", ctypes.c_void_p), ("sel_block", ctypes.c_int32),
        ("top_n", ctypes.c_int32), ("local_window", ctypes.c_int32),
        ("seqlens_q", ctypes.c_void_p), ("seqlens_kv", ctypes.c_void_p),
        ("bottom_right", ctypes.c_int32),
        ("sink", ctypes.c_void_p), ("dsink", ctypes.c_void_p),
        ("drop_threshold", ctypes.c_uint32), ("drop_seed_lo", ctypes.c_uint32),
        ("drop_seed_hi", ctypes.c_uint32),
    ]


_lib = None


def _bind(lib):
    """Declare the argument types of every exported oracle function."""
    P = ctypes.c_void_p
    dp = ctypes.POINTER(_Desc)
    i32 = ctypes.c_int32
    lib.ora_fwd.argtypes = [dp, P, P, P, P, P, P]
    lib.ora_bwd.argtypes = [dp, P, P, P, P, P, P, P, P, P, P]
    lib.ora_blockwise_fwd.argtypes = [dp, P, P, P, i32, i32, i32, P, P, P]
    lib.ora_rows.argtypes = [dp, P, P, P, P, i32, P, P, P, P, P]
    lib.ora_keys.argtypes = [dp, P, P, P, P, i32, i32, i32, P, P, P]
    lib.ora_select.argtypes = [P, P, i32, i32, i32, i32, i32, i32, i32, P]
    lib.ora_dropout_keep.argtypes = [dp, i32, i32, P]
    lib.ora_philox4x32_10.argtypes = [P, ctypes.c_uint32, ctypes.c_uint32, P]
    for f in ("ora_fwd", "ora_bwd", "ora_blockwise_fwd", "ora_rows", "ora_keys",
              "ora_select", "ora_num_threads", "ora_dropout_keep", "ora_philox4x32_10"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle runs on (OMP_NUM_THREADS, else all cores)."""
    return int(_load().ora_num_threads())


def _in(x):
    """Return (contiguous array, dtype code) for an input tensor."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float64:
        return x, _F64
    if x.dtype == np.float32:
        return x, _F32
    if x.dtype == np.uint16:
        return x, _BF16
    raise TypeError(f"oracle inputs must be float64, float32 or bf16 bits (uint16), got {x.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _desc(q, k, v, *, causal, window, scale, bias, block_idx, sel_block, top_n,
          local_window, in_dtype, seqlens_q=None, seqlens_kv=None, bottom_right=False, sink=None,
          dropout_p=0.0, dropout_seed=0):
    B, S, Hq, d = q.shape
    Hkv, dv = k.shape[2], v.shape[3]
    if k.shape != (B, S, Hkv, d) or v.shape != (B, S, Hkv, dv):
        raise ValueError("q, k, v shapes disagree")
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    D = _Desc()
    D.B, D.S, D.Hq, D.Hkv, D.d, D.dv = B, S, Hq, Hkv, d, dv
    D.scale = float(d ** -0.5 if scale is None else scale)
    D.causal = int(bool(causal))
    wl, wr = (-1, -1) if window is None else window
    D.window_left, D.window_right = int(wl), int(wr)
    D.in_dtype = in_dtype
    keep = []
    if bias is not None:
        b64 = np.asarray(bias, dtype=np.float64)
        if b64.ndim != 4:
            raise ValueError("bias must be 4-D [B|1, Hq|1, S|1, S|1]")
        full = (B, Hq, S, S)
        st = []
        for ax, (n, want) in enumerate(zip(b64.shape, full)):
            if n not in (1, want):
                raise ValueError(f"bias dim {ax} must be 1 or {want}")
        b64 = np.ascontiguousarray(b64)
        for ax in range(4):
            st.append(0 if b64.shape[ax] == 1 else b64.strides[ax] // 8)
        keep.append(b64)
        D.bias = b64.ctypes.data
        D.bias_strides[:] = st
    if block_idx is not None:
        bi = np.ascontiguousarray(block_idx, dtype=np.int32)
        if bi.shape != (B, Hq, S // sel_block, top_n):
            raise ValueError("block_idx must be [B, Hq, S/sel_block, top_n]")
        keep.append(bi)
        D.block_idx = bi.ctypes.data
        D.sel_block, D.top_n, D.local_window = sel_block, top_n, local_window
    for name, lens in (("seqlens_q", seqlens_q), ("seqlens_kv", seqlens_kv)):
        if lens is not None:
            ln = np.ascontiguousarray(lens, dtype=np.int32)
            if ln.shape != (B,) or ln.min() < 0 or ln.max() > S:
                raise ValueError(f"{name} must be [B] with values in [0, S]")
            keep.append(ln)
            setattr(D, name, ln.ctypes.data)
    D.bottom_right = int(bool(bottom_right))
    if sink is not None:
        sk = np.ascontiguousarray(sink, dtype=np.float64)
        if sk.shape != (Hq,):
            raise ValueError("sink must be [Hq]")
        keep.append(sk)
        D.sink = sk.ctypes.data
    _set_dropout(D, dropout_p, dropout_seed)
    return D, keep


def dropout_threshold(p: float) -> int:
    """Entries whose 32-bit draw is below this are dropped: round(p * 2^32)."""
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    return min(int(round(p * 2.0 ** 32)), 2 ** 32 - 1)


def _set_dropout(D, p, seed):
    D.drop_threshold = dropout_threshold(p)
    seed = int(seed) & (2 ** 64 - 1)
    D.drop_seed_lo, D.drop_seed_hi = seed & 0xFFFFFFFF, seed >> 32


def _check(rc, what):
    if rc:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def attention_fwd(q, k, v, *, causal=False, window=None, scale=None, bias=None,
                  block_idx=None, sel_block=32, top_n=8, local_window=32, seqlens_q=None,
                  seqlens_kv=None, bottom_right=False, sink=None, dropout_p=0.0, dropout_seed=0):
    """One-shot masked softmax attention.  Returns (o, m, l) in float64."""
    (q, dt), (k, _), (v, _) = _in(q), _in(k), _in(v)
    D, keep = _desc(q, k, v, causal=causal, window=window, scale=scale, bias=bias,
                    block_idx=block_idx, sel_block=sel_block, top_n=top_n,
                    local_window=local_window, in_dtype=dt, seqlens_q=seqlens_q,
                    seqlens_kv=seqlens_kv, bottom_right=bottom_right, sink=sink,
                    dropout_p=dropout_p, dropout_seed=dropout_seed)
    B, S, Hq, _ = q.shape
    o = np.zeros((B, S, Hq, v.shape[3]))
    m = np.zeros((B, Hq, S))
    l = np.zeros((B, Hq, S))
    _check(_load().ora_fwd(ctypes.byref(D), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(m),
                           _ptr(l)), "fwd")
    return o, m, l


def attention_bwd(q, k, v, dout, *, causal=False, window=None, scale=None, bias=None,
                  block_idx=None, sel_block=32, top_n=8, local_window=32, seqlens_q=None,
                  seqlens_kv=None, bottom_right=False, sink=None, want_dsink=False, dropout_p=0.0,
                  dropout_seed=0):
    """Analytic gradients.  Returns (dq, dk, dv, o, m, l) in float64, plus dsink [Hq]
    when want_dsink (a sink must be given)."""
    (q, dt), (k, _), (v, _), (dout, _) = _in(q), _in(k), _in(v), _in(dout)
    D, keep = _desc(q, k, v, causal=causal, window=window, scale=scale, bias=bias,
                    block_idx=block_idx, sel_block=sel_block, top_n=top_n,
                    local_window=local_window, in_dtype=dt, seqlens_q=seqlens_q,
                    seqlens_kv=seqlens_kv, bottom_right=bottom_right, sink=sink,
                    dropout_p=dropout_p, dropout_seed=dropout_seed)
    dsink = None
    if want_dsink:
        if sink is None:
            raise ValueError("want_dsink needs a sink")
        dsink = np.zeros(q.shape[2])
        D.dsink = dsink.ctypes.data
    B, S, Hq, d = q.shape
    Hkv, dv_ = k.shape[2], v.shape[3]
    dq = np.zeros((B, S, Hq, d))
    dk = np.zeros((B, S, Hkv, d))
    dv = np.zeros((B, S, Hkv, dv_))
    o = np.zeros((B, S, Hq, dv_))
    m = np.zeros((B, Hq, S))
    l = np.zeros((B, Hq, S))
    _check(_load().ora_bwd(ctypes.byref(D), _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq),
                           _ptr(dk), _ptr(dv), _ptr(o), _ptr(m), _ptr(l)), "bwd")
    if want_dsink:
        return dq, dk, dv, o, m, l, dsink
    return dq, dk, dv, o, m, l


def blockwise_fwd(q, k, v, *, query_chunk, key_chunk, ring_size=1, causal=False,
                  window=None, scale=None, bias=None):
    """The pages' blockwise carry, step by step, in ring order.  Returns (o, m, l)."""
    (q, dt), (k, _), (v, _) = _in(q), _in(k), _in(v)
    D, keep = _desc(q, k, v, causal=causal, window=window, scale=scale, bias=bias,
                    block_idx=None, sel_block=32, top_n=8, local_window=32, in_dtype=dt)
    B, S, Hq, _ = q.shape
    o = np.zeros((B, S, Hq, v.shape[3]))
    m = np.zeros((B, Hq, S))
    l = np.zeros((B, Hq, S))
    _check(_load().ora_blockwise_fwd(ctypes.byref(D), _ptr(q), _ptr(k), _ptr(v), query_chunk,
                                     key_chunk, ring_size, _ptr(o), _ptr(m), _ptr(l)),
           "blockwise_fwd")
    return o, m, l


def rows(q, k, v, dout, row_list, *, causal=False, window=None, scale=None, bias=None,
         seqlens_q=None, seqlens_kv=None, bottom_right=False):
    """O, m, l and dQ of the sampled (b, h, q) rows.  dout may be None (no dQ)."""
    (q, dt), (k, _), (v, _) = _in(q), _in(k), _in(v)
    if dout is not None:
        dout, _ = _in(dout)
    D, keep = _desc(q, k, v, causal=causal, window=window, scale=scale, bias=bias,
                    block_idx=None, sel_block=32, top_n=8, local_window=32, in_dtype=dt,
                    seqlens_q=seqlens_q, seqlens_kv=seqlens_kv, bottom_right=bottom_right)
    rl = np.ascontiguousarray(np.asarray(row_list, dtype=np.int32).reshape(-1, 3))
    n = rl.shape[0]
    o = np.zeros((n, v.shape[3]))
    m = np.zeros(n)
    l = np.zeros(n)
    dq = np.zeros((n, q.shape[3])) if dout is not None else None
    _check(_load().ora_rows(ctypes.byref(D), _ptr(q), _ptr(k), _ptr(v), _ptr(dout), n,
                            _ptr(rl), _ptr(o), _ptr(m), _ptr(l), _ptr(dq)), "rows")
    return o, m, l, dq


def keys(q, k, v, dout, b, g, key_list, *, causal=False, window=None, scale=None,
         bias=None, seqlens_q=None, seqlens_kv=None, bottom_right=False):
    """dK and dV of the sampled keys of kv head g at batch b."""
    (q, dt), (k, _), (v, _), (dout, _) = _in(q), _in(k), _in(v), _in(dout)
    D, keep = _desc(q, k, v, causal=causal, window=window, scale=scale, bias=bias,
                    block_idx=None, sel_block=32, top_n=8, local_window=32, in_dtype=dt,
                    seqlens_q=seqlens_q, seqlens_kv=seqlens_kv, bottom_right=bottom_right)
    kl = np.ascontiguousarray(np.asarray(key_list, dtype=np.int32).reshape(-1))
    n = kl.shape[0]
    dk = np.zeros((n, q.shape[3]))
    dv = np.zeros((n, v.shape[3]))
    _check(_load().ora_keys(ctypes.byref(D), _ptr(q), _ptr(k), _ptr(v), _ptr(dout), int(b),
                            int(g), n, _ptr(kl), _ptr(dk), _ptr(dv)), "keys")
    return dk, dv


def select_blocks(q, k, *, block_size=32, top_n=8):
    """Exact top-n earlier key blocks per query block.  q, k: [B,S,H,d] -> int32 [B,H,S/bs,top_n]."""
    (q, dt), (k, dt2) = _in(q), _in(k)
    if dt != dt2 or q.shape != k.shape:
        raise ValueError("q and k must share shape and dtype")
    B, S, H, d = q.shape
    if block_size < 1 or S % block_size:
        raise ValueError("S must be a multiple of block_size")
    out = np.zeros((B, H, S // block_size, top_n), dtype=np.int32)
    _check(_load().ora_select(_ptr(q), _ptr(k), dt, B, S, H, d, block_size, top_n, _ptr(out)),
           "select")
    return out


def dropout_keep(S, b, h, *, dropout_p, dropout_seed):
    """The dropout decisions of batch entry b, q head h: uint8 [S, S], 1 = kept."""
    D = _Desc()
    D.S = S
    _set_dropout(D, dropout_p, dropout_seed)
    keep = np.zeros((S, S), dtype=np.uint8)
    _check(_load().ora_dropout_keep(ctypes.byref(D), int(b), int(h), _ptr(keep)), "dropout_keep")
    return keep


def philox4x32_10(counter, key):
    """The oracle's Philox4x32-10: four uint32 counter words, two key words -> four words."""
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _check(_load().ora_philox4x32_10(_ptr(c), int(key[0]), int(key[1]), _ptr(out)), "philox")
    return out
