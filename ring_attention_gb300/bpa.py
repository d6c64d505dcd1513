"""ctypes binding of libbpa.so: the C entry points under the same names.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libbpa.  Tensors are torch CUDA tensors (PyTorch supplies device
memory and streams); their data pointers and strides are passed through the
C ABI declared in include/bpa.h.  There is no fallback: if the library is
missing or a call fails, a ``BpaError`` is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

BPA_OK, BPA_ERR_INVALID_ARG, BPA_ERR_UNSUPPORTED, BPA_ERR_WORKSPACE = 0, 1, 2, 3
BPA_ERR_CUDA, BPA_ERR_TIMEOUT, BPA_ERR_DEVICE_CHECK = 4, 5, 6
BPA_BF16, BPA_FP32 = 0, 1
BPA_OP_FWD, BPA_OP_BWD = 0, 1


class BpaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


class bpa_attn_desc(ctypes.Structure):
    _fields_ = [
        ("struct_size", ctypes.c_uint32), ("dtype", ctypes.c_int32),
        ("B", ctypes.c_int32), ("S", ctypes.c_int32), ("Hq", ctypes.c_int32),
        ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("q_strides", ctypes.c_int64 * 3), ("k_strides", ctypes.c_int64 * 3),
        ("v_strides", ctypes.c_int64 * 3),
        ("scale", ctypes.c_float), ("causal", ctypes.c_int32),
        ("window_left", ctypes.c_int32), ("window_right", ctypes.c_int32),
        ("bias", ctypes.c_void_p), ("bias_strides", ctypes.c_int64 * 4),
        ("query_chunk", ctypes.c_int32), ("key_chunk", ctypes.c_int32),
        ("ring_size", ctypes.c_int32), ("ring_step_begin", ctypes.c_int32),
        ("ring_step_end", ctypes.c_int32),
        ("block_idx", ctypes.c_void_p), ("sel_block", ctypes.c_int32),
        ("top_n", ctypes.c_int32), ("local_window", ctypes.c_int32),
        ("dv", ctypes.c_int32), ("o_strides", ctypes.c_int64 * 3),
        ("seqlens_q", ctypes.c_void_p), ("seqlens_kv", ctypes.c_void_p),
        ("bottom_right", ctypes.c_int32),
        ("sink", ctypes.c_void_p), ("dsink", ctypes.c_void_p),
        ("deterministic", ctypes.c_int32),
        ("dropout_threshold", ctypes.c_uint32), ("dropout_reserved", ctypes.c_uint32),
        ("dropout_seed", ctypes.c_uint64),
    ]


_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded libbpa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise BpaError(BPA_ERR_CUDA, f"{path} is missing: build it with ring_attention_gb300.build.build()")
        L = ctypes.CDLL(path)
        P, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
        dp = ctypes.POINTER(bpa_attn_desc)
        L.bpa_workspace_size.argtypes, L.bpa_workspace_size.restype = [i32, dp], sz
        L.bpa_fwd.argtypes, L.bpa_fwd.restype = [dp, P, P, P, P, sz, P], ctypes.c_int
        L.bpa_bwd.argtypes, L.bpa_bwd.restype = [dp, P, P, P, P, P, P, P, P, sz, P], ctypes.c_int
        L.bpa_select_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        L.bpa_select_workspace_size.restype = sz
        L.bpa_select_blocks.argtypes = [P, P, i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int64),
                                        ctypes.POINTER(ctypes.c_int64), i32, i32, P, P, sz, P]
        L.bpa_select_blocks.restype = ctypes.c_int
        L.bpa_check.argtypes, L.bpa_check.restype = [P], ctypes.c_int
        L.bpa_status_string.argtypes, L.bpa_status_string.restype = [ctypes.c_int], ctypes.c_char_p
        L.bpa_last_error.argtypes, L.bpa_last_error.restype = [], ctypes.c_char_p
        L.bpa_version.argtypes, L.bpa_version.restype = [], i32
        L.bpa_debug_wait_timeout.argtypes = [P, sz, ctypes.c_uint64, P]
        L.bpa_debug_wait_timeout.restype = ctypes.c_int
        L.bpa_select_noalloc_max_bytes.argtypes, L.bpa_select_noalloc_max_bytes.restype = [], sz
        L.bpa_select_blocks_noalloc.argtypes = [P, P, i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int64),
                                                ctypes.POINTER(ctypes.c_int64), i32, i32, P, P]
        L.bpa_select_blocks_noalloc.restype = ctypes.c_int
        L.bpa_set_phase_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32]
        L.bpa_set_phase_events.restype = None
        _lib = L
    return _lib


def _raise_if(status: int, what: str):
    if status != BPA_OK:
        L = lib()
        raise BpaError(status, f"{what}: {L.bpa_status_string(status).decode()}: {L.bpa_last_error().decode()}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BPA_BF16
    if t.dtype == torch.float32:
        return BPA_FP32
    raise TypeError(f"tensors must be bfloat16 or float32, got {t.dtype}")


def _bshd_strides(t: torch.Tensor, name: str):
    if t.dim() != 4:
        raise ValueError(f"{name} must be a 4-D BSHD tensor")
    if t.stride(3) != 1:
        raise ValueError(f"{name}: the head dimension must be contiguous")
    return (t.stride(0), t.stride(1), t.stride(2))


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def make_desc(q, k, v, *, o=None, causal=False, window=(-1, -1), scale=None, bias=None, query_chunk=0,
              key_chunk=0, ring_size=1, ring_steps=None, block_idx=None, sel_block=0, top_n=0,
              local_window=0, seqlens_q=None, seqlens_kv=None, bottom_right=False, sink=None,
              dsink=None, deterministic=False, dropout_p=0.0, dropout_seed=0) -> bpa_attn_desc:
    """Fill a bpa_attn_desc from torch tensors (no data is touched).  The value head dim
    is v's last dim; o (the output, or dout, which shares its strides) sets o_strides."""
    B, S, Hq, d = q.shape
    Hkv = k.shape[2]
    D = bpa_attn_desc()
    D.struct_size = ctypes.sizeof(bpa_attn_desc)
    D.dtype = _dtype_code(q)
    D.B, D.S, D.Hq, D.Hkv, D.d = B, S, Hq, Hkv, d
    D.q, D.k, D.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    D.q_strides[:] = _bshd_strides(q, "q")
    D.k_strides[:] = _bshd_strides(k, "k")
    D.v_strides[:] = _bshd_strides(v, "v")
    D.dv = v.shape[3]
    if o is not None:
        if o.shape[:3] != q.shape[:3] or o.shape[3] != v.shape[3]:
            raise ValueError("o / dout must be [B, S, Hq, dv]")
        D.o_strides[:] = _bshd_strides(o, "o")
    D.scale = 0.0 if scale is None else float(scale)
    D.causal = int(bool(causal))
    wl, wr = (-1, -1) if window is None else window
    D.window_left, D.window_right = int(wl), int(wr)
    if bias is not None:
        if bias.dtype != torch.float32 or bias.dim() != 4:
            raise ValueError("bias must be a 4-D float32 tensor [B|1, Hq|1, S|1, S|1]")
        D.bias = bias.data_ptr()
        D.bias_strides[:] = [0 if bias.shape[i] == 1 else bias.stride(i) for i in range(4)]
    D.query_chunk, D.key_chunk = int(query_chunk), int(key_chunk)
    D.ring_size = int(ring_size)
    if ring_steps is not None:
        D.ring_step_begin, D.ring_step_end = int(ring_steps[0]), int(ring_steps[1])
    if block_idx is not None:
        if block_idx.dtype != torch.int32 or not block_idx.is_contiguous():
            raise ValueError("block_idx must be a contiguous int32 tensor")
        D.block_idx = block_idx.data_ptr()
        D.sel_block, D.top_n, D.local_window = int(sel_block), int(top_n), int(local_window)
    for name, lens in (("seqlens_q", seqlens_q), ("seqlens_kv", seqlens_kv)):
        if lens is not None:
            if lens.dtype != torch.int32 or lens.shape != (B,) or not lens.is_contiguous() or lens.device != q.device:
                raise ValueError(f"{name} must be a contiguous int32 [B] tensor on q's device")
            setattr(D, name, lens.data_ptr())
    D.bottom_right = int(bool(bottom_right))
    for name, t in (("sink", sink), ("dsink", dsink)):
        if t is not None:
            if t.dtype != torch.float32 or t.shape != (Hq,) or not t.is_contiguous() or t.device != q.device:
                raise ValueError(f"{name} must be a contiguous float32 [Hq] tensor on q's device")
            setattr(D, name, t.data_ptr())
    D.deterministic = int(bool(deterministic))
    D.dropout_threshold = dropout_threshold(dropout_p)
    D.dropout_seed = int(dropout_seed) & (2 ** 64 - 1)
    return D


def dropout_threshold(p: float) -> int:
    """The descriptor's dropout threshold for drop probability p: round(p * 2^32), at most
    2^32 - 1 (entries whose 32-bit draw is below it are dropped)."""
    p = float(p)
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout_p must be in [0, 1)")
    return min(int(round(p * 4294967296.0)), 4294967295)


def bpa_workspace_size(op: int, desc: bpa_attn_desc) -> int:
    return int(lib().bpa_workspace_size(op, ctypes.byref(desc)))


def workspace(nbytes: int, device) -> torch.Tensor:
    """A device buffer of at least nbytes, 256-byte aligned (torch's allocator aligns to 512)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def bpa_fwd(q, k, v, *, o=None, m=None, l=None, workspace_buf=None, stream=None, **kw):
    """Forward pass.  Returns (o, m, l): o [B, S, Hq, dv] (v's head dim); m and l are
    float32 [B, Hq, S]."""
    B, S, Hq, _ = q.shape
    if o is None:
        if v.shape[3] == q.shape[3]:
            o = torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
        else:
            o = torch.empty(q.shape[:3] + (v.shape[3],), dtype=q.dtype, device=q.device)
    D = make_desc(q, k, v, o=o, **kw)
    if m is None:
        m = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    if l is None:
        l = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    if o.dtype != q.dtype:
        raise ValueError("o must have the dtype of q")
    need = bpa_workspace_size(BPA_OP_FWD, D)
    if need == 0:
        _raise_if(BPA_ERR_INVALID_ARG, "bpa_workspace_size")
    ws = workspace(need, q.device) if workspace_buf is None else workspace_buf
    st = lib().bpa_fwd(ctypes.byref(D), o.data_ptr(), m.data_ptr(), l.data_ptr(), ws.data_ptr(),
                       ws.numel(), _stream_ptr(stream))
    _raise_if(st, "bpa_fwd")
    return o, m, l


def bpa_bwd(q, k, v, o, dout, m, l, *, dq=None, dk=None, dv=None, workspace_buf=None, stream=None, **kw):
    """Backward pass.  Returns (dq, dk, dv) with the dtypes and strides of q, k, v;
    o and dout are [B, S, Hq, dv] with common strides."""
    D = make_desc(q, k, v, o=o, **kw)
    dq = torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device) if dq is None else dq
    dk = torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device) if dk is None else dk
    dv = torch.empty_strided(v.shape, v.stride(), dtype=v.dtype, device=v.device) if dv is None else dv
    for name, a, b in (("o", o, q), ("dout", dout, o), ("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if name == "o":
            if a.dtype != b.dtype:
                raise ValueError("o must have the dtype of q")
            continue
        if a.stride() != b.stride() or a.dtype != b.dtype:
            raise ValueError(f"{name} must share dtype and strides with its input")
    need = bpa_workspace_size(BPA_OP_BWD, D)
    if need == 0:
        _raise_if(BPA_ERR_INVALID_ARG, "bpa_workspace_size")
    ws = workspace(need, q.device) if workspace_buf is None else workspace_buf
    st = lib().bpa_bwd(ctypes.byref(D), o.data_ptr(), dout.data_ptr(), m.data_ptr(), l.data_ptr(),
                       dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(), ws.numel(),
                       _stream_ptr(stream))
    _raise_if(st, "bpa_bwd")
    return dq, dk, dv


def bpa_select_blocks(q, k, *, block_size=32, top_n=8, out=None, workspace_buf=None, stream=None):
    """Exact top-n block selection: int32 [B, H, S/block_size, top_n]."""
    B, S, H, d = q.shape
    if k.shape != q.shape or k.dtype != q.dtype:
        raise ValueError("q and k must share shape and dtype")
    qs = (ctypes.c_int64 * 3)(*_bshd_strides(q, "q"))
    ks = (ctypes.c_int64 * 3)(*_bshd_strides(k, "k"))
    nblk = S // block_size if block_size > 0 else 0
    if out is None:
        out = torch.empty((B, H, nblk, top_n), dtype=torch.int32, device=q.device)
    need = int(lib().bpa_select_workspace_size(B, S, H, d, block_size))
    if need == 0:
        raise BpaError(BPA_ERR_INVALID_ARG, "bpa_select_workspace_size: invalid sizes")
    ws = workspace(need, q.device) if workspace_buf is None else workspace_buf
    st = lib().bpa_select_blocks(q.data_ptr(), k.data_ptr(), _dtype_code(q), B, S, H, d, qs, ks,
                                 block_size, top_n, out.data_ptr(), ws.data_ptr(), ws.numel(),
                                 _stream_ptr(stream))
    _raise_if(st, "bpa_select_blocks")
    return out


def bpa_select_blocks_noalloc(q, k, *, block_size=32, top_n=8, out=None, stream=None):
    """bpa_select_blocks without a workspace: the library's built-in scratch buffer is used."""
    B, S, H, d = q.shape
    if k.shape != q.shape or k.dtype != q.dtype:
        raise ValueError("q and k must share shape and dtype")
    qs = (ctypes.c_int64 * 3)(*_bshd_strides(q, "q"))
    ks = (ctypes.c_int64 * 3)(*_bshd_strides(k, "k"))
    nblk = S // block_size if block_size > 0 else 0
    if out is None:
        out = torch.empty((B, H, nblk, top_n), dtype=torch.int32, device=q.device)
    st = lib().bpa_select_blocks_noalloc(q.data_ptr(), k.data_ptr(), _dtype_code(q), B, S, H, d, qs, ks,
                                         block_size, top_n, out.data_ptr(), _stream_ptr(stream))
    _raise_if(st, "bpa_select_blocks_noalloc")
    return out


def bpa_check(workspace_buf: torch.Tensor) -> None:
    """Raises BpaError if a kernel of the last call on this workspace reported a fault."""
    _raise_if(lib().bpa_check(workspace_buf.data_ptr()), "bpa_check")


def bpa_set_phase_events(events) -> None:
    """Record these torch.cuda.Event objects at the phase boundaries of the next
    bpa_fwd / bpa_bwd call on this thread (None clears the hook)."""
    if events is None:
        lib().bpa_set_phase_events(None, 0)
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    lib().bpa_set_phase_events(arr, len(events))


def bpa_debug_wait_timeout(workspace_buf: torch.Tensor, limit_ns: int, stream=None) -> None:
    st = lib().bpa_debug_wait_timeout(workspace_buf.data_ptr(), workspace_buf.numel(), int(limit_ns),
                                      _stream_ptr(stream))
    _raise_if(st, "bpa_debug_wait_timeout")
