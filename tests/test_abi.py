"""The C-ABI library builds, loads and exports what include/bpa.h declares.

Runs without a GPU: only host-side argument validation is exercised (every
call here fails its checks before anything touches the device).
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bpa.h")


@pytest.fixture(scope="module")
def bpa():
    from ring_attention_gb300 import build
    build.build()
    from ring_attention_gb300 import bpa as mod
    return mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bpa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("bpa_fwd", "bpa_bwd", "bpa_select_blocks", "bpa_workspace_size", "bpa_check"):
        assert want in names


def test_library_exports_every_declared_symbol(bpa):
    L = bpa.lib()
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, f"not exported: {missing}"
    out = subprocess.run(["nm", "-D", "--defined-only", bpa.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (bpa_\w+)", out))
    assert set(declared_functions()) <= exported


def test_descriptor_layout_matches_c(tmp_path, bpa):
    # compile a host-only probe of the header and compare sizeof / offsetof
    fields = [f[0] for f in bpa.bpa_attn_desc._fields_]
    src = tmp_path / "probe.c"
    body = "\n".join(f'printf("{f} %zu\\n", offsetof(bpa_attn_desc, {f}));' for f in fields)
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "bpa.h"\nint main(void){\n'
                   'printf("size %zu\\n", sizeof(bpa_attn_desc));\n' + body + "\nreturn 0;}\n")
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                         check=True).stdout.splitlines())
    assert int(got["size"]) == ctypes.sizeof(bpa.bpa_attn_desc)
    for f in fields:
        assert int(got[f]) == getattr(bpa.bpa_attn_desc, f).offset, f


def _desc(bpa, **over):
    D = bpa.bpa_attn_desc()
    D.struct_size = ctypes.sizeof(bpa.bpa_attn_desc)
    D.dtype = bpa.BPA_BF16
    D.B, D.S, D.Hq, D.Hkv, D.d = 2, 256, 8, 2, 128
    D.q, D.k, D.v = 0x10000, 0x20000, 0x30000    # never dereferenced by host checks
    D.q_strides[:] = (256 * 8 * 128, 8 * 128, 128)
    D.k_strides[:] = (256 * 2 * 128, 2 * 128, 128)
    D.v_strides[:] = (256 * 2 * 128, 2 * 128, 128)
    D.window_left = D.window_right = -1
    D.ring_size = 1
    for k, v in over.items():
        setattr(D, k, v)
    return D


@pytest.mark.parametrize("over,status", [
    (dict(struct_size=8), 1),
    (dict(dtype=7), 1),
    (dict(Hq=6, Hkv=4), 1),
    (dict(d=513), 2),
    (dict(S=0), 1),
    (dict(q=0), 1),
    (dict(window_left=-2), 1),
    (dict(ring_size=3), 1),
    (dict(ring_size=2, query_chunk=100), 1),
    (dict(ring_size=2, ring_step_begin=2, ring_step_end=2), 1),
])
def test_forward_rejects_bad_arguments(bpa, over, status):
    D = _desc(bpa, **over)
    st = bpa.lib().bpa_fwd(ctypes.byref(D), 0x40000, 0x50000, 0x60000, 0x70000, 1 << 20, None)
    assert st == status, bpa.lib().bpa_last_error().decode()
    assert bpa.lib().bpa_last_error().decode() != ""


def test_workspace_is_checked_before_launch(bpa):
    D = _desc(bpa)
    L = bpa.lib()
    need = L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(D))
    assert need >= 256 and need % 256 == 0
    assert L.bpa_fwd(ctypes.byref(D), 0x40000, 0x50000, 0x60000, None, need, None) == bpa.BPA_ERR_WORKSPACE
    assert L.bpa_fwd(ctypes.byref(D), 0x40000, 0x50000, 0x60000, 0x70010, need, None) == bpa.BPA_ERR_WORKSPACE
    assert L.bpa_fwd(ctypes.byref(D), 0x40000, 0x50000, 0x60000, 0x70000, need - 1, None) == bpa.BPA_ERR_WORKSPACE


def test_workspace_sizes(bpa):
    L = bpa.lib()
    D = _desc(bpa)
    assert L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(D)) == 256
    D2 = _desc(bpa, ring_size=4)
    assert L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(D2)) == 256 + 4 * 2 * 256 * 8 * 128
    bw = L.bpa_workspace_size(bpa.BPA_OP_BWD, ctypes.byref(D))
    assert bw == 256 + 2 * (4 * 2 * 8 * 256) + 4 * 2 * 256 * 8 * 128
    assert L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(_desc(bpa, Hq=3))) == 0
    assert L.bpa_workspace_size(7, ctypes.byref(D)) == 0


def test_backward_rejects_bad_arguments(bpa):
    L = bpa.lib()
    D = _desc(bpa, ring_size=2, ring_step_end=1)
    p = 0x80000
    st = L.bpa_bwd(ctypes.byref(D), p, p, p, p, p, p, p, p, 1 << 30, None)
    assert st == bpa.BPA_ERR_INVALID_ARG
    D = _desc(bpa, block_idx=0x1000, sel_block=32, top_n=8, local_window=32, ring_size=2)
    assert L.bpa_bwd(ctypes.byref(D), p, p, p, p, p, p, p, p, 1 << 30, None) == bpa.BPA_ERR_INVALID_ARG
    D = _desc(bpa)
    assert L.bpa_bwd(ctypes.byref(D), p, 0, p, p, p, p, p, p, 1 << 30, None) == bpa.BPA_ERR_INVALID_ARG


def test_select_rejects_bad_arguments(bpa):
    L = bpa.lib()
    st = (ctypes.c_int64 * 3)(8192 * 8 * 64, 8 * 64, 64)
    p = 0x80000
    assert L.bpa_select_blocks(p, p, 0, 4, 8192, 8, 64, st, st, 33, 8, p, p, 1 << 30, None) == 1
    assert L.bpa_select_blocks(p, p, 0, 4, 8192, 8, 64, st, st, 32, 0, p, p, 1 << 30, None) == 1
    assert L.bpa_select_blocks(p, p, 0, 4, 8192, 8, 64, st, st, 32, 8, p, p, 16, None) == 3
    assert L.bpa_select_workspace_size(4, 8192, 8, 64, 32) == 256 + 2 * 4 * 8 * 256 * 64 * 8 + 4 * 8 * 256 * 64 * 4
    # more blocks per sequence than the selection kernel holds
    assert L.bpa_select_blocks(p, p, 0, 1, 4097 * 8, 1, 8, st, st, 8, 4, p, p, 1 << 40, None) == 2


def test_select_noalloc_reports_argument_errors_first(bpa):
    # a problem beyond the built-in scratch with a bad argument reports the argument,
    # exactly like the workspace entry point, not the scratch limit
    L = bpa.lib()
    st = (ctypes.c_int64 * 3)(65536 * 8 * 512, 8 * 512, 512)
    p = 0x80000
    big = (4, 65536, 8, 512, 32)      # far more than 16 MiB of block sums
    assert L.bpa_select_workspace_size(*big) > L.bpa_select_noalloc_max_bytes()
    assert L.bpa_select_blocks_noalloc(p, p, 0, *big[:4], st, st, 32, 100, p, None) == bpa.BPA_ERR_INVALID_ARG
    assert b"top_n" in L.bpa_last_error()
    assert L.bpa_select_blocks_noalloc(p, p, 0, *big[:4], st, st, 32, 8, 0, None) == bpa.BPA_ERR_INVALID_ARG
    assert L.bpa_select_blocks_noalloc(p, p, 0, *big[:4], st, st, 32, 8, p, None) == bpa.BPA_ERR_UNSUPPORTED
    assert b"scratch" in L.bpa_last_error()


def test_status_strings(bpa):
    L = bpa.lib()
    assert L.bpa_status_string(5) == b"BPA_ERR_TIMEOUT"
    assert L.bpa_version() == 6


def test_version_1_descriptor_is_accepted(bpa):
    """A caller built against descriptor version 1 passes the shorter struct_size: the
    value head dim defaults to d and the output strides to q's."""
    L = bpa.lib()
    D = _desc(bpa)
    full = L.bpa_workspace_size(bpa.BPA_OP_BWD, ctypes.byref(D))
    D.struct_size = bpa.bpa_attn_desc.dv.offset
    assert L.bpa_workspace_size(bpa.BPA_OP_BWD, ctypes.byref(D)) == full
    D.struct_size = bpa.bpa_attn_desc.dv.offset + 4
    assert L.bpa_workspace_size(bpa.BPA_OP_BWD, ctypes.byref(D)) == 0
    # version 2: no sequence lengths; the fields past the shorter struct are not read
    D = _desc(bpa, seqlens_q=0x1000, ring_size=2)
    D.struct_size = bpa.bpa_attn_desc.seqlens_q.offset
    assert L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(D)) > 0


def test_deterministic_checks_and_workspace(bpa):
    L = bpa.lib()
    D = _desc(bpa, deterministic=1, ring_size=2)
    assert L.bpa_workspace_size(bpa.BPA_OP_BWD, ctypes.byref(D)) == 0
    assert b"deterministic" in L.bpa_last_error()
    # one dQ slice per 128-key tile: S = 256 -> two slices of 4 * B * Hq * S' * d bytes
    base = L.bpa_workspace_size(bpa.BPA_OP_BWD, ctypes.byref(_desc(bpa)))
    det = L.bpa_workspace_size(bpa.BPA_OP_BWD, ctypes.byref(_desc(bpa, deterministic=1)))
    assert det - base == 4 * 2 * 8 * 256 * 128
    # version 4: the flag past the shorter struct is not read
    D = _desc(bpa, deterministic=1, ring_size=2)
    D.struct_size = bpa.bpa_attn_desc.deterministic.offset
    assert L.bpa_workspace_size(bpa.BPA_OP_BWD, ctypes.byref(D)) > 0


def test_sink_checks(bpa):
    L = bpa.lib()
    D = _desc(bpa, sink=0x2000, ring_size=2)
    assert L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(D)) == 0
    assert b"sink" in L.bpa_last_error()
    D = _desc(bpa, dsink=0x2000)
    assert L.bpa_workspace_size(bpa.BPA_OP_BWD, ctypes.byref(D)) == 0
    assert b"dsink needs a sink" in L.bpa_last_error()
    D = _desc(bpa, sink=0x2000, dsink=0x3000)
    assert L.bpa_workspace_size(bpa.BPA_OP_BWD, ctypes.byref(D)) == L.bpa_workspace_size(
        bpa.BPA_OP_BWD, ctypes.byref(_desc(bpa)))
    # version 3: the sink fields past the shorter struct are not read
    D = _desc(bpa, sink=0x2000, ring_size=2)
    D.struct_size = bpa.bpa_attn_desc.sink.offset
    assert L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(D)) > 0


def test_sequence_lengths_checks(bpa):
    L = bpa.lib()
    p = 0x80000
    for over in (dict(ring_size=2), dict(block_idx=0x1000, sel_block=32, top_n=8, local_window=32)):
        for field in ("seqlens_q", "seqlens_kv"):
            D = _desc(bpa, **{field: 0x2000}, **over)
            assert L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(D)) == 0
            assert b"sequence lengths" in L.bpa_last_error()
            assert L.bpa_fwd(ctypes.byref(D), p, p, p, p, 1 << 30, None) == bpa.BPA_ERR_INVALID_ARG
    # lengths with the full-sequence layout need no more workspace
    D0 = _desc(bpa)
    D1 = _desc(bpa, seqlens_q=0x2000, seqlens_kv=0x3000, bottom_right=1)
    assert L.bpa_workspace_size(bpa.BPA_OP_BWD, ctypes.byref(D1)) == L.bpa_workspace_size(
        bpa.BPA_OP_BWD, ctypes.byref(D0))


def test_value_head_dim_checks_and_sizes(bpa):
    L = bpa.lib()
    D = _desc(bpa, ring_size=2)
    base = L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(D))
    D.dv = D.d // 2   # separate value head dim: the forward ring carry is [B, S, Hq, dv]
    half = L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(D))
    assert half == 256 + (base - 256) // 2
    D.dv = 513
    assert L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(D)) == 0
    assert b"value head dim" in L.bpa_last_error()
    D.dv = -1
    assert L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(D)) == 0


def test_dropout_fields(bpa):
    L = bpa.lib()
    D = _desc(bpa, dropout_threshold=1 << 30, dropout_seed=2 ** 63 + 5)
    assert L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(D)) > 0
    D = _desc(bpa, dropout_threshold=1 << 30, dropout_reserved=1)
    assert L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(D)) == 0
    assert b"dropout_reserved" in L.bpa_last_error()
    # version 5: the dropout fields past the shorter struct are not read
    D = _desc(bpa, dropout_reserved=1)
    D.struct_size = bpa.bpa_attn_desc.dropout_threshold.offset
    assert L.bpa_workspace_size(bpa.BPA_OP_FWD, ctypes.byref(D)) > 0
