"""One pass of a named workload through the library, for profilers.

    python -m ring_attention_gb300.run_once --workload NAME [--B b] [--S s] [--passes fwd,bwd]
                                            [--warmup W] [--repeat R]

Draws the workload's seeded synthetic inputs (``inputs.make_inputs``; --B / --S shrink the
recipe), builds the library if needed and runs W warm-up rounds then R measured rounds of
the requested passes on cuda:0: ``fwd`` / ``bwd`` (bpa_fwd / bpa_bwd with the workload's
masks, bias, ring size and, for the block-selected workloads, the selection of
``select``), ``select`` (bpa_select_blocks).  A profiler skips the warm-up launches
(ncu -s) and captures the rest; the kernels' launch counts per round are printed.
Nothing is timed here: bench.py measures.
"""
from __future__ import annotations

import argparse
import sys


def main(argv=None) -> int:
    from ring_attention_gb300.inputs import BLOCK_SEL, BLOCK_SEL_JOINT, MLA_CAUSAL, VARLEN_CAUSAL, WORKLOADS

    names = dict(WORKLOADS)
    for w in (BLOCK_SEL_JOINT, MLA_CAUSAL, VARLEN_CAUSAL):
        names[w.name] = w
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", required=True, choices=sorted(names))
    ap.add_argument("--B", type=int, default=None)
    ap.add_argument("--S", type=int, default=None)
    ap.add_argument("--passes", default="fwd,bwd")
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--repeat", type=int, default=1)
    args = ap.parse_args(argv)

    import numpy as np
    import torch

    from ring_attention_gb300 import bpa, build
    from ring_attention_gb300.inputs import make_inputs

    build.build()
    w = names[args.workload]
    dev = torch.device("cuda:0")
    q, k, v, do, bias = make_inputs(w, B=args.B, S=args.S)

    def t(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    tq, tk, tv, tdo, tb = t(q), t(k), t(v), t(do), t(bias)
    B, S = tq.shape[0], tq.shape[1]
    kw = dict(causal=w.causal, window=w.window, bias=tb, query_chunk=w.query_chunk if S == w.S else 0,
              key_chunk=w.key_chunk if S == w.S else 0, ring_size=w.ring_size)
    for name in ("seqlens_q", "seqlens_kv"):
        if getattr(w, name):
            kw[name] = torch.tensor([min(x, S) for x in getattr(w, name)][:B], dtype=torch.int32, device=dev)
    kw["bottom_right"] = w.bottom_right
    passes = args.passes.split(",")
    idx = None
    if w.sel_block:
        idx = bpa.bpa_select_blocks(tq, tk, block_size=w.sel_block, top_n=w.top_n)
        kw.update(block_idx=idx, sel_block=w.sel_block, top_n=w.top_n, local_window=w.local_window)
    o = m = l = None

    def one_round():
        nonlocal o, m, l
        if "select" in passes:
            bpa.bpa_select_blocks(tq, tk, block_size=w.sel_block, top_n=w.top_n, out=idx)
        if "fwd" in passes or ("bwd" in passes and o is None):
            o, m, l = bpa.bpa_fwd(tq, tk, tv, **kw)
        if "bwd" in passes:
            bpa.bpa_bwd(tq, tk, tv, o, tdo if tdo is not None else torch.randn_like(o), m, l, **kw)

    for _ in range(args.warmup):
        one_round()
    torch.cuda.synchronize()
    for _ in range(args.repeat):
        one_round()
    torch.cuda.synchronize()
    print(f"{w.name}: B={B} S={S} passes={','.join(passes)} warmup={args.warmup} repeat={args.repeat}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
