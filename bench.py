#!/usr/bin/env python
"""Attention forward + backward throughput on GB300, TFLOP/s over unmasked score entries.

One step = bpa_fwd + bpa_bwd over one batch of the GQA causal workload
(B=2, S=4096, Hq=32, Hkv=8, d=128, bf16, seed 1), inputs resident in HBM.
FLOPs count only allowed (query, key) entries: 2*(d + dv) per entry forward
(Q K^T and P V), 6*d + 4*dv backward (the five contractions, recompute included);
4*d and 10*d for this workload (dv = d).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun: every rank runs its own replica of the workload
(independent batches, no collective on the data path) -> "scaling": "weak".
--impl reference times the float64 CPU oracle on the host cores (rank 0).
Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from ring_attention_gb300.inputs import WORKLOADS, GQA_CAUSAL, make_inputs, unmasked_entries  # noqa: E402

METRIC = "attention fwd/bwd TFLOP/s (unmasked FLOPs) and % of GB300 BF16 tensor peak"
FLUSH_BYTES = 256 << 20     # > 129 MB L2: written between timed steps
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def flops(w, entries):
    """Algorithmic FLOPs per allowed (query, key) entry: forward Q K^T (2 d) and P V (2 dv);
    backward the recomputed Q K^T, dP = dO V^T, dV = P^T dO (2 dv each but the first, 2 d),
    dK = dS^T Q and dQ = dS K (2 d each)."""
    d, dv = w.d, w.d_v
    return (2.0 * d + 2.0 * dv) * entries, (6.0 * d + 4.0 * dv) * entries


def max_over_ranks(x: float, device=None) -> float:
    """The largest x over the ranks of the initialised process group (x itself on one
    process): every rank's timed region is measured, the slowest one counts."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput of weak-scaled replicas: the units all ranks processed over
    the slowest rank's time."""
    return flops_per_step * steps * world / (max_ms * 1e-3) / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def code_digest(path: str) -> str:
    """sha256[:16] of a C / CUDA source with its comments and white space removed: edits to
    comments alone keep the digest, any change to the code changes it."""
    import re
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()[:16]


def kernel_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current code of the kernel (else None)."""
    src = {"k_bwd_tc": "bwd_tc.cu", "k_fwd_tc": "fwd_tc.cuh"}[kernel]
    path = os.path.join(ROOT, "ring_attention_gb300", "csrc", src)
    digest = code_digest(path)
    table = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(table):
        return None
    for line in open(table):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == digest:
            return float(parts[3])
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.idx)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.2)
        self.out = ""
        if self.proc:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_oracle_sample(w, budget_s: float):
    """Time the float64 oracle (fwd + bwd) on the largest S (power of two, same
    recipe, B=1) that fits the budget.  Returns (TFLOP/s, seconds, description, cores)."""
    from oracle import oracle
    oracle.build()
    S = 64
    best = None
    while S <= w.S:
        q, k, v, do, bias = make_inputs(w, B=1, S=S)
        t0 = time.perf_counter()
        oracle.attention_bwd(q, k, v, do, causal=w.causal, window=w.window, bias=bias)
        dt = time.perf_counter() - t0
        ent = unmasked_entries(w, S) // w.B
        f_fwd, f_bwd = flops(w, ent)
        best = ((f_fwd + f_bwd) / dt / 1e12, dt, S)
        if dt * 4.5 > budget_s:    # doubling S roughly quadruples the causal work
            break
        S *= 2
    tf, dt, S = best
    desc = (f"float64 oracle fwd+bwd on B=1, S={S}, Hq={w.Hq}, Hkv={w.Hkv}, d={w.d} of the same recipe "
            f"(seed {w.seed}); {dt:.2f} s")
    return tf, dt, desc, oracle.num_threads(), S


def oracle_baselines(budget_s: float = 15.0):
    """The float64 oracle timed on the host cores beside the GPU path (a reported baseline,
    not a target): full runs of the tiny fp32, sliding-window and block-selected workloads;
    the long ring workload on a reduced S of the same recipe, its full-run time extrapolated
    by the ratio of unmasked entries and labelled as such.  (The headline workload's sample
    is the line's cpu_baseline.)"""
    from oracle import oracle
    from ring_attention_gb300.inputs import BLOCK_SEL, GQA_SWA, RING_LONG, TINY_F32
    oracle.build()
    out = {"cores": oracle.num_threads(), "kind": "oracle"}
    for w in (TINY_F32, GQA_SWA):
        q, k, v, do, bias = make_inputs(w)
        t0 = time.perf_counter()
        oracle.attention_bwd(q, k, v, do, causal=w.causal, window=w.window, bias=bias)
        dt = time.perf_counter() - t0
        f = sum(flops(w, unmasked_entries(w)))
        out[w.name] = {"run": "full", "fwd_bwd_s": dt, "tflops": f / dt / 1e12}
    w = BLOCK_SEL
    q, k, v, _, _ = make_inputs(w)
    t0 = time.perf_counter()
    idx = oracle.select_blocks(q, k, block_size=w.sel_block, top_n=w.top_n)
    t1 = time.perf_counter()
    oracle.attention_fwd(q, k, v, causal=True, block_idx=idx, sel_block=w.sel_block, top_n=w.top_n,
                         local_window=w.local_window)
    t2 = time.perf_counter()
    out[w.name] = {"run": "full", "select_s": t1 - t0, "fwd_s": t2 - t1}
    w = RING_LONG
    tf, dt, _, _, S = cpu_oracle_sample(w, budget_s)
    part = unmasked_entries(w, S) // w.B
    out[w.name] = {"run": f"B=1, S={S} of the same recipe; full run extrapolated by unmasked entries",
                   "fwd_bwd_s": dt, "tflops": tf,
                   "extrapolated_full_fwd_bwd_s": dt * unmasked_entries(w) / part}
    return out


def time_extra_workloads(bpa, dev, peak_tf):
    """Secondary workloads (not the headline): device-timed per-call times.
    Inputs are drawn on the device from seeded generators (timing only; the
    parity tests use the numpy recipe)."""
    import torch
    from ring_attention_gb300.inputs import (BLOCK_SEL, BLOCK_SEL_JOINT, GQA_SWA, MLA_CAUSAL, RING_LONG, TINY_F32,
                                             VARLEN_CAUSAL)

    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    out = {}

    def rnd(shape, dtype, seed):
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        return torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(dtype)

    def fwd_bwd(w, steps, warmup, deterministic=False, dropout_p=0.0):
        dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        q = rnd((w.B, w.S, w.Hq, w.d), dt, w.seed)
        k = rnd((w.B, w.S, w.Hkv, w.d), dt, w.seed + 1)
        v = rnd((w.B, w.S, w.Hkv, w.d_v), dt, w.seed + 2)
        do = rnd((w.B, w.S, w.Hq, w.d_v), dt, w.seed + 3)
        bias = None
        if w.pad_tail:
            bias = torch.zeros((1, 1, 1, w.S), device=dev, dtype=torch.float32)
            bias[..., w.S - w.pad_tail:] = -1e9
        kw = dict(causal=w.causal, window=w.window, bias=bias, query_chunk=w.query_chunk, key_chunk=w.key_chunk,
                  ring_size=w.ring_size, deterministic=deterministic)
        if dropout_p:
            kw.update(dropout_p=dropout_p, dropout_seed=w.seed)
        tok_q = tok_k = w.B * w.S
        if w.seqlens_q:
            lens_q = list(w.seqlens_q)
            lens_k = list(w.seqlens_kv) if w.seqlens_kv else lens_q
            kw.update(seqlens_q=torch.tensor(lens_q, dtype=torch.int32, device=dev),
                      seqlens_kv=torch.tensor(lens_k, dtype=torch.int32, device=dev), bottom_right=w.bottom_right)
            tok_q, tok_k = sum(lens_q), sum(lens_k)
        D = bpa.make_desc(q, k, v, **kw)
        wsf = bpa.workspace(bpa.bpa_workspace_size(bpa.BPA_OP_FWD, D), dev)
        wsb = bpa.workspace(bpa.bpa_workspace_size(bpa.BPA_OP_BWD, D), dev)
        o, m, l = bpa.bpa_fwd(q, k, v, workspace_buf=wsf, **kw)
        dq, dk, dv = bpa.bpa_bwd(q, k, v, o, do, m, l, workspace_buf=wsb, **kw)
        # the iterations are queued back to back (one synchronise at the end), so that the host's
        # argument marshalling overlaps the previous call's kernels instead of showing up as
        # idle device time between an event and the first kernel
        evs = []
        for it in range(warmup + steps):
            a, b, c = E(), E(), E()
            a.record()
            bpa.bpa_fwd(q, k, v, o=o, m=m, l=l, workspace_buf=wsf, **kw)
            b.record()
            bpa.bpa_bwd(q, k, v, o, do, m, l, dq=dq, dk=dk, dv=dv, workspace_buf=wsb, **kw)
            c.record()
            evs.append((a, b, c))
        torch.cuda.synchronize()
        tf = [a.elapsed_time(b) for a, b, c in evs[warmup:]]
        tb = [b.elapsed_time(c) for a, b, c in evs[warmup:]]
        bpa.bpa_check(wsf)
        bpa.bpa_check(wsb)
        ent = unmasked_entries(w)
        f_fwd, f_bwd = flops(w, ent)
        mf, mb = statistics.mean(tf), statistics.mean(tb)
        el = 2 if dt == torch.bfloat16 else 4
        d, dv = w.d, w.d_v
        # valid tokens only: Q, K, V read, O written; backward + dO, O read, dQ, dK, dV written
        fwd_bytes = el * (tok_q * (d + dv) * w.Hq + tok_k * (d + dv) * w.Hkv)
        bwd_bytes = el * (tok_q * (2 * d + 2 * dv) * w.Hq + tok_k * (2 * d + 2 * dv) * w.Hkv)
        res = {"fwd_ms": mf, "bwd_ms": mb, "fwd_tflops": f_fwd / mf / 1e9, "bwd_tflops": f_bwd / mb / 1e9,
               "fwd_pct_peak": 100 * f_fwd / mf / 1e9 / peak_tf, "bwd_pct_peak": 100 * f_bwd / mb / 1e9 / peak_tf,
               "fwd_min_bytes_gbs": fwd_bytes / mf / 1e6, "bwd_min_bytes_gbs": bwd_bytes / mb / 1e6,
               "unmasked_entries": ent, "steps": steps}
        del q, k, v, do, o, dq, dk, dv, wsf, wsb
        torch.cuda.empty_cache()
        return res

    out[GQA_SWA.name] = fwd_bwd(GQA_SWA, 20, 3)
    out[TINY_F32.name] = fwd_bwd(TINY_F32, 20, 3)
    out[RING_LONG.name] = fwd_bwd(RING_LONG, 2, 1)
    out[MLA_CAUSAL.name] = fwd_bwd(MLA_CAUSAL, 10, 3)
    out[VARLEN_CAUSAL.name] = fwd_bwd(VARLEN_CAUSAL, 10, 3)
    # the headline workload with the determinism knob (per-key-tile dQ slices, ordered sum)
    out[GQA_CAUSAL.name + "_deterministic"] = fwd_bwd(GQA_CAUSAL, 10, 3, deterministic=True)
    # the headline workload with attention dropout (Philox4x32-10 keep decisions in the kernels)
    out[GQA_CAUSAL.name + "_dropout0.1"] = fwd_bwd(GQA_CAUSAL, 10, 3, dropout_p=0.1)

    def block_selected(w):
        q = rnd((w.B, w.S, w.Hq, w.d), torch.bfloat16, w.seed)
        k = rnd((w.B, w.S, w.Hkv, w.d), torch.bfloat16, w.seed + 1)
        v = rnd((w.B, w.S, w.Hkv, w.d), torch.bfloat16, w.seed + 2)
        idx = bpa.bpa_select_blocks(q, k, block_size=w.sel_block, top_n=w.top_n)
        kw = dict(causal=True, block_idx=idx, sel_block=w.sel_block, top_n=w.top_n, local_window=w.local_window)
        do = rnd((w.B, w.S, w.Hq, w.d), torch.bfloat16, w.seed + 3)
        o, m, l = bpa.bpa_fwd(q, k, v, **kw)
        wsb = bpa.workspace(bpa.bpa_workspace_size(bpa.BPA_OP_BWD, bpa.make_desc(q, k, v, **kw)), dev)
        dq, dk, dv = bpa.bpa_bwd(q, k, v, o, do, m, l, workspace_buf=wsb, **kw)
        evs = []
        for it in range(23):   # queued back to back, as above
            a, b, c, e = E(), E(), E(), E()
            a.record()
            bpa.bpa_select_blocks(q, k, block_size=w.sel_block, top_n=w.top_n, out=idx)
            b.record()
            bpa.bpa_fwd(q, k, v, o=o, m=m, l=l, **kw)
            c.record()
            bpa.bpa_bwd(q, k, v, o, do, m, l, dq=dq, dk=dk, dv=dv, workspace_buf=wsb, **kw)
            e.record()
            evs.append((a, b, c, e))
        torch.cuda.synchronize()
        ts = [a.elapsed_time(b) for a, b, c, e in evs[3:]]
        ta = [b.elapsed_time(c) for a, b, c, e in evs[3:]]
        tb = [c.elapsed_time(e) for a, b, c, e in evs[3:]]
        # algorithmic bytes: Q, K, V read once and O written once (the gathered re-reads come from L2);
        # backward: Q, K, V, O, dO read, dQ, dK, dV written
        qkvo = 2 * w.B * w.S * w.d * (2 * w.Hq + 2 * w.Hkv)
        bwd_bytes = 2 * w.B * w.S * w.d * (4 * w.Hq + 4 * w.Hkv)
        nb = (idx >= 0).sum().item()
        return {"select_ms": statistics.mean(ts), "attention_ms": statistics.mean(ta),
                "attention_min_bytes_gbs": qkvo / statistics.mean(ta) / 1e6,
                "backward_ms": statistics.mean(tb),
                "backward_min_bytes_gbs": bwd_bytes / statistics.mean(tb) / 1e6,
                "selected_blocks": int(nb), "steps": 20}

    out[BLOCK_SEL.name] = block_selected(BLOCK_SEL)
    out[BLOCK_SEL_JOINT.name] = block_selected(BLOCK_SEL_JOINT)
    return out


def run_reference(args, w):
    """Reference arm: the float64 CPU oracle, as it stands, on bounded samples."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import oracle
    oracle.build()
    per_step = max(0.05, 120.0 / max(1, args.steps + args.warmup))
    # pick the sample size once, then run warmup + timed steps on it
    tf, dt, desc, cores, S = cpu_oracle_sample(w, per_step)
    q, k, v, do, bias = make_inputs(w, B=1, S=S)
    ent = unmasked_entries(w, S) // w.B
    f = sum(flops(w, ent))
    for _ in range(args.warmup):
        oracle.attention_bwd(q, k, v, do, causal=w.causal, window=w.window, bias=bias)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention_bwd(q, k, v, do, causal=w.causal, window=w.window, bias=bias)
    el = time.perf_counter() - t0
    val = f * args.steps / el / 1e12
    sample = f"each step: float64 oracle fwd+bwd on B=1, S={S} of the workload's recipe ({ent} unmasked entries)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "sample": sample},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=GQA_CAUSAL.name, choices=sorted(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary workloads")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from ring_attention_gb300 import build as _build
    if rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    from ring_attention_gb300 import bpa

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- inputs (each rank: its own replica of the workload) -------------
    q_np, k_np, v_np, do_np, bias_np = make_inputs(w)

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    q, k, v, do = to_dev(q_np), to_dev(k_np), to_dev(v_np), to_dev(do_np)
    bias = to_dev(bias_np) if bias_np is not None else None
    kw = dict(causal=w.causal, window=w.window, bias=bias, query_chunk=w.query_chunk, key_chunk=w.key_chunk,
              ring_size=w.ring_size)
    D = bpa.make_desc(q, k, v, **kw)
    ws_f = bpa.workspace(bpa.bpa_workspace_size(bpa.BPA_OP_FWD, D), dev)
    ws_b = bpa.workspace(bpa.bpa_workspace_size(bpa.BPA_OP_BWD, D), dev)
    o = torch.empty_like(q)
    m = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32, device=dev)
    l = torch.empty_like(m)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(ev_f=None, ev_b=None):
        bpa.bpa_set_phase_events(ev_f)
        bpa.bpa_fwd(q, k, v, o=o, m=m, l=l, workspace_buf=ws_f, **kw)
        bpa.bpa_set_phase_events(ev_b)
        bpa.bpa_bwd(q, k, v, o, do, m, l, dq=dq, dk=dk, dv=dv, workspace_buf=ws_b, **kw)

    for _ in range(args.warmup):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    bpa.bpa_check(ws_f)
    bpa.bpa_check(ws_b)

    # ---- timed region ---------------------------------------------------
    K = args.steps
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [(E(), E()) for _ in range(K)]
    evf = [[E() for _ in range(3)] for _ in range(K)]
    evb = [[E() for _ in range(4)] for _ in range(K)]
    for e in [x for row in evf + evb for x in row]:
        e.record()   # creates the CUDA event; the library re-records it at its phase boundary
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for i in range(K):
            ev[i][0].record()
            step(evf[i], evb[i])
            ev[i][1].record()
            flush.zero_()          # L2 flush between steps (not timed)
        torch.cuda.synchronize()
        barrier()
        wall = time.perf_counter() - wall0
    bpa.bpa_check(ws_f)
    bpa.bpa_check(ws_b)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    fwd_ms = [e[0].elapsed_time(e[1]) for e in evf]
    bwd_main_ms = [e[1].elapsed_time(e[2]) for e in evb]
    bwd_pre_ms = [e[0].elapsed_time(e[1]) for e in evb]
    bwd_post_ms = [e[2].elapsed_time(e[3]) for e in evb]
    total_ms = max_over_ranks(sum(step_ms), dev)

    entries = unmasked_entries(w)
    f_fwd, f_bwd = flops(w, entries)
    value = aggregate_tflops(f_fwd + f_bwd, K, world, total_ms)
    ms_per_step = total_ms / K
    peaks, peaks_kind = load_peaks()
    peak_tf = float(peaks["bf16_tflops"])
    fwd_tf = f_fwd / (statistics.mean(fwd_ms) * 1e-3) / 1e12
    bwd_main_tf = f_bwd / (statistics.mean(bwd_main_ms) * 1e-3) / 1e12
    bwd_tf = f_bwd / (statistics.mean([a + b + c for a, b, c in zip(bwd_pre_ms, bwd_main_ms, bwd_post_ms)]) * 1e-3) / 1e12
    traffic = kernel_traffic("k_bwd_tc")

    # ---- end to end through the public API: pinned host -> device -> host --
    # Every step uploads its inputs from pinned host memory and downloads its outputs.  The
    # copies run on their own streams against two device buffer sets, so step i + 1's
    # uploads and step i - 1's downloads overlap step i's kernels; events order the reuse of
    # each buffer set.
    h_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (q, k, v, do)]
    for h, t in zip(h_in, (q, k, v, do)):
        h.copy_(t)
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, dq, dk, dv)]
    d_in = [[torch.empty_like(t) for t in (q, k, v, do)] for _ in range(2)]
    d_out = [[torch.empty_like(t) for t in (o, dq, dk, dv)] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    s_up, s_run, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of a set uploaded
    ev_used = [torch.cuda.Event() for _ in range(2)]    # the kernels reading a set's inputs are done
    ev_done = [torch.cuda.Event() for _ in range(2)]    # outputs of a set written
    ev_out = [torch.cuda.Event() for _ in range(2)]     # outputs of a set downloaded
    started = [False, False]

    def e2e_steps(n, t_start=None, t_end=None):
        if t_start is not None:
            t_start.record(s_up)
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_up):
                if started[b]:
                    s_up.wait_event(ev_used[b])
                for d_, h in zip(d_in[b], h_in):
                    d_.copy_(h, non_blocking=True)
                ev_in[b].record(s_up)
            s_run.wait_event(ev_in[b])
            if started[b]:
                s_run.wait_event(ev_out[b])
            xo, xdq, xdk, xdv = d_out[b]
            xq, xk, xv, xdo = d_in[b]
            bpa.bpa_fwd(xq, xk, xv, o=xo, m=m, l=l, workspace_buf=ws_f, stream=s_run, **kw)
            bpa.bpa_bwd(xq, xk, xv, xo, xdo, m, l, dq=xdq, dk=xdk, dv=xdv, workspace_buf=ws_b, stream=s_run, **kw)
            ev_used[b].record(s_run)
            ev_done[b].record(s_run)
            with torch.cuda.stream(s_down):
                s_down.wait_event(ev_done[b])
                for h, d_ in zip(h_out, d_out[b]):
                    h.copy_(d_, non_blocking=True)
                ev_out[b].record(s_down)
            started[b] = True
        if t_end is not None:
            s_up.wait_stream(s_down)
            t_end.record(s_up)

    e2e_steps(3)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = E(), E()
    e2e_steps(args.e2e_steps, e0, e1)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    e2e_val = aggregate_tflops(f_fwd + f_bwd, args.e2e_steps, world, e2e_ms)

    extra = None
    if rank == 0 and world == 1 and not args.no_extra:   # at N > 1 the other GPUs would idle meanwhile
        extra = time_extra_workloads(bpa, dev, peak_tf)

    cpu = None
    oracle_others = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, dt, desc, cores, _ = cpu_oracle_sample(w, 20.0)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}
        if not args.no_extra:
            oracle_others = oracle_baselines()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                       "causal": w.causal, "window": list(w.window), "unmasked_entries": entries,
                       "flops_per_step": f_fwd + f_bwd, "l2": "flushed between timed steps (256 MiB write)",
                       "parallelism": f"replicas x{world}"},
            "pct_of_peak": {"fwd": 100 * fwd_tf / peak_tf, "bwd": 100 * bwd_tf / peak_tf,
                            "step": 100 * value / world / peak_tf, "peak": f"bf16_tflops ({peaks_kind})"},
            "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
            "roofline": {"kernel": "k_bwd_tc (backward main kernel)", "bound": "tensor",
                         "achieved": bwd_main_tf, "peak": peak_tf, "unit": "TFLOP/s", "frac": bwd_main_tf / peak_tf,
                         "peak_kind": f"bf16_tflops, burst ({peaks_kind})",
                         "traffic": traffic},
            "roofline_fwd": {"kernel": "k_fwd_tc", "bound": "tensor", "achieved": fwd_tf, "peak": peak_tf,
                             "unit": "TFLOP/s", "frac": fwd_tf / peak_tf, "traffic": kernel_traffic("k_fwd_tc")},
            "kernel_ms": {"fwd": statistics.mean(fwd_ms), "bwd_pre": statistics.mean(bwd_pre_ms),
                          "bwd_main": statistics.mean(bwd_main_ms), "bwd_post": statistics.mean(bwd_post_ms)},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": 4 * K,
            "clocks": clocks.summary(),
            "wall_s_timed_region": wall,
            "extra": extra,
            "oracle_baselines": oracle_others,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
