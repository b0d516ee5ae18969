#!/usr/bin/env python3
"""Benchmark of one padding-free packed attention step on GB300.

A step is one pass of the hot path over one synthetic batch of the
long-document indexing workload (32 documents of 2048..8192 tokens, 16 heads x
64, bf16, forward only): pack the lengths (one host read), gather q, k and v
from their padded grids into packed buffers, plan the tiles, run the packed
attention forward, and scatter the output back to a zero-padded grid.

The metric is real-token TFLOP/s, 4 * sum_i L_i^2 * H * d per step divided by
the step time (tokens/s and the fraction of the tensor-core peak ride along).
Inputs (three 0.5 GB padded grids) are larger than the 129 MB L2, so no L2
flush runs between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload on the host cores (the only other place this file runs the oracle
is the cpu_baseline leg).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "packed attention real-token TFLOP/s and tokens/s; % of GB300 tensor-core peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            return json.load(fh), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def visible_pairs(lengths, first_token=False, window=None):
    """(query, key) pairs that attention computes: L^2 per sequence (L with a
    first-token query); with a local window (left, right) each query at
    position r sees keys max(r - left, 0) .. min(r + right, L - 1)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    if window is None:
        return int(lengths.sum()) if first_token else int((lengths ** 2).sum())
    left, right = window
    total = 0
    for length in lengths:
        pos = np.zeros(1, np.int64) if first_token else np.arange(length, dtype=np.int64)
        lo = np.maximum(pos - left, 0) if left >= 0 else np.zeros_like(pos)
        hi = np.minimum(pos + right, length - 1) if right >= 0 else np.full_like(pos, length - 1)
        total += int((hi - lo + 1).sum())
    return total


def real_flops(lengths, heads, head_dim, first_token=False, window=None):
    return float(4 * visible_pairs(lengths, first_token, window) * heads * head_dim)


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str | None = None):
        self.gpu_index = gpu_index
        self.proc = None
        # The raw samples go where --clocks-csv says, else to a temporary file.
        self.keep = path is not None
        self.path = path.replace("{gpu}", str(gpu_index)) if path else os.path.join(
            tempfile.gettempdir(), f"pe_clocks_gpu{gpu_index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, flag in zip(names, parts[5:9]):
                    if flag.lower() == "active":
                        reasons.add(name)
        if not self.keep:
            os.remove(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- traffic

def source_sha1(files) -> str:
    """sha1 of the concatenated kernel sources (the kernel's .cu file and the
    csrc headers whose code it inlines)."""
    h = hashlib.sha1()
    for name in files:
        path = os.path.join(ROOT, "padding_free_packed_gb300", "csrc", name)
        if not os.path.exists(path):
            return ""
        h.update(open(path, "rb").read())
    return h.hexdigest()


def committed_traffic(kernel_name: str, source_files, config: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (their sha1 is recorded in the summary) and for
    the same workload and mode (`config`, e.g. "longdoc_bf16" or
    "graph_fp32 first-token")."""
    path = os.path.join(ROOT, "profiles", f"{kernel_name}_traffic.txt")
    if not os.path.exists(path) or not source_files:
        return None
    fields = {}
    with open(path) as fh:
        for line in fh:
            key, _, value = line.partition(":")
            fields[key.strip()] = value.strip()
    sha = source_sha1(source_files)
    if fields.get("source_sha1") != sha or fields.get("config") != config:
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


_HEADERS = ["pe_common.cuh", "pe_sm103.cuh"]
KERNEL_SOURCES = {"tcgen05_bf16_d64": ["pe_fwd_sm103.cu"] + _HEADERS,
                  "simt_ffma": ["pe_fwd_simt.cu", "pe_fwd_simt.cuh", "pe_common.cuh"],
                  "first_token_gemv": ["pe_first_token.cu", "pe_token_stream.cuh"] + _HEADERS,
                  "first_token_bwd": ["pe_first_token_bwd.cu", "pe_token_stream.cuh"] + _HEADERS,
                  "tcgen05_f32_d64": ["pe_fwd_sm103_f32.cu"] + _HEADERS,
                  "tcgen05_bf16_d128": ["pe_fwd_sm103_d128.cu"] + _HEADERS,
                  "tcgen05_bf16_d64_bwd": ["pe_bwd_sm103.cu", "pe_bwd_sm103.cuh",
                                           "pe_bwd_simt.cu"] + _HEADERS,
                  "tcgen05_bf16_d128_bwd": ["pe_bwd_sm103_d128.cu", "pe_bwd_sm103.cuh",
                                            "pe_bwd_simt.cu"] + _HEADERS}


# --------------------------------------------------------------------------- our arm

def run_ours(args, rank, world):
    import torch

    import padding_free_packed_gb300 as pe
    from padding_free_packed_gb300 import workloads

    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pe.load_library()
    wl = workloads.WORKLOADS[args.workload]
    if (args.dtype and args.dtype != wl.dtype) or args.heads or args.head_dim:
        if not args.packed:
            raise SystemExit("--dtype, --heads and --head-dim need --packed")
        import dataclasses
        dt = args.dtype or wl.dtype
        h_, d_ = args.heads or wl.num_heads, args.head_dim or wl.head_dim
        wl = dataclasses.replace(wl, dtype=dt, num_heads=h_, head_dim=d_,
                                 description=f"{wl.description}, as {h_}x{d_} {dt}")
    # Weak scaling: every rank draws its own batch of the same workload.
    train = wl.backward or args.backward
    rows_layout = args.layout == "rows"
    if rows_layout:
        # Documents packed several to a padded row (an indexed packing mask).
        drawn = workloads.make_packed_row_inputs(args.workload, args.row_len, seed=args.seed + rank,
                                                 with_dout=train, max_sequences=args.sequences)
        lengths, row_ids = drawn[0], drawn[1]
        host_grids = list(drawn[2:])
    elif args.packed:
        # Already-packed inputs (a pipeline that collates without padding):
        # the step is the attention forward (and backward) alone.
        lengths = workloads.draw_lengths(args.workload, np.random.default_rng(args.seed + rank))
        if args.sequences:
            lengths = np.ascontiguousarray(lengths[: args.sequences])
        xin = workloads.make_custom(lengths, wl.num_heads, wl.head_dim, wl.torch_dtype,
                                    seed=args.seed + rank, with_dout=train)
        host_grids = [xin.q, xin.k, xin.v] + ([xin.dout] if train else [])
    else:
        drawn = workloads.make_padded_inputs(args.workload, seed=args.seed + rank,
                                             max_sequences=args.sequences, with_dout=train)
        lengths = drawn[0]
        host_grids = list(drawn[1:])
    gq = host_grids[0]
    s, h, d = wl.max_seq_len, wl.num_heads, wl.head_dim
    n_tokens = int(lengths.astype(np.int64).sum())
    if args.first_token:
        if not args.packed:
            raise SystemExit("--first-token needs --packed")
        train = args.backward   # a workload's own backward step is for full attention
    window = tuple(args.window) if args.window else None
    fwd_flops = real_flops(lengths, h, d, first_token=args.first_token, window=window)
    bwd_flops = 2.5 * fwd_flops if train else 0.0   # 10 sum L^2 H d: five GEMM-shaped products
    flops = fwd_flops + bwd_flops
    kernel = pe.pe_attention_kernel(wl.torch_dtype, d, query_is_first_token=args.first_token,
                                    window=window, max_seq_len=s)
    bwd_kernel = pe.pe_attention_kernel(wl.torch_dtype, d, query_is_first_token=args.first_token,
                                        backward=True, window=window,
                                        max_seq_len=s) if train else None

    # The per-step layout metadata: lengths, or the packed rows' mask.
    meta_host = row_ids if rows_layout else lengths
    lengths_d = torch.from_numpy(meta_host).to(dev)
    dev_grids = [t.to(dev) for t in host_grids]
    og = (torch.empty((n_tokens, h, d), dtype=dev_grids[0].dtype, device=dev) if rows_layout
          else torch.empty_like(dev_grids[0]))
    grad_grids = ([torch.empty_like(og) for _ in range(3)] if rows_layout else
                  [torch.empty_like(dev_grids[0]) for _ in range(3)]) if train else None
    packed_cu = pe.pe_pack_sequences(lengths_d, s)[1] if args.packed else None
    q_first = (dev_grids[0][packed_cu[:-1].long()].contiguous()
               if args.packed and args.first_token else None)
    do_first = (dev_grids[3][packed_cu[:-1].long()].contiguous()
                if args.packed and args.first_token and train else None)
    stream = torch.cuda.current_stream(dev)
    fwd_events, bwd_events = [], []
    # One workspace per direction for every call (all attention calls run on
    # one stream); their status words are read once after the timed region.
    n_seq = int(len(lengths))
    ws_fwd = torch.empty(max(16, pe.attention_workspace_bytes(
        wl.torch_dtype, n_seq, n_tokens, h, d, s, args.first_token, False)),
        dtype=torch.uint8, device=dev)
    ws_bwd = torch.empty(max(16, pe.attention_workspace_bytes(
        wl.torch_dtype, n_seq, n_tokens, h, d, s, args.first_token, True)),
        dtype=torch.uint8, device=dev) if train else None

    # Full attention, or local attention with the --window bounds.
    def attention_fwd(*a, **kw):
        kw["workspace"] = ws_fwd
        if window is None:
            return pe.pe_packed_attention_fwd(*a, **kw)
        q_, k_, v_, cu_, s_, scale_ = a
        return pe.pe_packed_attention_fwd_local(q_, k_, v_, cu_, s_, window[0], window[1],
                                                scale_, **kw)

    def attention_bwd(*a):
        ft = bool(args.first_token)
        if window is None:
            return pe.pe_packed_attention_bwd(*a, query_is_first_token=ft, workspace=ws_bwd)
        return pe.pe_packed_attention_bwd_local(*a[:8], window[0], window[1], a[8],
                                                query_is_first_token=ft, workspace=ws_bwd)

    def timed(record, events, fn):
        if not record:
            return fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        result = fn()
        e1.record(stream)
        events.append((e0, e1))
        return result

    def step(lengths_t, grids, record, outs=None):
        # outs: (output buffer, gradient buffers) to write into; the shared
        # ones by default, a pipeline buffer set in the end-to-end leg.
        o_buf, g_bufs = outs if outs is not None else (og, grad_grids)
        if args.packed:
            cu = packed_cu
            q, k, v = grids[:3]
            if args.first_token:
                out, lse = timed(record, fwd_events, lambda: attention_fwd(
                    q_first, k, v, cu, s, wl.scale, query_is_first_token=True, need_lse=train))
                if train:
                    timed(record, bwd_events, lambda: attention_bwd(
                        do_first, q_first, k, v, out, lse, cu, s, wl.scale))
                return n_tokens
        elif rows_layout:
            flat, cu, n = pe.pe_pack_document_ids(lengths_t)
            q, k, v = (pe.pe_gather_packed(g, flat, n) for g in grids[:3])
        else:
            flat, cu, n = pe.pe_pack_sequences(lengths_t, s)
            q, k, v = (pe.pe_gather_packed(g, flat, n) for g in grids[:3])
        out, lse = timed(record, fwd_events,
                         lambda: attention_fwd(q, k, v, cu, s, wl.scale, need_lse=train))
        if args.packed or rows_layout:
            o_buf.copy_(out)       # packed rows: the output stays packed (a THD consumer)
        else:
            pe.pe_scatter_padded(out, cu, s, out=o_buf)
        if train:
            do = grids[3] if args.packed else pe.pe_gather_packed(grids[3], flat, n)
            grads = timed(record, bwd_events,
                          lambda: attention_bwd(do, q, k, v, out, lse, cu, s, wl.scale))
            for g, grid in zip(grads, g_bufs):
                if args.packed or rows_layout:
                    grid.copy_(g)
                else:
                    pe.pe_scatter_padded(g, cu, s, out=grid)
        return n_tokens

    # Padded steps: pack scan+fill, 3 gathers, plan+attention, scatter; training
    # adds the dO gather, the backward (delta, plan, key pass, plan, query pass)
    # and 3 scatters. Packed steps: plan+attention (+ the 5 backward launches).
    if args.packed and args.first_token:   # layout check, streaming kernel, merge (each way)
        launches_per_step = 3 + (3 if train else 0)
    elif args.packed:
        launches_per_step = 2 + (5 if train else 0)
    elif rows_layout:   # mask count, scan, fill, 3 gathers, plan + attention (+ dO gather, backward)
        launches_per_step = 3 + 3 + 2 + ((1 + 5) if train else 0)
    else:
        launches_per_step = 2 + 3 + 2 + 1 + ((1 + 5 + 3) if train else 0)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step(lengths_d, dev_grids, False)
    barrier()
    with ClockSampler(local_rank, args.clocks_csv) as clocks:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(args.steps):
            step(lengths_d, dev_grids, True)
        end.record(stream)
        barrier()
    elapsed_ms = start.elapsed_time(end)
    # What the kernels found (layout check, bounded waits): 0 when every call
    # of the timed region completed normally.
    device_status = {"forward": pe.pe_read_device_status(ws_fwd)}
    if train:
        device_status["backward"] = pe.pe_read_device_status(ws_bwd)
    fwd_ms = sum(a.elapsed_time(b) for a, b in fwd_events) / len(fwd_events)
    bwd_ms = sum(a.elapsed_time(b) for a, b in bwd_events) / len(bwd_events) if train else 0.0
    if world > 1:
        t = torch.tensor([elapsed_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    ms_per_step = elapsed_ms / args.steps

    # End to end through the same public calls: pinned host grids in, padded
    # output (and gradients) back to pinned host memory, every step's copies
    # inside the timed region. Steps are pipelined as a serving or training
    # loop would run them: the host-to-device copies of step i+1 (on their own
    # stream) and the device-to-host copy of step i-1's result (on a third)
    # overlap step i's compute, with two buffer sets alternating.
    e2e = None
    if not args.no_e2e and not (args.packed or rows_layout):
        e2e = e2e_padded(args, pe, torch, dev, stream, lengths, host_grids, s, wl, train,
                         flops, n_tokens, attention_fwd, attention_bwd, barrier, world)
    elif not args.no_e2e:
        host_in = [t.pin_memory() for t in host_grids]
        hlen = torch.from_numpy(meta_host).pin_memory()
        nbuf = 2
        dev_in = [[torch.empty_like(t, device=dev) for t in host_in] for _ in range(nbuf)]
        dlen = [torch.empty_like(lengths_d) for _ in range(nbuf)]
        outs = [(torch.empty_like(og), [torch.empty_like(g) for g in grad_grids] if train else None)
                for _ in range(nbuf)]
        host_out = [[torch.empty_like(t, device="cpu").pin_memory()
                     for t in [o] + (g if g is not None else [])] for o, g in outs]
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        comp = stream
        in_free = [torch.cuda.Event() for _ in range(nbuf)]    # compute done with inputs b
        in_ready = [torch.cuda.Event() for _ in range(nbuf)]   # inputs b uploaded
        out_ready = [torch.cuda.Event() for _ in range(nbuf)]  # results b computed
        out_free = [torch.cuda.Event() for _ in range(nbuf)]   # results b downloaded
        for b in range(nbuf):
            for ev in (in_free[b], out_free[b]):
                ev.record(comp)

        def upload(i):
            b = i % nbuf
            up.wait_event(in_free[b])
            with torch.cuda.stream(up):
                dlen[b].copy_(hlen, non_blocking=True)
                for dst, src in zip(dev_in[b], host_in):
                    dst.copy_(src, non_blocking=True)
                in_ready[b].record(up)

        def compute_and_download(i):
            b = i % nbuf
            comp.wait_event(in_ready[b])
            comp.wait_event(out_free[b])
            step(dlen[b], dev_in[b], False, outs[b])
            in_free[b].record(comp)
            out_ready[b].record(comp)
            down.wait_event(out_ready[b])
            with torch.cuda.stream(down):
                results = [outs[b][0]] + (outs[b][1] if train else [])
                for dst, src in zip(host_out[b], results):
                    dst.copy_(src, non_blocking=True)
                out_free[b].record(down)

        def run(n):
            upload(0)
            for i in range(n):
                if i + 1 < n:
                    upload(i + 1)              # the next step's inputs, during this compute
                compute_and_download(i)

        run(max(2, min(args.warmup, 3)))
        torch.cuda.synchronize(dev)
        barrier()
        e2e_steps = max(2, min(args.steps, 10))
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(comp)
        up.wait_event(t0)
        run(e2e_steps)
        comp.wait_stream(down)
        comp.wait_stream(up)
        t1.record(comp)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_ms = t0.elapsed_time(t1) / e2e_steps
        if world > 1:
            t = torch.tensor([e2e_ms], device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            e2e_ms = float(t.item())
        h2d = sum(x.numel() * x.element_size() for x in [hlen] + host_in)
        d2h = sum(x.numel() * x.element_size() for x in host_out[0])
        e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "pipelined": "uploads of step i+1 and downloads of step i-1 overlap step i"}

    peaks, peaks_src = load_peaks()
    # The dominant kernel: the forward, or the backward when it takes longer.
    if train and bwd_ms > fwd_ms:
        dom_kernel, dom_flops, dom_ms = bwd_kernel, bwd_flops, bwd_ms
    else:
        dom_kernel, dom_flops, dom_ms = kernel, fwd_flops, fwd_ms
    if dom_kernel == "tcgen05_f32_d64":
        # fp32 operands split into bf16 hi + lo: three bf16 products per fp32
        # product, so the ceiling for the useful flops is a third of bf16's.
        bound, peak, unit = "tensor", float(peaks["bf16_tflops"]) / 3.0, "TFLOP/s"
        peak_note = f"dense bf16 burst / 3 (three bf16 products per fp32 product), {peaks_src}"
    elif dom_kernel.startswith("tcgen05"):
        bound, peak, unit = "tensor", float(peaks["bf16_tflops"]), "TFLOP/s"
        peak_note = f"dense bf16 burst, {peaks_src}"
    elif dom_kernel in ("first_token_gemv", "first_token_bwd"):
        bound, peak, unit = "hbm", float(peaks["hbm_gbs"]), "GB/s"
        peak_note = f"HBM copy, {peaks_src}"
    else:
        ffma = (torch.cuda.get_device_properties(dev).multi_processor_count * 128 * 2
                * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12)
        bound, peak, unit = "alu", ffma, "TFLOP/s"
        peak_note = "FFMA: SMs x 128 lanes x 2 flop x max SM clock"
    if bound == "hbm":
        esize = 4 if wl.dtype == "fp32" else 2
        if dom_kernel == "first_token_bwd":
            # k, v read and dk, dv written once; q, dO, out read and dq written
            # once per sequence and head; lse read.
            hbm_bytes = (4 * n_tokens + 4 * len(lengths)) * h * d * esize + 4 * h * len(lengths)
        else:
            # k and v read once, q read and the output written once per sequence and head.
            hbm_bytes = (2 * n_tokens + 2 * len(lengths)) * h * d * esize
        achieved = hbm_bytes / (dom_ms * 1e-3) / 1e9
    else:
        achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    traffic_config = (args.workload + (f"[:{args.sequences}]" if args.sequences else "")
                      + (f" as {wl.num_heads}x{wl.head_dim} {wl.dtype}"
                         if (args.dtype or args.heads or args.head_dim) else "")
                      + (" first-token" if args.first_token else "")
                      + (f" window {window[0]} {window[1]}" if window else "")
                      + (" backward" if train and dom_kernel == bwd_kernel else "")
                      + (f" seed {args.seed + rank}" if args.seed + rank else ""))
    traffic = committed_traffic(dom_kernel, KERNEL_SOURCES.get(dom_kernel), traffic_config)
    value = world * flops / (ms_per_step * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": args.workload + (f"[:{args.sequences}]" if args.sequences else "")
                   + (f" as {wl.num_heads}x{wl.head_dim} {wl.dtype}"
                      if (args.dtype or args.heads or args.head_dim) else ""),
                   "description": wl.description,
                   "num_sequences": int(len(lengths)), "num_tokens": n_tokens,
                   "heads": h, "head_dim": d, "max_seq_len": s,
                   "attention": (f"local window ({window[0]}, {window[1]})" if window
                                 else "full") + (", first-token query" if args.first_token
                                                 else ""),
                   "layout": (f"documents packed into rows of {args.row_len} (indexed packing "
                              "mask)" if rows_layout else
                              "packed" if args.packed else "one sequence per padded row"),
                   "step": ("mask -> flat_index/cu_seqlens + gather q,k,v + tile plan + attention "
                            "forward" + (" + dO gather + backward" if train else "")
                            + " (outputs stay packed)") if rows_layout else
                           (("tile plan + attention forward + backward on packed inputs"
                             if train else "tile plan + attention forward on packed inputs")
                            if args.packed else
                            ("pack + gather q,k,v,dO + tile plan + attention forward + scatter "
                             "+ attention backward + scatter dq,dk,dv" if train else
                             "pack + gather q,k,v + tile plan + attention forward + scatter")),
                   "flops_per_step": flops,
                   "l2": (f"{len(host_grids)} {'packed buffers' if args.packed else 'padded grids'}"
                          f" of {gq.numel() * gq.element_size() / 1e9:.2f} GB"
                          + ("; larger than L2, no flush"
                             if gq.numel() * gq.element_size() > 129e6 else
                             "; smaller than L2 (profiling case)")),
                   "parallelism": f"dp{world} (independent batches per GPU, no collective)"},
        "tokens_per_s": world * n_tokens / (ms_per_step * 1e-3),
        "pct_of_tensor_peak": 100.0 * value / world / float(peaks["bf16_tflops"]),
        "attention_kernel": kernel,
        "attention_ms": fwd_ms,
        "backward_kernel": bwd_kernel,
        "backward_ms": bwd_ms if train else None,
        "roofline_kernel": dom_kernel,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_note,
                     "frac_of_sustained": (achieved / (float(peaks["bf16_tflops_sustained"]) * peak
                                                      / float(peaks["bf16_tflops"]))
                                           if bound == "tensor" else None)},
        "gpu_launches": launches_per_step * args.steps,
        "device_status": device_status,
        "clocks": clocks.summary(),
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_rows, args.seed, window)
    return line


# --------------------------------------------------------------------------- end to end

def e2e_padded(args, pe, torch, dev, comp, lengths, host_grids, s, wl, train, flops, n_tokens,
               attention_fwd, attention_bwd, barrier, world):
    """End to end from pinned host memory through the public calls, every step
    inside the timed region: upload the lengths and pack (its one host read),
    upload the real rows of the pinned padded q, k, v (and dO) grids straight
    into packed device buffers with the copy engines (pe_upload_packed: one
    copy per sequence, no padding crosses the host link), attention (and
    backward), scatter the padded output (and gradients) on the device and
    copy them back to pinned host memory. Steps are pipelined over four
    streams with two buffer sets: step i+1's uploads and step i-1's download
    overlap step i's attention (the copy engines need no SMs)."""
    host_in = [t.pin_memory() for t in host_grids]
    hlen = torch.from_numpy(lengths).pin_memory()
    nbuf = 2
    io, up, down = (torch.cuda.Stream(dev) for _ in range(3))
    row_shape = tuple(host_in[0].shape[2:])
    dlen = [torch.empty(lengths.shape, dtype=torch.int32, device=dev) for _ in range(nbuf)]
    packed = [[torch.empty((n_tokens,) + row_shape, dtype=t.dtype, device=dev) for t in host_in]
              for _ in range(nbuf)]
    n_out = 4 if train else 1
    dev_out = [[torch.empty_like(host_in[0], device=dev) for _ in range(n_out)]
               for _ in range(nbuf)]
    host_out = [[torch.empty_like(host_in[0]).pin_memory() for _ in range(n_out)]
                for _ in range(nbuf)]
    state = [None] * nbuf
    ev = {name: [torch.cuda.Event() for _ in range(nbuf)]
          for name in ("packed", "uploaded", "computed", "downloaded")}
    for b in range(nbuf):
        ev["computed"][b].record(comp)
        ev["downloaded"][b].record(comp)

    def prep(i):
        b = i % nbuf
        with torch.cuda.stream(io):
            io.wait_event(ev["computed"][b])      # buffer set b is free again
            dlen[b].copy_(hlen, non_blocking=True)
            _, cu, _ = pe.pe_pack_sequences(dlen[b], s)
            cu.record_stream(comp)
            state[b] = cu
            ev["packed"][b].record(io)
        with torch.cuda.stream(up):
            up.wait_event(ev["computed"][b])
            for src, dst in zip(host_in, packed[b]):
                pe.pe_upload_packed(src, lengths, out=dst)
            ev["uploaded"][b].record(up)

    def compute(i):
        b = i % nbuf
        comp.wait_event(ev["packed"][b])
        comp.wait_event(ev["uploaded"][b])
        comp.wait_event(ev["downloaded"][b])     # step i-2's results have left the device
        cu = state[b]
        q, k, v = packed[b][:3]
        out, lse = attention_fwd(q, k, v, cu, s, wl.scale, need_lse=train)
        results = [out]
        if train:
            results += list(attention_bwd(packed[b][3], q, k, v, out, lse, cu, s, wl.scale))
        for src, dst in zip(results, dev_out[b]):
            pe.pe_scatter_padded(src, cu, s, out=dst)
        ev["computed"][b].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(ev["computed"][b])
            for src, dst in zip(dev_out[b], host_out[b]):
                dst.copy_(src, non_blocking=True)
            ev["downloaded"][b].record(down)

    def run(n):
        prep(0)
        for i in range(n):
            if i + 1 < n:
                prep(i + 1)                       # overlaps step i's attention
            compute(i)

    run(max(2, min(args.warmup, 3)))
    torch.cuda.synchronize(dev)
    barrier()
    steps = max(2, min(args.steps, 10))
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    for st in (io, up, down):
        st.wait_event(t0)
    run(steps)
    for st in (io, up, down):
        comp.wait_stream(st)
    t1.record(comp)
    torch.cuda.synchronize(dev)
    barrier()
    ms = t0.elapsed_time(t1) / steps
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    row_bytes = host_in[0].element_size() * int(np.prod(row_shape))
    h2d = hlen.numel() * hlen.element_size() + len(host_in) * n_tokens * row_bytes
    d2h = n_out * host_in[0].numel() * host_in[0].element_size()
    return {"value": world * flops / (ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "path": "real rows of the pinned padded inputs uploaded by the copy engines "
                    "(pe_upload_packed), padded results copied back; step i+1's uploads and "
                    "step i-1's download overlap step i"}


# --------------------------------------------------------------------------- layer tail

# ModernBERT's feed-forward width for its hidden sizes (base, large).
FFN_WIDTH = {768: 1152, 1024: 2624}


def run_tail(args, rank, world):
    """The packed encoder layer tail on a workload's packed tokens: positions,
    RoPE on q and k, residual-LayerNorm on [N, H*d], GeGLU on [N, 2F] - all
    bandwidth kernels, reported as algorithmic bytes per second."""
    import torch

    import padding_free_packed_gb300 as pe
    from padding_free_packed_gb300 import workloads

    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pe.load_library()
    wl = workloads.WORKLOADS[args.workload]
    lengths = workloads.draw_lengths(args.workload, np.random.default_rng(args.seed + rank))
    n, h, d = int(lengths.sum()), wl.num_heads, wl.head_dim
    c = h * d
    f = FFN_WIDTH.get(c, 3 * c // 2)
    dt = wl.torch_dtype
    e = torch.empty((), dtype=dt).element_size()
    gen = torch.Generator(device=dev).manual_seed(args.seed + rank)
    mk = lambda *shape: torch.randn(*shape, generator=gen, device=dev).to(dt)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)).to(dev)
    q, k, x, resid, mlp_in = mk(n, h, d), mk(n, h, d), mk(n, c), mk(n, c), mk(n, 2 * f)
    w = torch.ones(c, dtype=dt, device=dev)
    b = len(lengths)
    algo = {"positions": 4 * n + 4 * (b + 1),
            "rope": 2 * 2 * n * c * e + 4 * n,
            "layernorm": 4 * n * c * e + c * e,
            "geglu": 3 * n * f * e}
    stream = torch.cuda.current_stream(dev)
    events = {key: [] for key in algo}

    def timed(record, key, fn):
        if not record:
            return fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        out = fn()
        e1.record(stream)
        events[key].append((e0, e1))
        return out

    def step(record):
        pos = timed(record, "positions", lambda: pe.pe_packed_positions(cu, n))
        timed(record, "rope", lambda: pe.pe_rope_packed(q, k, pos, 160000.0))
        timed(record, "layernorm", lambda: pe.pe_layernorm(x, w, None, 1e-5, residual=resid))
        timed(record, "geglu", lambda: pe.pe_geglu(mlp_in))

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank, args.clocks_csv) as clocks:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            step(True)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / args.steps
    per = {key: sum(a.elapsed_time(b) for a, b in ev) / len(ev) for key, ev in events.items()}
    gbs = {key: algo[key] / (per[key] * 1e-3) / 1e9 for key in algo}
    peaks, peaks_src = load_peaks()
    dom = max(per, key=per.get)
    total = sum(algo.values())
    return {
        "metric": "packed encoder layer tail HBM throughput", "value": world * total / (ms * 1e-3) / 1e9,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": args.workload, "num_tokens": n, "hidden": c, "heads": h,
                   "head_dim": d, "ffn_width": f,
                   "step": "positions + RoPE(q, k) + residual-LayerNorm + GeGLU",
                   "bytes_per_step": total,
                   "l2": "inputs larger than L2, no flush" if n * 2 * f * e > 129e6 else
                         "inputs smaller than L2"},
        "kernels": {key: {"ms": per[key], "gb_s": gbs[key], "bytes": algo[key]} for key in algo},
        "roofline": {"bound": "hbm", "achieved": gbs[dom], "peak": float(peaks["hbm_gbs"]),
                     "unit": "GB/s", "frac": gbs[dom] / float(peaks["hbm_gbs"]), "traffic": None,
                     "peak_source": f"copy bandwidth, {peaks_src}", "kernel": dom},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks.summary(),
    }


# --------------------------------------------------------------------------- oracle arms

def _oracle_sample(workload: str, rows: int, seed: int, window=None):
    """A bounded sample of the workload for the oracle: `rows` random (token,
    head) query rows, each attending over its whole sequence (or its window)."""
    from padding_free_packed_gb300 import workloads
    x = workloads.make_inputs(workload, seed=seed)
    import oracle
    _, cu, n = oracle.pack_sequences(x.lengths, x.workload.max_seq_len)
    rng = np.random.default_rng(1234)
    r = rng.integers(0, n, rows)
    hs = rng.integers(0, x.workload.num_heads, rows)
    seq = np.searchsorted(cu, r, side="right") - 1
    lens = (cu[1:] - cu[:-1]).astype(np.int64)[seq]
    if window is not None:   # keys each sampled query sees inside its window
        pos = r - cu[seq]
        lo = np.maximum(pos - window[0], 0) if window[0] >= 0 else np.zeros_like(pos)
        hi = np.minimum(pos + window[1], lens - 1) if window[1] >= 0 else lens - 1
        lens = hi - lo + 1
    flops = float(4 * lens.sum() * x.workload.head_dim)
    # Widen to fp64 once, outside any timed region.
    x.q, x.k, x.v = (t.double().numpy() for t in (x.q, x.k, x.v))
    return x, cu, r, hs, flops


def _time_oracle(x, cu, r, hs, window=None):
    import oracle
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.attention_fwd_rows(x.q, x.k, x.v, cu, x.workload.scale, False, r, hs, threads=threads,
                              window=window or (-1, -1))
    return time.perf_counter() - t0, threads


def cpu_baseline(workload: str, rows: int, seed: int, window=None):
    x, cu, r, hs, flops = _oracle_sample(workload, rows, seed, window)
    dt, threads = _time_oracle(x, cu, r, hs, window)
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "seconds": dt,
            "sample": f"{rows} random (token, head) query rows of {workload} (seed {seed}), each "
                      + ("over its whole sequence" if window is None else
                         f"over its local window {tuple(window)}") + ", fp64 oracle row path"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from padding_free_packed_gb300 import workloads
    wl = workloads.WORKLOADS[args.workload]
    window = tuple(args.window) if args.window else None
    x, cu, r, hs, flops = _oracle_sample(args.workload, args.ref_rows, args.seed, window)
    for _ in range(args.warmup):
        _time_oracle(x, cu, r, hs, window)
    times = []
    threads = 1
    for _ in range(args.steps):
        dt, threads = _time_oracle(x, cu, r, hs, window)
        times.append(dt)
    total = sum(times)
    value = flops * args.steps / total / 1e12
    sample = (f"{args.ref_rows} random (token, head) query rows of {args.workload} per step, "
              + ("each over its whole sequence" if window is None else
                 f"each over its local window {window}") + ", fp64 oracle row path")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload,
                                            "description": wl.description},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="longdoc_bf16")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--dtype", choices=["bf16", "fp32"], default=None,
                    help="with --packed: the workload's lengths in another dtype")
    ap.add_argument("--heads", type=int, default=None,
                    help="with --packed: the workload's lengths with another head count")
    ap.add_argument("--head-dim", type=int, default=None,
                    help="with --packed: the workload's lengths with another head_dim")
    ap.add_argument("--sequences", type=int, default=None,
                    help="keep only the first K sequences of the workload (profiling cases)")
    ap.add_argument("--packed", action="store_true",
                    help="inputs already packed: time the attention calls alone")
    ap.add_argument("--first-token", action="store_true",
                    help="with --packed: one query per sequence (its first token)")
    ap.add_argument("--layout", choices=["padded", "rows"], default="padded",
                    help="rows: documents packed several to a row of --row-len tokens, with an "
                         "indexed packing mask (document i of a row marked i)")
    ap.add_argument("--row-len", type=int, default=16384)
    ap.add_argument("--window", type=int, nargs=2, metavar=("LEFT", "RIGHT"), default=None,
                    help="local attention: query at position r sees keys r-LEFT .. r+RIGHT "
                         "(negative = unbounded); e.g. 64 64 for ModernBERT's local layers")
    ap.add_argument("--tail", action="store_true",
                    help="time the packed encoder layer tail (positions, RoPE, residual-"
                         "LayerNorm, GeGLU) on the workload's packed tokens instead")
    ap.add_argument("--backward", action="store_true",
                    help="add the attention backward (dO ~ N(0,1)) to a forward-only workload")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-csv", default=None,
                    help="keep the raw nvidia-smi clock samples of the timed region in this file "
                         "({gpu} is replaced by the GPU index)")
    ap.add_argument("--cpu-rows", type=int, default=98304,
                    help="query rows in the cpu_baseline sample (about 10-30 s of CPU work)")
    ap.add_argument("--ref-rows", type=int, default=2048,
                    help="query rows per reference-arm step")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    line = run_tail(args, rank, world) if args.tail else run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    # A kernel that reported a problem (a malformed layout, a pipeline wait
    # that gave up) makes the measurement invalid: fail the run.
    if any(v != 0 for v in line.get("device_status", {}).values()):
        raise SystemExit(f"device status {line['device_status']}: the timed calls did not "
                         "complete normally")


if __name__ == "__main__":
    main()
