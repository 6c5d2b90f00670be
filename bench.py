"""Benchmark: paged decode-attention KV GB/s (% of GB300 HBM peak) and seq-steps/s.

One step = the whole hot path for one decode step of one layer: the
quantize-on-write of every sequence's new token and paged decode attention
over the block-table-mapped cache, by default in one launch
(paged_decode_attention_with_write; --unfused: paged_kv_write, then
paged_decode_attention).  Inputs are seeded
and synthetic, shaped like the chosen workload (default: the Llama-3-8B-shaped
bf16 layer, batch 64, 32/8 heads, D 128, bs 16, context 4096).  The KV cache
(1 GiB) is far larger than L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]

Prints ONE JSON line (rank 0).  Under torchrun each rank runs an independent
replica on its own GPU (the path has no exchange step).
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode-attention KV GB/s (% of GB300 HBM peak) and seq-steps/sec, 1 GPU"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2**20


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s): the measured burst figure, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def _bits_to_tensor(bits, code):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16 if code == W.F16 else torch.bfloat16).cuda()


def _with_kv_dtype(w: W.Workload, name: str) -> W.Workload:
    """The workload with another cache dtype (16-bit caches take the query dtype)."""
    code = {v: k for k, v in W.DTYPE_NAMES.items()}[name]
    upd = dict(kv_dtype=code, name=f"{w.name}, {name} cache")
    if code in (W.F16, W.BF16):
        upd["q_dtype"] = code
    return dataclasses.replace(w, **upd)


def _kernel_launches_per_step(w: W.Workload, nparts: int, fused: bool = False) -> int:
    # paged_kv_write: one launch, three for one-byte caches (open, grow, encode)
    write = 0 if fused else (3 if w.kv_dtype in W.BLK8_TYPES else 1)
    return write + 1 + (1 if nparts > 1 else 0)


def run_ours(args, rank: int, world: int):
    import torch
    import paged_quantized_kv_write_gb300 as pkv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = W.CONFIGS[args.config]
    if args.partition:
        w = dataclasses.replace(w, partition_size=args.partition)
    if args.block_size:
        w = dataclasses.replace(w, block_size=args.block_size,
                                shared_prefix_tokens=(w.shared_prefix_tokens // args.block_size)
                                * args.block_size)
    if args.kv_dtype:
        w = _with_kv_dtype(w, args.kv_dtype)
    if args.batch:
        w = dataclasses.replace(w, batch=args.batch, pool_blocks=0)
    case = W.make_case(w, identity_tables=args.identity)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        k, v, s = pkv.alloc_cache(w.kv_dtype, case.num_blocks, w.num_kv_heads, w.head_dim,
                                  w.block_size)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        # prefill the context through the library's own write (untimed)
        chunk = 1 << 20
        for i in range(0, len(case.prefill_slots), chunk):
            sl = slice(i, i + chunk)
            pkv.paged_kv_write(_bits_to_tensor(case.prefill_k[sl], w.q_dtype),
                               _bits_to_tensor(case.prefill_v[sl], w.q_dtype),
                               torch.from_numpy(case.prefill_slots[sl]).to(dev), k, v, s,
                               w.kv_dtype, w.block_size, w.head_dim, status, stream)
        q = _bits_to_tensor(case.q, w.q_dtype)
        kn = _bits_to_tensor(case.k_new, w.q_dtype)
        vn = _bits_to_tensor(case.v_new, w.q_dtype)
        slots = torch.from_numpy(case.new_slots).to(dev)
        tables = torch.from_numpy(case.block_tables).to(dev)
        ctx = torch.from_numpy(case.context_lens).to(dev)
        out = torch.empty_like(q)
        mb = case.max_blocks_per_seq
        part = pkv.paged_decode_partition_size(w.batch, w.num_q_heads, w.num_kv_heads, mb,
                                               w.block_size, w.partition_size)
        nparts = -(-mb * w.block_size // part)
        ws = pkv.make_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, mb,
                                w.block_size, w.partition_size, device=dev)
    torch.cuda.synchronize()
    assert status.item() == 0, "prefill flagged an out-of-range slot"

    total_bytes = W.algorithmic_bytes(case, unique=True)
    attn_bytes = W.attention_bytes(case, unique=True)
    logical_bytes = W.algorithmic_bytes(case, unique=False)
    small = total_bytes < 4 * L2_BYTES
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev) if small else None

    def write(st):
        pkv.paged_kv_write(kn, vn, slots, k, v, s, w.kv_dtype, w.block_size, w.head_dim,
                           status, st)

    def attend(st):
        pkv.paged_decode_attention(q, k, v, tables, ctx, s, out, w.softmax_scale,
                                   w.num_kv_heads, w.kv_dtype, w.block_size, w.partition_size,
                                   ws, status, st)

    def fused(st):
        pkv.paged_decode_attention_with_write(q, kn, vn, slots, k, v, tables, ctx, s, out,
                                              w.softmax_scale, w.kv_dtype, w.block_size,
                                              w.partition_size, ws, status, st)

    def step(st):
        if not args.unfused:
            fused(st)
        else:
            write(st)
            attend(st)

    # Device-timed steps replay a CUDA graph of the step (the library's own
    # launches, captured once), so host-side submission gaps cannot leak into
    # the GPU timeline.  The attention alone is captured too, for the roofline.
    with torch.cuda.stream(stream):
        for _ in range(3):                     # first calls set kernel attributes
            step(stream)
    torch.cuda.synchronize()
    g_step, g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        step(stream)
    with torch.cuda.graph(g_attn, stream=stream):
        attend(stream)
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    aev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]

    def timed(graph, events):
        for _ in range(args.warmup):
            if flush is not None:
                flush.zero_()
            graph.replay()
        for a, b in events:
            if flush is not None:
                flush.zero_()
            a.record(stream)
            graph.replay()
            b.record(stream)

    with torch.cuda.stream(stream):
        torch.cuda.synchronize()
        _barrier(world)
        clocks = ClockSampler(dev.index)
        clocks.start()
        time.sleep(0.3)
        torch.cuda.synchronize()
        t_wall0 = time.perf_counter()
        timed(g_step, ev)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
        timed(g_attn, aev)
        torch.cuda.synchronize()
        clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    attn_ms = [a.elapsed_time(b) for a, b in aev]
    dev_ms = sum(step_ms)
    dev_ms = _max_over_ranks(dev_ms, world)
    write_avg_ms = max(0.0, statistics.mean(step_ms) - statistics.mean(attn_ms))
    assert status.item() == 0

    # End to end through the public API with host buffers.  Every step makes one
    # H2D copy of all of its inputs (packed back to back, 256-byte aligned, in
    # one pinned buffer), the eager calls on views of that device copy, and one
    # D2H copy of its output.
    #  * Inputs larger than L2: the staging is double-buffered, as a serving
    #    loop would do it -- step i + 1's inputs go up on their own stream while
    #    step i computes, and step i's output comes back on a third stream while
    #    step i + 1 computes; the timed region runs from the first timed step's
    #    H2D to the last timed step's D2H.
    #  * Small inputs (L2 flushed between steps): one stream, each step's H2D,
    #    calls and D2H between its own pair of events, the flush outside them.
    names = ("q", "kn", "vn", "slots", "tables", "ctx")
    srcs = {"q": q, "kn": kn, "vn": vn, "slots": slots, "tables": tables, "ctx": ctx}
    offs, packed = {}, 0
    for n in names:
        nb = srcs[n].numel() * srcs[n].element_size()
        offs[n] = (packed, nb)
        packed = (packed + nb + 255) // 256 * 256

    def packed_view(buf, n):
        o, nb = offs[n]
        return buf[o:o + nb].view(srcs[n].dtype).view(srcs[n].shape)

    host_in = torch.zeros(packed, dtype=torch.uint8).pin_memory()
    for n in names:
        packed_view(host_in, n).copy_(srcs[n].cpu())
    dev_in = [torch.empty(packed, dtype=torch.uint8, device=dev) for _ in range(2)]
    views = [tuple(packed_view(d, n) for n in names) for d in dev_in]
    outs = [torch.empty_like(out) for _ in range(2)]
    host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = packed
    d2h = host_out[0].numel() * host_out[0].element_size()
    torch.cuda.synchronize()
    if flush is not None:
        e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
        # the calls (write / attend / fused) read the first buffer set
        q, kn, vn, slots, tables, ctx = views[0]
        out = outs[0]
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.steps):
                flush.zero_()
                if i >= args.warmup:
                    e2e_ev[i - args.warmup][0].record(stream)
                dev_in[0].copy_(host_in, non_blocking=True)
                step(stream)
                host_out[0].copy_(out, non_blocking=True)
                if i >= args.warmup:
                    e2e_ev[i - args.warmup][1].record(stream)
        torch.cuda.synchronize()
        e2e_ms = _max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev), world)
        e2e_kind = "serial (L2 flushed between steps, outside the timed events)"
    else:
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs j are on the device
        ev_done = [torch.cuda.Event() for _ in range(2)]    # step on buffer j has finished
        ev_back = [torch.cuda.Event() for _ in range(2)]    # output j is back on the host
        e2e_t0 = torch.cuda.Event(enable_timing=True)
        e2e_t1 = torch.cuda.Event(enable_timing=True)
        for i in range(args.warmup + args.steps):
            j = i % 2
            if i == args.warmup:
                e2e_t0.record(s_in)
            if i >= 2:
                s_in.wait_event(ev_done[j])               # step i - 2 has read dev_in[j]
            with torch.cuda.stream(s_in):
                dev_in[j].copy_(host_in, non_blocking=True)
            ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            if i >= 2:
                stream.wait_event(ev_back[j])             # step i - 2's output has left outs[j]
            # the calls (write / attend / fused) read this step's buffers
            q, kn, vn, slots, tables, ctx = views[j]
            out = outs[j]
            with torch.cuda.stream(stream):
                step(stream)
            ev_done[j].record(stream)
            s_out.wait_event(ev_done[j])
            with torch.cuda.stream(s_out):
                host_out[j].copy_(outs[j], non_blocking=True)
            ev_back[j].record(s_out)
        e2e_t1.record(s_out)
        torch.cuda.synchronize()
        e2e_ms = _max_over_ranks(e2e_t0.elapsed_time(e2e_t1), world)
        e2e_kind = "pipelined (double-buffered staging: H2D and D2H on their own streams)"

    peak, peak_kind = _peaks()
    ms_per_step = dev_ms / args.steps
    gbs = whole_job_rate(total_bytes, args.steps, dev_ms, world) / 1e9
    attn_avg_ms = statistics.mean(attn_ms)
    achieved = attn_bytes / (attn_avg_ms * 1e-3) / 1e9
    result = {
        "metric": METRIC,
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {W.F16: "f16", W.BF16: "bf16", W.FP8_E4M3: "fp8_e4m3+bf16",
                  W.FP8_E5M2: "fp8_e5m2+bf16", W.INT8: "int8+bf16",
                  W.INT4_G32: "int4_g32+bf16"}[w.kv_dtype],
        "data": "synthetic (seeded N(0,1) q/K/V, shuffled block tables; no model weights)",
        "config": {
            "workload": f"config {args.config}: {w.name}",
            "batch": w.batch, "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "block_size": w.block_size,
            "kv_dtype": W.DTYPE_NAMES[w.kv_dtype],
            "context_tokens": int(case.context_lens.sum()),
            "partition_size": part, "num_partitions": nparts,
            "l2": "inputs larger than L2 (no flush)" if not small else "L2 flushed (256 MB write) between steps",
            "parallelism": f"replicas x{world}",
            "block_tables": "identity (contiguous)" if args.identity else "shuffled",
            "block_size_override": bool(args.block_size),
            "batch_override": bool(args.batch),
            "kv_dtype_override": bool(args.kv_dtype),
        },
        "seq_steps_per_s": round(whole_job_rate(w.batch, args.steps, dev_ms, world), 1),
        "pct_hbm_peak": round(100.0 * gbs / world / peak, 2),
        "bytes_per_step": total_bytes,
        "logical_bytes_per_step": logical_bytes,
        "e2e": {
            "value": round(whole_job_rate(total_bytes, args.steps, e2e_ms, world) / 1e9, 2),
            "unit": "GB/s",
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "ms_per_step": round(e2e_ms / args.steps, 5),
            "timing": e2e_kind,
        },
        "roofline": {
            "kernel": "paged_decode_kernel (+ pkv_lse_reduce when split)",
            "bound": "hbm",
            "achieved": round(achieved, 2),
            "peak": peak,
            "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback 6.8 TB/s",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": None if (args.kv_dtype or args.block_size or args.partition or args.batch)
                       else _traffic(args.config),
            "avg_launch_us": round(attn_avg_ms * 1e3, 3),
            "write_avg_us": round(write_avg_ms * 1e3, 3),
            "algorithmic_bytes": attn_bytes,
        },
        "gpu_launches": _kernel_launches_per_step(w, nparts, not args.unfused) * args.steps,
        "step_kind": "fused write + attention (one launch)" if not args.unfused
                     else "paged_kv_write, then paged_decode_attention",
        "clocks": clk,
        "wall_s_timed": round(t_wall, 4),
        "timing": "CUDA events around CUDA-graph replays of the step (write + attention); "
                  "roofline from replays of the attention alone",
    }
    return result


def measure_workload(cfg: int, reps: int, dev, flush, peak: float):
    """One workload's decode step on this GPU, in the library's launch configuration:
    CUDA-graph replays of the fused step (write + attention) and of the attention
    alone, each timed with the L2 flushed before every replay (a 256 MB write,
    outside the events) and warm (back to back, no flush).  The context is
    prefilled through paged_kv_write with K/V drawn on the device (the workload's
    distribution; host draws of a full-size context take longer than all of the
    timing).  Returns the figures as a dict."""
    import torch
    import paged_quantized_kv_write_gb300 as pkv

    w = W.CONFIGS[cfg]
    case = W.make_case(w, prefill_values=False)
    stream = torch.cuda.Stream(dev)
    n = len(case.prefill_slots)
    with torch.cuda.stream(stream):
        k, v, s = pkv.alloc_cache(w.kv_dtype, case.num_blocks, w.num_kv_heads, w.head_dim,
                                  w.block_size, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        if n:
            kp = W.draw_kv_device(w, n, w.seed * 2 + 1, dev)
            vp = W.draw_kv_device(w, n, w.seed * 2 + 2, dev)
            pkv.paged_kv_write(kp, vp, torch.from_numpy(case.prefill_slots).to(dev), k, v, s,
                               w.kv_dtype, w.block_size, w.head_dim, status, stream)
            del kp, vp
        q = _bits_to_tensor(case.q, w.q_dtype)
        kn = _bits_to_tensor(case.k_new, w.q_dtype)
        vn = _bits_to_tensor(case.v_new, w.q_dtype)
        slots = torch.from_numpy(case.new_slots).to(dev)
        tables = torch.from_numpy(case.block_tables).to(dev)
        ctx = torch.from_numpy(case.context_lens).to(dev)
        out = torch.empty_like(q)
        mb = case.max_blocks_per_seq
        part = pkv.paged_decode_partition_size(w.batch, w.num_q_heads, w.num_kv_heads, mb,
                                               w.block_size, w.partition_size)
        ws = pkv.make_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, mb,
                                w.block_size, w.partition_size, device=dev)
    torch.cuda.synchronize()

    def attend(st):
        pkv.paged_decode_attention(q, k, v, tables, ctx, s, out, w.softmax_scale,
                                   w.num_kv_heads, w.kv_dtype, w.block_size, w.partition_size,
                                   ws, status, st)

    def fused(st):
        pkv.paged_decode_attention_with_write(q, kn, vn, slots, k, v, tables, ctx, s, out,
                                              w.softmax_scale, w.kv_dtype, w.block_size,
                                              w.partition_size, ws, status, st)

    with torch.cuda.stream(stream):
        for _ in range(3):
            fused(stream)
    torch.cuda.synchronize()
    graphs = {}
    for name, fn in (("step", fused), ("attn", attend)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn(stream)
        graphs[name] = g
    torch.cuda.synchronize()

    def evict():
        # read (not write) 256 MB, twice L2, so that L2 holds only clean lines
        # of another buffer and no write-back competes with the timed launch
        torch.sum(flush, dtype=torch.int32)

    def time_graph(g, flushed):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        with torch.cuda.stream(stream):
            for _ in range(5):
                if flushed:
                    evict()
                g.replay()
            for a, b in ev:
                if flushed:
                    evict()
                a.record(stream)
                g.replay()
                b.record(stream)
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3     # us

    t = {(name, fl): time_graph(graphs[name], fl) for name in graphs for fl in (True, False)}
    assert status.item() == 0, f"config {cfg}: a kernel flagged an out-of-range id"
    attn_u = W.attention_bytes(case, unique=True)
    attn_l = W.attention_bytes(case, unique=False)
    step_u = W.algorithmic_bytes(case, unique=True)
    # the headline's rule: back-to-back replays when the step's inputs exceed L2
    # several times over (they evict themselves), cold L2 otherwise
    big = step_u >= 4 * L2_BYTES
    main = ("attn", not big)
    res = {
        "workload": w.name,
        "kv_dtype": W.DTYPE_NAMES[w.kv_dtype],
        "batch": w.batch,
        "partition_size": part,
        "decode_us": round(t[main], 2),
        "decode_gbs": round(attn_u / t[main] / 1e3, 1),
        "frac": round(attn_u / t[main] / 1e3 / peak, 4),
        "timed_as": "back-to-back (inputs > 4x L2)" if big else "L2 evicted before each replay",
        "decode_us_flushed": round(t[("attn", True)], 2),
        "decode_us_warm": round(t[("attn", False)], 2),
        "frac_flushed": round(attn_u / t[("attn", True)] / 1e3 / peak, 4),
        "frac_warm": round(attn_u / t[("attn", False)] / 1e3 / peak, 4),
        "step_us": round(t[("step", not big)], 2),
        "step_us_flushed": round(t[("step", True)], 2),
        "step_us_warm": round(t[("step", False)], 2),
        "seq_steps_per_s": round(w.batch / t[("step", not big)] * 1e6, 1),
        "algorithmic_bytes": attn_u,
        "traffic": _traffic(cfg),
    }
    if attn_l != attn_u:
        # shared-prefix blocks: counted once (unique) or once per sequence (logical)
        res["logical_bytes"] = attn_l
        res["decode_gbs_logical"] = round(attn_l / t[main] / 1e3, 1)
    del graphs, k, v, s, ws
    torch.cuda.empty_cache()
    return res


def run_per_config(args, dev):
    """Every workload's decode figures on this GPU (configs 1-5), with the clocks
    sampled over the whole sweep."""
    import torch
    peak, _ = _peaks()
    flush = torch.ones(256 * 2**20, dtype=torch.uint8, device=dev)
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    res = {}
    for cfg in sorted(W.CONFIGS):
        res[str(cfg)] = measure_workload(cfg, args.per_config_reps, dev, flush, peak)
    res["clocks"] = clocks.stop()
    res["timing"] = (f"median of {args.per_config_reps} CUDA-graph replays per figure; "
                     "'decode' = the attention call alone, 'step' = the fused write + "
                     "attention; flushed = a 256 MB read before each replay (outside the "
                     "events) evicts L2, warm = back-to-back replays; decode_us/frac use "
                     "the headline's rule (warm when the inputs exceed 4x L2)")
    return res


def run_copy(args, rank: int, world: int):
    """Copy-on-write block copies: time paged_kv_copy_blocks moving --copy-pairs
    random (src, dst) blocks of the workload's pool per step (K, V and scales)."""
    import torch
    import paged_quantized_kv_write_gb300 as pkv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = W.CONFIGS[args.config]
    if args.kv_dtype:
        w = _with_kv_dtype(w, args.kv_dtype)
    case = W.make_case(w)
    nb = case.num_blocks
    n = min(args.copy_pairs, nb // 2)
    rng = np.random.default_rng(7)
    perm = rng.permutation(nb)
    pairs = torch.from_numpy(np.stack([perm[:n], perm[n:2 * n]], 1).astype(np.int32)).to(dev)
    k, v, s = pkv.alloc_cache(w.kv_dtype, nb, w.num_kv_heads, w.head_dim, w.block_size,
                              device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    per_block = 2 * w.num_kv_heads * w.block_size * pkv.row_bytes(w.kv_dtype, w.head_dim)
    if w.kv_dtype in W.BLK8_TYPES:
        per_block += 2 * 4 * w.num_kv_heads
    elif w.kv_dtype == W.INT4_G32:
        per_block += 2 * w.num_kv_heads * w.block_size * (w.head_dim // 32) * 4
    step_bytes = 2 * n * per_block                   # read the sources, write the copies

    def copy(st):
        pkv.paged_kv_copy_blocks(k, v, s, w.kv_dtype, pairs, w.block_size, w.head_dim, status, st)

    with torch.cuda.stream(stream):
        for _ in range(3):
            copy(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        copy(stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        _barrier(world)
        clocks = ClockSampler(dev.index)
        clocks.start()
        time.sleep(0.3)
        for a, b in ev:
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        clk = clocks.stop()
    dev_ms = _max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), world)
    assert status.item() == 0
    peak, peak_kind = _peaks()
    gbs = whole_job_rate(step_bytes, args.steps, dev_ms, world) / 1e9
    return {
        "metric": "paged KV block copy GB/s (bytes read + written), 1 GPU",
        "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dev_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": W.DTYPE_NAMES[w.kv_dtype], "data": "synthetic pool (zeros), random disjoint pairs",
        "config": {"workload": f"config {args.config}: {w.name}, {n} block copies per step",
                   "num_blocks": nb, "pairs": n, "bytes_per_block_copy": per_block,
                   "l2": "moves far more than L2 per step (no flush)"},
        "roofline": {"kernel": "copy_blocks_kernel", "bound": "hbm",
                     "achieved": round(gbs / world, 2), "peak": peak,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "unit": "GB/s", "frac": round(gbs / world / peak, 4), "traffic": None},
        "gpu_launches": args.steps,
        "clocks": clk,
    }


def _prefill_kernel_name(kv_dtype: int) -> str:
    """The kernel paged_prefill_attention runs for this cache dtype."""
    if os.environ.get("PKV_PREFILL_MODE") == "mma":
        return "paged_decode_kernel (prefill mode, mma.sync)"
    return "prefill_ws_kernel (tcgen05, load / MMA / softmax warp roles)"


def run_prefill(args, rank: int, world: int):
    """Chunked prefill: time paged_prefill_attention on the prefill workload (8
    sequences of 4096 cached tokens, chunks of their last 512, Llama-3-8B-shaped)."""
    import torch
    import paged_quantized_kv_write_gb300 as pkv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w, n = W.prefill_workload()
    if args.kv_dtype:
        w = _with_kv_dtype(w, args.kv_dtype)
    case = W.make_case(w)
    chunk = [min(n, int(c)) for c in case.context_lens]
    q_bits, q_start = W.prefill_chunk(case, chunk)
    stream = torch.cuda.Stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):
        k, v, s = pkv.alloc_cache(w.kv_dtype, case.num_blocks, w.num_kv_heads, w.head_dim,
                                  w.block_size, device=dev)
        slots = np.concatenate([case.prefill_slots, case.new_slots[case.new_slots >= 0]])
        kk = np.concatenate([case.prefill_k, case.k_new[case.new_slots >= 0]])
        vv = np.concatenate([case.prefill_v, case.v_new[case.new_slots >= 0]])
        pkv.paged_kv_write(_bits_to_tensor(kk, w.q_dtype), _bits_to_tensor(vv, w.q_dtype),
                           torch.from_numpy(slots).to(dev), k, v, s, w.kv_dtype, w.block_size,
                           w.head_dim, status, stream)
        q = _bits_to_tensor(q_bits, w.q_dtype)
        out = torch.empty_like(q)
        qs = torch.from_numpy(q_start).to(dev)
        tables = torch.from_numpy(case.block_tables).to(dev)
        ctx = torch.from_numpy(case.context_lens).to(dev)
    torch.cuda.synchronize()

    def call(st):
        pkv.paged_prefill_attention(q, qs, k, v, tables, ctx, s, out, w.softmax_scale,
                                    w.num_kv_heads, w.kv_dtype, w.block_size, max(chunk),
                                    status, st)

    with torch.cuda.stream(stream):
        for _ in range(3):
            call(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call(stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        _barrier(world)
        clocks = ClockSampler(dev.index)
        clocks.start()
        time.sleep(0.3)
        for a, b in ev:
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        clk = clocks.stop()
    assert status.item() == 0
    dev_ms = _max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), world)
    flops = W.prefill_flops(case.context_lens, chunk, w.num_q_heads, w.head_dim)
    tflops = whole_job_rate(flops, args.steps, dev_ms, world) / 1e12
    peak, kind = _tensor_peak()
    kv_bytes = W.attention_bytes(case, unique=True)
    return {
        "metric": "chunked-prefill paged attention TFLOP/s (QK^T + PV over each query's causal range), 1 GPU",
        "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dev_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": W.DTYPE_NAMES[w.kv_dtype] + "+" + W.DTYPE_NAMES[w.q_dtype],
        "data": "synthetic (seeded N(0,1) q/K/V, shuffled block tables)",
        "config": {"workload": f"chunked prefill: {w.name}, {w.batch} sequences, chunks of "
                               f"{max(chunk)} over {int(case.context_lens.max())}-token contexts",
                   "query_tokens": int(q_start[-1]), "flops_per_step": flops,
                   "kv_bytes_per_step": kv_bytes},
        "roofline": {"kernel": _prefill_kernel_name(w.kv_dtype), "bound": "tensor",
                     "achieved": round(tflops / world, 2), "peak": peak,
                     "peak_kind": f"{kind} (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)",
                     "unit": "TFLOP/s", "frac": round(tflops / world / peak, 4), "traffic": None},
        "gpu_launches": args.steps,
        "clocks": clk,
    }


def _traffic(config: int):
    """DRAM bytes per launch of the decode kernel from a committed ncu summary, if one
    exists for this workload and the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(str(config))
        if not ent or ent.get("source_sha") != _kernel_sha():
            return None
        return ent["dram_bytes_per_launch"]
    except Exception:
        return None


def _kernel_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    for name in ("pkv_attn.cuh", "pkv_decode.cu", "pkv_decode_launch.cuh", "pkv_common.cuh"):
        with open(os.path.join(ROOT, "paged_quantized_kv_write_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def cpu_baseline(config: int, budget_s: float = 20.0):
    """The oracle as it stands on the host cores, over a bounded sample of the workload."""
    import oracle
    w = W.CONFIGS[config]
    # sample: the first n sequences of the workload, n sized to a few seconds of CPU work
    n = w.batch
    probe = W.make_case(w.scaled(batch=min(4, w.batch)))
    pk, pv, ps = oracle.prefill_case(probe)
    t0 = time.perf_counter()
    oracle.step_case(probe, pk, pv, ps)
    per_seq = (time.perf_counter() - t0) / probe.w.batch
    n = int(max(1, min(w.batch, budget_s / max(per_seq, 1e-6))))
    case = W.make_case(w.scaled(batch=n))
    k, v, s = oracle.prefill_case(case)
    reps = 0
    t0 = time.perf_counter()
    while True:                       # repeat the step for about budget_s / 2 seconds
        oracle.step_case(case, k, v, s)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s / 2 or reps >= 1000:
            break
    return {
        "value": round(W.algorithmic_bytes(case) * reps / dt / 1e9, 4),
        "unit": "GB/s",
        "seq_steps_per_s": round(n * reps / dt, 3),
        "cores": oracle.max_threads(),
        "kind": "oracle",
        "sample": f"{n} of {w.batch} sequences of config {config} (same heads, dims, lengths "
                  f"distribution), {reps} decode steps, fp64 C oracle with OpenMP",
        "seconds": round(dt, 3),
    }


def run_reference(args, rank: int, world: int):
    """The reference arm: the CPU oracle, timed on this machine's host cores."""
    import oracle
    w = W.CONFIGS[args.config]
    probe = W.make_case(w.scaled(batch=min(2, w.batch)))
    pk, pv, ps = oracle.prefill_case(probe)
    t0 = time.perf_counter()
    oracle.step_case(probe, pk, pv, ps)
    per_seq = (time.perf_counter() - t0) / probe.w.batch
    budget = args.ref_seconds / max(1, args.steps + args.warmup)   # the whole run's CPU time
    n = int(max(1, min(w.batch, budget / max(per_seq, 1e-6))))
    case = W.make_case(w.scaled(batch=n))
    k, v, s = oracle.prefill_case(case)
    for _ in range(args.warmup):
        oracle.step_case(case, k, v, s)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.step_case(case, k, v, s)
    dt = time.perf_counter() - t0
    val = W.algorithmic_bytes(case) * args.steps / dt / 1e9
    sample = (f"{n} of {w.batch} sequences of config {args.config} per step, fp64 C oracle "
              f"with OpenMP")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(val, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": f"config {args.config}: {w.name}", "sample": sample},
        "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    return rank, world


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time: replicas run in lockstep between barriers."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, steps: int, max_ms: float, world: int) -> float:
    """Units per second over all replicas: every rank processes units_per_rank per
    step; the job takes as long as its slowest rank."""
    return world * units_per_rank * steps / (max_ms * 1e-3)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=2, choices=sorted(W.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--identity", action="store_true",
                    help="lay every sequence out in consecutive blocks (paging-overhead comparator)")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="reference arm: CPU seconds the whole run may take (sizes its sample)")
    ap.add_argument("--block-size", type=int, default=0,
                    help="override the workload's block size (block-size sweep; 0: keep)")
    ap.add_argument("--kv-dtype", default="", choices=[""] + sorted(W.DTYPE_NAMES.values()),
                    help="override the workload's cache dtype (dtype comparison; empty: keep)")
    ap.add_argument("--unfused", action="store_true",
                    help="run the step as paged_kv_write then paged_decode_attention (two "
                         "launches) instead of paged_decode_attention_with_write (one)")
    ap.add_argument("--op", default="step", choices=["step", "copy", "prefill"],
                    help="step: the decode step (default); copy: copy-on-write block copies; "
                         "prefill: chunked-prefill attention")
    ap.add_argument("--copy-pairs", type=int, default=4096,
                    help="--op copy: block pairs copied per step")
    ap.add_argument("--partition", type=int, default=0,
                    help="override the workload's split-KV partition size (0: keep)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (wave-count sweep; 0: keep)")
    ap.add_argument("--per-config-reps", type=int, default=100,
                    help="replays per figure in the per-workload sweep (0: skip the sweep)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world = _dist()

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    if args.op in ("copy", "prefill"):
        res = (run_copy if args.op == "copy" else run_prefill)(args, rank, world)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    res = run_ours(args, rank, world)
    plain = not (args.identity or args.block_size or args.kv_dtype or args.unfused or
                 args.partition or args.batch)
    if args.per_config_reps > 0 and plain:
        import torch
        res["per_config"] = run_per_config(
            args, torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))))
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            res["cpu_baseline"] = cpu_baseline(args.config)
        elif not args.no_cpu_baseline:
            res["cpu_baseline"] = None
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
