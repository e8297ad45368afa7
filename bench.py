#!/usr/bin/env python
"""Benchmark of the paged GQA attention hot path on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the hot path over one batch: the append of the batch's new
tokens, then the attention call(s); for decode the two are one fused call
(paged_attn_decode_append), and the same step as two calls is timed alongside.
Default workload: batched decode (batch 32,
context ~U{128..4096}, 32 q / 8 KV heads x 128, 256-token blocks in a 1024-block
pool); the line also carries the causal-prefill half of the metric (4096-token
prompt appended into 16 blocks, then causal attention) measured in the same run.

Timing: W untimed warm-up steps, then K timed steps.  Before every timed step the
L2 is flushed (a 512 MiB device write, then a read of the same buffer so that the
flush's dirty lines are written back before the step: the step then starts from
an L2 holding only clean, unrelated lines; outside the timed region) and the GPU is
given a short head start so that every launch of the step is queued before it
begins; each step is bracketed by CUDA events on the launching stream.  Inputs are
resident in HBM for `value`; `e2e` repeats the step through the public API with
host (pinned) inputs copied in and the output copied back inside the timed region.

--impl reference times the fp64 CPU oracle on this host's cores on the same
workload (rank 0 only).  With N > 1 ranks (torchrun) every rank runs its own
replica of the workload (weak scaling, no collective on the data path); timing is
the max over ranks.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode KV-read GB/s (% of HBM peak); causal prefill attn TFLOP/s (% BF16 peak)"
FLUSH_BYTES = 512 << 20
HEAD_START_CYCLES = 200_000      # ~0.1 ms spin so a step's launches are all queued

# Per-launch DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) from an ncu
# capture, keyed by kernel, with the hash of the sources it was taken on.  A kernel
# whose sources changed since reports traffic null.
TRAFFIC = {
    # one ncu capture of the batched decode step (32 sequences, 243.9 MB of K/V)
    "decode": {"bytes_per_launch": 249650432 + 4694272, "sources": ("decode.cu", "common.cuh"),
               "sha": "8933af376eb543b1", "workload": "batched_decode"},
    # one ncu capture of the fused 8-bit decode step (batch 32, 126 MB of 8-bit K/V)
    "decode_fp8": {"bytes_per_launch": 131116800 + 4321280, "sources": ("decode_fp8.cu", "common.cuh"),
                   "sha": "fa1e86d11026bb58", "workload": "batched_decode_fp8"},
    # one ncu capture of the causal prefill of 4096 tokens with the prompt's append fused in
    "prefill": {"bytes_per_launch": 50459392 + 14682880, "sources": ("prefill.cu", "common.cuh"),
                "sha": "fec1d9b4cc5c409b", "workload": "causal_prefill"},
    # one ncu capture of the merged Q/K/V projection of 4096 tokens (hidden 4096)
    "qkv": {"bytes_per_launch": 117790208 + 35780352, "sources": ("qkv.cu", "common.cuh"),
            "sha": "2966bd0ce22b6d05", "workload": "qkv_append"},
}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default="batched_decode",
                   choices=["single_decode", "batched_decode", "causal_prefill", "mixed_batch",
                            "prefix_shared_decode", "layered_decode", "batched_decode_fp8",
                            "prefix_shared_decode_cascade", "qkv_append"])
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-prefill", action="store_true", help="skip the prefill sub-measurement")
    p.add_argument("--only-main", action="store_true",
                   help="measure only the named workload (no sub-objects for the other configurations)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target duration of the CPU oracle sample")
    return p.parse_args()


# ------------------------------------------------------------------ distributed plumbing

def dist_setup():
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def dist_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi in the background; clocks and throttle reasons of one GPU."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.windows = []

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark(self, t0: float, t1: float):
        self.windows.append((t0, t1))

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10], parts[5]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if any(a - 0.15 <= r[0] <= b + 0.15 for a, b in self.windows)]
        used = inside if len(inside) >= 3 else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in used for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median([r[1] for r in used]) if used else None,
                "sm_max_mhz": max(r[2] for r in used) if used else None,
                "reasons": reasons, "samples": len(used),
                "window": "timed region" if used is inside else "whole run (timed region too short)"}


# ------------------------------------------------------------------ helpers

def source_hash(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_gqa_attention_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class Timer:
    """Per-step CUDA events on one stream: marks[i] recorded between the step's calls."""

    def __init__(self, n_marks: int, stream):
        import torch

        self.stream = stream
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_marks)]

    def record(self, i):
        self.ev[i].record(self.stream)

    def spans_ms(self):
        return [self.ev[i].elapsed_time(self.ev[i + 1]) for i in range(len(self.ev) - 1)]


def flush_l2(buf):
    """Evict the L2: write a buffer 4x its size, then read it back (leaves clean lines)."""
    buf.zero_()
    buf.view(__import__("torch").int32).max()


def run_timed(step, n_marks, steps, warmup, flush_buf, stream, clocks=None):
    """W warm-up steps, then `steps` timed steps; returns per-step lists of span times (ms)."""
    import torch

    for _ in range(warmup):
        flush_l2(flush_buf)
        step(None)
    torch.cuda.synchronize()
    spans = []
    t0 = time.time()
    for _ in range(steps):
        flush_l2(flush_buf)
        torch.cuda._sleep(HEAD_START_CYCLES)
        tm = Timer(n_marks, stream)
        step(tm)
        spans.append(tm)
    torch.cuda.synchronize()
    t1 = time.time()
    if clocks is not None:
        clocks.mark(t0, t1)
    return [tm.spans_ms() for tm in spans], t1 - t0


def mean(xs):
    return sum(xs) / len(xs) if xs else float("nan")


def pcts(xs):
    """p10 / p50 / p90 of per-step times (ms), nearest rank."""
    if not xs:
        return None
    v = sorted(xs)
    at = lambda q: v[min(len(v) - 1, int(q * len(v)))]
    return {"p10": at(0.1), "p50": at(0.5), "p90": at(0.9)}


# ------------------------------------------------------------------ the two measured paths

def decode_measure(batch, steps, warmup, flush_buf, stream, clocks):
    """One decode step: the append of every sequence's new token fused with the decode
    (paged_attn_decode_append, one kernel).  The same step as two calls (kv_append, then
    paged_attn_decode) is timed too, over fewer steps, for comparison."""
    import torch

    from paged_gqa_attention_gb300 import ops

    ws = ops.make_workspace(batch.num_seqs, batch.max_blocks_per_seq)
    out = torch.empty_like(batch.q)

    def step(tm):
        if tm: tm.record(0)
        ops.paged_attn_decode_append(batch.q, batch.k_new, batch.v_new, batch.k_pool, batch.v_pool,
                                     batch.block_table, batch.seq_lens, ws, out=out)
        if tm: tm.record(1)

    def two_calls(tm):
        if tm: tm.record(0)
        ops.kv_append(batch.k_pool, batch.v_pool, batch.k_new, batch.v_new, batch.block_table,
                      batch.cu_q_lens, batch.seq_lens, ws)
        if tm: tm.record(1)
        ops.paged_attn_decode(batch.q, batch.k_pool, batch.v_pool, batch.block_table,
                              batch.seq_lens, ws, out=out)
        if tm: tm.record(2)

    spans, wall = run_timed(step, 2, steps, warmup, flush_buf, stream, clocks)
    spans2, _ = run_timed(two_calls, 3, max(10, min(steps, 200)), warmup, flush_buf, stream)
    ops.check_error(ws)
    return {"attn_ms": mean([s[0] for s in spans]), "step_ms": mean([s[0] for s in spans]),
            "step_pcts": pcts([s[0] for s in spans]),
            "two_call_append_ms": mean([s[0] for s in spans2]),
            "two_call_decode_ms": mean([s[1] for s in spans2]), "wall_s": wall, "launches": steps}


def prefill_measure(batch, steps, warmup, flush_buf, stream, clocks):
    """One prefill step: the append of the prompt's K/V fused with the causal attention
    (paged_attn_prefill_append, one kernel).  The same step as two calls (kv_append, then
    paged_attn_prefill) is timed too, over fewer steps, for comparison."""
    import torch

    from paged_gqa_attention_gb300 import ops

    ws = ops.make_workspace(batch.num_seqs, batch.max_blocks_per_seq)
    out = torch.empty_like(batch.q)

    def step(tm):
        if tm: tm.record(0)
        ops.paged_attn_prefill_append(batch.q, batch.k_new, batch.v_new, batch.k_pool, batch.v_pool,
                                      batch.block_table, batch.cu_q_lens, batch.seq_lens, batch.max_q_len, ws,
                                      out=out)
        if tm: tm.record(1)

    def two_calls(tm):
        if tm: tm.record(0)
        ops.kv_append(batch.k_pool, batch.v_pool, batch.k_new, batch.v_new, batch.block_table,
                      batch.cu_q_lens, batch.seq_lens, ws)
        if tm: tm.record(1)
        ops.paged_attn_prefill(batch.q, batch.k_pool, batch.v_pool, batch.block_table,
                               batch.cu_q_lens, batch.seq_lens, batch.max_q_len, ws, out=out)
        if tm: tm.record(2)

    spans, wall = run_timed(step, 2, steps, warmup, flush_buf, stream, clocks)
    spans2, _ = run_timed(two_calls, 3, max(10, min(steps, 200)), warmup, flush_buf, stream)
    ops.check_error(ws)
    return {"step_ms": mean([s[0] for s in spans]), "step_pcts": pcts([s[0] for s in spans]),
            "two_call_append_ms": mean([s[0] for s in spans2]), "two_call_prefill_ms": mean([s[1] for s in spans2]),
            "wall_s": wall, "launches": steps}


def mixed_measure(batch, steps, warmup, flush_buf, stream, clocks):
    """One continuous-batching step: the decode sequences' append fused into their decode
    (paged_attn_decode_append) and the chunks' append fused into their prefill
    (paged_attn_prefill_append): two kernels.  The same step as three calls (one kv_append for
    every new token, the decode, the prefill) is timed too."""
    import torch

    from paged_gqa_attention_gb300 import ops

    n_dec = batch.info["n_decode"]
    dec = batch.select(slice(0, n_dec))
    pre = batch.select(slice(n_dec, batch.num_seqs))
    ws = ops.make_workspace(batch.num_seqs, batch.max_blocks_per_seq)
    out_d = torch.empty_like(dec.q)
    out_p = torch.empty_like(pre.q)

    def step(tm):
        if tm: tm.record(0)
        ops.paged_attn_decode_append(dec.q, dec.k_new, dec.v_new, dec.k_pool, dec.v_pool, dec.block_table,
                                     dec.seq_lens, ws, out=out_d)
        if tm: tm.record(1)
        ops.paged_attn_prefill_append(pre.q, pre.k_new, pre.v_new, pre.k_pool, pre.v_pool, pre.block_table,
                                      pre.cu_q_lens, pre.seq_lens, pre.max_q_len, ws, out=out_p)
        if tm: tm.record(2)

    def three_calls(tm):
        if tm: tm.record(0)
        ops.kv_append(batch.k_pool, batch.v_pool, batch.k_new, batch.v_new, batch.block_table,
                      batch.cu_q_lens, batch.seq_lens, ws)
        if tm: tm.record(1)
        ops.paged_attn_decode(dec.q, dec.k_pool, dec.v_pool, dec.block_table, dec.seq_lens, ws,
                              out=out_d)
        if tm: tm.record(2)
        ops.paged_attn_prefill(pre.q, pre.k_pool, pre.v_pool, pre.block_table, pre.cu_q_lens,
                               pre.seq_lens, pre.max_q_len, ws, out=out_p)
        if tm: tm.record(3)

    spans, wall = run_timed(step, 3, steps, warmup, flush_buf, stream, clocks)
    spans3, _ = run_timed(three_calls, 4, max(10, min(steps, 200)), warmup, flush_buf, stream)
    ops.check_error(ws)
    return {"decode_ms": mean([s[0] for s in spans]), "prefill_ms": mean([s[1] for s in spans]),
            "step_ms": mean([sum(s) for s in spans]), "step_pcts": pcts([sum(s) for s in spans]),
            "three_call": {"kv_append_ms": mean([s[0] for s in spans3]), "decode_ms": mean([s[1] for s in spans3]),
                           "prefill_ms": mean([s[2] for s in spans3])},
            "wall_s": wall, "launches": 2 * steps, "dec": dec, "pre": pre}


def layered_measure(layers, steps, warmup, flush_buf, stream, clocks):
    """The decode step over all layers: one replay of the captured CUDA graph
    (pa_decode_graph_launch) against the same layers launched one call at a time."""
    import torch

    from paged_gqa_attention_gb300 import ops

    b0 = layers.base
    ws = ops.make_workspace(b0.num_seqs, b0.max_blocks_per_seq)
    out = torch.empty_like(layers.q)
    g = ops.decode_graph(layers.q, layers.k_new, layers.v_new, layers.k_pool, layers.v_pool,
                         b0.block_table, b0.seq_lens, ws, out=out)

    def graph_step(tm):
        if tm: tm.record(0)
        g.launch()
        if tm: tm.record(1)

    def eager_step(tm):
        if tm: tm.record(0)
        for l in range(layers.layers):
            ops.paged_attn_decode_append(layers.q[l], layers.k_new[l], layers.v_new[l], layers.k_pool[l],
                                         layers.v_pool[l], b0.block_table, b0.seq_lens, ws, out=out[l])
        if tm: tm.record(1)

    spans, wall = run_timed(graph_step, 2, steps, warmup, flush_buf, stream, clocks)
    spans2, _ = run_timed(eager_step, 2, max(10, min(steps, 200)), warmup, flush_buf, stream)
    ops.check_error(ws)
    return {"graph_ms": mean([x[0] for x in spans]), "step_pcts": pcts([x[0] for x in spans]),
            "eager_ms": mean([x[0] for x in spans2]),
            "graph": g, "ws": ws, "out": out, "launches": steps * layers.layers}


def e2e_layered_measure(layers, graph, out, steps, warmup, stream):
    """The graph step through the public API from pinned host memory: every step copies the
    layers' q / k_new / v_new in, replays the graph and copies the outputs back."""
    import torch

    host = {k: getattr(layers, k).cpu().pin_memory() for k in ("q", "k_new", "v_new")}
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()

    def step():
        for k, t in host.items():
            getattr(layers, k).copy_(t, non_blocking=True)
        graph.launch()
        out_host.copy_(out, non_blocking=True)

    return dict(e2e_run(step, steps, warmup, stream), h2d=h2d, d2h=d2h)


FP8_ROW_BYTES = 2 * (128 + 4)       # one token of one KV head in the 8-bit cache: K and V codes + scales


def fp8_prepare(batch):
    """Bench input: the 8-bit cache holding every sequence's context before its new token,
    quantised on the GPU (kv_append_fp8) from the batch's bf16 context rows."""
    from paged_gqa_attention_gb300 import ops
    from paged_gqa_attention_gb300 import workloads as wl

    ws = ops.make_workspace(batch.num_seqs, batch.max_blocks_per_seq)
    k_rows, v_rows, cu, lens = wl.context_rows(batch, drop_last=1)
    cache = ops.fp8_cache(batch.num_blocks)
    ops.kv_append_fp8(*cache, k_rows, v_rows, batch.block_table, cu, lens, ws)
    ops.check_error(ws)
    return cache


def fp8_decode_measure(batch, cache, steps, warmup, flush_buf, stream, clocks):
    """One decode step over the 8-bit cache: the append of every sequence's new token fused
    with the decode (paged_attn_decode_append_fp8, one kernel).  The same step as two calls
    (kv_append_fp8, then paged_attn_decode_fp8) is timed too, over fewer steps."""
    import torch

    from paged_gqa_attention_gb300 import ops

    ws = ops.make_workspace(batch.num_seqs, batch.max_blocks_per_seq)
    out = torch.empty_like(batch.q)

    def step(tm):
        if tm: tm.record(0)
        ops.paged_attn_decode_append_fp8(batch.q, batch.k_new, batch.v_new, *cache, batch.block_table,
                                         batch.seq_lens, ws, out=out)
        if tm: tm.record(1)

    def two_calls(tm):
        if tm: tm.record(0)
        ops.kv_append_fp8(*cache, batch.k_new, batch.v_new, batch.block_table, batch.cu_q_lens,
                          batch.seq_lens, ws)
        if tm: tm.record(1)
        ops.paged_attn_decode_fp8(batch.q, *cache, batch.block_table, batch.seq_lens, ws, out=out)
        if tm: tm.record(2)

    spans, wall = run_timed(step, 2, steps, warmup, flush_buf, stream, clocks)
    spans2, _ = run_timed(two_calls, 3, max(10, min(steps, 200)), warmup, flush_buf, stream)
    ops.check_error(ws)
    return {"step_ms": mean([x[0] for x in spans]), "decode_ms": mean([x[0] for x in spans]),
            "step_pcts": pcts([x[0] for x in spans]),
            "two_call_append_ms": mean([x[0] for x in spans2]), "two_call_decode_ms": mean([x[1] for x in spans2]),
            "wall_s": wall, "launches": steps}


def e2e_fp8_measure(batch, cache, steps, warmup, stream):
    """The 8-bit decode step through the public API with pinned host inputs and a host result."""
    import torch

    from paged_gqa_attention_gb300 import ops

    host = {k: getattr(batch, k).cpu().pin_memory()
            for k in ("q", "k_new", "v_new", "block_table", "seq_lens")}
    dev = {k: torch.empty_like(getattr(batch, k)) for k in host}
    out_host = torch.empty(batch.q.shape, dtype=batch.q.dtype).pin_memory()
    out_dev = torch.empty_like(batch.q)
    ws = ops.make_workspace(batch.num_seqs, batch.max_blocks_per_seq)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()

    def step():
        for k, t in host.items():
            dev[k].copy_(t, non_blocking=True)
        ops.paged_attn_decode_append_fp8(dev["q"], dev["k_new"], dev["v_new"], *cache, dev["block_table"],
                                         dev["seq_lens"], ws, out=out_dev)
        out_host.copy_(out_dev, non_blocking=True)

    r = e2e_run(step, steps, warmup, stream)
    ops.check_error(ws)
    return dict(r, h2d=h2d, d2h=d2h)


def oracle_sample_fp8(batch):
    """The oracle's 8-bit attention (as it stands) on a cache the oracle quantised itself from
    the batch's bf16 context; a pass covers the first n sequences (decode: one row each)."""
    import numpy as np
    import torch

    import oracle
    from paged_gqa_attention_gb300 import ops
    from paged_gqa_attention_gb300 import workloads as wl

    kp, vp = oracle.kv_append(batch.k_pool.cpu(), batch.v_pool.cpu(), batch.k_new.cpu(), batch.v_new.cpu(),
                              batch.block_table.cpu(), batch.cu_q_lens.cpu(), batch.seq_lens.cpu())
    as_bf16 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    k_rows, v_rows, cu_all, lens = wl.context_rows(batch, as_bf16(kp), as_bf16(vp))
    empty = [t.numpy() for t in ops.fp8_cache(batch.num_blocks, device="cpu")]
    cache = oracle.kv_append_fp8(*empty, k_rows, v_rows, batch.block_table.cpu(), cu_all, lens)
    q, bt, cu, sl = batch.q.cpu(), batch.block_table.cpu(), batch.cu_q_lens.cpu(), batch.seq_lens.cpu()
    seq_bytes = [n * 8 * FP8_ROW_BYTES for n in batch.seq_lens_host]

    def run(n):
        t0 = time.time()
        oracle.attention_fp8(q[:n], *cache, bt[:n], cu[:n + 1], sl[:n], scale=wl.SCALE)
        return time.time() - t0, float(sum(seq_bytes[:n]))

    return {"run": run, "units": batch.num_seqs, "unit": "GB/s", "scale": 1e9,
            "what": "sequences x 32 heads of the batch", "how": "fp64 C oracle over the 8-bit cache with OpenMP"}


def cascade_measure(batch, shared_blocks, steps, warmup, flush_buf, stream, clocks):
    """The decode step of a batch sharing a prefix, as a cascade: kv_append of the new tokens,
    then paged_attn_decode_cascade (the shared prefix for every query on the tensor cores,
    then each private suffix with the LSE merge)."""
    import torch

    from paged_gqa_attention_gb300 import ops

    ws = ops.make_workspace(batch.num_seqs, batch.max_blocks_per_seq)
    cws = ops.make_cascade_workspace(batch.num_seqs, batch.max_blocks_per_seq, shared_blocks)
    out = torch.empty_like(batch.q)

    def step(tm):
        if tm: tm.record(0)
        ops.kv_append(batch.k_pool, batch.v_pool, batch.k_new, batch.v_new, batch.block_table, batch.cu_q_lens,
                      batch.seq_lens, ws)
        if tm: tm.record(1)
        ops.paged_attn_decode_cascade(batch.q, batch.k_pool, batch.v_pool, batch.block_table, batch.seq_lens,
                                      shared_blocks, cws, out=out)
        if tm: tm.record(2)

    spans, wall = run_timed(step, 3, steps, warmup, flush_buf, stream, clocks)
    ops.check_error(ws)
    ops.check_error(cws)
    return {"append_ms": mean([x[0] for x in spans]), "cascade_ms": mean([x[1] for x in spans]),
            "step_ms": mean([x[0] + x[1] for x in spans]), "step_pcts": pcts([x[0] + x[1] for x in spans]),
            "wall_s": wall, "launches": 3 * steps}


E2E_HOW = ("value / ms_per_step: steps issued back to back through the public call, each reading its inputs "
           "from pinned host memory and leaving its result in host memory, the run bracketed by CUDA events; "
           "latency_ms_per_step: the same step with the host waiting for each result; host_call_us: the host's "
           "time to issue one step")


def e2e_run(step, steps, warmup, stream):
    """Time one end-to-end step (inputs from pinned host memory, result back to host memory,
    through the public call) two ways: back to back, the whole run bracketed by events and
    the host issuing each step without waiting for the last (the throughput a serving loop
    sees; every step still reads its inputs from and leaves its result in host memory), and
    one at a time, the host waiting for each step's result before issuing the next (the
    latency of one request).  Also the host's own time per call (issue only)."""
    import torch

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    host_s = 0.0
    e0.record(stream)
    for _ in range(steps):
        h0 = time.perf_counter()
        step()
        host_s += time.perf_counter() - h0
    e1.record(stream)
    e1.synchronize()
    piped = e0.elapsed_time(e1) / steps
    times = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        b.synchronize()          # the result is on the host when the step ends
        times.append(a.elapsed_time(b))
    return {"step_ms": piped, "latency_ms": mean(times), "host_call_us": host_s / steps * 1e6}


def e2e_decode_measure(batch, steps, warmup, stream, flush_buf=None):
    """The decode step through the C ABI with host buffers (pa_decode_step_host): pinned
    host inputs read in place over the host link, fused append + decode, output written back
    to host memory, every step.  With flush_buf, also the same step device-timed as the
    device-input step is (L2 flushed, queued behind a spin): the cost of the host inputs
    alone."""
    import torch

    from paged_gqa_attention_gb300 import ops

    host = {k: getattr(batch, k).cpu().pin_memory()
            for k in ("q", "k_new", "v_new", "block_table", "seq_lens")}
    out_host = torch.empty(batch.q.shape, dtype=batch.q.dtype).pin_memory()
    staging = ops.decode_step_host_staging(batch.num_seqs, batch.max_blocks_per_seq)
    ws = ops.make_workspace(batch.num_seqs, batch.max_blocks_per_seq)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()

    def step():
        ops.decode_step_host(out_host, host["q"], host["k_new"], host["v_new"], host["block_table"],
                             host["seq_lens"], batch.k_pool, batch.v_pool, staging, ws)

    r = e2e_run(step, steps, warmup, stream)
    # the host's time to issue one step through the C entry point alone (no Python checks)
    lib = ops.load()
    args = (ops.SHAPE, out_host.data_ptr(), None, host["q"].data_ptr(), host["k_new"].data_ptr(),
            host["v_new"].data_ptr(), host["block_table"].data_ptr(), host["seq_lens"].data_ptr(), batch.num_seqs,
            batch.max_blocks_per_seq, batch.k_pool.data_ptr(), batch.v_pool.data_ptr(), batch.k_pool.shape[0],
            ops.DEFAULT_SCALE, staging.data_ptr(), staging.numel(), ws.data_ptr(), ws.numel(), stream.cuda_stream)
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    for _ in range(steps):
        if lib.pa_decode_step_host(*args) != 0:
            raise RuntimeError("pa_decode_step_host failed")
    r["host_call_c_abi_us"] = (time.perf_counter() - h0) / steps * 1e6
    torch.cuda.synchronize()
    if flush_buf is not None:
        def timed(tm):
            if tm: tm.record(0)
            step()
            if tm: tm.record(1)
        spans, _ = run_timed(timed, 2, steps, warmup, flush_buf, stream)
        r["device_timed_ms"] = mean([x[0] for x in spans])
    ops.check_error(ws)
    return dict(r, h2d=h2d, d2h=d2h)


def e2e_measure(batch, kind, steps, warmup, stream):
    """The same step through the public API with pinned host inputs and a host result."""
    import torch

    from paged_gqa_attention_gb300 import ops

    host = {k: getattr(batch, k).cpu().pin_memory()
            for k in ("q", "k_new", "v_new", "block_table", "seq_lens", "cu_q_lens")}
    dev = {k: torch.empty_like(getattr(batch, k)) for k in host}
    out_host = torch.empty(batch.q.shape, dtype=batch.q.dtype).pin_memory()
    out_dev = torch.empty_like(batch.q)
    ws = ops.make_workspace(batch.num_seqs, batch.max_blocks_per_seq)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()
    n_dec = batch.info.get("n_decode", 0)
    t_dec = n_dec          # decode tokens come first in a mixed batch (one per sequence)
    shared = batch.info.get("shared_blocks", 0)
    cws = (ops.make_cascade_workspace(batch.num_seqs, batch.max_blocks_per_seq, shared)
           if kind == "cascade" else None)

    def step():
        for k in host:
            dev[k].copy_(host[k], non_blocking=True)
        if kind == "decode":
            ops.paged_attn_decode_append(dev["q"], dev["k_new"], dev["v_new"], batch.k_pool,
                                         batch.v_pool, dev["block_table"], dev["seq_lens"], ws,
                                         out=out_dev)
        elif kind == "cascade":
            ops.kv_append(batch.k_pool, batch.v_pool, dev["k_new"], dev["v_new"], dev["block_table"],
                          dev["cu_q_lens"], dev["seq_lens"], ws)
            ops.paged_attn_decode_cascade(dev["q"], batch.k_pool, batch.v_pool, dev["block_table"],
                                          dev["seq_lens"], shared, cws, out=out_dev)
        elif kind == "prefill":
            ops.paged_attn_prefill_append(dev["q"], dev["k_new"], dev["v_new"], batch.k_pool, batch.v_pool,
                                          dev["block_table"], dev["cu_q_lens"], dev["seq_lens"], batch.max_q_len, ws,
                                          out=out_dev)
        else:  # mixed: decode sequences, then prefill chunks, from the same device copies
            ops.paged_attn_decode_append(dev["q"][:t_dec], dev["k_new"][:t_dec], dev["v_new"][:t_dec],
                                         batch.k_pool, batch.v_pool, dev["block_table"][:n_dec],
                                         dev["seq_lens"][:n_dec], ws, out=out_dev[:t_dec])
            cu_p = dev["cu_q_lens"][n_dec:] - t_dec
            ops.paged_attn_prefill_append(dev["q"][t_dec:], dev["k_new"][t_dec:], dev["v_new"][t_dec:],
                                          batch.k_pool, batch.v_pool, dev["block_table"][n_dec:], cu_p,
                                          dev["seq_lens"][n_dec:], batch.max_q_len, ws, out=out_dev[t_dec:])
        out_host.copy_(out_dev, non_blocking=True)

    r = e2e_run(step, steps, warmup, stream)
    ops.check_error(ws)
    return dict(r, h2d=h2d, d2h=d2h)


# ------------------------------------------------------------------ CPU oracle

def compact_subset(batch, n_seqs):
    """Host copy of the first n_seqs sequences of a batch with only the pool blocks they use
    (tables renumbered to a compact pool): input preparation for the oracle's sample, so that
    a sample of a large workload does not copy its whole pools.  Pure data movement."""
    import torch

    from paged_gqa_attention_gb300 import workloads as wl

    sub = batch.select(slice(0, n_seqs))
    rows = sub.block_table
    used = torch.unique(rows[rows >= 0])
    remap = torch.full((batch.num_blocks,), -1, dtype=torch.int64, device=rows.device)
    remap[used] = torch.arange(used.numel(), device=rows.device)
    bt = torch.where(rows >= 0, remap[rows.clamp(min=0).long()], torch.full_like(rows.long(), -1))
    return wl.Batch(name=sub.name, q=sub.q.cpu(), k_new=sub.k_new.cpu(), v_new=sub.v_new.cpu(),
                    k_pool=batch.k_pool.index_select(0, used).cpu(),
                    v_pool=batch.v_pool.index_select(0, used).cpu(),
                    block_table=bt.to(torch.int32).cpu(), seq_lens=sub.seq_lens.cpu(),
                    cu_q_lens=sub.cu_q_lens.cpu(), max_q_len=sub.max_q_len,
                    seq_lens_host=list(sub.seq_lens_host), q_lens_host=list(sub.q_lens_host),
                    info=dict(sub.info))


def oracle_sample_attention(batch, kind, rows_cap=None, threads=0):
    """The oracle (as it stands) on a bounded sample of the workload: (token, head) rows of the
    first sequences (at least one; capped for prefill), each pass over n of them (evenly
    spaced).  The throughput is scaled to the metric's unit by the rows' own bytes or flops.
    threads: OpenMP threads of the oracle (0 = every core)."""
    import numpy as np

    import oracle
    from paged_gqa_attention_gb300 import workloads as wl

    n_seqs, rows_so_far = 0, 0
    for ql in batch.q_lens_host:
        n_seqs += 1
        rows_so_far += ql * 32
        if rows_cap and rows_so_far >= rows_cap:
            break
    sb = compact_subset(batch, n_seqs)
    kp, vp = oracle.kv_append(sb.k_pool, sb.v_pool, sb.k_new, sb.v_new, sb.block_table, sb.cu_q_lens,
                              sb.seq_lens)
    q, bt, cu, sl = sb.q, sb.block_table, sb.cu_q_lens, sb.seq_lens
    toks_all = list(range(int(cu[-1])))
    toks = np.repeat(np.array(toks_all, dtype=np.int32), 32)
    heads = np.tile(np.arange(32, dtype=np.int32), len(toks_all))
    if rows_cap and len(toks) > rows_cap:
        sel = np.linspace(0, len(toks) - 1, rows_cap).astype(np.int64)
        toks, heads = toks[sel], heads[sel]
    # work per row: the (query, key) pairs it attends to
    cu_l, sl_l, ql_l = [int(x) for x in cu], sb.seq_lens_host, sb.q_lens_host
    seqs = np.searchsorted(cu_l, toks, side="right") - 1
    pairs = np.array([sl_l[s] - ql_l[s] + (t - cu_l[s]) + 1 for t, s in zip(toks.tolist(), seqs.tolist())],
                     dtype=np.float64)
    # decode: KV bytes, every (sequence, KV head) context row read once -> per query-head row
    # the share is (p + 1) tokens x 2 (K, V) x 128 x 2 B / 4 heads; prefill: 4 x 128 flops a pair
    per_pair = (2 * 128 * 2) / 4 if kind == "decode" else 4 * 128

    def run(n):
        pick = np.linspace(0, len(toks) - 1, n).astype(np.int64) if n < len(toks) else np.arange(len(toks))
        t0 = time.time()
        oracle.attention(q, kp, vp, bt, cu, sl, scale=wl.SCALE, rows=(toks[pick], heads[pick]),
                         num_threads=threads)
        return time.time() - t0, float(pairs[pick].sum()) * per_pair

    return {"run": run, "units": len(toks), "unit": "GB/s" if kind == "decode" else "TFLOP/s",
            "scale": 1e9 if kind == "decode" else 1e12,
            "what": f"(token, head) rows of the first {n_seqs} sequence(s) of the workload",
            "how": "fp64 C oracle with OpenMP", "threads": threads}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def timed_oracle(sample, target_s):
    """Full passes over the sample for about target_s (at least one): the cpu_baseline object."""
    import oracle

    reps, dt, work = 0, 0.0, 0.0
    while True:
        d, w = sample["run"](sample["units"])
        reps, dt, work = reps + 1, dt + d, work + w
        if dt >= target_s:
            break
    threads = sample.get("threads") or oracle.max_threads()
    return {"value": work / dt / sample["scale"], "unit": sample["unit"], "cores": threads,
            "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"{sample['units']} {sample['what']}, {reps} pass(es), {dt:.1f} s, {sample['how']}"
                      f" on {threads} thread(s)"}


def cpu_baseline(batch, kind, target_s, rows_cap=None, threads=0):
    return timed_oracle(oracle_sample_attention(batch, kind, rows_cap, threads), target_s)


def cpu_baseline_fp8(batch, target_s):
    return timed_oracle(oracle_sample_fp8(batch), target_s)


def cpu_baseline_qkv(tokens, target_s):
    return timed_oracle(oracle_sample_qkv(tokens), target_s)


# ------------------------------------------------------------------ merged Q/K/V projection

QKV_HIDDEN = 4096                  # Qwen3-8B's hidden size


def qkv_inputs(tokens, seed, device="cuda"):
    """Synthetic x [tokens, 4096] ~ N(0, 1) and stacked weights [6144, 4096] ~ N(0, 1/4096), bf16."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(tokens, QKV_HIDDEN, generator=g, device=device).to(torch.bfloat16)
    w = (torch.randn(6144, QKV_HIDDEN, generator=g, device=device) / 64).to(torch.bfloat16)
    return x, w


def qkv_measure(batch, x, w, steps, warmup, flush_buf, stream, clocks, qk_norm=False):
    """One paged_qkv_append call (one kernel): q of every new token out, k and v into the cache,
    q and k rotated by Qwen3's rotary embedding (theta 1e6) at each token's position.  With
    qk_norm, the call with Qwen3's per-head normalisation of q and k first (synthetic gains;
    two kernels: the projection, then the in-place norm and rotation)."""
    import torch

    from paged_gqa_attention_gb300 import ops

    ws = ops.make_workspace(batch.num_seqs, batch.max_blocks_per_seq)
    q = torch.empty(x.shape[0], 32, 128, dtype=torch.bfloat16, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    gq, gk = ((1.0 + 0.5 * torch.randn(128, generator=g, device="cuda")).to(torch.bfloat16) if qk_norm else None
              for _ in range(2))

    def step(tm):
        if tm: tm.record(0)
        ops.paged_qkv_append(x, w, batch.k_pool, batch.v_pool, batch.block_table, batch.cu_q_lens,
                             batch.seq_lens, ws, rope_theta=ops.QWEN3_ROPE_THETA, q_norm_weight=gq,
                             k_norm_weight=gk, q_out=q)
        if tm: tm.record(1)

    spans, wall = run_timed(step, 2, steps, warmup, flush_buf, stream, clocks)
    ops.check_error(ws)
    return {"step_ms": mean([sp[0] for sp in spans]), "step_pcts": pcts([sp[0] for sp in spans]), "wall_s": wall,
            "launches": steps * (2 if qk_norm else 1)}


def e2e_qkv_measure(batch, x, w, steps, warmup, stream):
    """End to end through the public call: x copied from pinned host memory, the projection,
    q copied back to pinned host memory, all inside the timed region (w stays resident, as a
    layer's weights do)."""
    import torch

    from paged_gqa_attention_gb300 import ops

    ws = ops.make_workspace(batch.num_seqs, batch.max_blocks_per_seq)
    x_host = x.cpu().pin_memory()
    q_host = torch.empty(x.shape[0], 32, 128, dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x)
    q_dev = torch.empty(x.shape[0], 32, 128, dtype=torch.bfloat16, device="cuda")

    def step():
        x_dev.copy_(x_host, non_blocking=True)
        ops.paged_qkv_append(x_dev, w, batch.k_pool, batch.v_pool, batch.block_table, batch.cu_q_lens,
                             batch.seq_lens, ws, rope_theta=ops.QWEN3_ROPE_THETA, q_out=q_dev)
        q_host.copy_(q_dev, non_blocking=True)

    r = e2e_run(step, steps, warmup, stream)
    ops.check_error(ws)
    return dict(r, h2d=x_host.numel() * 2, d2h=q_host.numel() * 2)


def oracle_sample_qkv(tokens):
    """The oracle's fp64 projection on the host cores; a pass covers n of 16 token rows spread
    over the workload's tokens."""
    import oracle

    x, w = qkv_inputs(tokens, 7, device="cpu")
    rows = list(range(0, tokens, max(1, tokens // 16)))[:16]

    def run(n):
        t0 = time.time()
        oracle.qkv_project(x, w, rows=rows[:n])
        return time.time() - t0, 2.0 * n * QKV_HIDDEN * 6144

    return {"run": run, "units": len(rows), "unit": "TFLOP/s", "scale": 1e12,
            "what": f"token rows x 6144 outputs x {QKV_HIDDEN}", "how": "fp64 C oracle with OpenMP"}


# ------------------------------------------------------------------ main paths

def reference_arm(args, world, rank):
    """--impl reference: the oracle on the host cores, rank 0 only.  The inputs are prepared
    once; one warm-up pass over the whole sample sizes each step's share of it so that the K
    steps together take about --cpu-seconds."""
    if rank != 0:
        return
    import oracle
    import torch

    from paged_gqa_attention_gb300 import workloads as wl

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    if args.workload == "batched_decode_fp8":
        sample = oracle_sample_fp8(wl.batched_decode(device=dev))
    elif args.workload == "qkv_append":
        sample = oracle_sample_qkv(4096)
    else:
        if args.workload == "layered_decode":
            batch = wl.layered_decode(device=dev).base     # GB/s of one layer: the same per layer
        elif args.workload == "prefix_shared_decode_cascade":
            batch = wl.prefix_shared_decode(device=dev)    # the cascade computes the same attention
        else:
            batch = wl.WORKLOADS[args.workload](device=dev)
        kind = "decode" if "decode" in args.workload or args.workload == "mixed_batch" else "prefill"
        sample = oracle_sample_attention(batch, kind, rows_cap_for(args.workload))
    steps = max(args.steps, 1)
    d_full, _ = sample["run"](sample["units"])                      # warm-up, sizes the steps
    per_step = args.cpu_seconds / steps
    n = max(1, min(sample["units"], int(sample["units"] * per_step / max(d_full, 1e-9))))
    vals, secs = [], 0.0
    for _ in range(steps):
        d, w = sample["run"](n)
        secs += d
        vals.append(w / d / sample["scale"])
    value = mean(vals)
    cpu = {"value": value, "unit": sample["unit"], "cores": oracle.max_threads(), "kind": "oracle",
           "sample": f"{n} of {sample['units']} {sample['what']} per step, {steps} steps, {secs:.1f} s, "
                     f"{sample['how']}"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": sample["unit"],
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload}, "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": sample["unit"], "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def rows_cap_for(workload):
    """Bound on the (token, head) rows of one oracle pass (keeps a pass to seconds)."""
    return {"single_decode": None, "batched_decode": None, "mixed_batch": 1024,
            "causal_prefill": 2048, "prefix_shared_decode": 256, "layered_decode": None,
            "prefix_shared_decode_cascade": 256}[workload]


def roofline(achieved, peak, unit, bound, traffic):
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak if peak else None, "traffic": traffic}


def traffic_for(kernel, workload=None):
    """DRAM bytes of one launch from the committed capture, or None when the sources changed
    since, or when the line's workload is not the one captured (a launch of another size)."""
    t = TRAFFIC.get(kernel)
    if not t or source_hash(*t["sources"]) != t["sha"]:
        return None
    if workload is not None and workload != t["workload"]:
        return None
    return t["bytes_per_launch"]


DEFAULT_SUBS = ("single_decode", "causal_prefill", "mixed_batch", "prefix_shared_decode",
                "prefix_shared_decode_cascade", "batched_decode_fp8", "layered_decode", "qkv_append")


def load_workload(wname):
    """The batch (and, for the layered step, the layers) a workload measures, on the GPU."""
    from paged_gqa_attention_gb300 import workloads as wl

    layers = wl.layered_decode(device="cuda") if wname == "layered_decode" else None
    if layers is not None:
        return layers.base, layers
    if wname == "batched_decode_fp8":
        return wl.batched_decode(device="cuda"), None
    if wname == "prefix_shared_decode_cascade":
        return wl.prefix_shared_decode(device="cuda"), None
    if wname == "qkv_append":
        return wl.causal_prefill(device="cuda"), None   # the 4096-token prompt's new tokens
    return wl.WORKLOADS[wname](device="cuda"), None


def timing_floor(flush_buf, stream, steps=300):
    """The time this method gives a step that does almost nothing: one torch kernel adding 1 to
    32 floats, timed like every step (L2 flushed, queued behind a device spin, CUDA events
    around it).  The launch after the step's first event is part of every measured step."""
    import torch

    x = torch.zeros(32, device="cuda")

    def step(tm):
        if tm: tm.record(0)
        x.add_(1.0)
        if tm: tm.record(1)

    spans, _ = run_timed(step, 2, steps, 20, flush_buf, stream)
    return mean([s[0] for s in spans]) * 1e3


def warm_l2_latency(batch, stream, steps=200):
    """The fused decode step back to back with nothing flushed in between (the whole working
    set stays in L2): mean latency of one call, in us."""
    import torch

    from paged_gqa_attention_gb300 import ops

    ws = ops.make_workspace(batch.num_seqs, batch.max_blocks_per_seq)
    out = torch.empty_like(batch.q)
    call = lambda: ops.paged_attn_decode_append(batch.q, batch.k_new, batch.v_new, batch.k_pool, batch.v_pool,
                                                batch.block_table, batch.seq_lens, ws, out=out)
    for _ in range(20):
        call()
    torch.cuda.synchronize()
    # every call is queued behind a device spin first, so that the events bracket device time
    # and not the host's launch rate
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda._sleep(HEAD_START_CYCLES * max(1, steps // 2))
    for e0, e1 in ev:
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    ops.check_error(ws)
    v = [a.elapsed_time(b) * 1e3 for a, b in ev]
    return {"mean_us": mean(v), "p50_us": pcts(v)["p50"], "steps": steps,
            "how": "fused append + decode, all calls queued behind a device spin, no L2 flush between "
                   "them (the 2 MiB context stays in L2), CUDA events around each call"}


def measure(wname, steps, warmup, e2e_steps, peaks, flush_buf, stream, clocks, world):
    """One workload's entry of the JSON line: value, unit, ms_per_step, roofline, kernels,
    gpu_launches, e2e and config.  Returns (entry, kind, batch, layers)."""
    import torch

    from paged_gqa_attention_gb300 import workloads as wl

    batch, layers = load_workload(wname)
    e = {}
    cfg = {"workload": wname, **batch.info, "heads": "32 q / 8 kv x 128", "block_tokens": 256,
           **({"layers": layers.layers} if layers is not None else {}),
           "l2": f"flushed before every timed step ({FLUSH_BYTES >> 20} MiB write + read)",
           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}

    if wname in ("single_decode", "batched_decode", "prefix_shared_decode"):
        r = decode_measure(batch, steps, warmup, flush_buf, stream, clocks)
        kv_bytes = batch.kv_bytes()
        io_bytes = batch.num_seqs * 32 * 128 * 2 * 2 + batch.num_seqs * (batch.max_blocks_per_seq + 1) * 4
        step_ms = dist_max(r["step_ms"], world)
        attn_ms = dist_max(r["attn_ms"], world)
        e.update(value=world * kv_bytes / (step_ms * 1e-3) / 1e9, unit="GB/s", ms_per_step=step_ms)
        # algorithmic bytes: every distinct K/V byte once (the shared prefix of the prefix-shared
        # workload is one set of blocks, however many sequences read it)
        alg_bytes = wl.unique_kv_bytes(batch) + io_bytes
        ach = alg_bytes / (attn_ms * 1e-3) / 1e9
        e["roofline"] = roofline(ach, peaks["hbm_gbs"], "GB/s", "hbm", traffic_for("decode", wname))
        e["roofline"]["kernel"] = "decode_kernel"
        e["roofline"]["algorithmic_bytes_per_launch"] = alg_bytes
        e["kernels"] = {"decode_append_us": r["attn_ms"] * 1e3,
                        "two_call_step": {"kv_append_us": r["two_call_append_ms"] * 1e3,
                                          "decode_us": r["two_call_decode_ms"] * 1e3},
                        "kv_bytes_per_step": kv_bytes,
                        "unique_kv_bytes": wl.unique_kv_bytes(batch)}
        if wname == "prefix_shared_decode":
            uniq = wl.unique_kv_bytes(batch)
            e["kernels"]["unique_kv_gbs"] = uniq / (attn_ms * 1e-3) / 1e9
            e["kernels"]["unique_kv_frac"] = e["kernels"]["unique_kv_gbs"] / peaks["hbm_gbs"]
        if wname == "single_decode":
            e["warm_l2_latency"] = warm_l2_latency(batch, stream)
        e["gpu_launches"] = r["launches"]
        x = e2e_decode_measure(batch, e2e_steps, 5, stream, flush_buf)
        x_ms = dist_max(x["step_ms"], world)
        e["e2e"] = {"value": world * kv_bytes / (x_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": x["h2d"], "d2h_bytes_per_step": x["d2h"], "ms_per_step": x_ms,
                    "via": "pa_decode_step_host (C ABI, host buffers)",
                    "latency_ms_per_step": x["latency_ms"], "host_call_us": x["host_call_us"], "how": E2E_HOW,
                    "device_timed_step_us": x["device_timed_ms"] * 1e3, "host_call_c_abi_us": x["host_call_c_abi_us"]}
        kind = "decode"
    elif wname == "layered_decode":
        r = layered_measure(layers, steps, warmup, flush_buf, stream, clocks)
        kv_bytes = layers.kv_bytes()
        io_bytes = layers.layers * (batch.num_seqs * 32 * 128 * 2 * 2 +
                                    batch.num_seqs * (batch.max_blocks_per_seq + 1) * 4)
        step_ms = dist_max(r["graph_ms"], world)
        e.update(value=world * kv_bytes / (step_ms * 1e-3) / 1e9, unit="GB/s", ms_per_step=step_ms)
        e["roofline"] = roofline((kv_bytes + io_bytes) / (step_ms * 1e-3) / 1e9, peaks["hbm_gbs"],
                                 "GB/s", "hbm", traffic_for("decode", wname))
        e["roofline"]["kernel"] = "decode_kernel"
        e["roofline"]["algorithmic_bytes_per_launch"] = (kv_bytes + io_bytes) // layers.layers
        e["kernels"] = {"layers": layers.layers, "graph_step_us": r["graph_ms"] * 1e3,
                        "graph_us_per_layer": r["graph_ms"] * 1e3 / layers.layers,
                        "one_call_per_layer_step_us": r["eager_ms"] * 1e3,
                        "one_call_per_layer_us_per_layer": r["eager_ms"] * 1e3 / layers.layers,
                        "kv_bytes_per_step": kv_bytes}
        e["gpu_launches"] = r["launches"]
        x = e2e_layered_measure(layers, r["graph"], r["out"], e2e_steps, 5, stream)
        x_ms = dist_max(x["step_ms"], world)
        e["e2e"] = {"value": world * kv_bytes / (x_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": x["h2d"], "d2h_bytes_per_step": x["d2h"], "ms_per_step": x_ms,
                    "latency_ms_per_step": x["latency_ms"], "host_call_us": x["host_call_us"], "how": E2E_HOW}
        r["graph"].close()
        kind = "decode"
    elif wname == "prefix_shared_decode_cascade":
        shared = batch.info["shared_blocks"]
        r = cascade_measure(batch, shared, steps, warmup, flush_buf, stream, clocks)
        kv_bytes = batch.kv_bytes()
        uniq = wl.unique_kv_bytes(batch)
        step_ms = dist_max(r["step_ms"], world)
        casc_ms = dist_max(r["cascade_ms"], world)
        e.update(value=world * kv_bytes / (step_ms * 1e-3) / 1e9, unit="GB/s", ms_per_step=step_ms)
        e["roofline"] = roofline(uniq / (casc_ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s", "hbm", None)
        e["roofline"]["kernel"] = "cascade (prefix pass on prefill_kernel + suffix decode_kernel)"
        e["roofline"]["algorithmic_bytes_per_launch"] = uniq
        e["kernels"] = {"kv_append_us": r["append_ms"] * 1e3, "cascade_us": r["cascade_ms"] * 1e3,
                        "kv_bytes_per_step": kv_bytes, "unique_kv_bytes": uniq,
                        "unique_kv_gbs": uniq / (casc_ms * 1e-3) / 1e9}
        e["gpu_launches"] = r["launches"]
        cfg["cascade"] = f"{shared} shared blocks attended once per KV head, then the private suffixes"
        x = e2e_measure(batch, "cascade", max(10, min(e2e_steps, 50)), 3, stream)
        x_ms = dist_max(x["step_ms"], world)
        e["e2e"] = {"value": world * kv_bytes / (x_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": x["h2d"], "d2h_bytes_per_step": x["d2h"], "ms_per_step": x_ms,
                    "latency_ms_per_step": x["latency_ms"], "host_call_us": x["host_call_us"], "how": E2E_HOW}
        kind = "decode"
    elif wname == "batched_decode_fp8":
        cache = fp8_prepare(batch)
        r = fp8_decode_measure(batch, cache, steps, warmup, flush_buf, stream, clocks)
        ntok = sum(batch.seq_lens_host)
        kv_bytes = ntok * 8 * FP8_ROW_BYTES
        bf16_bytes = batch.kv_bytes()
        io_bytes = batch.num_seqs * 32 * 128 * 2 * 2 + batch.num_seqs * (batch.max_blocks_per_seq + 1) * 4
        step_ms = dist_max(r["step_ms"], world)
        dec_ms = dist_max(r["decode_ms"], world)
        e.update(value=world * kv_bytes / (step_ms * 1e-3) / 1e9, unit="GB/s", ms_per_step=step_ms)
        e["roofline"] = roofline((kv_bytes + io_bytes) / (dec_ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s",
                                 "hbm", traffic_for("decode_fp8", wname))
        e["roofline"]["kernel"] = "decode_fp8_kernel"
        e["roofline"]["algorithmic_bytes_per_launch"] = kv_bytes + io_bytes
        e["kernels"] = {"decode_append_fp8_us": r["step_ms"] * 1e3,
                        "two_call_step": {"kv_append_fp8_us": r["two_call_append_ms"] * 1e3,
                                          "decode_fp8_us": r["two_call_decode_ms"] * 1e3},
                        "fp8_kv_bytes_per_step": kv_bytes, "bf16_kv_bytes_per_step": bf16_bytes,
                        "bf16_equivalent_gbs": world * bf16_bytes / (step_ms * 1e-3) / 1e9}
        e["gpu_launches"] = r["launches"]
        x = e2e_fp8_measure(batch, cache, e2e_steps, 5, stream)
        x_ms = dist_max(x["step_ms"], world)
        e["e2e"] = {"value": world * kv_bytes / (x_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": x["h2d"], "d2h_bytes_per_step": x["d2h"], "ms_per_step": x_ms,
                    "latency_ms_per_step": x["latency_ms"], "host_call_us": x["host_call_us"], "how": E2E_HOW}
        cfg["kv_cache"] = "8-bit: E4M3 codes + one fp32 scale per token and KV head"
        e["dtype"] = "f16 products over e4m3 codes"
        kind = "decode_fp8"
    elif wname == "qkv_append":
        x_in, w = qkv_inputs(batch.total_tokens, 7)
        r = qkv_measure(batch, x_in, w, steps, warmup, flush_buf, stream, clocks)
        flops = 2.0 * batch.total_tokens * QKV_HIDDEN * 6144
        step_ms = dist_max(r["step_ms"], world)
        e.update(value=world * flops / (step_ms * 1e-3) / 1e12, unit="TFLOP/s", ms_per_step=step_ms)
        e["roofline"] = roofline(flops / (step_ms * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s", "tensor",
                                 traffic_for("qkv", wname))
        e["roofline"]["kernel"] = "qkv_pair_kernel"
        e["roofline"]["algorithmic_flops_per_launch"] = flops
        # the same call for a decode step's batch: 32 new tokens, the weights dominate the bytes
        db = wl.batched_decode(device="cuda")
        dx, _ = qkv_inputs(db.total_tokens, 8)
        dr = qkv_measure(db, dx, w, max(20, min(steps, 200)), warmup, flush_buf, stream, None)
        wbytes = 6144 * QKV_HIDDEN * 2 + db.total_tokens * (QKV_HIDDEN + 6144) * 2
        e["kernels"] = {"qkv_us": r["step_ms"] * 1e3, "tokens": batch.total_tokens, "hidden": QKV_HIDDEN,
                        "decode_batch": {"tokens": db.total_tokens, "qkv_us": dr["step_ms"] * 1e3,
                                         "bytes": wbytes, "gbs": wbytes / (dr["step_ms"] * 1e-3) / 1e9,
                                         "hbm_frac": wbytes / (dr["step_ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"]}}
        # the same call with Qwen3's QK-norm: the projection without the rotation, then one
        # memory-bound pass that reads and rewrites every new q and k row
        nr = qkv_measure(batch, x_in, w, max(20, min(steps, 200)), warmup, flush_buf, stream, None, qk_norm=True)
        pr = qkv_measure(batch, x_in, w, max(20, min(steps, 200)), warmup, flush_buf, stream, None)
        norm_bytes = 2 * batch.total_tokens * (32 + 8) * 128 * 2
        extra_us = (nr["step_ms"] - pr["step_ms"]) * 1e3
        e["kernels"]["qk_norm"] = {
            "call_us": nr["step_ms"] * 1e3, "plain_call_us": pr["step_ms"] * 1e3, "extra_us": extra_us,
            "norm_pass_bytes": norm_bytes,
            "norm_pass_gbs_if_extra": norm_bytes / (extra_us * 1e-6) / 1e9 if extra_us > 0 else None,
            "how": "the call with QK-norm and the plain call, each timed over the same steps; extra_us is "
                   "their difference (the norm pass plus the launch between the two kernels)"}
        e["gpu_launches"] = r["launches"] + dr["launches"] + nr["launches"] + pr["launches"]
        x = e2e_qkv_measure(batch, x_in, w, max(10, min(e2e_steps, 50)), 3, stream)
        x_ms = dist_max(x["step_ms"], world)
        e["e2e"] = {"value": world * flops / (x_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": x["h2d"], "d2h_bytes_per_step": x["d2h"], "ms_per_step": x_ms,
                    "latency_ms_per_step": x["latency_ms"], "host_call_us": x["host_call_us"], "how": E2E_HOW}
        cfg["projection"] = ("x [4096, 4096] @ w_qkv [6144, 4096]^T; rotary embedding of q and k (theta 1e6); "
                             "q out, k and v into their cache slots")
        kind = "qkv"
    elif wname == "causal_prefill":
        r = prefill_measure(batch, steps, warmup, flush_buf, stream, clocks)
        flops = batch.attention_flops()
        step_ms = dist_max(r["step_ms"], world)
        e.update(value=world * flops / (step_ms * 1e-3) / 1e12, unit="TFLOP/s", ms_per_step=step_ms)
        # the step is one kernel: the prefill with the prompt's append fused in
        e["roofline"] = roofline(flops / (step_ms * 1e-3) / 1e12, peaks["bf16_tflops"],
                                 "TFLOP/s", "tensor", traffic_for("prefill", wname))
        e["roofline"]["kernel"] = "prefill_kernel (append fused)"
        e["roofline"]["algorithmic_flops_per_launch"] = flops
        e["kernels"] = {"prefill_append_us": r["step_ms"] * 1e3,
                        "two_call_step": {"kv_append_us": r["two_call_append_ms"] * 1e3,
                                          "prefill_us": r["two_call_prefill_ms"] * 1e3}}
        e["gpu_launches"] = r["launches"]
        x = e2e_measure(batch, "prefill", max(10, min(e2e_steps, 50)), 3, stream)
        x_ms = dist_max(x["step_ms"], world)
        e["e2e"] = {"value": world * flops / (x_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": x["h2d"], "d2h_bytes_per_step": x["d2h"], "ms_per_step": x_ms,
                    "latency_ms_per_step": x["latency_ms"], "host_call_us": x["host_call_us"], "how": E2E_HOW}
        kind = "prefill"
    else:  # mixed_batch
        r = mixed_measure(batch, steps, warmup, flush_buf, stream, clocks)
        dec, pre = r["dec"], r["pre"]
        kv_bytes = dec.kv_bytes()
        flops = pre.attention_flops()
        step_ms = dist_max(r["step_ms"], world)
        t_bw = kv_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3
        t_tc = flops / (peaks["bf16_tflops"] * 1e12) * 1e3
        e.update(value=world * kv_bytes / (step_ms * 1e-3) / 1e9, unit="GB/s", ms_per_step=step_ms)
        e["roofline"] = roofline(kv_bytes / (r["decode_ms"] * 1e-3) / 1e9, peaks["hbm_gbs"],
                                 "GB/s", "hbm", traffic_for("decode", wname))
        e["roofline"]["kernel"] = "decode_kernel (append fused)"
        e["roofline"]["algorithmic_bytes_per_launch"] = kv_bytes
        e["prefill_roofline"] = dict(roofline(flops / (r["prefill_ms"] * 1e-3) / 1e12, peaks["bf16_tflops"],
                                              "TFLOP/s", "tensor", traffic_for("prefill", wname)),
                                     kernel="prefill_kernel (append fused; + planning kernel)",
                                     algorithmic_flops_per_launch=flops)
        e["kernels"] = {"decode_append_us": r["decode_ms"] * 1e3, "prefill_append_us": r["prefill_ms"] * 1e3,
                        "prefill_tflops": flops / (r["prefill_ms"] * 1e-3) / 1e12,
                        "combined_roofline_frac": (t_bw + t_tc) / step_ms,
                        "three_call_step": {k.replace("_ms", "_us"): v * 1e3 for k, v in r["three_call"].items()}}
        e["gpu_launches"] = r["launches"]
        x = e2e_measure(batch, "mixed", max(10, min(e2e_steps, 100)), 3, stream)
        x_ms = dist_max(x["step_ms"], world)
        e["e2e"] = {"value": world * kv_bytes / (x_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": x["h2d"], "d2h_bytes_per_step": x["d2h"], "ms_per_step": x_ms,
                    "latency_ms_per_step": x["latency_ms"], "host_call_us": x["host_call_us"], "how": E2E_HOW}
        kind = "decode"
    if r.get("step_pcts"):
        e["step_ms_percentiles"] = r["step_pcts"]   # this rank's timed steps (rank 0 prints)
    e["config"] = cfg
    return e, kind, batch, layers


def cpu_for(wname, kind, batch, seconds, threads=0):
    """The oracle timed on the host cores over a bounded sample of the workload."""
    from paged_gqa_attention_gb300 import workloads as wl

    if kind == "decode_fp8":
        return cpu_baseline_fp8(batch, seconds)
    if kind == "qkv":
        return cpu_baseline_qkv(batch.total_tokens, seconds)
    return cpu_baseline(batch, kind, seconds, rows_cap_for(wname), threads)


def main():
    args = parse_args()
    if args.impl == "reference":
        # host-only: rank 0 runs the oracle, the other ranks exit at once (no process group)
        reference_arm(args, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
        return
    world, rank, local = dist_setup()
    import torch

    from paged_gqa_attention_gb300 import build as pa_build
    from paged_gqa_attention_gb300 import ops

    torch.cuda.set_device(local)
    pa_build.build()
    ops.load()
    peaks = measured_peaks()
    stream = torch.cuda.current_stream()
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    clocks = ClockSampler(local)
    clocks.start()
    wname = args.workload
    cpu_ok = rank == 0 and world == 1 and not args.no_cpu_baseline
    dist_barrier(world)

    e2e_steps = max(20, min(args.steps, 200))
    entry, kind, batch, layers = measure(wname, args.steps, args.warmup, e2e_steps, peaks, flush_buf, stream,
                                         clocks, world)
    line = {"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic"}
    line.update(entry)
    if cpu_ok:
        line["cpu_baseline"] = cpu_for(wname, kind, batch, args.cpu_seconds)
        if wname in ("single_decode", "batched_decode"):
            one = cpu_for(wname, kind, batch, max(2.0, args.cpu_seconds / 4), threads=1)
            line["cpu_baseline"]["one_core"] = {"value": one["value"], "unit": one["unit"], "cores": 1,
                                                "sample": one["sample"]}
    del batch, layers
    torch.cuda.empty_cache()

    # The default run also measures every other configuration of the metric (one sub-object
    # each, fewer steps, a shorter CPU baseline): the causal prefill as "prefill" (the other
    # half of the metric), the rest under "configs".
    sub_steps = max(10, min(args.steps, 200))
    sub_warm = max(3, min(args.warmup, 10))
    sub_cpu = max(2.0, args.cpu_seconds / 4)
    if wname == "batched_decode" and not args.only_main:
        subs = {}
        for sname in DEFAULT_SUBS:
            if sname == "causal_prefill" and args.no_prefill:
                continue
            se, skind, sbatch, slayers = measure(sname, sub_steps, sub_warm, max(10, min(sub_steps, 50)), peaks,
                                                 flush_buf, stream, clocks, world)
            se["steps"] = sub_steps
            se["warmup"] = sub_warm
            if cpu_ok:
                se["cpu_baseline"] = cpu_for(sname, skind, sbatch, sub_cpu)
                if sname == "single_decode":
                    one = cpu_for(sname, skind, sbatch, sub_cpu, threads=1)
                    se["cpu_baseline"]["one_core"] = {"value": one["value"], "unit": one["unit"], "cores": 1,
                                                      "sample": one["sample"]}
            if sname == "causal_prefill":
                line["prefill"] = se
            else:
                subs[sname] = se
            del sbatch, slayers
            torch.cuda.empty_cache()
        line["configs"] = subs
    line["clocks"] = clocks.stop()
    line["peaks"] = peaks
    line["timing_floor_us"] = timing_floor(flush_buf, stream)
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist_barrier(world)


if __name__ == "__main__":
    main()
