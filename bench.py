#!/usr/bin/env python
"""Benchmark of the lightning-indexer hot path on one GB300 (or N replicas).

One step = one fused decode (block scores + top-k) over the spec-decode batch:
64 requests x 4 query tokens (positions seq_len-4..seq_len-1), seq_lens uniform
in [4096, 32768], 1 index head, topk 16, init 1, local 2, pages shuffled in a
pool 1.25x the need.  Inputs are resident in HBM; the L2 is flushed (a read of
a 2x-L2 buffer) before every timed step and the flush is not timed.  Each
timed step replays a CUDA graph of the public call (as a serving loop runs
decode steps); the same call timed eagerly is reported beside it.

Printed: one JSON line with rows/s (value), the roofline of the decode kernel
against the measured HBM copy bandwidth, the CPU oracle timed on one host
core and on all of them, an end-to-end figure through the public API with
host buffers, clocks sampled during the run, and (under "extra") the other
workloads: high-batch decode, NVFP4 decode, causal prefill at topk 16 and 32,
NVFP4 prefill, a chunked prefill batch, the sparse page table and a mixed
decode + prefill batch.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs its own replica of the batch (weak scaling);
value is the rows of all ranks over the slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode score+top-k rows/s & HBM GB/s; prefill index TFLOP/s vs peak"
HEADLINE = "spec_decode"
# the headline batch, as both arms (ours and the oracle's) name it
HEADLINE_WORKLOAD = ("spec-decode batch: 64 requests x query_len 4, seq_lens U[4096,32768], "
                     "1 index head, topk 16, init 1, local 2, pool 1.25x need (shuffled)")
BLOCK = 128
L2_BYTES = 129 * 1024 * 1024
# kernel sources whose hash a committed ncu summary must match for its
# dram traffic to be reported
DECODE_SOURCES = ["decode.cu", "decode_common.cuh", "ptx.cuh", "internal.h", "warp_select.cuh"]
NVFP4_DECODE_SOURCES = ["decode_fp4.cu", "decode_common.cuh", "ptx.cuh", "internal.h",
                        "warp_select.cuh", "nvfp4.cuh"]
PREFILL_SOURCES = ["prefill.cu", "ptx.cuh", "internal.h", "warp_select.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="bound on the CPU oracle sample")
    ap.add_argument("--only", choices=["high_batch", "nvfp4_decode", "prefill", "prefill_topk32",
                                       "nvfp4_prefill", "chunked_prefill", "mixed_batch"],
                    help="run just this extra workload and print its result (for profiling)")
    return ap.parse_args()


# ---------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                source="fallback")


def kernel_sources_sha(names):
    h = hashlib.sha256()
    for n in names:
        h.update(open(os.path.join(ROOT, "sparse_attention_block_paged_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(profile_name, sources):
    """dram bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", txt)
    s = re.search(r"source_sha256:\s*([0-9a-f]+)", txt)
    if not m or not s or s.group(1) != kernel_sources_sha(sources):
        return None
    return int(m.group(1))


class ClockSampler:
    """nvidia-smi sampling of clocks and throttle reasons while the GPU works."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.f = None

    def start(self):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.f.flush()
        rows = [l.strip().split(", ") for l in open(self.f.name) if l.strip()]
        os.unlink(self.f.name)
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows if len(r) >= 9 for k in range(4)
                          if r[5 + k].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(sm)}


def device_inputs(wl, torch, dev):
    q = torch.from_numpy(wl.q.view(np.int16)).view(torch.bfloat16).to(dev)
    d = dict(q=q, table=torch.from_numpy(wl.block_table).to(dev),
             lens=torch.from_numpy(wl.seq_lens).to(dev))
    if wl.kv_format == "bf16":
        d["cache"] = torch.from_numpy(wl.cache.view(np.int16)).view(torch.bfloat16).to(dev)
    else:
        d["codes"] = torch.from_numpy(wl.codes).to(dev)
        d["scales"] = torch.from_numpy(wl.scales).to(dev)
    return d


def decode_bytes(wl):
    """Algorithmic bytes of one fused decode: the visible keys of every request
    (tokens 0..seq_len-1), the queries, the block-table entries and lengths
    read, and the ids written."""
    per_tok = 256 if wl.kv_format == "bf16" else 72
    nb = (wl.seq_lens.astype(np.int64) + BLOCK - 1) // BLOCK
    return int(wl.seq_lens.astype(np.int64).sum() * per_tok + wl.q.nbytes + nb.sum() * 4
               + wl.seq_lens.nbytes + wl.heads * wl.rows * wl.topk * 4)


def prefill_flops(wl):
    """2 * 128 * (visible keys of every query row), token-level causal."""
    pos = []
    for i, s in enumerate(wl.seq_lens.astype(np.int64)):
        ql = (int(wl.cu_seqlens[i + 1] - wl.cu_seqlens[i]) if wl.cu_seqlens is not None
              else wl.query_len)
        start = s - ql
        pos.append((s * (s + 1) - start * (start + 1)) // 2)   # sum of (p+1) over rows
    return 2.0 * 128 * float(sum(pos)) * wl.heads


def graph_of(torch, fn, stream):
    """fn() (which launches on `stream`) run once, then captured once in a
    CUDA graph; returns the graph's replay."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g.replay


def timed_steps(torch, fn, steps, warmup, flush, stream, min_warm_s=0.0):
    """Per-step CUDA-event times (ms) of fn() on `stream`, L2 flushed (untimed)
    before each step."""
    for _ in range(warmup):
        fn()
    if min_warm_s > 0:
        t0 = time.time()
        while time.time() - t0 < min_warm_s:
            flush()
            fn()
        torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


# ---------------------------------------------------------------- our arm

def bench_decode(mm, torch, wl, steps, warmup, flush, stream, pk, min_warm_s=0.0):
    dev = torch.device("cuda", torch.cuda.current_device())
    d = device_inputs(wl, torch, dev)
    out = torch.empty((wl.heads, wl.rows, wl.topk), dtype=torch.int32, device=dev)
    ws = mm.new_workspace(mm.OP_DECODE, wl.heads, wl.num_reqs, wl.query_len, wl.max_seq_len,
                          wl.topk, dev)
    kw = dict(query_len=wl.query_len, max_seq_len=wl.max_seq_len, topk=wl.topk,
              init_blocks=wl.init_blocks, local_blocks=wl.local_blocks, sm_scale=wl.sm_scale,
              out=out, workspace=ws, stream=stream)
    if wl.kv_format == "bf16":
        fn = lambda: mm.decode(d["q"], d["cache"], d["table"], d["lens"], **kw)  # noqa: E731
        sources = DECODE_SOURCES
    else:
        fn = lambda: mm.decode_nvfp4(d["q"], d["codes"], d["scales"], d["table"], d["lens"], **kw)  # noqa: E731
        sources = NVFP4_DECODE_SOURCES
    # Each timed step replays a CUDA graph of the call: eagerly, the
    # binding's host time can outlast the untimed flush and leave the GPU
    # idle inside the timed region.  The eager time is reported beside it.
    with torch.cuda.stream(stream):
        ms_eager = timed_steps(torch, fn, steps, warmup, flush, stream, min_warm_s)
        ms = timed_steps(torch, graph_of(torch, fn, stream), steps, warmup, flush, stream)
    assert mm.get_device_error(stream) == 0, "device status word set"
    t = statistics.mean(ms) * 1e-3
    nbytes = decode_bytes(wl)
    res = dict(value=wl.rows / t, unit="rows/s", ms_per_step=t * 1e3,
               ms_median=statistics.median(ms), steps=steps,
               timing="CUDA-graph replay of the call", eager_ms_per_step=statistics.mean(ms_eager),
               roofline=dict(bound="hbm", achieved=nbytes / t / 1e9, peak=pk["hbm_gbs"],
                             unit="GB/s", frac=nbytes / t / 1e9 / pk["hbm_gbs"],
                             traffic=None, algorithmic_bytes=nbytes,
                             peak_source=pk["source"] + " burst copy"))
    return res, d, out, ws, kw, sources


def _packed_inputs(torch, wl, dev, n_slots):
    """The step's queries, block table and lengths packed in one pinned host
    buffer, and n_slots device buffers with views of the three."""
    parts = [wl.q.view(np.uint8).reshape(-1), wl.block_table.view(np.uint8).reshape(-1),
             wl.seq_lens.view(np.uint8).reshape(-1)]
    offs, n = [], 0
    for p in parts:
        offs.append(n)
        n += (p.nbytes + 255) // 256 * 256
    host = torch.empty(n, dtype=torch.uint8).pin_memory()
    for p, o in zip(parts, offs):
        host[o:o + p.nbytes] = torch.from_numpy(p)
    slots = []
    for _ in range(n_slots):
        buf = torch.empty(n, dtype=torch.uint8, device=dev)
        q = buf[offs[0]:offs[0] + parts[0].nbytes].view(torch.bfloat16).view(wl.q.shape)
        table = buf[offs[1]:offs[1] + parts[1].nbytes].view(torch.int32).view(wl.block_table.shape)
        lens = buf[offs[2]:offs[2] + parts[2].nbytes].view(torch.int32).view(wl.seq_lens.shape)
        slots.append((buf, q, table, lens))
    return host, slots, int(sum(p.nbytes for p in parts))


def bench_e2e_graph(mm, torch, wl, d, kw, steps, warmup, stream, k_steps=4):
    """End to end as a pipelined serving loop runs it: every step copies its
    packed inputs host -> device (pinned), runs the decode through the public
    API and copies its ids device -> host.  k_steps consecutive steps (own
    input and output buffers each) are captured once as one CUDA graph: the
    decodes in order on the main stream, each step's copies on a second
    stream, so that a step's H2D copy and D2H read overlap its neighbours'
    decodes.  `serial` is one step per graph, copies and decode in order on
    one stream.  No L2 flush: the key cache the decode streams (about 283 MB)
    is larger than the L2.  Time = the whole run, host clock, device
    synchronised on both sides."""
    dev = d["q"].device
    host, slots, h2d = _packed_inputs(torch, wl, dev, k_steps)
    outs = [torch.empty((wl.heads, wl.rows, wl.topk), dtype=torch.int32, device=dev)
            for _ in range(k_steps)]
    o_hs = [torch.empty(o.shape, dtype=torch.int32).pin_memory() for o in outs]
    ws = mm.new_workspace(mm.OP_DECODE, wl.heads, wl.num_reqs, wl.query_len, wl.max_seq_len,
                          wl.topk, dev)
    kw = {k: v for k, v in kw.items() if k not in ("out", "workspace", "stream")}
    copy = torch.cuda.Stream(device=dev)

    def run(g, n_rep):
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n_rep):
            g.replay()
        torch.cuda.synchronize()
        return time.perf_counter() - t0

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        _, q0, t0_, l0 = slots[0]
        mm.decode(q0, d["cache"], t0_, l0, out=outs[0], workspace=ws, stream=stream, **kw)  # warm
        torch.cuda.synchronize()
        # serial: one step per graph
        g1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1, stream=stream):
            slots[0][0].copy_(host, non_blocking=True)
            mm.decode(q0, d["cache"], t0_, l0, out=outs[0], workspace=ws,
                      stream=torch.cuda.current_stream(), **kw)
            o_hs[0].copy_(outs[0], non_blocking=True)
        el1 = run(g1, steps)
        # pipelined: k_steps per graph
        gk = torch.cuda.CUDAGraph()
        n_rep = max(1, steps // k_steps)
        with torch.cuda.graph(gk, stream=stream):
            main = torch.cuda.current_stream()
            copy.wait_stream(main)   # fork the copy stream into the capture
            ins = []
            for i in range(k_steps):
                with torch.cuda.stream(copy):
                    slots[i][0].copy_(host, non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(copy)
                ins.append(ev)
            for i in range(k_steps):
                main.wait_event(ins[i])
                _, q, tb, ln = slots[i]
                mm.decode(q, d["cache"], tb, ln, out=outs[i], workspace=ws, stream=main, **kw)
                done = torch.cuda.Event()
                done.record(main)
                copy.wait_event(done)
                with torch.cuda.stream(copy):
                    o_hs[i].copy_(outs[i], non_blocking=True)
            main.wait_stream(copy)
        elk = run(gk, n_rep)
    want = outs[0].cpu().numpy()
    for o_h in o_hs:
        assert np.array_equal(o_h.numpy(), want)
    assert mm.get_device_error(stream) == 0, "device status word set"
    total = n_rep * k_steps
    return dict(value=wl.rows * total / elk, unit="rows/s",
                h2d_bytes_per_step=h2d, d2h_bytes_per_step=int(o_hs[0].nbytes),
                steps=total, ms_per_step=elk / total * 1e3,
                timing="host clock around the whole run, device synchronised on both sides",
                copies=f"per step one H2D of the packed inputs and one D2H of the ids; "
                       f"{k_steps} steps per CUDA graph, each step's copies on a second stream "
                       f"overlapping its neighbours' decodes",
                serial=dict(value=wl.rows * steps / el1, unit="rows/s", steps=steps,
                            ms_per_step=el1 / steps * 1e3,
                            copies="one step per CUDA graph: H2D, decode, D2H in order on one stream"))


def bench_e2e(mm, torch, wl, d, out, ws, kw, steps, warmup, flush, stream):
    """Same decode through the public API with host buffers: one H2D copy of
    the step's queries, block table and lengths (packed in one pinned
    buffer), the call on device views of them, and a D2H copy of the ids."""
    parts = [wl.q.view(np.uint8).reshape(-1), wl.block_table.view(np.uint8).reshape(-1),
             wl.seq_lens.view(np.uint8).reshape(-1)]
    offs, n = [], 0
    for p in parts:
        offs.append(n)
        n += (p.nbytes + 255) // 256 * 256
    host = torch.empty(n, dtype=torch.uint8).pin_memory()
    for p, o in zip(parts, offs):
        host[o:o + p.nbytes] = torch.from_numpy(p)
    dev = torch.empty(n, dtype=torch.uint8, device=d["q"].device)
    q = dev[offs[0]:offs[0] + parts[0].nbytes].view(torch.bfloat16).view(d["q"].shape)
    table = dev[offs[1]:offs[1] + parts[1].nbytes].view(torch.int32).view(d["table"].shape)
    lens = dev[offs[2]:offs[2] + parts[2].nbytes].view(torch.int32).view(d["lens"].shape)
    o_h = torch.empty(out.shape, dtype=torch.int32).pin_memory()

    def fn():
        dev.copy_(host, non_blocking=True)
        mm.decode(q, d["cache"], table, lens, **kw)
        o_h.copy_(out, non_blocking=True)

    with torch.cuda.stream(stream):
        ms = timed_steps(torch, fn, steps, warmup, flush, stream)
    torch.cuda.synchronize()
    assert np.array_equal(o_h.numpy(), out.cpu().numpy())
    t = statistics.mean(ms) * 1e-3
    return dict(value=wl.rows / t, unit="rows/s",
                h2d_bytes_per_step=int(sum(p.nbytes for p in parts)),
                d2h_bytes_per_step=int(o_h.nbytes),
                copies="one H2D of the packed inputs, one D2H of the ids")


def bench_sparse_table(mm, torch, wl, steps, flush, stream):
    """The headline decode with the sparse page table (2 pages per block,
    stride 4) against the plain decode, both timed the same way."""
    dev = torch.device("cuda", torch.cuda.current_device())
    d = device_inputs(wl, torch, dev)
    attn = torch.from_numpy(_attention_table(wl)).to(dev)
    st = torch.empty((wl.rows, wl.topk * 2), dtype=torch.int32, device=dev)
    ctx = torch.empty((wl.rows,), dtype=torch.int32, device=dev)
    out = torch.empty((wl.heads, wl.rows, wl.topk), dtype=torch.int32, device=dev)
    ws = mm.new_workspace(mm.OP_DECODE, wl.heads, wl.num_reqs, wl.query_len, wl.max_seq_len,
                          wl.topk, dev)
    kw = dict(query_len=wl.query_len, max_seq_len=wl.max_seq_len, topk=wl.topk,
              init_blocks=wl.init_blocks, local_blocks=wl.local_blocks, sm_scale=wl.sm_scale,
              out=out, workspace=ws, stream=stream)
    fn = lambda: mm.decode_sparse_table(d["q"], d["cache"], d["table"], d["lens"], **kw,  # noqa: E731
                                        attention_block_table=attn, sparse_block_table_out=st,
                                        sparse_context_lens_out=ctx, block_page_stride=4,
                                        pages_per_block=2)
    with torch.cuda.stream(stream):
        ms = timed_steps(torch, fn, steps, 3, flush, stream)
    assert mm.get_device_error(stream) == 0, "device status word set"
    t = statistics.mean(ms) * 1e-3
    return dict(value=wl.rows / t, unit="rows/s", ms_per_step=t * 1e3, steps=steps,
                pages_per_block=2, block_page_stride=4, workload=wl.name + " + sparse page table")


def _attention_table(wl):
    import workloads as W
    return W.attention_block_table(wl, 1)


def bench_prefill(mm, torch, wl, steps, warmup, flush, stream, pk, time_scorer=True):
    dev = torch.device("cuda", torch.cuda.current_device())
    d = device_inputs(wl, torch, dev)
    out = torch.empty((wl.heads, wl.rows, wl.topk), dtype=torch.int32, device=dev)
    nvfp4 = wl.kv_format == "nvfp4"
    ragged = wl.cu_seqlens is not None
    n = mm.workspace_bytes(mm.OP_PREFILL_NVFP4 if nvfp4 else mm.OP_PREFILL, wl.heads, wl.num_reqs,
                           wl.query_len, wl.max_seq_len, wl.topk)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    kw = dict(max_seq_len=wl.max_seq_len, topk=wl.topk,
              init_blocks=wl.init_blocks, local_blocks=wl.local_blocks, sm_scale=wl.sm_scale,
              out=out, workspace=ws, stream=stream)
    cache = d["codes"] if nvfp4 else d["cache"]
    if ragged:
        cu = torch.from_numpy(wl.cu_seqlens).to(dev)
        fn = lambda: mm.prefill_ragged(d["q"], cache, d["table"], d["lens"], cu,  # noqa: E731
                                       max_query_len=wl.query_len, index_scales=d.get("scales"),
                                       **kw)
    elif nvfp4:
        fn = lambda: mm.prefill_nvfp4(d["q"], cache, d["scales"], d["table"], d["lens"],  # noqa: E731
                                      query_len=wl.query_len, **kw)
    else:
        fn = lambda: mm.prefill(d["q"], cache, d["table"], d["lens"], query_len=wl.query_len, **kw)  # noqa: E731
    # Each step is a CUDA-graph replay of the same call (the calls are
    # capturable): eagerly, the binding's marshalling and the launches (tens
    # of microseconds of host time) can outlast the untimed L2 flush before
    # the step and leave the GPU idle inside the timed region.  The eager
    # step time is reported beside it.
    with torch.cuda.stream(stream):
        ms_eager = timed_steps(torch, fn, steps, warmup, flush, stream)
        ms_all = timed_steps(torch, graph_of(torch, fn, stream), steps, warmup, flush, stream)
    # The scorer keeps each row's candidates and a small merge kernel writes
    # the ids (after the dequant pass for NVFP4); `value` is the whole step's
    # rate.  The roofline is the scorer kernel's: the same kernel in score
    # mode, timed alone through the score call (bf16, uniform rows), which
    # also writes -inf past each row's block.  time_scorer=False: the whole
    # step is the roofline's kernel time.
    assert mm.get_device_error(stream) == 0, "device status word set"
    t_all = statistics.mean(ms_all) * 1e-3
    fl = prefill_flops(wl)
    res = dict(value=fl / t_all / 1e12, unit="TFLOP/s (scores + top-k)",
               rows_per_s=wl.rows / t_all, ms_per_step=t_all * 1e3,
               timing="CUDA-graph replay of the call",
               eager_ms_per_step=statistics.mean(ms_eager))
    t_sc = None
    if time_scorer and not nvfp4 and not ragged:
        width = -(-wl.max_seq_len // BLOCK)
        sc_out = torch.empty((wl.heads, wl.rows, width), dtype=torch.float32, device=dev)
        scf = lambda: mm.score(d["q"], cache, d["table"], d["lens"], query_len=wl.query_len,  # noqa: E731
                               max_seq_len=wl.max_seq_len, sm_scale=wl.sm_scale, out=sc_out,
                               stream=stream)
        with torch.cuda.stream(stream):
            ms_sc = timed_steps(torch, graph_of(torch, scf, stream), steps, warmup, flush, stream)
            # the standalone selector (mm3idx_topk) on the same scores
            self_sel = lambda: mm.topk(sc_out, d["lens"], query_len=wl.query_len,  # noqa: E731
                                       max_seq_len=wl.max_seq_len, topk=wl.topk,
                                       init_blocks=wl.init_blocks,
                                       local_blocks=wl.local_blocks, out=out, stream=stream)
            ms_sel = timed_steps(torch, self_sel, steps, warmup, flush, stream)
        t_sc = statistics.mean(ms_sc) * 1e-3
        res["scorer_ms"] = t_sc * 1e3
        res["selector_alone_ms"] = statistics.mean(ms_sel)
        del sc_out
    t_roof = t_sc if t_sc is not None else t_all
    res["roofline"] = dict(bound="tensor", achieved=fl / t_roof / 1e12,
                           peak=pk["bf16_tflops"], unit="TFLOP/s",
                           frac=fl / t_roof / 1e12 / pk["bf16_tflops"],
                           traffic=profiled_traffic("prefill_scorer_causal_prefill.md",
                                                    PREFILL_SOURCES) if t_sc else None,
                           algorithmic_flops=fl,
                           kernel="score-mode prefill kernel alone" if t_sc
                           else "whole step (scores + top-k)",
                           peak_source=pk["source"] + " cuBLAS bf16 burst")
    return res


def bench_forward(mm, torch, wl, steps, warmup, flush, stream, pk):
    """A mixed batch through mm3idx_forward (decode rows first, then two
    chunked prefills, one call) against the same work as two calls (the
    decode, then the ragged prefill) on the same stream."""
    dev = torch.device("cuda", torch.cuda.current_device())
    d = device_inputs(wl, torch, dev)
    nd = int(np.sum(np.diff(wl.cu_seqlens) == 4))           # the leading 4-row requests
    dec_rows = nd * 4
    cu = wl.cu_seqlens
    pcu = torch.from_numpy((cu[nd:] - cu[nd]).astype(np.int32)).to(dev)
    pmax = int(np.diff(cu[nd:]).max())
    out = torch.empty((wl.heads, wl.rows, wl.topk), dtype=torch.int32, device=dev)
    n = mm.forward_workspace_bytes(wl.heads, nd, 4, wl.num_reqs - nd, pmax, wl.max_seq_len, wl.topk)
    ws = torch.zeros(n, dtype=torch.uint8, device=dev)
    kw = dict(max_seq_len=wl.max_seq_len, topk=wl.topk, init_blocks=wl.init_blocks,
              local_blocks=wl.local_blocks, sm_scale=wl.sm_scale)
    fn = lambda: mm.forward(d["q"], d["cache"], d["table"], d["lens"], pcu, num_decodes=nd,  # noqa: E731
                            decode_query_len=4, prefill_max_query_len=pmax, out=out,
                            workspace=ws, stream=stream, **kw)
    # the same work as two calls
    dws = mm.new_workspace(mm.OP_DECODE, wl.heads, nd, 4, wl.max_seq_len, wl.topk, dev)
    pws = mm.new_workspace(mm.OP_PREFILL, wl.heads, wl.num_reqs - nd, pmax, wl.max_seq_len,
                           wl.topk, dev)
    qd, qp = d["q"][:dec_rows], d["q"][dec_rows:]

    def two():
        mm.decode(qd, d["cache"], d["table"][:nd], d["lens"][:nd], query_len=4, out=out[:, :dec_rows],
                  workspace=dws, stream=stream, **kw)
        mm.prefill_ragged(qp, d["cache"], d["table"][nd:], d["lens"][nd:], pcu,
                          max_query_len=pmax, out=out[:, dec_rows:], workspace=pws, stream=stream,
                          **kw)

    # Both as CUDA-graph replays, as the other workloads are timed.
    with torch.cuda.stream(stream):
        ms = timed_steps(torch, graph_of(torch, fn, stream), steps, warmup, flush, stream)
        ms2 = timed_steps(torch, graph_of(torch, two, stream), steps, warmup, flush, stream)
    assert mm.get_device_error(stream) == 0, "device status word set"
    t = statistics.mean(ms) * 1e-3
    return dict(value=wl.rows / t, unit="rows/s", ms_per_step=t * 1e3,
                timing="CUDA-graph replay of the call",
                two_calls_ms=statistics.mean(ms2), decode_requests=nd,
                prefill_rows=int(wl.rows - dec_rows), steps=steps)


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(wl, seconds):
    """The oracle as it stands, single-threaded, on whole batches of the
    workload until `seconds` of CPU time are spent (at least one request)."""
    import oracle
    rows = 0
    t0 = time.perf_counter()
    i = 0
    while True:
        sub = oracle.subset(wl, [i % wl.num_reqs])
        oracle.problem(sub, want_scores=False)
        rows += sub.rows
        i += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return dict(value=rows / el, unit="rows/s", cores=1, kind="oracle", cpu=cpu_model(),
                host_cores=os.cpu_count(),
                sample=f"{i} requests ({rows} rows) of the {wl.name} workload, "
                       f"request by request, {el:.1f} s on one host core")


def cpu_baseline_all_cores(wl, seconds):
    """The same oracle call, one request per task, on a thread per host core
    (the C oracle runs with the interpreter lock released).  The ids of the
    first requests are checked against a single-threaded run of the same
    requests."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    cores = os.cpu_count() or 1
    check = min(wl.num_reqs, 2 * cores)
    want = {i: oracle.problem(oracle.subset(wl, [i]), want_scores=False)[1]
            for i in range(check)}

    def one(i):
        return i, oracle.problem(oracle.subset(wl, [i % wl.num_reqs]), want_scores=False)[1]

    rows, done, same = 0, 0, True
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=cores) as ex:
        while True:
            for i, ids in ex.map(one, range(done, done + 4 * cores)):
                rows += ids.shape[1]
                if i in want:
                    same = same and bool(np.array_equal(ids, want[i]))
            done += 4 * cores
            el = time.perf_counter() - t0
            if el >= seconds:
                break
    return dict(value=rows / el, unit="rows/s", cores=cores, kind="oracle", cpu=cpu_model(),
                identical_to_single_core=same,
                sample=f"{done} requests ({rows} rows) of the {wl.name} workload, "
                       f"one request per task on {cores} threads, {el:.1f} s")


def max_over_ranks(t_ms, device):
    """The slowest rank's time (ms); the local time when running alone."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return t_ms
    tt = torch.tensor([t_ms], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_value(rows_per_rank, world, t_ms):
    """Whole-job throughput: every rank's rows over the slowest rank's time."""
    return world * rows_per_rank / (t_ms * 1e-3)


def run_ours(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    import sparse_attention_block_paged_gb300 as mm
    import workloads as W

    pk = peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream()
    flush_buf = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)

    def flush():
        torch.amax(flush_buf, dim=0, out=flush_out)

    if args.only:
        w = W.make(args.only)
        if args.only in ("prefill", "prefill_topk32", "nvfp4_prefill", "chunked_prefill"):
            r = bench_prefill(mm, torch, w, args.steps, max(args.warmup, 3), flush, stream, pk)
        elif args.only == "mixed_batch":
            r = bench_forward(mm, torch, w, args.steps, max(args.warmup, 3), flush, stream, pk)
        else:
            r = bench_decode(mm, torch, w, args.steps, max(args.warmup, 3), flush, stream, pk)[0]
        r["workload"] = w.name
        print(json.dumps(r), flush=True)
        return

    wl = W.make(HEADLINE)
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    res, d, out, ws, kw, sources = bench_decode(mm, torch, wl, args.steps, max(args.warmup, 3),
                                                flush, stream, pk, min_warm_s=1.5)
    res["roofline"]["traffic"] = profiled_traffic("decode_spec_decode.md", sources)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t = max_over_ranks(res["ms_per_step"], dev)
    t_eager = max_over_ranks(res["eager_ms_per_step"], dev)
    e2e_serial = bench_e2e(mm, torch, wl, d, out, ws, kw, args.steps, max(args.warmup, 3), flush,
                           stream)
    e2e = bench_e2e_graph(mm, torch, wl, d, kw, args.steps, max(args.warmup, 3), stream)
    e2e["eager"] = e2e_serial
    extra = {}
    if not args.no_extra and rank == 0:
        for key in ("high_batch", "nvfp4_decode"):
            w2 = W.make(key)
            r2, _, _, _, _, src2 = bench_decode(mm, torch, w2, max(20, args.steps // 4), 3, flush,
                                                stream, pk)
            r2["roofline"]["traffic"] = profiled_traffic(f"decode_{key}.md", src2)
            r2["workload"] = w2.name
            extra[key] = r2
            del w2
        w4 = W.make("prefill")
        r4 = bench_prefill(mm, torch, w4, max(10, args.steps // 10), 3, flush, stream, pk)
        r4["workload"] = w4.name
        extra["prefill"] = r4
        del w4
        w8 = W.make("prefill_topk32")
        r8 = bench_prefill(mm, torch, w8, max(10, args.steps // 10), 3, flush, stream, pk,
                           time_scorer=False)
        r8["workload"] = w8.name
        extra["prefill_topk32"] = r8
        del w8
        w5 = W.make("nvfp4_prefill")
        r5 = bench_prefill(mm, torch, w5, max(10, args.steps // 10), 3, flush, stream, pk)
        r5["workload"] = w5.name
        r5["unit"] = "TFLOP/s (dequant + scores + top-k)"
        r5["roofline"]["traffic"] = None      # two kernels; the summaries cover the bf16 scorer
        extra["nvfp4_prefill"] = r5
        del w5
        w6 = W.make("chunked_prefill")
        r6 = bench_prefill(mm, torch, w6, max(10, args.steps // 10), 3, flush, stream, pk)
        r6["workload"] = w6.name
        r6["roofline"]["traffic"] = None      # not the workload the scorer summary was taken on
        extra["chunked_prefill"] = r6
        del w6
        extra["sparse_table"] = bench_sparse_table(mm, torch, wl, max(20, args.steps // 4), flush,
                                                   stream)
        w7 = W.make("mixed_batch")
        r7 = bench_forward(mm, torch, w7, max(20, args.steps // 4), 3, flush, stream, pk)
        r7["workload"] = w7.name
        extra["mixed_batch"] = r7
        del w7
    clk = clocks.stop()
    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    line = {
        "metric": METRIC,
        "value": job_value(wl.rows, world, t),
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": t,
        "timing": res["timing"],
        "eager_ms_per_step": t_eager,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded numpy draws, bf16 q/k ~ N(0,1))",
        "config": {"workload": HEADLINE_WORKLOAD,
                   "rows_per_step": wl.rows, "key_bytes_per_step": wl.key_bytes(),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed before each timed step (read of a 2x-L2 buffer), flush not timed"},
        "roofline": res["roofline"],
        "cpu_baseline": cpu_baseline(wl, args.cpu_seconds),
        "cpu_baseline_all_cores": cpu_baseline_all_cores(wl, args.cpu_seconds / 2),
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clk,
        "extra": extra,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle as it stands on the headline workload: each step is a
    bounded sample (4 requests = 16 rows) of the spec-decode batch."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    import workloads as W
    wl = W.make(HEADLINE)
    per_step = 4

    def step(k):
        reqs = [(k * per_step + j) % wl.num_reqs for j in range(per_step)]
        oracle.problem(oracle.subset(wl, reqs), want_scores=False)

    for k in range(max(args.warmup, 3)):
        step(k)
    t0 = time.perf_counter()
    for k in range(args.steps):
        step(k)
    el = time.perf_counter() - t0
    rows = args.steps * per_step * wl.query_len
    value = rows / el
    line = {
        "metric": METRIC, "impl": "reference", "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded numpy draws)",
        "config": {"workload": HEADLINE_WORKLOAD,
                   "sample_per_step": f"{per_step} requests ({per_step * wl.query_len} rows)"},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"{per_step} requests per step, {args.steps} steps"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
