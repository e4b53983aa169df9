#!/usr/bin/env python3
"""Benchmark of the indexer decode step: FP8 paged MQA logits, then per-row top-k.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload wide|decode|tiny|mtp|kv2g|wide_b<B>|sweep:P,next_n,H,B,ctx]
                    [--sweep subset|all]

One step = one logits launch plus one top-k launch over one batch of synthetic
inputs (by default the wide workload, the largest configuration on one GPU:
B=256, next_n=4 -> 1024 rows, H=64, D=128, P=16, ctx U[4096, 16384],
W = stride = 2^20, k=2048).  Metric: row-tokens per second, sum_r ctx_r /
time, in Gtok/s, whole job over all ranks.

Timing: inputs are resident in HBM; several input sets rotate so that the
bytes one cycle touches exceed the 129 MB L2; each measurement times exactly
K steps, run as replays of a CUDA graph of S steps, bracketed by a barrier
and a device synchronise on both sides, with CUDA events; the measurement is
repeated until about half a second has been timed, and the median
measurement (the slowest rank's) counts.  A second graph of the same steps
with timing events around every kernel is replayed after the timed region
and gives the per-launch durations.

`--sweep` runs the throughput sweep instead (one JSON line per point).

Multi-GPU: one process per GPU (torchrun), each running its own batch of
requests; no data-path collective (requests are independent), so scaling is
weak.  `--impl reference` times the CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "indexer Gtokens/s (rows x context tokens) and % of FP8/HBM roofline, 1 GB300"
UNIT = "Gtok/s"
L2_BYTES = 129 * 2**20
MEASURE_SECONDS = 0.5          # timed per bench line, over repeated K-step measurements


# ------------------------------------------------------------------ helpers
def row_tokens(w) -> int:
    """sum_r ctx_r: tokens each query row scores (row j of a request sees
    ctx - next_n + j + 1 of them, clamped to [0, W])."""
    ctx = w.context_lens.astype(np.int64)[:, None]
    j = np.arange(w.next_n)[None, :]
    cap = min(w.max_model_len, w.block_table.shape[1] * w.page_size)
    return int(np.clip(ctx - w.next_n + j + 1, 0, cap).sum())


def logits_bytes(w) -> int:
    """Algorithmic HBM bytes of one logits launch: K values and scales once per
    request, the block-table entries read, q and weights, context lengths, and
    the full-width fp32 output."""
    cap = min(w.max_model_len, w.block_table.shape[1] * w.page_size)
    ctx = np.clip(w.context_lens.astype(np.int64), 0, cap)
    kv = int(ctx.sum()) * (w.head_dim + 4)
    table = int(np.ceil(ctx / w.page_size).sum()) * 4
    qw = w.batch * w.next_n * w.heads * (w.head_dim + 4)
    out = w.rows * w.max_model_len * 4
    return kv + table + qw + out + 4 * w.batch


def logits_flops(w) -> int:
    return row_tokens(w) * 2 * w.heads * w.head_dim


def epilogue_fp32_ops(w) -> int:
    """FP32 lane operations of the logits epilogue: per row, valid token and
    head one max (the ReLU) and one fused multiply-add (the weighted sum)."""
    return row_tokens(w) * w.heads * 2


FP32_LANES_PER_SM = 128          # FP32 lanes of a Blackwell SM (4 partitions x 32)


def topk_bytes(w) -> int:
    return row_tokens(w) * 4 + w.rows * w.topk * 4


TILE_TOKENS, FILL_COLS = 128, 4096     # the logits kernel's MMA tile and -inf fill unit


def fill_heavy(w) -> bool:
    """The logits kernel's rule for a launch whose -inf fill outweighs its
    tiles four times over (fill units of 4096 columns against 128-token
    tiles); the fused launch then shares the fill over the whole grid."""
    ce = np.clip(np.asarray(w.context_lens, dtype=np.int64), 0, w.max_model_len)
    tiles = (ce + TILE_TOKENS - 1) // TILE_TOKENS
    fs = np.minimum(w.max_model_len, tiles * TILE_TOKENS)
    units = w.next_n * ((w.max_model_len - fs + FILL_COLS - 1) // FILL_COLS)
    return int(units.sum()) > 4 * int(tiles.sum())


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def make_workload(name: str, layout: str = "split"):
    import synth

    if name.startswith("sweep:"):
        p, n, h, b, c = (int(x) for x in name.split(":", 1)[1].split(","))
        return synth.sweep_point(p, n, h, b, c, layout=layout)
    if name.startswith("wide_b"):
        return synth.wide(layout, batch=int(name[len("wide_b"):]))
    return synth.NAMED[name](layout)


def describe(w) -> str:
    return (f"{w.name}: B={w.batch}, next_n={w.next_n}, H={w.heads}, D={w.head_dim}, P={w.page_size}, "
            f"W={w.max_model_len}, stride={w.logits_stride}, k={w.topk}, seed={w.seed}")


# The logits kernel's source: its file and the headers it includes (the
# fused launch's row selection lives in select.cuh).
LOGITS_SOURCES = ("logits.cu", "select.cuh", "ptx.cuh", "common.cuh")


def source_sha(paths) -> str:
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def logits_source_sha() -> str:
    csrc = os.path.join(ROOT, "sparse_attention_indexer_03_gb300", "csrc")
    return source_sha([os.path.join(csrc, f) for f in LOGITS_SOURCES])


def profiled_traffic(workload: str, fused: bool = False):
    """DRAM bytes per logits launch from the committed ncu summary, if it was
    taken on the current kernel source (logits_source_sha); else None."""
    path = os.path.join(ROOT, "profiles", f"logits_tc{'_topk' if fused else ''}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    s = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != logits_source_sha():
        return None
    return int(m.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self) -> dict:
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = [r.split(", ") for r in self.out.strip().splitlines() if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        under_load = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": float(np.median(under_load)) if under_load else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows)}


def aggregate(ms: float, tokens: int, world: int, device=None):
    """Whole-job figures over the ranks: the slowest rank's time and the sum of
    the row-tokens every rank processed per step.  Ranks hold independent
    requests, so this is the only cross-rank exchange, and it lies outside the
    timed region."""
    if world <= 1:
        return ms, tokens
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    n = torch.tensor([tokens], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())


def rank_workload(name: str, rank: int, layout: str = "split"):
    """The batch of requests rank `rank` serves: the named workload (the same
    shapes on every rank, weak scaling)."""
    return make_workload(name, layout)


# ------------------------------------------------------------------ CPU oracle
def oracle_step_sample(w, budget_s: float):
    """Time the CPU oracle (logits, then top-k) over the workload's requests in
    order until `budget_s` seconds have passed; returns (row_tokens, seconds, requests)."""
    import oracle

    ctx_rows = oracle.row_context_lengths(w.context_lens, w.next_n, w.max_model_len,
                                          w.max_model_len, 1)
    done_tok, reqs, t0 = 0, 0, time.perf_counter()
    b = 0
    while time.perf_counter() - t0 < budget_s:
        rows = list(range(b * w.next_n, (b + 1) * w.next_n))
        lg = oracle.paged_mqa_logits(w.q, w.pool.ids, w.pool.data, w.pool.num_pages, w.page_size,
                                     w.weights, w.context_lens, w.block_table, w.next_n,
                                     w.max_model_len, layout=w.layout, rows=rows)
        oracle.top_k_per_row(lg.astype(np.float32), ctx_rows[rows], w.topk)
        done_tok += int(ctx_rows[rows].sum())
        reqs += 1
        b = (b + 1) % w.batch
    return done_tok, time.perf_counter() - t0, reqs


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return 0
    w = make_workload(args.workload)
    # Each step is a bounded sample: about 150 s of oracle work for the whole run.
    budget = min(2.0, 150.0 / (args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_step_sample(w, min(budget, 0.5))
    tok, sec = 0, 0.0
    reqs_total = 0
    for _ in range(args.steps):
        t, s, r = oracle_step_sample(w, budget)
        tok += t
        sec += s
        reqs_total += r
    value = tok / sec / 1e9
    sample = (f"{reqs_total} requests of the {w.name} batch over {args.steps} steps "
              f"(each step about {budget:.1f} s of oracle work: fp64 logits of the request's rows, then top-k)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": describe(w)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def run_ours(args, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist

    import sparse_attention_indexer_03_gb300 as sai

    torch.cuda.set_device(local_rank)
    sai.build()
    dev = torch.device("cuda", local_rank)
    w = rank_workload(args.workload, rank, args.layout)
    tok = row_tokens(w)

    # Rotating input sets: enough that one cycle touches more bytes than L2.
    touched = logits_bytes(w) + topk_bytes(w)
    R = max(2, min(16, math.ceil(2.0 * L2_BYTES / max(touched, 1))))
    sets = []
    for _ in range(R):
        d = w.to_device(dev)
        d["logits"] = torch.empty((w.rows, w.logits_stride), dtype=torch.float32, device=dev)
        d["indices"] = torch.empty((w.rows, w.topk), dtype=torch.int32, device=dev)
        d["ws"] = torch.zeros(max(1, sai.logits_topk_workspace_bytes(w.batch) // 4), dtype=torch.int32, device=dev)
        sets.append(d)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    fused = args.path == "fused" or (args.path == "auto" and fill_heavy(w))

    def logits_call(d):
        sai.paged_mqa_logits(d["q"], d["kv"], w.page_size, d["weights"], d["context_lens"],
                             d["block_table"], d["logits"], w.max_model_len, num_pages=w.pool.num_pages,
                             status=status, kv_layout=w.layout, stream=stream)

    def topk_call(d):
        sai.top_k_per_row_decode(d["logits"], d["context_lens"], w.next_n, w.max_model_len, w.topk,
                                 d["indices"], stream=stream)

    def fused_call(d):
        sai.paged_mqa_logits_topk(d["q"], d["kv"], w.page_size, d["weights"], d["context_lens"],
                                  d["block_table"], d["logits"], w.max_model_len, w.topk, d["indices"],
                                  d["ws"], num_pages=w.pool.num_pages, status=status, stream=stream)

    def step(d):
        if fused:
            fused_call(d)
        else:
            logits_call(d)
            topk_call(d)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(sets[i % R])
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"status {int(status.item()):#x}"

    # The timed region replays a graph of S steps (logits, then top-k) with no
    # other nodes: event nodes between kernels cost time and break the
    # programmatic overlap of one kernel's start with the previous one's tail.
    K = args.steps
    S = K if K <= 200 else 100
    K = S * math.ceil(K / S)
    reps = K // S
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(S):
            step(sets[i % R])
    # A second graph brackets every kernel with timing events; it is replayed
    # right after the timed region and gives the per-launch kernel durations.
    try:
        ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)] for _ in range(S)]
    except TypeError:              # a torch without graph-recordable timing events
        ev = None
    probe = None
    if ev:
        probe = torch.cuda.CUDAGraph()
        with torch.cuda.graph(probe, stream=stream):
            for i in range(S):
                d = sets[i % R]
                ev[i][0].record(stream)
                fused_call(d) if fused else logits_call(d)
                ev[i][1].record(stream)
                if not fused:
                    topk_call(d)
                ev[i][2].record(stream)
    with torch.cuda.stream(stream):
        graph.replay()                  # untimed: graph upload and warm-up
        if probe is not None:
            probe.replay()
    torch.cuda.synchronize()
    # Rough length of one measurement, to choose how many to take.
    c0 = time.perf_counter()
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    est = max(1e-6, (time.perf_counter() - c0) * reps)
    M = max(3, min(2000, math.ceil(args.measure_seconds / est)))
    if world > 1:                      # every rank takes the same number of measurements
        m_t = torch.tensor([M], dtype=torch.int64, device=dev)
        dist.all_reduce(m_t, op=dist.ReduceOp.MAX)
        M = int(m_t.item())

    # Each measurement times exactly K steps (reps replays of the S-step
    # graph), bracketed by a barrier and a synchronise on both sides.
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    meas = []
    with ClockSampler(local_rank) as clocks:
        for _ in range(M):
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):          # replay() launches on the current stream
                t_start.record(stream)
                for _ in range(reps):
                    graph.replay()
                t_end.record(stream)
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            meas.append(t_start.elapsed_time(t_end))
        with torch.cuda.stream(stream):
            if probe is not None:
                probe.replay()
        torch.cuda.synchronize()
    ms = float(np.median(meas))
    ms_mean = float(np.mean(meas))
    if ev:
        logits_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(S)]
        topk_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(S)]
    else:                          # per-kernel events on an eager pass over the same sets
        logits_ms, topk_ms = [], []
        with torch.cuda.stream(stream):
            for i in range(S):
                a, b2, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
                d = sets[i % R]
                a.record(stream)
                fused_call(d) if fused else logits_call(d)
                b2.record(stream)
                if not fused:
                    topk_call(d)
                c.record(stream)
                torch.cuda.synchronize()
                logits_ms.append(a.elapsed_time(b2))
                topk_ms.append(b2.elapsed_time(c))
    ms, tok_all = aggregate(ms, tok, world, dev)
    assert int(status.item()) == 0, f"status {int(status.item()):#x}"

    # End to end through the Python API: each step copies its inputs (q,
    # weights, context lengths, block table, packed in one pinned host buffer)
    # to the device with one copy, runs the step, and copies the indices back
    # to pinned host memory.  As a serving loop would, two buffer sets
    # alternate so that one step's copies overlap the other's kernels (copy
    # engines in, kernels, copy engines out, on three streams); the copies and
    # the calls are captured in a CUDA graph of E_STEPS steps.  The K-cache
    # pool stays on the device.
    parts = [("q", w.q), ("weights", w.weights), ("context_lens", w.context_lens),
             ("block_table", w.block_table)]
    offs, total = {}, 0
    for name, arr in parts:
        offs[name] = total
        total += (arr.nbytes + 255) // 256 * 256
    host_in, dev_in, de, out_host = [], [], [], []
    for b in range(2):
        hb = torch.empty(total, dtype=torch.uint8).pin_memory()
        for name, arr in parts:
            hb[offs[name]:offs[name] + arr.nbytes].copy_(
                torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1)))
        host_in.append(hb)
        dev_in.append(torch.empty(total, dtype=torch.uint8, device=dev))
        db = dict(sets[b % R])
        for name, arr in parts:
            db[name] = dev_in[b][offs[name]:offs[name] + arr.nbytes].view(db[name].dtype).view(db[name].shape)
        de.append(db)
        out_host.append(torch.empty((w.rows, w.topk), dtype=torch.int32).pin_memory())
    h2d = sum(arr.nbytes for _, arr in parts)
    d2h = out_host[0].numel() * out_host[0].element_size()
    cp_in, cp_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    E_STEPS = 32                     # each replay starts and ends with the copy pipeline drained

    def e2e_steps():
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_comp = [torch.cuda.Event(), torch.cuda.Event()]
        ev_out = [torch.cuda.Event(), torch.cuda.Event()]
        fork = torch.cuda.Event()
        fork.record(stream)
        cp_in.wait_event(fork)
        cp_out.wait_event(fork)
        for i in range(E_STEPS):
            b = i % 2
            if i >= 2:
                cp_in.wait_event(ev_comp[b])            # step i - 2 is done with dev_in[b]
            with torch.cuda.stream(cp_in):
                dev_in[b].copy_(host_in[b], non_blocking=True)
            ev_in[b].record(cp_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])            # step i - 2's indices are copied out
            with torch.cuda.stream(stream):
                step(de[b])
            ev_comp[b].record(stream)
            cp_out.wait_event(ev_comp[b])
            with torch.cuda.stream(cp_out):
                out_host[b].copy_(de[b]["indices"], non_blocking=True)
            ev_out[b].record(cp_out)
        join = torch.cuda.Event()
        join.record(cp_in)
        stream.wait_event(join)
        stream.wait_event(ev_out[0])
        stream.wait_event(ev_out[1])

    e2e_steps()
    torch.cuda.synchronize()
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph, stream=stream):
        e2e_steps()
    with torch.cuda.stream(stream):
        e2e_graph.replay()
    torch.cuda.synchronize()
    c0 = time.perf_counter()
    with torch.cuda.stream(stream):
        e2e_graph.replay()
    torch.cuda.synchronize()
    Me = max(3, min(500, math.ceil(0.5 * args.measure_seconds / max(1e-6, time.perf_counter() - c0))))
    Ke = E_STEPS
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e_meas = []
    for _ in range(Me):
        with torch.cuda.stream(stream):
            e0.record(stream)
            e2e_graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        e_meas.append(e0.elapsed_time(e1))
    e2e_ms = float(np.median(e_meas))
    e2e_ms, _ = aggregate(e2e_ms, tok, world, dev)
    assert int(status.item()) == 0, f"status {int(status.item()):#x}"

    if rank != 0:
        return 0
    peaks = load_peaks()
    lg_ms = float(np.mean(logits_ms))
    tk_ms = float(np.mean(topk_ms))
    # The fused kernel's compulsory HBM bytes add the index rows it writes;
    # the logits it selects from are re-read through L2.
    lbytes = logits_bytes(w) + (w.rows * w.topk * 4 if fused else 0)
    lflops = logits_flops(w)
    fp8_peak_tflops = 2.0 * peaks["bf16_tflops"]          # nominal fp8 : bf16 dense ratio 4.5 : 2.25
    t_hbm = lbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = lflops / (fp8_peak_tflops * 1e12)
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": lbytes / (lg_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": lflops / (lg_ms * 1e-3) / 1e12, "peak": fp8_peak_tflops,
                "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    il = w.layout == "interleaved"
    roof["traffic"] = None if il else profiled_traffic(w.name, fused)
    roof["kernel"] = "logits_tc_kernel" + (" (interleaved K)" if il else "") + (" (fused top-k)" if fused else "")
    roof["algorithmic_per_launch"] = lbytes if roof["bound"] == "hbm" else lflops
    roof["peak_source"] = peaks["source"] + (" (fp8 = 2 x measured bf16)" if roof["bound"] == "tensor" else "")
    # Diagnostic, not a roofline term of the copy/GEMM peaks: the epilogue's
    # FP32 work at one lane operation per FP32 lane and clock, at the SM clock
    # sampled during the timed region.
    clk = clocks.summary()
    sm_mhz = clk.get("sm_mhz") or clk.get("sm_max_mhz") or 2070.0
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    t_fp32_ms = epilogue_fp32_ops(w) / (sms * FP32_LANES_PER_SM * sm_mhz * 1e6) * 1e3
    roof["fp32_epilogue"] = {"ops_per_launch": epilogue_fp32_ops(w), "bound_ms": t_fp32_ms,
                             "frac_of_kernel_time": t_fp32_ms / lg_ms,
                             "lanes": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes at {sm_mhz:.0f} MHz"}
    value = tok_all * K / (ms * 1e-3) / 1e9

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        ctok, csec, creqs = oracle_step_sample(w, float(os.environ.get("SAI_CPU_BASELINE_SECONDS", "12")))
        cpu = {"value": ctok / csec / 1e9, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{creqs} requests of the {w.name} batch in order ({ctok} row-tokens), "
                         f"fp64 logits then top-k, {csec:.1f} s"}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": max(args.warmup, 3), "ms_per_step": ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic",
            "config": {"workload": describe(w), "row_tokens_per_step": tok,
                       "l2": f"{R} rotating input sets, {R * touched / 2**20:.0f} MB touched per cycle > 129 MB L2",
                       "timing": f"median of {M} measurements, each of exactly {K} steps ({K // S} replays of a "
                                 f"CUDA graph of {S} steps, barrier and synchronise on both sides); kernel "
                                 f"durations from a replay of the same steps with timing events around each kernel",
                       "ms_per_step_mean": ms_mean / K,
                       "ms_per_step_min_max": [min(meas) / K, max(meas) / K],
                       "path": ("one fused launch (logits; rows of completed requests queued and selected by "
                                "every CTA while its other warps write the -inf fill"
                                + (", fill units shared by the whole grid through one counter)"
                                   if fill_heavy(w) else ")")
                                if fused else "two launches (logits, top-k)"),
                       "logits_ms": lg_ms, "topk_ms": None if fused else tk_ms,
                       "logits_ms_median": float(np.median(logits_ms)),
                       "topk_ms_median": None if fused else float(np.median(topk_ms)),
                       "topk_gbs": None if fused else topk_bytes(w) / (tk_ms * 1e-3) / 1e9,
                       "topk_exposed_ms": None if fused else max(0.0, ms / K - lg_ms),
                       "topk_note": None if fused else ("the top-k launch is a programmatic dependent of the "
                                                        "logits launch: its duration includes waiting for "
                                                        "the logits; topk_exposed_ms is the step time past "
                                                        "the logits launch's"),
                       "parallelism": f"replicas x{world} (independent requests per GPU)"},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": tok_all * Ke / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "how": "per step: one pinned H2D copy of the packed inputs, the step, one D2H copy "
                           "of the indices; two buffer sets alternate so copies overlap kernels; "
                           f"median of {Me} replays of a graph of {E_STEPS} steps"},
            "gpu_launches": (1 if fused else 2) * K,
            "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ K-cache write
KC_METRIC = "K-cache FP8 quantise + insert GB/s (bf16 K rows -> paged e4m3 cache), 1 GB300"
KC_TOKENS, KC_PAGE, KC_PAGES = 16384, 64, 8192      # a 16384-token batch into the decode pool


def kcache_bytes(T: int) -> int:
    """Algorithmic HBM bytes: bf16 rows and int64 slots read, 132 bytes written per token."""
    return T * (2 * 128 + 8 + 132)


def run_kcache(args, rank: int, world: int, local_rank: int):
    import torch

    import sparse_attention_indexer_03_gb300 as sai
    import synth

    torch.cuda.set_device(local_rank)
    sai.build()
    dev = torch.device("cuda", local_rank)
    T, P, NP = KC_TOKENS, KC_PAGE, KC_PAGES
    per_set = T * (2 * 128 + 8)
    R = max(2, min(64, math.ceil(2.0 * L2_BYTES / per_set)))
    sets = []
    for i in range(R):
        bits, slots = synth.kcache_batch(T, P, NP, seed=100 + i)
        sets.append((torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev),
                     torch.from_numpy(slots).to(dev)))
    cache = torch.zeros(NP * P * 132, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i):
        k, s = sets[i % R]
        sai.indexer_k_quant_insert(k, s, cache, P, status=status, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    torch.cuda.synchronize()
    K = args.steps
    S = K if K <= 200 else 100
    K = S * math.ceil(K / S)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(S):
            step(i)
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        with torch.cuda.stream(stream):
            t0.record(stream)
            for _ in range(K // S):
                graph.replay()
            t1.record(stream)
        torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    ms, _ = aggregate(ms, T, world, dev)
    assert int(status.item()) == 0

    # End to end: pinned host rows and slots in, the status word out.
    hk = torch.from_numpy(synth.kcache_batch(T, P, NP, seed=99)[0].view(np.int16)).pin_memory()
    hs = torch.from_numpy(synth.kcache_batch(T, P, NP, seed=99)[1]).pin_memory()
    hst = torch.zeros(1, dtype=torch.int32).pin_memory()
    dk, ds = sets[0]
    Ke = min(args.steps, 200)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(Ke + 3):
            if i == 3:
                e0.record(stream)
            dk.view(torch.int16).copy_(hk, non_blocking=True)
            ds.copy_(hs, non_blocking=True)
            sai.indexer_k_quant_insert(dk, ds, cache, P, status=status, stream=stream)
            hst.copy_(status, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms, _ = aggregate(e0.elapsed_time(e1), T, world, dev)
    if rank != 0:
        return 0
    peaks = load_peaks()
    nbytes = kcache_bytes(T)
    gbs = nbytes * world * K / (ms * 1e-3) / 1e9
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle

        bits, slots = synth.kcache_batch(2048, P, NP, seed=7)
        c0 = time.perf_counter()
        reps = 0
        small = np.zeros(NP * P * 132, np.uint8)
        while time.perf_counter() - c0 < 5.0:
            codes, scales = oracle.kcache.quantize_k_rows(bits)
            oracle.kcache.insert_k_rows(small, slots, codes, scales, NP, P)
            reps += 1
        csec = time.perf_counter() - c0
        cpu = {"value": kcache_bytes(2048) * reps / csec / 1e9, "unit": "GB/s", "cores": cpu_threads(),
               "kind": "oracle", "sample": f"{reps} x 2048 tokens quantised and inserted, {csec:.1f} s"}
    line = {"metric": KC_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": max(args.warmup, 3), "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16->e4m3", "data": "synthetic",
            "config": {"workload": f"kcache: T={T} bf16 rows, P={P}, pool {NP} pages, split layout",
                       "tokens_per_step": T, "l2": f"{R} rotating input sets > 129 MB L2",
                       "timing": f"{K // S} replays of a CUDA graph of {S} steps"},
            "roofline": {"bound": "hbm", "achieved": gbs / world, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / world / peaks["hbm_gbs"], "traffic": None,
                         "kernel": "k_quant_insert_kernel", "algorithmic_per_launch": nbytes,
                         "peak_source": peaks["source"]},
            "cpu_baseline": cpu,
            "e2e": {"value": nbytes * world * Ke / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": T * (256 + 8), "d2h_bytes_per_step": 4},
            "gpu_launches": K, "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ consumer gather
GA_METRIC = "selected-KV gather GB/s (top-k indices -> int64 row ids -> 576-byte rows), 1 GB300"
GA_ROW, GA_PAGE, GA_PAGES = 576, 64, 8192            # FP8 MLA rows, the decode pool's pages


def run_gather(args, rank: int, world: int, local_rank: int):
    import torch

    import sparse_attention_indexer_03_gb300 as sai
    import synth

    torch.cuda.set_device(local_rank)
    sai.build()
    dev = torch.device("cuda", local_rank)
    idx, table, ctx = synth.gather_batch(page_size=GA_PAGE, num_pages=GA_PAGES)
    rows, k = idx.shape
    gen = torch.Generator(device=dev)
    gen.manual_seed(6)
    pool = torch.randint(0, 256, (GA_PAGES * GA_PAGE * GA_ROW,), dtype=torch.uint8, device=dev, generator=gen)
    out_bytes = rows * k * GA_ROW
    R = max(2, math.ceil(2.0 * L2_BYTES / out_bytes))
    sets = [(torch.from_numpy(idx).to(dev), torch.from_numpy(table).to(dev),
             torch.empty((rows, k), dtype=torch.int64, device=dev),
             torch.empty((rows, k, GA_ROW), dtype=torch.uint8, device=dev)) for _ in range(R)]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i):
        d_idx, d_tab, ids, out = sets[i % R]
        sai.gather_selected_kv(d_idx, 1, d_tab, GA_PAGE, pool, GA_ROW, row_ids=ids, out=out, status=status,
                               stream=stream)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    torch.cuda.synchronize()
    K = args.steps
    S = K if K <= 200 else 100
    K = S * math.ceil(K / S)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(S):
            step(i)
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        with torch.cuda.stream(stream):
            t0.record(stream)
            for _ in range(K // S):
                graph.replay()
            t1.record(stream)
        torch.cuda.synchronize()
    ms, _ = aggregate(t0.elapsed_time(t1), rows, world, dev)
    assert int(status.item()) == 0
    # Algorithmic bytes: the selected rows read, every output row written, the
    # indices read and the row ids written (table reads are a few KB).
    selected = int((idx >= 0).sum())
    nbytes = selected * GA_ROW + out_bytes + rows * k * (4 + 8)
    # End to end: pinned indices in, gathered rows out.
    h_idx = torch.from_numpy(idx).pin_memory()
    h_out = torch.empty((rows, k, GA_ROW), dtype=torch.uint8).pin_memory()
    d_idx, d_tab, ids, out = sets[0]
    Ke = min(args.steps, 50)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(Ke + 3):
            if i == 3:
                e0.record(stream)
            d_idx.copy_(h_idx, non_blocking=True)
            sai.gather_selected_kv(d_idx, 1, d_tab, GA_PAGE, pool, GA_ROW, row_ids=ids, out=out, status=status,
                                   stream=stream)
            h_out.copy_(out, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms, _ = aggregate(e0.elapsed_time(e1), rows, world, dev)
    if rank != 0:
        return 0
    peaks = load_peaks()
    gbs = nbytes * world * K / (ms * 1e-3) / 1e9
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle

        host_pool = pool[: 1 << 26].cpu().numpy()                   # a 64 MB slice of the pool
        sub = idx[:4] % (host_pool.size // GA_ROW // GA_PAGE * GA_PAGE)
        sub_tab = (table[:4] % (host_pool.size // GA_ROW // GA_PAGE)).astype(np.int32)
        c0, reps = time.perf_counter(), 0
        while time.perf_counter() - c0 < 5.0:
            ids_h = oracle.gather.kv_row_ids(sub, sub_tab, 1, GA_PAGE, host_pool.size // GA_ROW // GA_PAGE)
            oracle.gather.gather_kv_rows(host_pool, ids_h, GA_ROW)
            reps += 1
        csec = time.perf_counter() - c0
        per = int((sub >= 0).sum()) * GA_ROW + sub.size * (GA_ROW + 12)
        cpu = {"value": per * reps / csec / 1e9, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{reps} x 4 rows of 2048 selected tokens gathered, {csec:.1f} s"}
    line = {"metric": GA_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": max(args.warmup, 3), "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": {"workload": f"gather: {rows} rows x k={k}, {GA_ROW}-byte rows, P={GA_PAGE}, "
                                   f"pool {GA_PAGES} pages ({GA_PAGES * GA_PAGE * GA_ROW >> 20} MB)",
                       "selected_rows_per_step": selected, "l2": f"{R} rotating output sets > 129 MB L2",
                       "timing": f"{K // S} replays of a CUDA graph of {S} steps"},
            "roofline": {"bound": "hbm", "achieved": gbs / world, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / world / peaks["hbm_gbs"], "traffic": None, "kernel": "gather_rows_kernel",
                         "algorithmic_per_launch": nbytes, "peak_source": peaks["source"]},
            "cpu_baseline": cpu,
            "e2e": {"value": nbytes * world * Ke / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": idx.nbytes, "d2h_bytes_per_step": out_bytes},
            "gpu_launches": K, "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ throughput sweep
def sweep_subset():
    """The declared subset: every (P, next_n, H) at B in {64, 256} and ctx in
    {8192, 65536} (96 of the 600 points)."""
    import synth

    return [(p, n, h, b, c) for _, p, n, h, b, c in synth.sweep_points() if b in (64, 256) and c in (8192, 65536)]


def run_sweep(args, rank: int, world: int, local_rank: int):
    """One JSON line per sweep point: Gtok/s of the step (logits, then top-k)
    and the logits kernel against its binding roofline."""
    import torch

    import sparse_attention_indexer_03_gb300 as sai
    import synth

    torch.cuda.set_device(local_rank)
    sai.build()
    dev = torch.device("cuda", local_rank)
    if args.sweep == "subset":
        points = sweep_subset()
    elif args.sweep == "all":
        points = [(p, n, h, b, c) for _, p, n, h, b, c in synth.sweep_points()]
    else:
        points = [tuple(int(x) for x in pt.split(",")) for pt in args.sweep.split(";")]
    index = {(p, n, h, b, c): i for i, p, n, h, b, c in synth.sweep_points()}
    peaks = load_peaks()
    fp8_peak_tflops = 2.0 * peaks["bf16_tflops"]
    stream = torch.cuda.Stream(device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for pt in points:
        seed = 1000 + index.get(pt, 999)
        w0 = synth.sweep_point_device(*pt, device=dev, seed=seed)
        tok = row_tokens(w0)
        touched = logits_bytes(w0) + topk_bytes(w0)
        R = max(2, min(16, math.ceil(2.0 * L2_BYTES / max(touched, 1))))
        sets = [w0.dev] + [synth.sweep_point_device(*pt, device=dev, seed=seed + 7919 * r).dev for r in range(1, R)]
        for d in sets:
            d["logits"] = torch.empty((w0.rows, w0.logits_stride), dtype=torch.float32, device=dev)
            d["indices"] = torch.empty((w0.rows, w0.topk), dtype=torch.int32, device=dev)

        def lcall(d):
            sai.paged_mqa_logits(d["q"], d["kv"], w0.page_size, d["weights"], d["context_lens"], d["block_table"],
                                 d["logits"], w0.max_model_len, num_pages=w0.num_pages, status=status, stream=stream)

        def tcall(d):
            sai.top_k_per_row_decode(d["logits"], d["context_lens"], w0.next_n, w0.max_model_len, w0.topk,
                                     d["indices"], stream=stream)

        with torch.cuda.stream(stream):
            for i in range(3):
                lcall(sets[i % R])
                tcall(sets[i % R])
        torch.cuda.synchronize()
        S = max(R, min(100, 2 * R * math.ceil(50 / R)))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(S):
                lcall(sets[i % R])
                tcall(sets[i % R])
        ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)] for _ in range(S)]
        probe = torch.cuda.CUDAGraph()
        with torch.cuda.graph(probe, stream=stream):
            for i in range(S):
                ev[i][0].record(stream)
                lcall(sets[i % R])
                ev[i][1].record(stream)
                tcall(sets[i % R])
                ev[i][2].record(stream)
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        c0 = time.perf_counter()
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        M = max(3, min(200, math.ceil(0.1 / max(1e-6, time.perf_counter() - c0))))
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        meas = []
        with ClockSampler(local_rank) as clocks:
            for _ in range(M):
                torch.cuda.synchronize()
                with torch.cuda.stream(stream):
                    t0.record(stream)
                    graph.replay()
                    t1.record(stream)
                torch.cuda.synchronize()
                meas.append(t0.elapsed_time(t1))
            with torch.cuda.stream(stream):
                probe.replay()
            torch.cuda.synchronize()
        assert int(status.item()) == 0, f"status {int(status.item()):#x} at {pt}"
        ms = float(np.median(meas)) / S
        lg_ms = float(np.median([ev[i][0].elapsed_time(ev[i][1]) for i in range(S)]))
        tk_ms = float(np.median([ev[i][1].elapsed_time(ev[i][2]) for i in range(S)]))
        lbytes, lflops = logits_bytes(w0), logits_flops(w0)
        t_hbm = lbytes / (peaks["hbm_gbs"] * 1e9)
        t_tc = lflops / (fp8_peak_tflops * 1e12)
        bound = "hbm" if t_hbm >= t_tc else "tensor"
        frac = max(t_hbm, t_tc) / (lg_ms * 1e-3)
        line = {"sweep_point": {"page_size": pt[0], "next_n": pt[1], "heads": pt[2], "batch": pt[3], "ctx": pt[4]},
                "metric": METRIC, "value": tok / (ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": ms,
                "logits_ms": lg_ms, "topk_ms": tk_ms, "row_tokens_per_step": tok,
                "roofline": {"bound": bound, "frac": frac,
                             "achieved": (lbytes / (lg_ms * 1e-3) / 1e9) if bound == "hbm"
                             else (lflops / (lg_ms * 1e-3) / 1e12),
                             "peak": peaks["hbm_gbs"] if bound == "hbm" else fp8_peak_tflops,
                             "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
                             "algorithmic_per_launch": lbytes if bound == "hbm" else lflops},
                "timing": f"median of {M} replays of a graph of {S} steps, {R} rotating input sets",
                "clocks": clocks.summary()}
        if rank == 0:
            print(json.dumps(line), flush=True)
        del sets, graph, probe, w0
        torch.cuda.empty_cache()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="wide")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--measure-seconds", type=float, default=MEASURE_SECONDS,
                    help="time to spend on repeated K-step measurements (the median counts)")
    ap.add_argument("--op", choices=["indexer", "kcache", "gather"], default="indexer",
                    help="the indexer decode path (logits, top-k), the K-cache write before it, "
                         "or the consumer's gather of the selected KV rows after it")
    ap.add_argument("--layout", choices=["split", "interleaved"], default="split",
                    help="K-cache layout of the indexer workload (interleaved: pages staged as stored, "
                         "rewritten for the MMA)")
    ap.add_argument("--sweep", default=None,
                    help="run the throughput sweep instead: 'subset' (every P, next_n, H at B in {64, 256}, "
                         "ctx in {8192, 65536}), 'all' (600 points) or 'P,n,H,B,ctx;...'")
    ap.add_argument("--path", choices=["auto", "fused", "separate"], default="auto",
                    help="one fused logits + top-k launch per step, or the two launches; auto: fused "
                         "where the -inf fill outweighs the logits tiles four times over (the wide "
                         "workload), where the fused launch spreads the fill over the whole grid")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.path == "fused" and args.layout != "split":
        ap.error("the fused logits + top-k launch reads page-split caches only")
    if args.path == "auto" and args.layout != "split":
        args.path = "separate"

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        print(f"note: WORLD_SIZE={world} but --gpus {args.gpus}", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        if args.op == "kcache":
            return run_kcache(args, rank, world, local_rank)
        if args.op == "gather":
            return run_gather(args, rank, world, local_rank)
        if args.sweep:
            return run_sweep(args, rank, world, local_rank)
        return run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
