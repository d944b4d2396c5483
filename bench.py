#!/usr/bin/env python
"""Benchmark of the FP8 indexer logits on GB300.

One step = one call of the hot path on one batch of synthetic input.  The
default workload is the MTP-verify decode batch (batch 16, next_n 6, 32 heads,
131072-token contexts, max_model_len 1048576, KV block size 64) -- the shape
the indexer pages quote their decode figure on.  Other workloads:
--workload {decode_b1, decode_ragged, decode_mtp_verify, decode_mtp_verify_n1,
prefill_4x1024, decode_blk1, prefill_paged_4x1024 and prefill_paged_blk1_4x1024
(the prefill shape with K read from a paged cache, block 64 or the co-packed
block-1 cache), prefill_2048x65536, prefill_1024x131072 (the prefill page's
other real chunk shapes)}, the top-k consumer of the logits (k = 2048) on two
of those shapes: --workload {topk_decode_mtp_verify, topk_prefill_4x1024}, and
the fused decode logits + top-k: --workload fused_topk_decode_mtp_verify.

Prints ONE JSON line (rank 0):
  value      = us per call (all ranks' calls / max-over-ranks device time),
               each call a CUDA-graph replay, timed with CUDA events on the
               launching stream.  When a call's inputs are larger than the
               L2 (the long-context decode workloads) the calls run back to
               back; otherwise the L2 is flushed before every call (512 MB
               written, then read back so no dirty lines are left to the
               timed call) outside the events around each call.
  roofline   = the dominant kernel's algorithmic bytes / its mean duration
               against the measured HBM copy bandwidth.
  e2e        = the same call driven from pinned host memory: per-step inputs
               copied host->device and the results back on the host, all
               inside the timed region.  Decode writes its logits straight
               into a pinned host output (e2e.copy_back: the same with a
               device output and the written columns copied back); prefill
               copies its logits back; the top-k workloads copy the indices
               back.
  cpu_baseline = the CPU oracle (fp64, OpenMP) on a bounded random sample of
               the same workload's logits, scaled to the whole workload.
--impl reference times that oracle alone as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "indexer logits us/call; essential GB/s and % of roofline (1 GB300)"
UNIT = "us/call"
HEAD_DIM = 128
KV_TOKEN_BYTES = HEAD_DIM + 4  # 128 e4m3 bytes + f32 scale per token

WORKLOADS = {
    "decode_b1": (0, None),
    "decode_ragged": (1, None),
    "decode_mtp_verify": (2, None),
    "decode_mtp_verify_n1": (2, 1),
    "prefill_4x1024": (3, None),
    "decode_blk1": (4, None),
    "prefill_paged_4x1024": (3, None),  # config 3 with K in a paged cache (block 64), gathered in the kernel
    "prefill_paged_blk1_4x1024": (3, None),  # the same with the co-packed block-size-1 cache
    "prefill_2048x65536": (5, None),
    "prefill_1024x131072": (6, None),
}
PAGED_PREFILL = {"prefill_paged_4x1024": 64, "prefill_paged_blk1_4x1024": 1}  # workload -> cache block size
# top-k consumer workloads: (config index, k); the logits are the library's
# own output for that configuration, produced before the timed region
TOPK_WORKLOADS = {
    "topk_decode_mtp_verify": (2, 2048),
    "topk_prefill_4x1024": (3, 2048),
}
TOPK_METRIC = "top-k of the indexer logits us/call; essential GB/s and % of HBM roofline (1 GB300)"
# fused decode logits + top-k (fp8_paged_mqa_topk): (config index, k)
FUSED_WORKLOADS = {
    "fused_topk_decode_mtp_verify": (2, 2048),
}
FUSED_METRIC = "fused indexer logits + top-k us/call; essential GB/s and % of HBM roofline (1 GB300)"
DEFAULT_WORKLOAD = "decode_mtp_verify"
L2_FLUSH_BYTES = 512 << 20
L2_BYTES = 126 << 20  # GB300 L2 (nvidia-smi reports about 126 MiB)
GRAPH_CALLS = 10      # calls per captured graph in back-to-back timing
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- byte model
def decode_window_elems(context_lens, next_n, max_model_len) -> int:
    """Written logits: sum over rows of |{p : p <= ctx - next_n + n, p < max_model_len}|."""
    tot = 0
    for c in np.asarray(context_lens, dtype=np.int64).tolist():
        for n in range(next_n):
            tot += max(0, min(c - next_n + n, max_model_len - 1) + 1)
    return tot


def decode_bytes(batch, next_n, heads, context_lens, max_model_len, block_size=64, k_reads=1):
    """Essential HBM bytes of one decode call: every K token (128 B + 4 B
    scale) read k_reads times per request (1 for a shared K walk), Q, weights,
    and the written output.  The block table is reported separately."""
    ctx = np.minimum(np.maximum(np.asarray(context_lens, dtype=np.int64), 0), max_model_len)
    k = int(ctx.sum()) * KV_TOKEN_BYTES * k_reads
    q = batch * next_n * heads * HEAD_DIM
    w = batch * next_n * heads * 4
    out = decode_window_elems(context_lens, next_n, max_model_len) * 4
    table = int(np.ceil(ctx / block_size).sum()) * 4
    return {"k": k, "q": q, "w": w, "out": out, "total": k + q + w + out, "table": table}


def decode_flops(heads, context_lens, next_n, max_model_len) -> int:
    return 2 * HEAD_DIM * heads * decode_window_elems(context_lens, next_n, max_model_len)


def prefill_bytes(m, n, heads):
    """Essential bytes of one prefill call: K + scale, Q, weights, and the full
    [M, N] f32 output (every element is written)."""
    k = n * KV_TOKEN_BYTES
    q = m * heads * HEAD_DIM
    w = m * heads * 4
    out = m * n * 4
    return {"k": k, "q": q, "w": w, "out": out, "total": k + q + w + out, "table": 0}


def prefill_window_pairs(ks, ke, n) -> int:
    lo = np.maximum(np.asarray(ks, np.int64), 0)
    hi = np.minimum(np.asarray(ke, np.int64), n)
    return int(np.maximum(hi - lo, 0).sum())


def prefill_flops(heads, ks, ke, n) -> int:
    return 2 * HEAD_DIM * heads * prefill_window_pairs(ks, ke, n)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# The source file of each workload's dominant kernel; every kernel also
# builds from the shared headers and is planned and launched by the host.
KERNEL_SOURCE = {"decode": "paged_logits.cu", "prefill": "mqa_logits.cu", "topk": "topk.cu"}
SHARED_SOURCES = ("api.cpp", "common.cuh", "kernels.h", "ptx.cuh")


def workload_kernel(workload: str) -> str:
    if workload in TOPK_WORKLOADS:
        return "topk"
    if workload in FUSED_WORKLOADS:
        return "decode"  # the filter pass of the decode kernel dominates
    return workloads.CONFIGS[WORKLOADS[workload][0]]["kind"]


def kernel_source_hash(workload: str) -> str:
    """Hash of the sources that build and launch the workload's dominant
    kernel: a recorded ncu traffic figure is reported only while they are
    unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_fp8_gb300", "csrc")
    for f in sorted(SHARED_SOURCES + (KERNEL_SOURCE[workload_kernel(workload)],)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """dram read+write bytes per launch from the committed ncu summary, if the
    kernels are unchanged since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel_hash") != kernel_source_hash(workload):
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------ multi-rank
def reduce_max(value: float, world: int, device) -> float:
    """Max of a per-rank time over all ranks (identity on one rank).  Ranks
    run independent replicas of the workload: no data-path collective, only
    this timing reduction."""
    if world <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_call(max_total_ms: float, steps_per_rank: int, world: int) -> float:
    """All ranks' calls divided by the slowest rank's device time, in us/call."""
    return max_total_ms * 1e3 / (steps_per_rank * world)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None
        self.marks = []

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        return rows

    @staticmethod
    def summarize(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------- helpers
def make_case(workload):
    idx, next_n = WORKLOADS[workload]
    if workload in PAGED_PREFILL:
        c = workloads.CONFIGS[idx]
        lens = [c["n"] // c["requests"]] * c["requests"]
        rows = [c["m"] // c["requests"]] * c["requests"]
        blk = PAGED_PREFILL[workload]
        return idx, workloads.paged_prefill_case(lens, rows, c["heads"], block_size=blk, seed=1000 + idx,
                                                 name=c["desc"] + f", K paged (block {blk})")
    return idx, workloads.make_config(idx, next_n=next_n)


def contiguous_view(case):
    """The gathered-K prefill case the CPU oracle reads (oracle gather)."""
    import oracle
    if not isinstance(case, workloads.PagedPrefillCase):
        return case
    k, s = oracle.gather_paged_k(case.kv_cache, case.block_tables, case.cu_seq_lens, case.block_size)
    return workloads.PrefillCase(q=case.q, k=k, kv_scale=s, weights=case.weights, ks=case.ks, ke=case.ke,
                                 name=case.name)


def case_bytes_flops(idx, case):
    if workloads.CONFIGS[idx]["kind"] == "decode":
        b = decode_bytes(case.batch, case.next_n, case.heads, case.context_lens, case.max_model_len,
                         case.block_size)
        f = decode_flops(case.heads, case.context_lens, case.next_n, case.max_model_len)
        units = decode_window_elems(case.context_lens, case.next_n, case.max_model_len)
    else:
        b = prefill_bytes(case.rows, case.cols, case.heads)
        f = prefill_flops(case.heads, case.ks, case.ke, case.cols)
        units = prefill_window_pairs(case.ks, case.ke, case.cols)
    return b, f, units


def oracle_sample_us(o, case, kind, n_elems, rng):
    """Oracle time (s) for n_elems random in-window logits of the workload."""
    if kind == "decode":
        rows_total = case.batch * case.next_n
        rows = rng.integers(0, rows_total, n_elems * 2)
        last = np.minimum(case.context_lens.astype(np.int64)[rows // case.next_n] - case.next_n + rows % case.next_n,
                          case.max_model_len - 1)
        keep = last >= 0
        rows, last = rows[keep][:n_elems], last[keep][:n_elems]
        cols = (rng.random(rows.size) * (last + 1)).astype(np.int64)
        t0 = time.perf_counter()
        o.paged_mqa_logits_at(case.q, case.kv_cache, case.weights, case.context_lens, case.block_tables,
                              case.block_size, case.max_model_len, rows, cols)
        return time.perf_counter() - t0, rows.size
    lo = np.maximum(case.ks.astype(np.int64), 0)
    hi = np.minimum(case.ke.astype(np.int64), case.cols)
    ok = np.nonzero(hi > lo)[0]
    rows = ok[rng.integers(0, ok.size, n_elems)]
    cols = lo[rows] + (rng.random(rows.size) * (hi[rows] - lo[rows])).astype(np.int64)
    t0 = time.perf_counter()
    o.mqa_logits_at(case.q, case.k, case.kv_scale, case.weights, case.ks, case.ke, rows, cols)
    return time.perf_counter() - t0, rows.size


def cpu_baseline(case, kind, units, budget_s=12.0, seed=0):
    """The oracle as it stands on this host's cores, on a bounded sample."""
    import oracle
    o = oracle.Oracle()
    rng = np.random.default_rng(seed)
    t, n = oracle_sample_us(o, case, kind, 2000, rng)  # calibrate
    rate = n / max(t, 1e-6)
    n_elems = int(min(max(2000, rate * budget_s), 5_000_000))
    t, n = oracle_sample_us(o, case, kind, n_elems, rng)
    us_per_call = t / n * units * 1e6
    return {"value": us_per_call, "unit": UNIT, "cores": o.max_threads(), "kind": "oracle",
            "sample": f"{n} random in-window logits of {units} ({t:.1f} s), scaled to the whole workload"}


def run_conditions(workload, world, nbytes=None):
    """The config keys that say how a workload's calls are timed (the same in
    both arms, so that their configs compare equal)."""
    if workload in TOPK_WORKLOADS:
        l2 = "flushed before every call (512 MB written, then read back)"
    elif workload in FUSED_WORKLOADS:
        l2 = f"inputs larger than L2: back-to-back calls (graphs of {GRAPH_CALLS} calls), one event pair around the timed region"
    else:
        input_bytes = int(nbytes["total"] - nbytes["out"])
        l2 = (f"inputs ({input_bytes / 1e6:.0f} MB per call) larger than L2: back-to-back calls "
              f"(graphs of {GRAPH_CALLS} calls), one event pair around the timed region"
              if input_bytes > L2_BYTES else "flushed before every call (512 MB written, then read back)")
    return {"l2": l2, "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world):
    import torch
    import sparse_attention_fp8_gb300 as fp8idx

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    idx, case = make_case(args.workload)
    kind = workloads.CONFIGS[idx]["kind"]
    nbytes, flops, units = case_bytes_flops(idx, case)
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(device=dev)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    if kind == "decode":
        d = {k: up(getattr(case, k)) for k in ("q", "kv_cache", "weights", "context_lens", "block_tables")}
        rows = case.batch * case.next_n
        out = torch.full((rows, case.max_model_len), float("-inf"), device=dev)  # caller's pre-fill, once

        def call(s=stream):
            fp8idx.fp8_paged_mqa_logits(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                                        case.max_model_len, out, stream=s)
        step_inputs = ("q", "weights", "context_lens", "block_tables")
        result_cols = int(min(case.max_model_len, max(int(case.context_lens.max()), 1)))
    elif args.workload in PAGED_PREFILL:
        d = {k: up(getattr(case, k)) for k in ("q", "kv_cache", "block_tables", "cu_seq_lens", "weights", "ks", "ke")}
        out = torch.empty((case.rows, case.cols), device=dev)

        def call(s=stream):
            fp8idx.fp8_mqa_logits_paged(d["q"], d["kv_cache"], d["block_tables"], d["cu_seq_lens"], d["weights"],
                                        d["ks"], d["ke"], out, stream=s)
        step_inputs = ("q", "weights", "ks", "ke", "cu_seq_lens", "block_tables")
        result_cols = case.cols
    else:
        d = {k: up(getattr(case, k)) for k in ("q", "k", "kv_scale", "weights", "ks", "ke")}
        out = torch.empty((case.rows, case.cols), device=dev)

        def call(s=stream):
            fp8idx.fp8_mqa_logits(d["q"], d["k"], d["kv_scale"], d["weights"], d["ks"], d["ke"], out, stream=s)
        step_inputs = ("q", "k", "kv_scale", "weights", "ks", "ke")
        result_cols = case.cols

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2():
        # Write a buffer 4x the L2, then read it back: the write evicts the
        # previous contents and the read writes back the dirty lines here,
        # outside the timed region, so each timed call starts from a clean L2.
        flush.zero_()
        torch.sum(flush, dim=0, dtype=torch.int64, out=flush_sink)

    # One call captured in a CUDA graph; a step is one replay (one kernel).
    # When the inputs a call reads are larger than L2, steps run back to back
    # (every call streams its inputs from HBM anyway); otherwise L2 is
    # flushed before every step, outside the timed events.
    input_bytes = int(nbytes["total"] - nbytes["out"])
    back_to_back = input_bytes > L2_BYTES
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        call()  # first call: lazy initialisation outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    torch.cuda.synchronize()
    # back-to-back steps replay GRAPH_CALLS captured calls at a time
    graph_n = None
    if back_to_back:
        graph_n = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_n, stream=stream):
            for _ in range(GRAPH_CALLS):
                call()
        torch.cuda.synchronize()

    sampler = ClockSampler(dev.index)
    sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            if not back_to_back:
                flush_l2()
            graph.replay()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def timed_steps(n, flushed):
        """n calls; per-call device times (ms) from CUDA events on the stream."""
        barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        if flushed:
            starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
            ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
            with torch.cuda.stream(stream):
                for i in range(n):
                    flush_l2()
                    starts[i].record(stream)
                    graph.replay()
                    ends[i].record(stream)
            torch.cuda.synchronize()
            times = [st.elapsed_time(en) for st, en in zip(starts, ends)]
        else:
            # back to back: one event pair around all n calls
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(n // GRAPH_CALLS):
                    graph_n.replay()
                for _ in range(n % GRAPH_CALLS):
                    graph.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            times = [e0.elapsed_time(e1) / n] * n
        barrier()
        return times, time.time() - t0

    per_call_ms, t_wall = timed_steps(args.steps, not back_to_back)
    # clocks: if the timed region was too short for the sampler, soak the same step for ~1 s
    soak_t0 = time.time()
    if t_wall < 1.0:
        with torch.cuda.stream(stream):
            while time.time() - soak_t0 < 1.0:
                for _ in range(50):
                    if back_to_back:
                        graph_n.replay()
                    else:
                        flush_l2()
                        graph.replay()
                torch.cuda.synchronize()
    clocks = ClockSampler.summarize(sampler.stop())
    clocks["window"] = "timed region" if t_wall >= 1.0 else "timed region + 1 s soak of the same step"

    total_ms = reduce_max(float(sum(per_call_ms)), world, dev)
    us_per_call = whole_job_us_per_call(total_ms, args.steps, world)
    mean_ms = total_ms / args.steps
    median_us = statistics.median(per_call_ms) * 1e3
    # for reference: the same step with L2 flushed before every call
    flushed_us = None
    if back_to_back:
        fl_ms, _ = timed_steps(min(args.steps, 200), True)
        flushed_us = statistics.median(fl_ms) * 1e3
    del graph, graph_n

    # end to end from pinned host memory
    host_in = {k: torch.from_numpy(np.ascontiguousarray(getattr(case, k))).pin_memory() for k in step_inputs}
    host_out = torch.empty((out.shape[0], result_cols), dtype=torch.float32).pin_memory()
    # the written columns, packed on the device, then one contiguous D2H copy
    staging = torch.empty((out.shape[0], result_cols), dtype=torch.float32, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out.numel() * 4
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_time(step):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            step()  # warm-up (first touch of the host pages)
        torch.cuda.synchronize()
        barrier()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(e2e_steps):
                for k, t in host_in.items():
                    d[k].copy_(t, non_blocking=True)
                step()
            e1.record(stream)
        torch.cuda.synchronize()
        return whole_job_us_per_call(reduce_max(e0.elapsed_time(e1), world, dev), e2e_steps, world)

    def copy_back():
        call()
        staging.copy_(out[:, :result_cols])
        host_out.copy_(staging, non_blocking=True)

    e2e_copy_us = e2e_time(copy_back)
    e2e_us, e2e_direct = e2e_copy_us, None
    if kind == "decode":
        # The decode kernel writes its logits with plain stores, so the output
        # can be pinned host memory itself (written over NVLink-C2C while the
        # kernel runs); the caller's -inf pre-fill, once, as on the device.
        host_full = torch.full((rows, case.max_model_len), float("-inf"), dtype=torch.float32).pin_memory()

        def direct():
            fp8idx.fp8_paged_mqa_logits(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                                        case.max_model_len, host_full, stream=stream)
        e2e_direct = e2e_time(direct)
        torch.cuda.synchronize()
        if not torch.equal(host_full[:, :result_cols], out[:, :result_cols].cpu()):
            raise RuntimeError("logits written into host memory differ from the device logits")
        del host_full
        e2e_us = e2e_direct

    # Eager calls (no graph), back to back: the host cost of one public-API
    # call (binding, validation, tensor maps, launch) and the device time per
    # call when every call is launched on its own.
    n_eager = 200
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ea.record(stream)
        h0 = time.perf_counter()
        for _ in range(n_eager):
            call()
        host_us = (time.perf_counter() - h0) / n_eager * 1e6
        eb.record(stream)
    torch.cuda.synchronize()
    eager = {"host_us_per_call": round(host_us, 2), "device_us_per_call": round(ea.elapsed_time(eb) * 1e3 / n_eager, 2),
             "calls": n_eager, "note": "eager back-to-back calls through the public API, no graph"}

    status = fp8idx.device_status()
    hbm_peak = float(peaks["hbm_gbs"])
    fp8_peak = 2.0 * float(peaks["bf16_tflops"])  # nominal fp8:bf16 dense ratio 2
    achieved_gbs = nbytes["total"] / (mean_ms * 1e-3) / 1e9
    tflops = flops / (mean_ms * 1e-3) / 1e12
    roof_t_us = max(nbytes["total"] / (hbm_peak * 1e9), flops / (fp8_peak * 1e12)) * 1e6
    # the bound is whichever term of the roofline is larger: HBM bytes for the
    # decode and the 4x1024 prefill, fp8 tensor FLOPs for the long-window
    # prefill chunks
    if flops / (fp8_peak * 1e12) > nbytes["total"] / (hbm_peak * 1e9):
        roofline = {"bound": "tensor", "achieved": round(tflops, 1), "peak": fp8_peak, "unit": "TFLOP/s",
                    "frac": round(tflops / fp8_peak, 4), "traffic": recorded_traffic(args.workload),
                    "peak_source": f"{peak_src} bf16_tflops x2 (the nominal fp8:bf16 dense ratio)"}
    else:
        roofline = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(achieved_gbs / hbm_peak, 4), "traffic": recorded_traffic(args.workload),
                    "peak_source": f"{peak_src} hbm_gbs"}
    line = {
        "metric": METRIC, "value": round(us_per_call, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(mean_ms, 6), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 x e4m3 -> f32", "data": "synthetic",
        "config": {"workload": args.workload, "desc": case.name, **run_conditions(args.workload, world, nbytes)},
        "median_us": round(median_us, 3),
        "l2_flushed_median_us": round(flushed_us, 3) if flushed_us is not None else round(median_us, 3),
        "essential_bytes": nbytes, "fp8_flops": flops,
        "essential_gbs": round(achieved_gbs, 1),
        "roofline_fraction": round(roof_t_us / (mean_ms * 1e3), 4),
        "roofline": roofline,
        "tensor": {"achieved_tflops": round(tflops, 1), "peak_tflops": fp8_peak,
                   "frac": round(tflops / fp8_peak, 4), "peak_source": f"{peak_src} bf16_tflops x2 (fp8:bf16)"},
        "e2e": {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": ("per-step inputs H2D from pinned memory, call with a pinned host output (the kernel "
                         "writes the logits windows into host memory); the paged K cache stays resident"
                         if kind == "decode" else
                         "per-step inputs H2D from pinned memory, call, written logits D2H; "
                         + ("the paged K cache stays resident" if args.workload in PAGED_PREFILL else "")),
                **({"copy_back": {"value": round(e2e_copy_us, 3),
                                  "note": "the same with a device output and the written columns copied back"}}
                   if e2e_direct is not None else {})},
        "gpu_launches": args.steps,
        "eager": eager,
        "clocks": clocks,
        "device_status": "ok" if status == 0 else f"watchdog {status}",
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(contiguous_view(case), kind, units)
    return line


# ---------------------------------------------------------- top-k arm
def topk_windows(idx, case):
    from oracle import topk as T  # window arithmetic only (no selection)
    if workloads.CONFIGS[idx]["kind"] == "decode":
        return T.decode_windows(case.context_lens, case.next_n, case.max_model_len)
    return T.prefill_windows(case.ks, case.ke, case.cols)


def topk_cpu_baseline(logits_host_rows, rows, lo, hi, k, n_rows_total, budget_s=10.0):
    """The numpy top-k oracle on a bounded sample of rows, scaled to all rows."""
    from oracle import topk as T
    done, t_total = 0, 0.0
    while done < len(rows) and t_total < budget_s:
        r = rows[done]
        t0 = time.perf_counter()
        T.topk_rows(logits_host_rows[done:done + 1], lo[r:r + 1], hi[r:r + 1], k)
        t_total += time.perf_counter() - t0
        done += 1
    return {"value": t_total / done * n_rows_total * 1e6, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done} of {n_rows_total} rows ({t_total:.1f} s), scaled to all rows"}


def run_topk(args, rank, world):
    import torch
    import sparse_attention_fp8_gb300 as fp8idx

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    idx, k = TOPK_WORKLOADS[args.workload]
    case = workloads.make_config(idx)
    kind = workloads.CONFIGS[idx]["kind"]
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(device=dev)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    # the logits this top-k consumes: the library's own output for the configuration
    if kind == "decode":
        d = {key: up(getattr(case, key)) for key in ("q", "kv_cache", "weights", "context_lens", "block_tables")}
        rows = case.batch * case.next_n
        logits = torch.full((rows, case.max_model_len), float("-inf"), device=dev)
        fp8idx.fp8_paged_mqa_logits(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                                    case.max_model_len, logits)
        win = {"context_lens": d["context_lens"]}
        del d

        def call(s=stream):
            fp8idx.fp8_paged_topk(logits, win["context_lens"], case.next_n, case.max_model_len, k, indices, stream=s)
    else:
        d = {key: up(getattr(case, key)) for key in ("q", "k", "kv_scale", "weights", "ks", "ke")}
        rows = case.rows
        logits = torch.empty((rows, case.cols), device=dev)
        fp8idx.fp8_mqa_logits(d["q"], d["k"], d["kv_scale"], d["weights"], d["ks"], d["ke"], logits)
        win = {"ks": d["ks"], "ke": d["ke"]}
        del d

        def call(s=stream):
            fp8idx.fp8_mqa_topk(logits, win["ks"], win["ke"], k, indices, stream=s)
    indices = torch.empty((rows, k), dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    lo, hi = topk_windows(idx, case)
    window_elems = int(np.maximum(hi - lo, 0).sum())
    nbytes = {"logits": window_elems * 4, "indices": rows * k * 4, "windows": int(sum(t.numel() * 4 for t in win.values())),
              "total": window_elems * 4 + rows * k * 4 + int(sum(t.numel() * 4 for t in win.values()))}

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)
    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index)
    sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    # L2 flushed before every call (written, then read back), outside the events
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush.zero_()
            torch.sum(flush, dim=0, dtype=torch.int64, out=flush_sink)
            starts[i].record(stream)
            graph.replay()
            ends[i].record(stream)
    torch.cuda.synchronize()
    per_call_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    if time.time() - t0 < 1.0:  # soak so the clock sampler sees the load
        with torch.cuda.stream(stream):
            t1 = time.time()
            while time.time() - t1 < 1.0:
                for _ in range(50):
                    graph.replay()
                torch.cuda.synchronize()
    clocks = ClockSampler.summarize(sampler.stop())
    clocks["window"] = "timed region + 1 s soak of the same step"
    total_ms = reduce_max(float(sum(per_call_ms)), world, dev)
    us_per_call = whole_job_us_per_call(total_ms, args.steps, world)
    mean_ms = total_ms / args.steps
    median_us = statistics.median(per_call_ms) * 1e3

    # end to end: the windows' logits from pinned host memory, indices back
    if kind == "decode":
        width = int(hi.max()) if rows else 0
    else:
        width = case.cols
    host_logits = torch.empty((rows, width), dtype=torch.float32).pin_memory()
    host_logits.copy_(logits[:, :width].cpu())
    host_idx = torch.empty((rows, k), dtype=torch.int32).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            logits[:, :width].copy_(host_logits, non_blocking=True)
            call()
            host_idx.copy_(indices, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_us = whole_job_us_per_call(reduce_max(e0.elapsed_time(e1), world, dev), e2e_steps, world)

    hbm_peak = float(peaks["hbm_gbs"])
    achieved_gbs = nbytes["total"] / (mean_ms * 1e-3) / 1e9
    line = {
        "metric": TOPK_METRIC, "value": round(us_per_call, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(mean_ms, 6), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 -> i32", "data": "synthetic (logits of the library's kernel)",
        "config": {"workload": args.workload, "desc": f"top-{k} per row of: {case.name}",
                   **run_conditions(args.workload, world)},
        "median_us": round(median_us, 3),
        "essential_bytes": nbytes,
        "essential_gbs": round(achieved_gbs, 1),
        "roofline_fraction": round(achieved_gbs / hbm_peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved_gbs / hbm_peak, 4), "traffic": recorded_traffic(args.workload),
                     "peak_source": f"{peak_src} hbm_gbs"},
        "e2e": {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": rows * width * 4,
                "d2h_bytes_per_step": rows * k * 4,
                "note": "per-step logits windows H2D from pinned memory, call, indices D2H"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rng = np.random.default_rng(0)
        sample = np.sort(rng.choice(rows, size=min(rows, 64), replace=False))
        line["cpu_baseline"] = topk_cpu_baseline(logits[torch.from_numpy(sample).to(dev)].cpu().numpy(), sample,
                                                 lo, hi, k, rows)
    return line


# ------------------------------------------------------------ fused arm
def run_fused(args, rank, world):
    """The fused decode logits + top-k call (six launches, the logits of every
    row never written) on the MTP-verify batch; inputs larger than L2, so
    calls run back to back (graphs of GRAPH_CALLS calls)."""
    import torch
    import sparse_attention_fp8_gb300 as fp8idx

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    idx, k = FUSED_WORKLOADS[args.workload]
    case = workloads.make_config(idx)
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(device=dev)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    d = {key: up(getattr(case, key)) for key in ("q", "kv_cache", "weights", "context_lens", "block_tables")}
    rows = case.batch * case.next_n
    indices = torch.empty((rows, k), dtype=torch.int32, device=dev)
    ws = torch.empty(fp8idx.paged_mqa_topk_workspace(case.batch, case.next_n, case.max_model_len, k) + 256,
                     dtype=torch.uint8, device=dev)

    def call(s=stream):
        fp8idx.fp8_paged_mqa_topk(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                                  case.max_model_len, k, indices, workspace=ws, stream=s)
    b = decode_bytes(case.batch, case.next_n, case.heads, case.context_lens, case.max_model_len, case.block_size)
    nbytes = {"k": b["k"], "q": b["q"], "w": b["w"], "indices": rows * k * 4,
              "total": b["k"] + b["q"] + b["w"] + rows * k * 4, "table": b["table"]}
    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    graph_n = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_n, stream=stream):
        for _ in range(GRAPH_CALLS):
            call()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index)
    sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup // GRAPH_CALLS)):
            graph_n.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    n_rep = max(1, args.steps // GRAPH_CALLS)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n_rep):
            graph_n.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    steps = n_rep * GRAPH_CALLS
    if time.time() - t0 < 1.0:
        with torch.cuda.stream(stream):
            t1 = time.time()
            while time.time() - t1 < 1.0:
                for _ in range(10):
                    graph_n.replay()
                torch.cuda.synchronize()
    clocks = ClockSampler.summarize(sampler.stop())
    clocks["window"] = "timed region + 1 s soak of the same step"
    total_ms = reduce_max(e0.elapsed_time(e1), world, dev)
    us_per_call = whole_job_us_per_call(total_ms, steps, world)
    mean_ms = total_ms / steps
    # e2e: per-step queries, weights, lengths and tables from pinned memory, indices back
    step_inputs = ("q", "weights", "context_lens", "block_tables")
    host_in = {key: torch.from_numpy(np.ascontiguousarray(getattr(case, key))).pin_memory() for key in step_inputs}
    host_idx = torch.empty((rows, k), dtype=torch.int32).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        a0.record(stream)
        for _ in range(e2e_steps):
            for key, t in host_in.items():
                d[key].copy_(t, non_blocking=True)
            call()
            host_idx.copy_(indices, non_blocking=True)
        a1.record(stream)
    torch.cuda.synchronize()
    e2e_us = whole_job_us_per_call(reduce_max(a0.elapsed_time(a1), world, dev), e2e_steps, world)
    hbm_peak = float(peaks["hbm_gbs"])
    achieved_gbs = nbytes["total"] / (mean_ms * 1e-3) / 1e9
    return {
        "metric": FUSED_METRIC, "value": round(us_per_call, 3), "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(mean_ms, 6), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 x e4m3 -> f32 -> i32", "data": "synthetic",
        "config": {"workload": args.workload, "desc": f"top-{k} per row of the logits of: {case.name}",
                   **run_conditions(args.workload, world)},
        "essential_bytes": nbytes,
        "essential_gbs": round(achieved_gbs, 1),
        "roofline_fraction": round(achieved_gbs / hbm_peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved_gbs / hbm_peak, 4), "traffic": recorded_traffic(args.workload),
                     "peak_source": f"{peak_src} hbm_gbs",
                     "note": "the whole call (six launches) against the bytes of K, Q, weights and indices"},
        "e2e": {"value": round(e2e_us, 3), "unit": UNIT,
                "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in host_in.values())),
                "d2h_bytes_per_step": rows * k * 4,
                "note": "per-step inputs H2D from pinned memory, call, indices D2H; the paged K cache stays resident"},
        "gpu_launches": steps * 6,
        "clocks": clocks,
        "device_status": "ok" if fp8idx.device_status() == 0 else "watchdog",
    }


# ---------------------------------------------------------- reference arm
def run_reference_topk(args):
    """Reference arm of a top-k workload: the numpy oracle on a bounded
    sample of rows of the same shape and windows (normal random logits)."""
    from oracle import topk as T
    idx, k = TOPK_WORKLOADS[args.workload]
    case = workloads.make_config(idx)
    lo, hi = topk_windows(idx, case)
    rows = lo.size
    rng = np.random.default_rng(1)
    vals = []
    for _ in range(args.warmup + args.steps):
        r = np.sort(rng.choice(rows, size=min(rows, 8), replace=False))
        width = int(hi[r].max())
        sample = rng.normal(size=(r.size, width)).astype(np.float32)
        t0 = time.perf_counter()
        T.topk_rows(sample, lo[r], hi[r], k)
        vals.append((time.perf_counter() - t0) / r.size * rows * 1e6)
    v = float(np.mean(vals[args.warmup:]))
    return {
        "impl": "reference", "metric": TOPK_METRIC, "value": round(v, 1), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(v / 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 -> i32", "data": "synthetic",
        "config": {"workload": args.workload, "desc": f"top-{k} per row of: {case.name}",
                   **run_conditions(args.workload, int(os.environ.get("WORLD_SIZE", "1")))},
        "cpu_baseline": {"value": round(v, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "8 random rows per step, scaled to all rows"},
        "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference(args):
    import oracle
    if args.workload in TOPK_WORKLOADS:
        return run_reference_topk(args)
    if args.workload in FUSED_WORKLOADS:
        # the oracle logits of the same decode batch (sampled, scaled), plus
        # the numpy top-k over rows of that length (sampled, scaled)
        idx, k = FUSED_WORKLOADS[args.workload]
        a = argparse.Namespace(**vars(args))
        a.workload = next(w for w, (i, nn) in WORKLOADS.items() if i == idx and nn is None)
        line = run_reference(a)
        TOPK_WORKLOADS.setdefault("_fused_topk", (idx, k))
        a.workload = "_fused_topk"
        topk_line = run_reference_topk(a)
        v = line["value"] + topk_line["value"]
        line.update({"metric": FUSED_METRIC, "value": round(v, 1), "ms_per_step": round(v / 1e3, 3),
                     "config": {"workload": args.workload, "desc": f"top-{k} per row of the logits of: "
                                + line["config"]["desc"],
                                **run_conditions(args.workload, int(os.environ.get("WORLD_SIZE", "1")))}})
        line["cpu_baseline"]["value"] = round(v, 1)
        line["cpu_baseline"]["sample"] += "; plus the numpy top-k on 8 random rows per step, scaled"
        line["e2e"]["value"] = round(v, 1)
        return line
    idx, case = make_case(args.workload)
    nbytes, _, _ = case_bytes_flops(idx, case)
    case = contiguous_view(case)
    kind = workloads.CONFIGS[idx]["kind"]
    _, _, units = case_bytes_flops(idx, case)
    o = oracle.Oracle()
    rng = np.random.default_rng(1)
    t, n = oracle_sample_us(o, case, kind, 2000, rng)
    rate = n / max(t, 1e-6)
    per_step_s = max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    n_elems = int(min(max(2000, rate * per_step_s), 5_000_000))
    for _ in range(args.warmup):
        oracle_sample_us(o, case, kind, n_elems, rng)
    vals = []
    for _ in range(args.steps):
        t, n = oracle_sample_us(o, case, kind, n_elems, rng)
        vals.append(t / n * units * 1e6)
    v = float(np.mean(vals))
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(v / 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "desc": case.name,
                   **run_conditions(args.workload, int(os.environ.get("WORLD_SIZE", "1")), nbytes)},
        "cpu_baseline": {"value": round(v, 1), "unit": UNIT, "cores": o.max_threads(), "kind": "oracle",
                         "sample": f"{n_elems} random in-window logits per step of {units}, scaled"},
        "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(TOPK_WORKLOADS) + sorted(FUSED_WORKLOADS),
                    default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group("nccl")
    if args.workload in TOPK_WORKLOADS:
        line = run_topk(args, rank, world)
    elif args.workload in FUSED_WORKLOADS:
        line = run_fused(args, rank, world)
    else:
        line = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
