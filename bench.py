#!/usr/bin/env python
"""MoE layer hot-path benchmark: tokens/s of route + permute + grouped SwiGLU GEMM
+ combine on one GB300 (N GPUs = N independent replicas), with the dominant
kernel's roofline fraction, an end-to-end number through host buffers, the SM
clocks seen during the timed region, and the CPU oracle timed on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config decode|tiny|prefill|v3|pooled]
                  [--tokens T] [--impl ours|reference]

The default workload is the pooled 8-of-384 layer (T = 65,536 tokens, d = 3072,
64 destinations x 6 local experts, top-8, 3 waves, I = 1536), the largest one that
fits one GPU; the others are selected with --config.

One JSON line on stdout (rank 0).  ``--impl reference`` times the CPU oracle on
the same workload and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import subprocess
import statistics
import sys
import threading
import time
import types

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "MoE layer tokens/s (route+permute+grouped GEMM+combine); % HBM / TC roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="pooled",
                    choices=["decode", "tiny", "prefill", "v3", "pooled"])
    ap.add_argument("--tokens", type=int, default=None,
                    help="token count T (decode: 1, 8, 32 or 128, default 128; other workloads: "
                         "a smaller T for short profiling runs)")
    ap.add_argument("--experts", type=int, default=None,
                    help="a smaller expert count E (the same recipe otherwise; for short "
                         "profiling runs that keep per-expert shapes, e.g. v3 with 32 experts "
                         "and 1,024 tokens has the full workload's 256 rows per expert)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--bucket", default="",
                    help="decode: replay one captured graph over a fixed bucket of this many "
                         "token slots, serving --tokens real tokens per step; a comma list "
                         "(e.g. 1,2,4,8,16,32,64,128) is a ladder of buckets, each step "
                         "replaying the smallest that holds its tokens")
    ap.add_argument("--extras", action="store_true",
                    help="also time the backward of the transpose and the telemetry/bias calls "
                         "on this workload's buffers")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager launches instead of CUDA-graph replays of the step")
    ap.add_argument("--payload", default="bf16", choices=["bf16", "fp8_row", "fp8_block128"],
                    help="dispatch payload of the expert input rows (not for --config pooled)")
    ap.add_argument("--fp8-loader", default="auto", choices=["auto", "fused", "dequantize"],
                    help="FP8 payload: dequantize in the gate/up loader ('fused'), once into bf16 "
                         "rows before the bf16 pass ('dequantize'), or by rows per expert ('auto')")
    ap.add_argument("--decode-path", default="auto", choices=["auto", "fused", "separate"],
                    help="decode-sized batches: the one-launch layer (fused), the per-stage "
                         "calls (separate), or whichever the layer picks for the size (auto)")
    ap.add_argument("--expert-passes", default="auto", choices=["auto", "separate", "onepass"],
                    help="the two expert passes as two launches (separate) or one persistent "
                         "launch (onepass), or whichever the layer picks (auto)")
    ap.add_argument("--pool-sequential", action="store_true",
                    help="pooled: run every stage of every wave on one stream (the default "
                         "overlaps pack, compact and combine with the expert passes)")
    ap.add_argument("--gather", action="store_true",
                    help="bf16 payload: permute the maps only and gather the expert rows in the "
                         "gate/up loader instead of copying them in the permute")
    ap.add_argument("--jsonl", default=None,
                    help="also append the JSON line to this file (a results log for sweeps)")
    ap.add_argument("--resume", action="store_true",
                    help="with --jsonl: if the file already holds a line for the same run "
                         "arguments, print that line and run nothing")
    ap.add_argument("--route-only", action="store_true",
                    help="time the router alone on this workload's logits (a few MB on the "
                         "device; for kernel profiling), one JSON line with its duration")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the CPU baseline sample")
    return ap.parse_args()


def workload_for(args) -> workloads.Workload:
    if args.config == "decode":
        return workloads.decode(args.tokens or 128)
    w = {"tiny": workloads.tiny, "prefill": workloads.prefill, "v3": workloads.v3,
         "pooled": workloads.pooled}[args.config]()
    if args.tokens:
        w = workloads.scaled(w, T=args.tokens, name=f"{w.name}_T{args.tokens}")
    if args.experts:
        if w.pooled:
            raise SystemExit("--experts applies to the routed (non-pooled) workloads")
        w = workloads.scaled(w, E=args.experts, name=f"{w.name}_E{args.experts}")
    return w


# default timed steps: a timed region of at least about one second on every workload
DEFAULT_STEPS = {"decode": 5000, "tiny": 2000, "prefill": 600, "v3": 240, "pooled": 120}


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only: barrier and a max over ranks)
# ----------------------------------------------------------------------------

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if self.pg is None:
            return v
        t = torch.tensor([v], dtype=torch.float64,
                         device=f"cuda:{self.local}" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------
# SM clock sampling during the timed region (NVML read-only queries)
# ----------------------------------------------------------------------------

_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """Polls the SM clock and the clock-event reasons of this process's GPU every ~2 ms."""

    def __init__(self, device_index: int):
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self.ok = False
        self._stop = threading.Event()
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.dev = ctypes.c_void_p()
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if self.nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) != 0:
                if self.nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.dev)) != 0:
                    return
            m = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(m)) == 0:
                self.max_mhz = m.value
            self.ok = True
        except OSError:
            pass

    def _run(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        get_r = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(c)) == 0:
                self.samples.append(c.value)
            if get_r(self.dev, ctypes.byref(r)) == 0:
                self.reasons |= r.value
            time.sleep(0.002)

    def __enter__(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        return {"sm_mhz": float(statistics.median(self.samples)), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(self.samples), "sm_mhz_max_seen": max(self.samples),
                "reasons": sorted(n for b, n in _REASONS.items() if self.reasons & b),
                "reasons_mask": hex(self.reasons), "samples": len(self.samples)}


# ----------------------------------------------------------------------------
# algorithmic work per stage (bytes that must move, flops that must be done)
# ----------------------------------------------------------------------------

def stage_work(w, layer, name, counts, acc_rows, n_seg_w, I, d, pool=None):
    """(bytes, flops) the method needs for one launch of stage `name`.

    For the pooled stages `pool` holds the last wave's measured unit counts:
    placed (rows packed into pools), tokens (tokens with at least one placed
    row: each such token row is read once) and kept (rows compacted)."""
    T, k, E = w.T, w.k, w.E
    touched = int((counts > 0).sum())
    # bytes of one dispatched row: bf16 data, or E4M3 data plus its fp32 scales
    row_b = d * 2
    fused = getattr(layer, "fused_fp8", False)
    if getattr(layer, "payload", "bf16") != "bf16":
        row_b = d + layer.xs.shape[1] * 4
    if name == "route":
        return T * E * 4 + T * k * 8, 0
    if name == "decode_layer":
        # the whole layer in one launch: logits in, routes out, token rows in, the
        # permuted copy, the touched experts' weights, H and y written, the fp32 output
        # and the maps
        b = (T * E * 4 + T * k * 8 + T * d * 2 + acc_rows * d * 2 + touched * 3 * d * I * 2
             + acc_rows * I * 2 + acc_rows * d * 2 + T * d * 4 + 3 * T * k * 4 + (2 * E + 1) * 4)
        return b, 6 * acc_rows * d * I
    if name == "quantize":
        return T * d * 2 + T * row_b, 0
    gather = getattr(layer, "gather", False)
    if name == "permute":
        if gather:  # the maps only: the gate/up loader gathers the rows itself
            return T * k * 4 + 2 * T * k * 4 + (2 * E + 1) * 4, 0
        return T * k * 4 + T * row_b + acc_rows * row_b + 2 * T * k * 4 + (2 * E + 1) * 4, 0
    if name == "dequantize":
        return acc_rows * row_b + acc_rows * d * 2, 0
    if name == "gate_up":
        if gather:  # every token row at least once (the k copies of a row come from L2)
            return touched * 2 * d * I * 2 + T * d * 2 + acc_rows * I * 2, 4 * acc_rows * d * I
        a_row = row_b if fused else d * 2  # the unfused FP8 path reads the dequantized bf16 rows
        return touched * 2 * d * I * 2 + acc_rows * a_row + acc_rows * I * 2, 4 * acc_rows * d * I
    if name == "down":
        return touched * I * d * 2 + acc_rows * I * 2 + acc_rows * d * 2, 2 * acc_rows * I * d
    if name == "gate_up_down":  # both passes in one launch: their bytes and flops added
        gb, gf = stage_work(w, layer, "gate_up", counts, acc_rows, n_seg_w, I, d, pool)
        db, df = stage_work(w, layer, "down", counts, acc_rows, n_seg_w, I, d, pool)
        return gb + db, gf + df
    if name == "shared_expert":
        Is = w.shared_I
        return 3 * d * Is * 2 + T * d * 2 * 2 + 2 * T * Is * 2, 6 * T * d * Is
    if name == "combine":
        b = acc_rows * d * 2 + T * k * 8 + T * d * 4 + (T * d * 2 if w.shared_I else 0)
        if w.pooled:
            # map composition (route -> pool row -> compact row) and, in every wave
            # after the first, the read of the fp32 accumulator
            b += T * k * 4 * 2 + acc_rows * 4 + T * d * 4 * (w.n_waves - 1) / w.n_waves
        return int(b), 0
    if name == "pool_pack":
        return (T * k * 4 + pool["tokens"] * d * 2 + pool["placed"] * d * 2 + w.n_dest * d * 2
                + T * k * 4), 0
    if name == "pool_compact":
        return 2 * pool["kept"] * d * 2 + w.n_dest * d * 2 + 2 * w.n_dest * layer.pool_cap * 4, 0
    return 0, 0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return (float(j["hbm_gbs"]), float(j["bf16_tflops"]), float(j["bf16_tflops_sustained"]),
                "measured")
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def kernel_source_sha(name):
    src = {"gate_up": "grouped_swiglu.cu", "down": "grouped_swiglu.cu",
           "gate_up_down": "grouped_swiglu.cu",
           "decode_layer": "decode.cu",
           "shared_expert": "grouped_swiglu.cu", "route": "route.cu", "permute": "permute.cu",
           "quantize": "fp8.cu", "dequantize": "fp8.cu",
           "combine": "combine.cu", "pool_pack": "pool.cu", "pool_compact": "pool.cu"}[name]
    h = hashlib.sha256()
    # the kernel's own file, the router's device header where it is used, and the
    # header of helpers every kernel includes
    extra = ("route_dev.cuh",) if name in ("route", "decode_layer") else ()
    for fn in (src,) + extra + ("common.cuh",):
        with open(os.path.join(ROOT, "grouped_expert_gemm_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def lookup_traffic(stage, workload_name):
    """DRAM bytes per launch of `stage` from a committed ncu summary, if it was taken
    on the current kernel source: (bytes, note) from profiles/*.md lines
    'traffic: <stage> <workload> <bytes_per_launch> <source sha256[:16]> [note]', the
    note saying how a capture of a smaller case was scaled to a full launch; else
    (None, None)."""
    prof = os.path.join(ROOT, "profiles")
    if not os.path.isdir(prof):
        return None, None
    sha = kernel_source_sha(stage)
    pat = re.compile(r"^traffic:\s+(\S+)\s+(\S+)\s+(\d+)\s+([0-9a-f]{16})(?:\s+(.*))?$")
    for fn in sorted(os.listdir(prof)):
        if not fn.endswith(".md"):
            continue
        with open(os.path.join(prof, fn)) as f:
            for line in f:
                m = pat.match(line.strip())
                if m and m.group(1) == stage and m.group(2) == workload_name and m.group(4) == sha:
                    return int(m.group(3)), (m.group(5) or None)
    return None, None


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def build_layer(w, device, payload="bf16", gather=False, fp8_loader="auto", decode_path="auto",
                overlap=True, expert_passes="auto"):
    import grouped_expert_gemm_gb300 as g
    if w.pooled and payload != "bf16":
        raise SystemExit("--payload applies to the routed (non-pooled) workloads")
    logits, sel_bias = workloads.make_router_inputs(w, device)
    x = workloads.make_activations(w, device)
    wg, wu, wd = workloads.make_expert_weights(w, device)
    if w.pooled:
        pool_cap = g.capacity_from_factor(w.sender_cf, w.R, w.n_dest * w.n_waves)
        local_cap = g.capacity_from_factor(w.receiver_cf, w.R, w.local_per_dest * w.n_waves)
        layer = g.PooledMoELayer(w.T, w.d, w.k, w.I, w.n_dest, w.local_per_dest, w.n_waves,
                                 pool_cap, local_cap, wg, wu, wd, device=device,
                                 overlap=overlap)
    else:
        cap = -1 if w.capacity_factor is None else g.capacity_from_factor(w.capacity_factor, w.R, w.E)
        score = g.MOE_SCORE_SOFTMAX if w.score_fn == "softmax" else g.MOE_SCORE_SIGMOID_GROUP
        layer = g.MoELayer(w.T, w.d, w.E, w.k, w.I, wg, wu, wd, capacity=cap, score_fn=score,
                           n_group=w.n_group, topk_group=w.topk_group, route_scale=w.route_scale,
                           sel_bias=sel_bias, shared_weights=workloads.make_shared_weights(w, device),
                           payload=payload, gather=gather, fp8_loader=fp8_loader,
                           decode_path=decode_path, expert_passes=expert_passes, device=device)
    return layer, logits, sel_bias, x


_LIBCUDA = None


def record_external(ev, stream):
    """Record `ev` on `stream` as an event node of the graph being captured (an external
    event record, so it keeps a timestamp on every replay)."""
    global _LIBCUDA
    if _LIBCUDA is None:
        _LIBCUDA = ctypes.CDLL("libcuda.so.1")
        _LIBCUDA.cuEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
    r = _LIBCUDA.cuEventRecordWithFlags(ev.cuda_event, stream.cuda_stream, 1)  # ..._EXTERNAL
    if r != 0:
        raise RuntimeError(f"cuEventRecordWithFlags failed ({r})")


def isolated_stage_ms(layer, logits, x, stream, reps=3):
    """Milliseconds per launch of each stage of a pooled layer's sequential schedule (every
    stage on `stream`, CUDA events between the stages, eager launches), the layer switched
    back to its overlapped schedule afterwards."""
    layer.overlap = False
    try:
        stages = layer.stages(logits, x)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
               for _ in range(reps)]
        with torch.cuda.stream(stream):
            for _, fn, _ in stages:  # one untimed pass first
                fn(stream)
            for r in range(reps):
                evs[r][0].record(stream)
                for i, (_, fn, _) in enumerate(stages):
                    fn(stream)
                    evs[r][i + 1].record(stream)
        stream.synchronize()
    finally:
        layer.overlap = True
    tot, cnt = {}, {}
    for r in range(reps):
        for i, (n, _, _) in enumerate(stages):
            tot[n] = tot.get(n, 0.0) + evs[r][i].elapsed_time(evs[r][i + 1])
            cnt[n] = cnt.get(n, 0) + 1
    return {n: tot[n] / cnt[n] for n in tot}


def run_ours(args, dist, w):
    import grouped_expert_gemm_gb300 as g
    from grouped_expert_gemm_gb300 import abi, build
    build.build()
    device = torch.device(f"cuda:{dist.local}")
    torch.cuda.set_device(device)
    steps = args.steps if args.steps is not None else DEFAULT_STEPS[args.config]
    layer, logits, sel_bias, x = build_layer(w, device, args.payload, args.gather,
                                             args.fp8_loader, args.decode_path,
                                             overlap=not getattr(args, "pool_sequential", False),
                                             expert_passes=getattr(args, "expert_passes", "auto"))
    stream = torch.cuda.Stream(device)
    stages = layer.stages(logits, x)
    names = [n for n, _, _ in stages]
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for _, fn, _ in stages:
                fn(stream)
    stream.synchronize()
    if int(layer.dev_status.item()) != 0:
        raise RuntimeError(f"device status {int(layer.dev_status.item())} after warm-up")

    # Per step: an event at the start and one after every stage, on the stream the
    # stage runs on; a stage on a side stream also gets an event before it there.
    # A main-stream stage's time runs from the previous main-stream event.
    def new_ev():
        return torch.cuda.Event(enable_timing=True)
    evs = [{"start": new_ev(), "after": [new_ev() for _ in stages],
            "before": [new_ev() if side is not None else None for _, _, side in stages]}
           for _ in range(steps)]

    def instrumented_step(s_idx, cur, record):
        ev = evs[s_idx]
        record(ev["start"], cur)
        for i, (_, fn, side) in enumerate(stages):
            if side is not None:
                record(ev["before"][i], side)
            fn(None if record is record_external else cur)
            record(ev["after"][i], side if side is not None else cur)
    # A step whose working set fits L2 would find it resident from the step before
    # (the same inputs every step): such workloads flush L2 before every timed step
    # by reading a buffer four times the L2 size, outside the timed spans, and are
    # timed step by step.  With graphs, the flush and the step are one captured graph
    # with event nodes right after the flush and after the step: a step's span runs
    # from the end of the flush to the end of its last kernel (the device time of the
    # step), with the graph's own launch before the flush.  Without graphs the step's
    # launches follow the flush eagerly (the flush gives the host time to queue them).
    ws_bytes = working_set_bytes(w, layer)
    flush_l2 = ws_bytes < 2 * L2_BYTES
    flush_buf = torch.empty(4 * L2_BYTES // 4, dtype=torch.int32, device=device) if flush_l2 else None
    use_graph = not args.no_graph and not flush_l2
    spans = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(steps)]
    step_graph = None
    span_ms = []
    if flush_l2 and not args.no_graph:
        # flush + step as one graph, with event nodes after the flush and after the step
        step_graph = torch.cuda.CUDAGraph()
        g_start = torch.cuda.Event(enable_timing=True)
        g_end = torch.cuda.Event(enable_timing=True)
        for e in (g_start, g_end):
            e.record(stream)  # creates the event objects
        stream.synchronize()
        with torch.cuda.graph(step_graph, stream=stream):
            flush_buf.max()  # reads 4 x L2 of clean lines
            record_external(g_start, stream)
            l0 = abi.launch_count()
            for _, fn, _ in stages:
                fn(None)
            step_launches = abi.launch_count() - l0
            record_external(g_end, stream)
        with torch.cuda.stream(stream):
            step_graph.replay()
        stream.synchronize()
    if use_graph:
        # The K timed steps as one CUDA graph (every call is asynchronous and
        # allocation-free), plus an instrumented copy of it with the stage events as
        # external event nodes.  Event nodes add a few microseconds of gap each, so
        # the step time comes from the plain graph and the kernel durations from the
        # instrumented one, replayed right after it.
        for row in evs:
            for e in [row["start"]] + row["after"] + [b for b in row["before"] if b is not None]:
                e.record(stream)  # creates the event objects
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        l0 = abi.launch_count()
        with torch.cuda.graph(graph, stream=stream):
            for s in range(steps):
                for _, fn, _ in stages:
                    fn(None)
        graph_launches = abi.launch_count() - l0
        graph_inst = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_inst, stream=stream):
            cur = torch.cuda.current_stream()
            for s in range(steps):
                instrumented_step(s, cur, record_external)
        with torch.cuda.stream(stream):
            graph.replay()  # warm replays (untimed)
            graph_inst.replay()
        stream.synchronize()

    # timed region: K whole steps
    launches0 = abi.launch_count()
    sampler = ClockSampler(dist.local)
    dist.barrier()
    torch.cuda.synchronize(device)
    with sampler:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        with torch.cuda.stream(stream):
            if use_graph:
                graph.replay()
            elif step_graph is not None:
                # one replay per step; its span is read before the next replay re-records
                # the events (only the step boundaries carry events: an event between two
                # kernels would cut their programmatic launch overlap)
                for s in range(steps):
                    step_graph.replay()
                    stream.synchronize()
                    span_ms.append(g_start.elapsed_time(g_end))
            elif flush_l2:
                for s in range(steps):
                    flush_buf.max()  # reads 4 x L2 of clean lines
                    spans[s][0].record(stream)
                    for _, fn, _ in stages:
                        fn(stream)
                    spans[s][1].record(stream)
            else:
                for s in range(steps):
                    instrumented_step(s, stream, lambda e, st: e.record(st))
        t_end.record(stream)
        stream.synchronize()
        launches_timed = abi.launch_count() - launches0
        if flush_l2:  # stage times: the same steps again with events between stages
            with torch.cuda.stream(stream):
                for s in range(steps):
                    flush_buf.max()
                    instrumented_step(s, stream, lambda e, st: e.record(st))
            stream.synchronize()
        if use_graph:
            with torch.cuda.stream(stream):
                graph_inst.replay()
            stream.synchronize()
    torch.cuda.synchronize(device)
    dist.barrier()
    launches = graph_launches if use_graph else launches_timed
    if step_graph is not None:
        launches = step_launches * steps
    elapsed_ms = t_start.elapsed_time(t_end)
    if flush_l2:  # the steps' own spans, without the flushes between them
        if not span_ms:
            span_ms = [a.elapsed_time(b) for a, b in spans]
        elapsed_ms = sum(span_ms)
    max_ms = dist.max(elapsed_ms)
    quantiles = step_quantiles(span_ms if flush_l2 else None, stages, stream, steps, use_graph)
    if int(layer.dev_status.item()) != 0:
        raise RuntimeError(f"device status {int(layer.dev_status.item())} after timed steps")

    stage_ms = {}
    for s in range(steps):
        prev = evs[s]["start"]
        for i, (n, _, side) in enumerate(stages):
            if side is not None:
                dt = evs[s]["before"][i].elapsed_time(evs[s]["after"][i])
            else:
                dt = prev.elapsed_time(evs[s]["after"][i])
                prev = evs[s]["after"][i]
            # ordering steps launch no kernels
            if not (n.endswith("_fork") or n.endswith("_join") or n.startswith("sync_")):
                stage_ms[n] = stage_ms.get(n, 0.0) + dt
    per_step = {n: names.count(n) for n in names}
    # stages on a side stream overlap others; a layer's compute stream (the expert passes
    # of the overlapped pooled layer) holds the step's critical path like a main stream
    compute = getattr(layer, "compute_stream", None)
    side_names = {n for n, _, side in stages if side is not None and side is not compute}
    step_ms = max_ms / steps
    value = dist.world * w.T * steps / (max_ms / 1e3)

    # algorithmic work and the dominant kernel's roofline
    pool = None
    if w.pooled:
        acc_rows = int(layer.local_counts.sum().item())  # last wave's rows (per-wave unit)
        counts = layer.local_counts.cpu().numpy()
        placed = layer.route_to_poolrow.view(w.T, w.k) >= 0
        pool = {"placed": int(placed.sum().item()), "tokens": int(placed.any(1).sum().item()),
                "kept": acc_rows}
    else:
        acc_rows = int(layer.offsets[-1].item())
        counts = layer.counts.cpu().numpy()
    I, d = w.I, w.d
    hbm, tf_burst, tf_sust, peak_src = load_peaks()
    # a timed region of a second or more runs under the steady power cap: tensor-bound
    # kernels are measured against the sustained bf16 peak there, the burst one otherwise
    long_region = max_ms > 1000.0
    tf_peak = tf_sust if long_region else tf_burst
    per_stage = {}
    for n in stage_ms:
        per_launch_ms = stage_ms[n] / (steps * per_step[n])
        b, f = stage_work(w, layer, n, counts, acc_rows, w.E, I, d, pool)
        t_hbm = b / (hbm * 1e9)
        t_tc = f / (tf_peak * 1e12) if f else 0.0
        bound = "tensor" if t_tc > t_hbm else "hbm"
        if bound == "tensor":
            achieved = f / (per_launch_ms * 1e-3) / 1e12
            frac = achieved / tf_peak
        else:
            achieved = b / (per_launch_ms * 1e-3) / 1e9
            frac = achieved / hbm
        per_stage[n] = {"ms_per_launch": round(per_launch_ms, 5),
                        "share": round(stage_ms[n] / sum(stage_ms.values()), 4),
                        "bound": bound, "achieved": round(achieved, 2),
                        "unit": "TFLOP/s" if bound == "tensor" else "GB/s",
                        "frac": round(frac, 4), "alg_bytes": int(b), "alg_flops": int(f),
                        "traffic": lookup_traffic(n, traffic_key(w, layer))[0]}
        if n == "permute" and getattr(layer, "gather", False):
            per_stage[n]["note"] = ("maps only (counts, offsets, both maps): the gate/up loader "
                                    "gathers the expert rows from token order, so no row is "
                                    "copied here; --extras times the copying permute")
        if n in side_names:
            per_stage[n]["timing"] = ("side stream, overlapping the main-stream stages: the "
                                      "figure is the wall-clock span of its work, not a kernel "
                                      "duration")
    if side_names and getattr(layer, "overlap", False):
        # the side-stream stages once more, alone: a few eager steps of the same layer's
        # sequential schedule on one stream, events between the stages, so each of those
        # stages also carries its own kernel time beside its span in the overlapped step
        iso = isolated_stage_ms(layer, logits, x, stream, reps=3)
        for n in side_names & set(iso):
            b, _ = stage_work(w, layer, n, counts, acc_rows, w.E, I, d, pool)
            ach = b / (iso[n] * 1e-3) / 1e9
            per_stage[n]["isolated"] = {"ms_per_launch": round(iso[n], 5),
                                        "achieved": round(ach, 2), "unit": "GB/s",
                                        "frac": round(ach / hbm, 4)}
    # the dominant kernel among the main-stream stages (a side-stream figure is a span)
    dom = max((n for n in stage_ms if n not in side_names), key=lambda n: stage_ms[n])
    ds = per_stage[dom]
    traffic, traffic_note = lookup_traffic(dom, traffic_key(w, layer))
    roofline = {"kernel": dom, "bound": ds["bound"], "achieved": ds["achieved"],
                "peak": tf_peak if ds["bound"] == "tensor" else hbm, "unit": ds["unit"],
                "frac": ds["frac"], "traffic": traffic,
                "peak_source": f"{peak_src} ({'sustained' if long_region and ds['bound'] == 'tensor' else 'burst'})"}
    if traffic_note:
        roofline["traffic_note"] = traffic_note

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": dist.world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the workload, random-init expert weights)",
        "config": config_dict(w, layer, ws_bytes, flush_l2),
        "roofline": roofline, "stages": per_stage,
        "timing": ("the K steps replayed from one captured CUDA graph; stage times from CUDA "
                   "events between the stages of every step (on the stream each stage runs on) "
                   "of an instrumented replay of the "
                   "same K steps right after, on the launching stream" if use_graph else
                   "L2 flushed before every step: flush and step replayed as one captured graph "
                   "with event nodes after the flush and after the step (eager launches after "
                   "the flush with --no-graph); value from the sum of the steps' own spans "
                   "(events at each step's start and end only), stage times from a second "
                   "eager pass of the same steps with events between the stages"
                   if flush_l2 else
                   "eager launches with CUDA events between the stages of every timed step"),
        "clocks": sampler.summary(),
        "step_ms_quantiles": quantiles,
        "gpu_launches": int(launches),
    }
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, dist, w, layer, logits, x, stream, steps, use_graph,
                                flush_buf)
    if args.extras:
        result["extras"] = run_extras(args, w, layer, stream, steps, x)
    result["routing"] = routing_report(w, layer, stream)
    return result, layer, logits, sel_bias, x


def nearest_rank(xs, q):
    """The nearest-rank q-quantile: the ceil(q n)-th smallest of n values."""
    xs = sorted(xs)
    return xs[max(0, min(len(xs) - 1, int(np.ceil(q * len(xs))) - 1))]


def step_quantiles(span_ms, stages, stream, steps, use_graph):
    """Nearest-rank p50 / p90 of single steps, beside the K-step mean `value`: the spans
    (ms) of the timed steps when they were timed one by one (L2 flushed), else K more
    steps replayed one at a time from a one-step graph (or launched eagerly) with events
    at each step's start and end only."""
    spans = None
    if span_ms is None:
        spans = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(steps)]
        g1 = None
        if use_graph:
            g1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1, stream=stream):
                for _, fn, _ in stages:
                    fn(None)
        with torch.cuda.stream(stream):
            for a, b in spans:
                a.record(stream)
                if g1 is not None:
                    g1.replay()
                else:
                    for _, fn, _ in stages:
                        fn(stream)
                b.record(stream)
        stream.synchronize()
    ms = span_ms if span_ms is not None else [a.elapsed_time(b) for a, b in spans]
    return {"p50": round(nearest_rank(ms, 0.5), 5), "p90": round(nearest_rank(ms, 0.9), 5),
            "n": len(ms), "note": "single-step spans; nearest-rank quantiles"}


def routing_report(w, layer, stream):
    """Route accounting of the timed batch, read after the timed region: T*k routes,
    accepted, sender drops S and receiver drops R with the rates S/(T*k), R/(T*k) and
    R/(T*k - S), and the per-expert demand before capacity with its skew summaries
    (computed on the device by the library's demand and load-statistics calls)."""
    from grouped_expert_gemm_gb300 import abi
    routes = w.T * w.k
    demand = layer.expert_demand(stream)
    stats = torch.empty(5, dtype=torch.float64, device=demand.device)
    abi.moe_load_stats(w.E, demand, stats, stream)
    stream.synchronize()
    if w.pooled:
        S = int(layer.sender_drops.sum().item())
        Rr = int(layer.receiver_drops.sum().item())
    else:
        S = int(layer.n_dropped.item())
        Rr = 0
    st = stats.cpu().tolist()
    dem = demand.cpu().tolist()
    rep = {"routes": routes, "accepted": routes - S - Rr, "sender_drops": S,
           "receiver_drops": Rr,
           "sender_drop_rate": round(S / routes, 6) if routes else 0.0,
           "receiver_drop_rate": round(Rr / routes, 6) if routes else 0.0,
           "receiver_drop_rate_given_sent": round(Rr / (routes - S), 6) if routes > S else 0.0,
           "demand_summary": {"min": min(dem), "max": max(dem), "mean": routes / w.E,
                              "cv2": round(st[0], 6), "rho_max": round(st[1], 6),
                              "h_norm": round(st[2], 6), "e_eff": round(st[3], 3),
                              "max_vio": round(st[4], 6)},
           "demand_per_expert": dem}
    if not w.pooled:
        rep["admitted_per_expert"] = layer.counts.cpu().tolist()
    return rep


def run_bucket(args, dist, w):
    """Decode steps served from a fixed token bucket (one captured graph, device-side
    valid count; each step copies its inputs into the stable buffers and replays)."""
    import grouped_expert_gemm_gb300 as g
    from grouped_expert_gemm_gb300 import build
    build.build()
    device = torch.device(f"cuda:{dist.local}")
    torch.cuda.set_device(device)
    steps = args.steps if args.steps is not None else DEFAULT_STEPS[args.config]
    sizes = sorted({int(v) for v in str(args.bucket).split(",")})
    B = sizes[-1]
    wb = workloads.scaled(w, T=B)
    wg, wu, wd = workloads.make_expert_weights(wb, device)
    if len(sizes) == 1:
        bucket = g.DecodeBucket(B, w.d, w.E, w.k, w.I, wg, wu, wd, device=device)
    else:
        bucket = g.DecodeBucketLadder(sizes, w.d, w.E, w.k, w.I, wg, wu, wd, device=device)
    stream = torch.cuda.Stream(device)
    bucket.capture(stream)
    served = bucket if len(sizes) == 1 else bucket.pick(w.T)
    if served is None:
        raise SystemExit(f"--tokens {w.T} exceeds every bucket ({args.bucket})")
    logits, _ = workloads.make_router_inputs(w, device)
    x = workloads.make_activations(w, device)
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            out, path = bucket.forward(logits, x, stream=stream)
    stream.synchronize()
    assert path.startswith("replay"), path
    # the same L2 rule as the exact-shape steps: a working set that fits L2 is
    # flushed before every step and the steps' own spans are summed
    touched = int((served.layer.counts > 0).sum().item())
    ws_bytes = touched * 3 * w.d * w.I * 2 + served.B * (w.E * 4 + w.d * 2 + w.d * 4)
    flush_l2 = ws_bytes < 2 * L2_BYTES
    flush_buf = torch.empty(L2_BYTES, dtype=torch.int32, device=device) if flush_l2 else None
    spans = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(steps)]
    sampler = ClockSampler(dist.local)
    dist.barrier()
    torch.cuda.synchronize(device)
    with sampler:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        with torch.cuda.stream(stream):
            for i in range(steps):
                if flush_l2:
                    flush_buf.max()
                spans[i][0].record(stream)
                bucket.forward(logits, x, stream=stream)
                spans[i][1].record(stream)
        b.record(stream)
        stream.synchronize()
    dist.barrier()
    ms = a.elapsed_time(b)
    if flush_l2:
        ms = sum(e0.elapsed_time(e1) for e0, e1 in spans)
    ms = dist.max(ms)
    if int(served.layer.dev_status.item()) != 0:
        raise RuntimeError("device status after bucket steps")
    return {"metric": METRIC, "value": round(dist.world * w.T * steps / (ms / 1e3), 2),
            "unit": "tokens/s", "n_gpus": dist.world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": round(ms / steps, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "T": w.T, "bucket": served.B,
                       "buckets": sizes, "d": w.d, "E": w.E, "top_k": w.k, "I": w.I,
                       "path": "graph replay over the bucket, device-side valid count",
                       "step_working_set_bytes": int(ws_bytes),
                       "l2": ("flushed before every step (working set fits L2); value from "
                              "the steps' own spans" if flush_l2 else
                              "the step's working set is over twice L2")},
            "timing": "each step: one staging kernel (input copies into the stable buffers and "
                      "the valid count), graph replay", "clocks": sampler.summary(),
            "gpu_launches": steps * (1 + served.graph_launches)}


def run_route_only(args, dist, w):
    """The router alone on the workload's seeded logits: `steps` launches timed with
    CUDA events on the launching stream after `warmup` untimed ones, with the logits
    (and outputs) rotated over enough copies that together they exceed twice the L2,
    so every launch reads its logits from HBM."""
    import grouped_expert_gemm_gb300 as g
    from grouped_expert_gemm_gb300 import abi, build
    build.build()
    device = torch.device(f"cuda:{dist.local}")
    torch.cuda.set_device(device)
    logits, sel_bias = workloads.make_router_inputs(w, device)
    nbytes = w.T * w.E * 4 + w.T * w.k * 8
    copies = max(1, int(np.ceil(2 * L2_BYTES / max(nbytes, 1))) + 1)
    banks = [logits] + [logits.clone() for _ in range(copies - 1)]
    ids = [torch.empty((w.T, w.k), dtype=torch.int32, device=device) for _ in banks]
    gates = [torch.empty((w.T, w.k), dtype=torch.float32, device=device) for _ in banks]
    st = torch.zeros(1, dtype=torch.int32, device=device)
    score = abi.MOE_SCORE_SOFTMAX if w.score_fn == "softmax" else abi.MOE_SCORE_SIGMOID_GROUP
    p = abi.RouteParams(w.T, w.E, w.k, score, w.n_group, w.topk_group, w.route_scale)
    stream = torch.cuda.Stream(device)
    steps = args.steps if args.steps is not None else 200
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            b = i % copies
            abi.moe_route(p, banks[b], sel_bias, ids[b], gates[b], st, stream)
        stream.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            b = i % copies
            abi.moe_route(p, banks[b], sel_bias, ids[b], gates[b], st, stream)
        e.record(stream)
        stream.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    us = a.elapsed_time(e) / steps * 1e3
    hbm, _, _, src = load_peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"kernel": "route", "workload": w.name, "T": w.T, "E": w.E, "top_k": w.k,
            "router": w.score_fn, "us_per_launch": round(us, 3), "alg_bytes": nbytes,
            "achieved_gbs": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
            "peak_source": src, "launches": steps, "banks": copies}


def run_extras(args, w, layer, stream, steps, layer_x=None):
    """Time the calls beyond the forward path on this workload's buffers (events on the
    launching stream, eager launches): the copying permute (when the step gathers its
    rows instead), combine backward, token-gradient unpermute, the demand histogram,
    load telemetry and the bias step on that demand.  Not part of the step or of
    `value`."""
    from grouped_expert_gemm_gb300 import abi
    if w.pooled:
        return None
    hbm, _, _, _ = load_peaks()
    T, k, d = w.T, w.k, w.d
    R = max(T * k, 1)
    acc = int(layer.offsets[-1].item())
    dev = layer.out.device
    dout = torch.randn((T, d), device=dev, dtype=torch.float32)
    dy = torch.empty((R, d), dtype=torch.bfloat16, device=dev)
    dg = torch.empty((R,), dtype=torch.float32, device=dev)
    dx = torch.empty((T, d), dtype=torch.float32, device=dev)
    stats = torch.empty(5, dtype=torch.float64, device=dev)
    bias = torch.zeros(w.E, dtype=torch.float32, device=dev)
    calls = {}
    if getattr(layer, "gather", False):
        # the dispatch as a standalone copy (what the gathered gate/up pass replaces)
        xp = torch.empty((R, d), dtype=torch.bfloat16, device=dev)
        calls["permute_with_copy"] = (lambda: abi.moe_permute(
            T, d, w.E, k, layer.capacity, layer.topk_ids, layer_x, xp, layer.counts,
            layer.offsets, layer.row_to_route, layer.route_to_row, layer.n_dropped,
            layer.perm_ws, layer.perm_ws_bytes, layer.dev_status, stream),
            T * k * 4 + T * d * 2 + acc * d * 2 + 2 * T * k * 4 + (2 * w.E + 1) * 4)
    calls.update({
        "combine_backward": (lambda: abi.moe_combine_backward(
            T, k, d, dout, layer.y, R, layer.route_to_row, layer.gates, dy, dg, layer.dev_status,
            stream), T * d * 4 + 2 * acc * d * 2 + T * k * 8),
        "unpermute_grad": (lambda: abi.moe_unpermute_grad(
            T, k, d, dy, R, layer.route_to_row, dx, 0, layer.dev_status, stream),
            acc * d * 2 + T * d * 4 + T * k * 4),
        "expert_demand": (lambda: layer.expert_demand(stream), T * k * 4 + w.E * 4),
        "load_stats": (lambda: abi.moe_load_stats(w.E, layer.demand, stats, stream), w.E * 4),
        "bias_update": (lambda: abi.moe_bias_update(w.E, layer.demand, bias, 1e-3,
                                                     abi.MOE_BIAS_SIGN, stream), w.E * 12),
    })
    out = {}
    for name, (fn, nbytes) in calls.items():
        for _ in range(3):
            fn()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        stream.synchronize()
        ms = a.elapsed_time(b) / steps
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms_per_launch": round(ms, 5), "alg_bytes": int(nbytes),
                     "achieved_gbs": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4)}
    return out


def traffic_key(w, layer):
    """Workload name under which profiles/ records a stage's DRAM traffic."""
    p = getattr(layer, "payload", "bf16")
    key = w.name if p == "bf16" else f"{w.name}+{p}"
    if getattr(layer, "gather", False):
        key += "+gather"
    return key


L2_BYTES = 129 * 1024 * 1024


def working_set_bytes(w, layer, touched=None):
    """Bytes one step touches: the experts that received rows (all of them for the
    pooled layout; `touched` overrides the count read from the layer's last step),
    the shared expert, and the step's activations and buffers."""
    if w.pooled:
        b = sum(t.numel() * 2 for t in (layer.w_gate, layer.w_up, layer.w_down))
        b += w.T * w.E * 4 + w.T * w.d * 2                      # logits, token rows
        b += (layer.pools.numel() + layer.compact.numel() + layer.y.numel()) * 2
        return b + layer.rows * w.I * 2 + w.T * w.d * 4         # H, fp32 output
    if touched is None:
        touched = int((layer.counts > 0).sum().item())
    R = w.T * w.k
    b = touched * 3 * w.d * w.I * 2 + (3 * w.d * w.shared_I * 2 if w.shared_I else 0)
    b += w.T * w.E * 4 + w.T * w.d * 2 + 2 * R * w.d * 2 + R * w.I * 2 + w.T * w.d * 4
    return b


def config_dict(w, layer, ws_bytes=None, flush_l2=False):
    c = {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "top_k": w.k, "I": w.I,
         "router": w.score_fn, "parallelism": "replicas only (no data-path collective)"}
    if not w.pooled:
        c["payload"] = layer.payload
        if layer.payload == "bf16":
            c["expert_rows"] = ("gathered from token order by the gate/up loader"
                                if layer.gather else "permuted copy written by the permute")
        if layer.payload != "bf16":
            c["payload_bytes_per_row"] = w.d + layer.xs.shape[1] * 4
    if w.pooled:
        c["capacity"] = ("fixed pools: sender factor {} (pool_cap rows per destination per "
                         "wave), receiver factor {} (local_cap rows per local expert per wave)"
                         .format(w.sender_cf, w.receiver_cf))
    elif w.capacity_factor is not None:
        c["capacity_factor"] = w.capacity_factor
        c["capacity"] = layer.capacity
    else:
        c["capacity"] = "dropless"
    if w.shared_I:
        c["shared_I"] = w.shared_I
    if w.pooled:
        c.update({"n_dest": w.n_dest, "local_per_dest": w.local_per_dest, "n_waves": w.n_waves,
                  "pool_cap": layer.pool_cap, "local_cap": layer.local_cap,
                  "wave_policy": "stripe",
                  "schedule": ("pack, compact and combine of the waves on a second stream beside "
                               "the expert passes (double-buffered wave buffers)"
                               if getattr(layer, "overlap", False) else
                               "every stage of every wave in order on one stream")})
    wbytes = sum(t.numel() * 2 for t in (layer.w_gate, layer.w_up, layer.w_down))
    c["expert_weight_bytes"] = wbytes
    if ws_bytes is not None:
        c["step_working_set_bytes"] = int(ws_bytes)
        c["l2"] = ("the step's working set ({:.1f} MB) fits L2 (129 MiB): L2 flushed before every "
                   "timed step by reading a 516 MiB buffer, outside the timed spans"
                   .format(ws_bytes / 1e6) if flush_l2 else
                   "the step's working set ({:.2f} GB) is over twice L2 (129 MiB): every step "
                   "streams it from HBM".format(ws_bytes / 1e9))
    return c


def run_e2e(args, dist, w, layer, logits, x, stream, steps, use_graph, flush_buf=None):
    """Same metric through the host-buffer API (`HostPipeline`): every step copies its
    inputs host->device from pinned memory, runs the layer and copies the fp32 result
    device->host; copies of one step overlap the layer of its neighbours.  The K steps
    are one CUDA graph (or eager with --no-graph), timed between events on `stream`
    that bracket all three streams' work."""
    import grouped_expert_gemm_gb300 as g
    lh = logits.cpu().pin_memory()
    xh = x.cpu().pin_memory()
    oh = torch.empty(layer.out.shape, dtype=torch.float32).pin_memory()
    pipe = g.HostPipeline(layer)

    def run(n):
        pipe.begin(stream)
        for _ in range(n):
            pipe.submit(lh, xh, oh)
        pipe.end(stream)

    with torch.cuda.stream(stream):
        run(max(args.warmup, 3))
    stream.synchronize()
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            run(steps)
        with torch.cuda.stream(stream):
            graph.replay()  # warm replay (untimed)
        stream.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    if flush_buf is not None:
        # working set below L2: one step at a time, L2 flushed before each, the
        # steps' own spans summed (no overlap between steps)
        spans = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(steps)]
        with torch.cuda.stream(stream):
            for a, b in spans:
                flush_buf.max()
                a.record(stream)
                run(1)
                b.record(stream)
        stream.synchronize()
        dist.barrier()
        ms = dist.max(sum(a.elapsed_time(b) for a, b in spans))
        return {"value": round(dist.world * w.T * steps / (ms / 1e3), 2), "unit": "tokens/s",
                "h2d_bytes_per_step": int(lh.numel() * 4 + xh.numel() * 2),
                "d2h_bytes_per_step": int(oh.numel() * 4),
                "copies": "pinned host buffers; per step one H2D of logits and x, the layer and "
                          "one D2H of the fp32 output, L2 flushed before each step, no overlap "
                          "between steps"}
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    with torch.cuda.stream(stream):
        if use_graph:
            graph.replay()
        else:
            run(steps)
    b.record(stream)
    stream.synchronize()
    dist.barrier()
    ms = dist.max(a.elapsed_time(b))
    return {"value": round(dist.world * w.T * steps / (ms / 1e3), 2), "unit": "tokens/s",
            "h2d_bytes_per_step": int(lh.numel() * 4 + xh.numel() * 2),
            "d2h_bytes_per_step": int(oh.numel() * 4),
            "copies": "pinned host buffers; per step one H2D of logits and x and one D2H of "
                      "the fp32 output, overlapped with the neighbouring steps' layer "
                      "(double-buffered device inputs and outputs)"}


# ----------------------------------------------------------------------------
# the CPU oracle on a bounded sample (baseline leg and --impl reference)
# ----------------------------------------------------------------------------

def oracle_batch(w, inputs):
    """One pass of the oracle over a whole batch of tokens: routing, admission and
    permutation (or, pooled, pack and compact in every wave), the SwiGLU of every
    accepted route, and the fp32 combine.  `inputs` holds host copies of the batch's
    logits and token rows (the batch's size is its number of rows), the selection
    bias, a per-expert weight fetcher, the shared expert and the FP8 scale group.
    Capacities follow the workload's capacity factors for this batch size."""
    import oracle
    logits, sel_bias, xb, weights_of, shared, scale_group = inputs
    T, k = xb.shape[0], w.k
    if w.score_fn == "softmax":
        ids, gates = oracle.route_softmax(logits, k)
    else:
        ids, gates = oracle.route_sigmoid_group(logits, sel_bias, k, w.n_group, w.topk_group,
                                                w.route_scale)
    if w.pooled:
        # each route's fate over all waves; its expert is the local id at its destination
        pc = oracle.pool_capacity(w.sender_cf, T, k, w.n_dest, w.n_waves)
        lc = oracle.local_capacity(w.receiver_cf, T, k, w.local_per_dest, w.n_waves)
        row_of = np.full(T * k, -1)
        for wave in range(w.n_waves):
            rp = oracle.pool_pack(ids, xb, w.n_dest, w.local_per_dest, w.n_waves, pc, wave)
            rc = oracle.pool_compact(rp["pools"], pc, w.local_per_dest, lc)
            comp = oracle.compose_map(rp["route_to_poolrow"], rc["poolrow_to_row"])
            ok = comp >= 0
            row_of[ok] = comp[ok] + wave * w.local_per_dest * lc
        route_to_row = row_of
        eids = ids % w.local_per_dest
    else:
        cap = -1 if w.capacity_factor is None else oracle.capacity(w.capacity_factor, T, k, w.E)
        route_to_row = oracle.permute(ids, w.E, cap)["route_to_row"]
        eids = ids
    by_expert = {}
    for r in np.nonzero(route_to_row >= 0)[0]:
        by_expert.setdefault(int(eids.reshape(-1)[r]), []).append(int(r))
    y = {}
    for e, routes in by_expert.items():
        wg, wu, wd = weights_of(e)
        xr = xb[np.array(routes) // k]
        if scale_group is not None:  # FP8 payload: the experts see the dequantized rows
            xr = oracle.dequantize_fp8(*oracle.quantize_fp8(xr, scale_group), scale_group)
        _, ye = oracle.swiglu(oracle.bf16_to_f64(xr), oracle.bf16_to_f64(wg),
                              oracle.bf16_to_f64(wu), oracle.bf16_to_f64(wd))
        for i, r in enumerate(routes):
            y[int(route_to_row[r])] = ye[i]
    sh = None
    if shared is not None:
        sg, su, sd = shared
        _, sh = oracle.swiglu(oracle.bf16_to_f64(xb), oracle.bf16_to_f64(sg[0]),
                              oracle.bf16_to_f64(su[0]), oracle.bf16_to_f64(sd[0]))
    return [oracle.combine_token(lambda r: y[r], route_to_row[t * k:(t + 1) * k], gates[t],
                                 None if sh is None else sh[t]) for t in range(T)]


def host_inputs(logits, sel_bias, x, w_gate, w_up, w_down, shared=None, scale_group=None):
    """Host copies of the inputs (expert weights fetched per expert on demand)."""
    cache = {}

    def weights_of(e):
        if e not in cache:
            cache[e] = tuple(workloads.bf16_bits(t[e]) for t in (w_gate, w_up, w_down))
        return cache[e]
    sh = None if shared is None else tuple(workloads.bf16_bits(t) for t in shared)
    return (logits.cpu().numpy(), None if sel_bias is None else sel_bias.cpu().numpy(),
            workloads.bf16_bits(x), weights_of, sh, scale_group)


def first_tokens(inputs, n):
    """The batch of the first n tokens of `inputs`."""
    logits, sel_bias, xb, weights_of, shared, scale_group = inputs
    return (logits[:n], sel_bias, xb[:n], weights_of, shared, scale_group)


def oracle_sample(w, inputs, budget_s):
    """A batch of the workload's first tokens (16, 32, 64, ... or all T) whose oracle
    pass takes about `budget_s` seconds: doubled while a pass takes under half the
    budget.  Returns (n, seconds of its last pass)."""
    n = min(16, w.T)
    while True:
        t0 = time.perf_counter()
        oracle_batch(w, first_tokens(inputs, n))
        dt = time.perf_counter() - t0
        if n >= w.T or dt * 2 > budget_s:
            return n, dt
        n = min(w.T, n * 2)


def sample_text(w, n):
    caps = "the capacities recomputed from the same factors for that batch size" \
        if (w.pooled or w.capacity_factor is not None) else "dropless"
    return (f"the first {n} of {w.T} tokens of {w.name} as a batch of their own ({caps}); "
            f"each pass runs the whole oracle path on it: routing, "
            f"{'pool pack and compact in every wave' if w.pooled else 'admission and permutation'}"
            f", the fp64 SwiGLU of every accepted route, the combine")


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


CORES_NOTE = ("threads available to the process; numpy runs its matrix products on the BLAS "
              "thread pool over these cores and the rest of the oracle on one thread")


def run_cpu_baseline(args, w, layer, logits, sel_bias, x):
    inp = host_inputs(logits, sel_bias, x, layer.w_gate, layer.w_up, layer.w_down,
                      getattr(layer, "shared", None), getattr(layer, "scale_group", None))
    n, dt = oracle_sample(w, inp, args.cpu_budget)
    # repeat the pass until the oracle has worked about the budget, so the rate is not
    # one short pass
    passes, total = 1, dt
    while total < args.cpu_budget * 0.75 and passes < 64:
        t0 = time.perf_counter()
        oracle_batch(w, first_tokens(inp, n))
        total += time.perf_counter() - t0
        passes += 1
    return {"value": round(n * passes / total, 4), "unit": "tokens/s", "cores": cores(),
            "cores_note": CORES_NOTE, "cpu_model": cpu_model(), "kind": "oracle",
            "sample": f"{sample_text(w, n)}; {passes} pass{'es' if passes > 1 else ''}, "
                      f"{total:.1f} s"}


def oracle_layer_shape(w, wg, wu, wd):
    """What the config line and the working-set count read from a layer, taken from the
    workload and the oracle's capacities (the reference arm builds no layer)."""
    import oracle
    ns = types.SimpleNamespace(payload="bf16", gather=False, w_gate=wg, w_up=wu, w_down=wd)
    if w.pooled:
        ns.pool_cap = oracle.pool_capacity(w.sender_cf, w.T, w.k, w.n_dest, w.n_waves)
        ns.local_cap = oracle.local_capacity(w.receiver_cf, w.T, w.k, w.local_per_dest,
                                             w.n_waves)
        ns.rows = w.local_per_dest * ns.local_cap
        m = dict(dtype=torch.bfloat16, device="meta")
        ns.pools = torch.empty((w.n_dest, ns.pool_cap + 1, w.d), **m)
        ns.compact = torch.empty((ns.rows, w.d), **m)
        ns.y = torch.empty((ns.rows, w.d), **m)
    else:
        ns.capacity = -1 if w.capacity_factor is None else \
            oracle.capacity(w.capacity_factor, w.T, w.k, w.E)
    return ns


def run_reference(args, dist, w):
    """The oracle, as it stands, on this workload's seeded inputs (drawn with the same
    generators and device as our arm's, so the tensors are the same), timed on the host
    cores.  Nothing of the CUDA library is built, loaded or called."""
    if dist.rank != 0:
        return None
    import oracle
    steps = args.steps if args.steps is not None else 5
    if not torch.cuda.is_available():
        raise RuntimeError("the reference arm draws the same seeded inputs on the GPU")
    device = torch.device("cuda:0")
    logits, sel_bias = workloads.make_router_inputs(w, device)
    x = workloads.make_activations(w, device)
    wg, wu, wd = workloads.make_expert_weights(w, device)
    shared = workloads.make_shared_weights(w, device)
    inp = host_inputs(logits, sel_bias, x, wg, wu, wd, shared)
    shape = oracle_layer_shape(w, wg, wu, wd)
    touched = None
    if not w.pooled:
        if w.score_fn == "softmax":
            ids, _ = oracle.route_softmax(inp[0], w.k)
        else:
            ids, _ = oracle.route_sigmoid_group(inp[0], inp[1], w.k, w.n_group, w.topk_group,
                                                w.route_scale)
        touched = int((oracle.permute(ids, w.E, shape.capacity)["counts"] > 0).sum())
    ws_bytes = working_set_bytes(w, shape, touched)
    config = config_dict(w, shape, ws_bytes, ws_bytes < 2 * L2_BYTES)
    # per step a sample sized so that the whole --steps K --warmup W run takes a few
    # minutes at most
    budget = min(4.0, max(0.25, 150.0 / (steps + args.warmup + 2)))
    n, _ = oracle_sample(w, inp, budget)
    batch = first_tokens(inp, n)
    for _ in range(args.warmup):
        oracle_batch(w, batch)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_batch(w, batch)
    dt = time.perf_counter() - t0
    value = n * steps / dt
    sample = f"{sample_text(w, n)}; one pass per step"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
            "n_gpus": 1, "steps": steps, "warmup": args.warmup,
            "ms_per_step": round(dt / steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": config,
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores(),
                             "cores_note": CORES_NOTE, "cpu_model": cpu_model(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


RUN_KEYS = ("impl", "gpus", "steps", "warmup", "config", "tokens", "bucket", "payload",
            "fp8_loader", "gather", "no_graph", "no_e2e", "no_cpu_baseline", "extras",
            "route_only", "decode_path", "experts", "pool_sequential", "expert_passes")


def run_key(args) -> dict:
    """The arguments that decide what a run measures (the identity of a results-log line)."""
    return {k: getattr(args, k) for k in RUN_KEYS}


def logged_line(path, key):
    """The last line of the results log `path` recorded for run arguments `key`, or None."""
    if not path or not os.path.exists(path):
        return None
    found = None
    with open(path) as f:
        for line in f:
            try:
                rec = json.loads(line)
            except ValueError:
                continue  # a torn last line of an interrupted append
            if isinstance(rec, dict) and rec.get("run") == key:
                found = rec
    return found


def emit(res, args):
    """Print the run's JSON line and, with --jsonl, append it to the results log."""
    if args.jsonl:
        res = dict(res, run=run_key(args))
    line = json.dumps(res)
    print(line, flush=True)
    if args.jsonl:
        with open(args.jsonl, "a") as f:
            f.write(line + "\n")


def main():
    args = parse_args()
    if args.resume and args.jsonl and int(os.environ.get("RANK", "0")) == 0:
        prev = logged_line(args.jsonl, run_key(args))
        if prev is not None and int(os.environ.get("WORLD_SIZE", "1")) == 1:
            print(json.dumps(prev), flush=True)
            return
    dist = Dist()
    w = workload_for(args)
    try:
        if args.impl == "reference":
            res = run_reference(args, dist, w)
            if res is not None:
                emit(res, args)
            return
        if args.route_only:
            res = run_route_only(args, dist, w)
            if dist.rank == 0:
                print(json.dumps(res), flush=True)
            return
        if args.bucket:
            res = run_bucket(args, dist, w)
            if dist.rank == 0:
                emit(res, args)
            return
        res, layer, logits, sel_bias, x = run_ours(args, dist, w)
        if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
            # the oracle on the host cores: at N = 1 only, so N replicas' timing is unaffected
            res["cpu_baseline"] = run_cpu_baseline(args, w, layer, logits, sel_bias, x)
        if dist.rank == 0:
            emit(res, args)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
