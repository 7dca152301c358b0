#!/usr/bin/env python
"""Benchmark of the multi-adapter LoRA linear layer (lora_linear_forward) on GB300.

One step = one lora_linear_forward call over one batch, for every projection
of the workload: the LoRA kernels, then the tensor-core base GEMM that adds
the LoRA term before rounding.  For M <= 512 (the GEMM's swapped
orientation) the LoRA kernels write the whole correction s_i B_i A_i x as an
fp32 [M][N] array (per-row kernel, or the adapter-grouped shrink and
expand).  For larger M a plan kernel lists each 256-token tile's pool
blocks; then the two-SM GEMM computes V itself (tensor-core V items over
the same x) and adds the expand as extra MMAs from the pool's B blocks, or,
with fewer than 256 output columns, a tensor-core shrink and a convert
kernel compute V before the one-SM GEMM.  Prints ONE JSON line per workload (default: the
prefill SGMV workload, 8192 tokens of a 4096->4096 projection in 16 sorted
segments over adapters of ranks {8, 16, 32, 64}: the largest workload, and
the one whose base GEMM is bound by the tensor cores).

Timing: W warm-up steps, then K steps; L2 is flushed before every step,
outside the timed intervals: a 2 x L2 write, then a 2 x L2 read of another
buffer (so that no dirty lines of the flush are written back inside the
next step).  The timed steps replay one
forward call captured in a CUDA graph (the launch mode of a decode server);
a step's time is the interval between two CUDA events recorded as nodes of
that graph, right before the forward's first kernel and after its last, so
it excludes the latency of launching the graph (reported beside it as
`replay_ms_per_step`, from events recorded around each replay); step times
are summed.  The dominant kernel's roofline uses stage events the library
records around each kernel in an eager pass over the same K steps; the eager
step rate is reported beside the graph one.  `e2e` repeats the measurement through the C ABI
with pinned host buffers: the host->device copy of x and the row ids and the
device->host copy of the outputs are inside each timed step, all on one
stream of the caller's (not the legacy default stream).  The step is captured
in a CUDA graph and replayed (`e2e.value`); issued from the host call by call
it gives `e2e.eager_value`.  `e2e.streamed_value` streams the steps as a
serving loop would: two buffer sets, the copy-in of step i + 1 and the
copy-out of step i - 1 on streams of their own beside the forward of step i,
timed from the first copy-in to the last copy-out.

--impl reference times the float64 CPU oracle on the host cores on a bounded
row sample of the same workload (the reference arm of this comparison).
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "adapted tokens/s per LoRA linear; TC util (base GEMM) and HBM GB/s (LoRA path)"
DEFAULT_CONFIG = "prefill_sgmv"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_SOURCES = ["tc_gemm.cu", "sm100_ptx.cuh", "lora_device.cuh", "lora_internal.h", "tensor_map.cu", "tensor_map.h"]
# the small-M LoRA stage's kernels and their launch sequence
LORA_SOURCES = ["lora_pipe.cu", "lora_grouped.cu", "lora_kernels.cu", "sm100_ptx.cuh", "lora_device.cuh",
                "lora_internal.h"]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: ~1.5 s of GPU work)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["lora", "reference"], default="lora")
    ap.add_argument("--config", default=DEFAULT_CONFIG,
                    help="workload name, or 'all' for one line per workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU work of the oracle baseline")
    ap.add_argument("--w-int8", action="store_true",
                    help="base weights as int8 with per-row scales (decode shapes, M <= 64)")
    ap.add_argument("--w-int4", action="store_true",
                    help="base weights as packed int4 with per-row scales (decode shapes, M <= 64)")
    ap.add_argument("--reference-seconds", type=float, default=90.0,
                    help="oracle work of the whole --impl reference run")
    return ap.parse_args()


# ----------------------------------------------------------------------------- helpers

def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_hash(names) -> str:
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "adapter_gemm_linear_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def gemm_source_hash() -> str:
    return source_hash(GEMM_SOURCES)


def ncu_traffic(workload: str, stage: str = "gemm"):
    """dram bytes from a committed ncu capture, if it was taken on the
    current kernel sources: per launch of the GEMM kernel (stage "gemm"), or
    per forward summed over the small-M LoRA stage's kernels (stage "lora")."""
    try:
        with open(TRAFFIC_PATH) as f:
            entries = json.load(f)
    except (OSError, ValueError):
        return None
    src = source_hash(GEMM_SOURCES if stage == "gemm" else LORA_SOURCES)
    for e in entries.get("entries", []):
        if e.get("workload") == workload and e.get("stage", "gemm") == stage and e.get("source_hash") == src:
            return e.get("dram_bytes_per_launch" if stage == "gemm" else "dram_bytes_per_forward")
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(device_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        smax = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in self.samples:
            for name, v in zip(names, s[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(self.samples)}


def workload_stats(wl):
    """Distinct adapters, adapted rows and rank sums the byte counts need."""
    ids = wl.row_adapter
    used = wl.used_slots
    adapted = ids[ids >= 0]
    return {
        "distinct": int(used.size),
        "adapted_rows": int(adapted.size),
        "sum_r_distinct": int(sum(int(wl.ranks[s]) for s in used)),
        "sum_r_rows": int(sum(int(wl.ranks[s]) for s in adapted)),
    }


SWAPPED_MAX_M = 512  # the library's GEMM takes the swapped orientation up to this many rows


def algorithmic(wl, w_bits=0):
    """Per-call algorithmic bytes and flops, as the method defines them.

    Base GEMM (every projection): flops 2MNK, bytes (NK + MK + MN) * eb (a
    quantized W counts its packed bytes and one fp32 scale per row).
    LoRA term, standalone kernels (small M: the LoRA kernels read x and the
    distinct adapters and produce the correction the GEMM adds):
        sum_distinct r (K + N) eb + M_a (K + 2N) eb + 2 M_a r 4
    (adapters once each, the adapted rows of x read and of y read and
    written, the rank-r intermediate written and read).  Large M with the
    two-SM GEMM ("pair": shrink and expand inside the GEMM, only the tile
    plans before it): the GEMM's bytes are the base bytes plus the fused
    form below, its flops 2MNK plus the LoRA flops; the plan kernel's bytes
    are the row ids and the plans.  Large M otherwise ("rows": the shrink is
    its own kernel, the expand runs inside the GEMM): the shrink's share,
        sum_distinct r K eb + M_a K eb + M_a r 4,
    and the GEMM's share, sum_distinct r N eb + M_a r 4, beside the base
    bytes.  The fused form of the LoRA bytes (x and y shared with the base
    GEMM), sum_distinct r (K + N) eb + 2 M_a r 4, is reported beside them.
    LoRA flops: 2 r (K + N) per adapted row.
    The implementation's own intermediates (the fp32 correction array of the
    small-M path, the bf16 hi/lo V operand of the large-M path) are not
    algorithmic: they are reported separately as ``intermediate_bytes``
    (written once and read once).
    """
    eb = 2 if wl.dtype == "bf16" else 4
    st = workload_stats(wl)
    wb = {8: 1, 4: 0.5}.get(w_bits, eb)  # bytes per base weight
    M, K = wl.M, wl.K
    swapped = wl.dtype == "bf16" and M <= SWAPPED_MAX_M
    pair = wl.dtype == "bf16" and not swapped and not w_bits and all(p.N >= PAIR_BN for p in wl.projections)
    out = {"gemm_bytes": 0, "gemm_flops": 0, "lora_bytes": 0, "lora_flops": 0, "lora_bytes_fused": 0,
           "intermediate_bytes": 0, "per_proj": [],
           "orientation": "swapped" if swapped else "pair" if pair else "rows"}
    Ma, rd, rr = st["adapted_rows"], st["sum_r_distinct"], st["sum_r_rows"]
    for p in wl.projections:
        N = p.N
        base = int(N * K * wb) + (N * 4 if w_bits else 0) + (M * K + M * N) * eb
        fused = rd * (K + N) * eb + 2 * rr * 4
        gf, lf = 2 * M * N * K, 2 * rr * (K + N)
        if swapped:
            gb, lb = base, rd * (K + N) * eb + Ma * (K + 2 * N) * eb + 2 * rr * 4
            inter = 2 * M * N * 4  # the fp32 correction array
        elif pair:
            gb, lb = base + fused, 4 * M + 48 * 4 * (-(-M // PLAN_ROWS))
            gf, lf = gf + lf, 0
            inter = large_m_intermediates(wl, N, pair=True)
        else:
            gb = base + rd * N * eb + rr * 4
            lb = rd * K * eb + Ma * K * eb + rr * 4
            inter = large_m_intermediates(wl, N)
        out["gemm_bytes"] += gb
        out["gemm_flops"] += gf
        out["lora_bytes"] += lb
        out["lora_bytes_fused"] += fused
        out["lora_flops"] += lf
        out["intermediate_bytes"] += inter
        out["per_proj"].append({"N": N, "gemm_bytes": gb, "gemm_flops": gf, "lora_bytes": lb})
    out.update(st)
    return out


PLAN_ROWS = 256  # tokens per plan tile of the library's large-M LoRA path
PAIR_BN = 256    # output columns per tile of its two-SM GEMM
V_SLICES = 2     # K-slices of a tile's V in the two-SM GEMM


def large_m_intermediates(wl, N, pair=False):
    """Bytes of the large-M path's own intermediates for one projection: per
    256-token tile, the fp32 V of the pool blocks its rows use -- with the
    two-SM GEMM, all K-slices but one written and read once; otherwise an
    accumulator written by reductions and read once -- and Vt, its bf16 hi
    and lo parts (written once, read by every one of the GEMM's column
    tiles)."""
    ids = wl.row_adapter
    blocks = 0
    for t0 in range(0, wl.M, PLAN_ROWS):
        used = np.unique(ids[t0:t0 + PLAN_ROWS])
        blocks += sum(-(-int(wl.ranks[s]) // 16) for s in used if s >= 0)
    cols = 16 * blocks  # accumulator columns over all tiles
    col_tiles = -(-N // PAIR_BN)
    fp32 = cols * PLAN_ROWS * 4 * 2 * ((V_SLICES - 1) if pair else 1)
    return fp32 + cols * PLAN_ROWS * 2 * 2 * (1 + col_tiles)


def percentiles(values):
    """Median, 10th and 90th percentile of a list of step times."""
    a = np.asarray(values, dtype=np.float64)
    return {"p10": float(np.percentile(a, 10)), "p50": float(np.percentile(a, 50)),
            "p90": float(np.percentile(a, 90))}


# ----------------------------------------------------------------------------- GPU arm

def build_case(wl, device, w_bits=0):
    import torch
    from adapter_gemm_linear_gb300 import Int4Weight, Int8Weight, LinearCall, LoraPool

    td = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    max_rank = max(16, -(-int(wl.ranks.max()) // 16) * 16)
    used = set(int(s) for s in wl.used_slots)
    pools = []
    for p, proj in enumerate(wl.projections):
        pool = LoraPool(wl.K, proj.N, wl.num_slots, max_rank, wl.blocks_needed(), dtype=td,
                        device=device, free_list_seed=wl.free_list_seed + p)
        gen = torch.Generator(device=device)
        gen.manual_seed(1234 + p)
        for s in range(wl.num_slots):
            r = int(wl.ranks[s])
            if s in used or wl.num_slots <= 256:
                A, B = wl.adapter(p, s)
                pool.load(s, torch.from_numpy(A).to(td), torch.from_numpy(B).to(td), float(wl.alphas[s]))
            else:
                # resident but unused by this batch: device-random contents
                A = (torch.randn(r, wl.K, device=device, generator=gen) * 0.02).to(td)
                B = (torch.randn(proj.N, r, device=device, generator=gen) * 0.02).to(td)
                pool.load(s, A, B, float(wl.alphas[s]))
        pools.append(pool)
    x = torch.from_numpy(wl.x).to(td).to(device)
    Ws = [torch.from_numpy(p.W).to(td).to(device) for p in wl.projections]
    if w_bits:  # symmetric per-row int8 / int4 of the same weights
        Ws = [(Int8Weight if w_bits == 8 else Int4Weight).quantize(W) for W in Ws]
    outs = [torch.empty((wl.M, p.N), dtype=td, device=device) for p in wl.projections]
    seg = None
    if wl.mode == "sgmv":
        seg = (torch.from_numpy(wl.seg_offsets).to(device), torch.from_numpy(wl.seg_adapter).to(device))
        call = LinearCall(x, list(zip(Ws, pools, outs)), seg_offsets=seg[0], seg_adapter=seg[1])
        ids = None
    else:
        ids = torch.from_numpy(wl.row_adapter).to(device)
        call = LinearCall(x, list(zip(Ws, pools, outs)), row_adapter=ids)
    torch.cuda.synchronize(device)
    return {"pools": pools, "x": x, "Ws": Ws, "outs": outs, "ids": ids, "seg": seg, "call": call}


class L2Flush:
    """Evicts the workload from L2 before a step: a write of 2 x L2 bytes,
    then a read of another 2 x L2 bytes, so that L2 holds none of the
    workload's data and no dirty lines whose write-back would fall into the
    next timed interval."""

    def __init__(self, l2, device):
        import torch

        self.w = torch.empty(2 * l2, dtype=torch.uint8, device=device)
        self.r = torch.ones(2 * l2 // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def zero_(self):
        import torch

        self.w.zero_()
        self.sink.copy_(self.r.sum())


def graph_event_pair():
    """Two timing events that a CUDA graph records as nodes of its own, and
    the function that records one on the capturing stream."""
    import torch

    try:
        a = torch.cuda.Event(enable_timing=True, external=True)
        b = torch.cuda.Event(enable_timing=True, external=True)
        return a, b, lambda ev: ev.record()
    except TypeError:  # a torch without external events: the runtime's own call
        import ctypes

        lib = None
        for name in ("libcudart.so.13", "libcudart.so", "/usr/local/cuda/lib64/libcudart.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None:
            raise RuntimeError("no CUDA runtime library for in-graph timing events")
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        for ev in (a, b):  # create the raw events
            ev.record()
        torch.cuda.synchronize()

        def record(ev):
            stream = torch.cuda.current_stream()
            rc = lib.cudaEventRecordWithFlags(ctypes.c_void_p(ev.cuda_event), ctypes.c_void_p(stream.cuda_stream),
                                              ctypes.c_uint(1))  # cudaEventRecordExternal
            if rc != 0:
                raise RuntimeError(f"cudaEventRecordWithFlags failed ({rc})")

        return a, b, record


def time_device(case, wl, steps, warmup, flush, clocks_index):
    """Eager pass with per-stage events (kernel durations for the roofline),
    then the timed pass: one forward captured in a CUDA graph and replayed
    once per step, an L2 flush before each replay.  A step's time is the
    interval between two events recorded inside the graph around the
    forward; the interval between events recorded around each replay (which
    adds the graph's launch latency) is reported beside it."""
    import torch
    from adapter_gemm_linear_gb300 import kernel_launches

    call = case["call"]
    n_ev = 1 + 2 * len(wl.projections)
    for _ in range(warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    # ---- eager pass: stage durations of every kernel
    stage = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(steps)]
    e_starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e_ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for ev in stage:  # materialise the raw events before timing
        for e in ev:
            e.record()
    torch.cuda.synchronize()
    for i in range(steps):
        flush.zero_()
        call.set_stage_events(stage[i])
        e_starts[i].record()
        call()
        e_ends[i].record()
    torch.cuda.synchronize()
    call.set_stage_events(None)
    n_proj = len(wl.projections)
    shrink_ms = [sum(ev[2 * p].elapsed_time(ev[2 * p + 1]) for p in range(n_proj)) for ev in stage]
    gemm_ms = [sum(ev[2 * p + 1].elapsed_time(ev[2 * p + 2]) for p in range(n_proj)) for ev in stage]
    eager_ms = [s.elapsed_time(e) for s, e in zip(e_starts, e_ends)]
    # ---- timed pass: CUDA graph of one forward
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    g_start, g_end, record_in_graph = graph_event_pair()
    n_cap = kernel_launches()
    with torch.cuda.graph(graph):
        # timing events as nodes of the graph itself, right around the
        # forward's kernels: they measure the forward's device time without
        # the latency of launching the graph
        record_in_graph(g_start)
        call()
        record_in_graph(g_end)
    kernels_per_call = kernel_launches() - n_cap
    for _ in range(warmup):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    sampler = ClockSampler(clocks_index)
    time.sleep(0.3)
    step_ms = []
    for i in range(steps):
        flush.zero_()
        starts[i].record()
        graph.replay()
        ends[i].record()
        ends[i].synchronize()  # the in-graph events are recorded again by the next replay
        step_ms.append(g_start.elapsed_time(g_end))
    torch.cuda.synchronize()
    clocks = sampler.stop()
    replay_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    del graph
    return {"step_ms": step_ms, "replay_ms": replay_ms, "eager_ms": eager_ms, "shrink_ms": shrink_ms,
            "gemm_ms": gemm_ms,
            "launches": kernels_per_call * steps, "kernels_per_call": kernels_per_call, "clocks": clocks}


def _time_loads(K, N, r, td, device, reps):
    """Median load time of one rank-r adapter (K -> N) into a pool slot from
    each source; every load is followed by an unload."""
    import torch
    from adapter_gemm_linear_gb300 import LoraPool

    nbytes = r * (K + N) * (2 if td == torch.bfloat16 else 4)
    pool = LoraPool(K, N, 2, r, r // 16, dtype=td, device=device)
    gen = torch.Generator().manual_seed(7)
    A = (torch.randn(r, K, generator=gen) * 0.02).to(td)
    B = (torch.randn(N, r, generator=gen) * 0.02).to(td)
    srcs = {"host": (A, B), "mapped_host": (A.pin_memory(), B.pin_memory()),
            "device": (A.to(device), B.to(device))}
    out = {"rank": r, "bytes": nbytes}
    stream = torch.cuda.current_stream()
    for name, (a, b) in srcs.items():
        ms = []
        for _ in range(reps + 1):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            pool.load(0, a, b, float(2 * r), stream=stream, src=name.replace("_host", ""))
            torch.cuda.synchronize()
            ms.append((time.perf_counter() - t0) * 1e3)
            pool.unload(0, stream=stream)
        med = statistics.median(ms[1:])
        out[name] = {"ms": round(med, 4), "gbs": round(nbytes / (med / 1e3) / 1e9, 2)}
    torch.cuda.synchronize()
    pool.close()
    return out


def time_adapter_loads(wl, device, reps=8):
    """Pool residency: time to load one adapter of the workload's largest
    rank into a slot of its first projection's pool shape, by source --
    staged pageable host memory (synchronous), page-locked host memory read
    by the scatter kernel over the host link (asynchronous), and device
    memory -- and the same for an adapter of the residency page's size
    (rank 1024 on an 8192 -> 28672 projection, 75.5 MB)."""
    import torch

    td = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    r = max(16, -(-int(wl.ranks.max()) // 16) * 16)
    out = _time_loads(wl.K, wl.projections[0].N, r, td, device, reps)
    big = _time_loads(8192, 28672, 1024, torch.bfloat16, device, reps)
    big["shape"] = "rank 1024, 8192 -> 28672"
    out["page_scale"] = big
    return out


def time_e2e(case, wl, steps, flush, device):
    """Through the C ABI with pinned host buffers; copies inside each step."""
    import torch

    call = case["call"]
    x_host = torch.from_numpy(wl.x).to(case["x"].dtype).pin_memory()
    ids_host = None if case["ids"] is None else torch.from_numpy(wl.row_adapter).pin_memory()
    outs_host = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in case["outs"]]
    h2d = x_host.numel() * x_host.element_size() + (0 if ids_host is None else ids_host.numel() * 4)
    d2h = sum(o.numel() * o.element_size() for o in outs_host)

    def step():
        case["x"].copy_(x_host, non_blocking=True)
        if ids_host is not None:
            case["ids"].copy_(ids_host, non_blocking=True)
        call()
        for o, oh in zip(case["outs"], outs_host):
            oh.copy_(o, non_blocking=True)

    # a stream of the caller's own, as a serving loop would use (on the legacy
    # default stream the GEMM could not start beside the LoRA kernel)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    eager_ms, graph_ms = 0.0, 0.0
    with torch.cuda.stream(side):
        for _ in range(3):
            step()
        side.synchronize()
        # eager: the copies and the forward call issued from the host every step
        for i in range(steps):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(side)
            step()
            e.record(side)
            e.synchronize()
            eager_ms += s.elapsed_time(e)
        # graph: the same step (both copies and the forward) captured once and
        # replayed, as a decode loop replays its step
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            step()
        g.replay()
        side.synchronize()
        for i in range(steps):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(side)
            g.replay()
            e.record(side)
            e.synchronize()
            graph_ms += s.elapsed_time(e)
    torch.cuda.current_stream().wait_stream(side)
    return {"ms": graph_ms, "eager_ms": eager_ms, "h2d": h2d, "d2h": d2h}


def time_e2e_streamed(case, wl, steps):
    """Through the C ABI with pinned host buffers, as a serving loop streams
    its batches: two device buffer sets, the copy-in of step i + 1 (x and the
    row ids) and the copy-out of step i - 1 (the outputs) on streams of their
    own beside the forward of step i.  Every step moves its own bytes both
    ways; the time runs from the first copy-in to the last copy-out."""
    import torch
    from adapter_gemm_linear_gb300 import LinearCall

    x_host = torch.from_numpy(wl.x).to(case["x"].dtype).pin_memory()
    ids_host = None if case["ids"] is None else torch.from_numpy(wl.row_adapter).pin_memory()
    x1 = torch.empty_like(case["x"])
    outs1 = [torch.empty_like(o) for o in case["outs"]]
    if case["seg"] is not None:
        call1 = LinearCall(x1, list(zip(case["Ws"], case["pools"], outs1)), seg_offsets=case["seg"][0],
                           seg_adapter=case["seg"][1])
        ids1 = None
    else:
        ids1 = torch.empty_like(case["ids"])
        call1 = LinearCall(x1, list(zip(case["Ws"], case["pools"], outs1)), row_adapter=ids1)
    bufs = [(case["x"], case["ids"], case["outs"], case["call"]), (x1, ids1, outs1, call1)]
    outs_host = [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in case["outs"]] for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    for s in (s_in, s_comp, s_out):
        s.wait_stream(torch.cuda.current_stream())

    def issue(i):
        b = i % 2
        x, ids, outs, call = bufs[b]
        with torch.cuda.stream(s_in):
            s_in.wait_event(comp_done[b])  # the forward two steps back has read x_b
            x.copy_(x_host, non_blocking=True)
            if ids is not None:
                ids.copy_(ids_host, non_blocking=True)
            in_done[b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(in_done[b])
            s_comp.wait_event(out_done[b])  # the copy-out two steps back has read outs_b
            call()
            comp_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            for o, oh in zip(outs, outs_host[b]):
                oh.copy_(o, non_blocking=True)
            out_done[b].record(s_out)

    for i in range(4):
        issue(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for i in range(steps):
        issue(i)
    end.record(s_out)
    end.synchronize()
    ms = start.elapsed_time(end)
    torch.cuda.synchronize()
    torch.cuda.current_stream().wait_stream(s_out)
    return ms


def time_comparators(case, wl, flush, reps=20):
    """Context only: the same base GEMMs through torch.matmul (cuBLAS), and
    the whole layer as sequential passes in torch -- the base GEMM, then for
    every adapter in the batch its rows gathered, multiplied by A^T and B^T,
    scaled and added (the per-adapter loop the S-LoRA page contrasts with a
    batched operator).  Eager launches, L2 flushed before each step, CUDA
    events around each step; medians."""
    import torch

    x, Ws = case["x"], case["Ws"]
    if not all(isinstance(W, torch.Tensor) for W in Ws):
        return None
    outs = [torch.empty((wl.M, W.shape[0]), dtype=x.dtype, device=x.device) for W in Ws]
    ids = wl.row_adapter
    groups = []
    for p, proj in enumerate(wl.projections):
        per = []
        for s in wl.used_slots:
            rows = torch.from_numpy(np.nonzero(ids == s)[0].astype(np.int64)).to(x.device)
            A, B = wl.adapter(p, int(s))
            per.append((rows, torch.from_numpy(A).to(x.dtype).to(x.device), torch.from_numpy(B).to(x.dtype).to(x.device),
                        float(wl.alphas[s]) / float(wl.ranks[s])))
        groups.append(per)

    def base():
        for W, o in zip(Ws, outs):
            torch.matmul(x, W.t(), out=o)

    def looped():
        base()
        for per, o in zip(groups, outs):
            for rows, A, B, sc in per:
                xr = x.index_select(0, rows)
                o.index_add_(0, rows, torch.matmul(torch.matmul(xr, A.t()), B.t()), alpha=sc)

    res = {}
    for name, fn in (("cublas_base_gemm", base), ("torch_adapter_loop", looped)):
        for _ in range(3):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        ms = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            ms.append(a.elapsed_time(b))
        med = statistics.median(ms)
        res[name] = {"us": round(med * 1e3, 2), "tokens_per_s": round(wl.M / (med / 1e3), 1)}
    flops = sum(2 * wl.M * W.shape[0] * wl.K for W in Ws)
    res["cublas_base_gemm"]["tflops"] = round(flops / (res["cublas_base_gemm"]["us"] / 1e6) / 1e12, 1)
    res["torch_adapter_loop"]["adapters"] = int(wl.used_slots.size)
    return res


SINGLE_THREAD_WORKLOADS = ("tiny_fp32", "decode_bgmv", "decode_70b_qv")


def _oracle_rate(wl, seconds, threads):
    """Rows per second of the float64 oracle over every projection, on a
    seeded row sample sized so that one pass takes about a second."""
    import oracle

    rng = np.random.default_rng(0)
    t = time.perf_counter()
    for p in range(len(wl.projections)):
        oracle.workload_forward(wl, p, rows=[0], threads=1)
    row_s = max(time.perf_counter() - t, 1e-5)
    n = int(max(1, min(wl.M, 1.0 * threads / row_s)))
    done, reps = 0, 0
    t0 = time.perf_counter()
    while True:
        rows = np.sort(rng.choice(wl.M, size=n, replace=False))
        for p in range(len(wl.projections)):
            oracle.workload_forward(wl, p, rows=rows, threads=threads)
        done += n
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return done / dt, f"{reps} pass(es) of {n} random rows of {wl.M} x {len(wl.projections)} projection(s), " \
                      f"float64 oracle, {threads} thread(s), {dt:.1f} s"


def cpu_baseline(wl, seconds):
    import oracle

    cores = oracle.usable_cores()
    value, sample = _oracle_rate(wl, seconds, cores)
    out = {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample}
    if wl.name in SINGLE_THREAD_WORKLOADS:
        v1, s1 = _oracle_rate(wl, min(5.0, seconds / 2), 1)
        out["single_thread"] = {"value": v1, "unit": "tokens/s", "cores": 1, "sample": s1}
    return out


def max_over_ranks(values, device):
    """Each value's maximum over the ranks of the default process group (a
    job's time is its slowest rank's); the values themselves without one."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def rank0_value(value, device):
    """Rank 0's value on every rank (so that all ranks time the same number
    of steps); the value itself without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.broadcast(t, src=0)
    return type(value)(t.item())


def whole_job_rate(units_per_rank, world, ms):
    """Units processed by all ranks per second, over the slowest rank's time."""
    return units_per_rank * world / (ms / 1e3)


def run_gpu(cfg_name, args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from workloads import make_config

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    import __graft_entry__
    __graft_entry__.build()
    wl = make_config(cfg_name)
    w_bits = 8 if args.w_int8 else 4 if args.w_int4 else 0
    case = build_case(wl, device, w_bits)
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20) or (128 << 20))
    flush = L2Flush(l2, device)
    if args.steps is None:
        # about 1.5 s of forwards plus flushes
        case["call"]()
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(20):
            flush.zero_()
            case["call"]()
        torch.cuda.synchronize()
        per = (time.perf_counter() - t) / 20
        steps = int(min(20000, max(50, 1.5 / max(per, 1e-6))))
    else:
        steps = args.steps
    steps = rank0_value(steps, device)
    warmup = max(3, args.warmup)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    dev_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[local_rank]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else local_rank
    res = time_device(case, wl, steps, warmup, flush, dev_index)
    torch.cuda.synchronize()
    comparators = time_comparators(case, wl, flush) if world == 1 else None
    if world > 1:
        dist.barrier()
    total_ms = sum(res["step_ms"])
    gemm_ms = sum(res["gemm_ms"])
    shrink_ms = sum(res["shrink_ms"])
    e2e_steps = max(3, min(steps, 200))
    e2e = time_e2e(case, wl, e2e_steps, flush, device)
    e2e_streamed_ms = time_e2e_streamed(case, wl, e2e_steps)
    loads = time_adapter_loads(wl, device) if world == 1 else None
    total_ms, e2e_ms, e2e_eager_ms, e2e_streamed_ms = max_over_ranks(
        [total_ms, e2e["ms"], e2e["eager_ms"], e2e_streamed_ms], device)
    if rank != 0:
        return None

    peaks, peak_src = load_peaks()
    alg = algorithmic(wl, w_bits)
    value = whole_job_rate(wl.M * steps, world, total_ms)
    # dominant stage: the GEMM or the LoRA kernels, by their share of the
    # eager stage time
    gemm_avg_s = gemm_ms / steps / 1e3
    lora_avg_s = shrink_ms / steps / 1e3
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    gemm_dominant = gemm_ms >= shrink_ms
    if gemm_dominant:
        b, f, t = alg["gemm_bytes"], alg["gemm_flops"], gemm_avg_s
        kernel = "tc_gemm_pair_kernel (V items and LoRA steps inside)" if alg["orientation"] == "pair" \
            else "tc_gemm_lora_kernel"
    else:
        b, f, t = alg["lora_bytes"], alg["lora_flops"], lora_avg_s
        kernel = ("lora_rows_kernel, or pipe_shrink_kernel + pipe_expand_kernel (max_rank <= 128), or "
                  "group_rows_kernel + shrink_grouped_kernel + expand_grouped_kernel"
                  if alg["orientation"] == "swapped" else "shrink kernel")
    if f / b > ridge:
        roof = {"bound": "tensor", "achieved": round(f / t / 1e12, 2), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": round(b / t / 1e9, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    if gemm_dominant:
        roof["traffic"] = ncu_traffic(wl.name + (f"+int{w_bits}w" if w_bits else ""))
        roof["traffic_scope"] = "per launch of the GEMM kernel"
    else:
        roof["traffic"] = None if w_bits else ncu_traffic(wl.name, "lora")
        roof["traffic_scope"] = "per forward, the LoRA stage's kernels summed"
    roof["kernel"] = kernel
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured" else "fallback"
    roof["algorithmic_bytes_per_call"] = b
    roof["algorithmic_flops_per_call"] = f
    eager_total = sum(res["eager_ms"])
    roof["time_share"] = round((gemm_ms if gemm_dominant else shrink_ms) / eager_total, 3) if eager_total else None
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": round(total_ms / steps, 5),
        "step_ms_percentiles": {k: round(v, 5) for k, v in percentiles(res["step_ms"]).items()},
        "replay_ms_per_step": round(sum(res["replay_ms"]) / steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic (seeded, shapes and distributions of the workload)",
        "config": {
            "workload": wl.name, "M": wl.M, "K": wl.K, "N": [p.N for p in wl.projections],
            "slots": wl.num_slots, "ranks": sorted(set(int(r) for r in wl.ranks)),
            "mode": wl.mode, "distinct_adapters": alg["distinct"], "adapted_rows": alg["adapted_rows"],
            "l2": "flushed before every step (2 x L2 write, then 2 x L2 read of another buffer; outside the "
                  "timed intervals)",
            "launch": "CUDA graph of one lora_linear_forward call, replayed per step; step = events recorded "
                      "inside the graph around the forward",
            "parallelism": f"replicas x{world}",
            "base_weights": {8: "int8, one fp32 scale per row", 4: "int4 packed, one fp32 scale per row"}.get(
                w_bits, wl.dtype),
        },
        "roofline": roof,
        "stages": {
            "orientation": alg["orientation"],
            "lora_us": round(lora_avg_s * 1e6, 3),
            "lora_gbs": round(alg["lora_bytes"] / lora_avg_s / 1e9, 1) if lora_avg_s > 0 else None,
            "lora_frac_hbm": round(alg["lora_bytes"] / lora_avg_s / 1e9 / peaks["hbm_gbs"], 4)
            if lora_avg_s > 0 else None,
            "lora_bytes": alg["lora_bytes"],
            "lora_bytes_fused_form": alg["lora_bytes_fused"],
            "intermediate_bytes": alg["intermediate_bytes"],
            "gemm_us": round(gemm_avg_s * 1e6, 3),
            "gemm_tc_frac": round(alg["gemm_flops"] / gemm_avg_s / 1e12 / peaks["bf16_tflops"], 4),
            "gemm_hbm_frac": round(alg["gemm_bytes"] / gemm_avg_s / 1e9 / peaks["hbm_gbs"], 4),
            "gemm_us_percentiles": {k: round(v * 1e3, 3) for k, v in percentiles(res["gemm_ms"]).items()},
            "lora_us_percentiles": {k: round(v * 1e3, 3) for k, v in percentiles(res["shrink_ms"]).items()},
        },
        "comparators": comparators,
        "e2e": {"value": round(whole_job_rate(wl.M * e2e_steps, world, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "launch": "CUDA graph of the step (copies and forward) replayed per step",
                "eager_value": round(whole_job_rate(wl.M * e2e_steps, world, e2e_eager_ms), 1),
                "streamed_value": round(whole_job_rate(wl.M * e2e_steps, world, e2e_streamed_ms), 1),
                "streamed_launch": "two buffer sets; copy-in of step i+1 and copy-out of step i-1 on their "
                                   "own streams beside the forward of step i"},
        "adapter_load": loads,
        "gpu_launches": int(res["launches"]),
        "kernels_per_step": int(res["kernels_per_call"]),
        "eager": {"value": round(whole_job_rate(wl.M * steps, world, sum(res["eager_ms"])), 1), "unit": "tokens/s",
                  "ms_per_step": round(sum(res["eager_ms"]) / steps, 5)},
        "clocks": res["clocks"],
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    for pool in case["pools"]:
        pool.close()
    return line


# ----------------------------------------------------------------------------- reference arm

def run_reference(cfg_name, args):
    import oracle
    from workloads import make_config

    wl = make_config(cfg_name)
    cores = oracle.usable_cores()
    oracle.build()
    steps = args.steps if args.steps is not None else 10
    warmup = max(3, args.warmup)
    # calibrate: time of one row through every projection
    t = time.perf_counter()
    for p in range(len(wl.projections)):
        oracle.workload_forward(wl, p, rows=[0], threads=1)
    row_s = max(time.perf_counter() - t, 1e-4)
    budget = args.reference_seconds  # seconds of oracle work for the whole run
    rows_per_step = int(max(1, min(wl.M, budget * cores / (steps + warmup) / row_s)))
    rng = np.random.default_rng(0)

    def step():
        rows = rng.choice(wl.M, size=rows_per_step, replace=False)
        for p in range(len(wl.projections)):
            oracle.workload_forward(wl, p, rows=rows, threads=cores)

    for _ in range(warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    dt = time.perf_counter() - t0
    value = rows_per_step * steps / dt
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "tokens/s",
        "n_gpus": 1,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": round(dt / steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded, shapes and distributions of the workload)",
        "config": {"workload": wl.name, "M": wl.M, "K": wl.K, "N": [p.N for p in wl.projections],
                   "rows_per_step": rows_per_step},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows_per_step} random rows of {wl.M} per step, float64 oracle, "
                                   f"{cores} threads"},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    from workloads import CONFIG_NAMES, WIDENING_NAMES
    names = list(CONFIG_NAMES[1:]) + list(WIDENING_NAMES) if args.config == "all" else [args.config]
    if args.impl == "reference":
        if rank != 0:
            return 0
        for name in names:
            print(json.dumps(run_reference(name, args)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        for name in names:
            line = run_gpu(name, args, rank, world, local_rank)
            if line is not None:
                print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
