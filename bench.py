#!/usr/bin/env python3
"""Benchmark of the MoE dispatch / combine layout path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
layout (one or two kernels) -> dispatch -> combine, through the library's
C ABI (with --fused, layout and dispatch in one call).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload prefill]
  python bench.py --impl reference ...   (the CPU oracle, timed on host cores)

Prints ONE JSON line on rank 0.  Everything else goes to stderr.

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and torch.cuda.synchronize() on both sides.  Each step is timed on the
launching stream with one pair of CUDA events around the whole step, and the
L2 is flushed before every step, outside the events: a 256 MiB write evicts
the workload's lines, then a 256 MiB read evicts the write's dirty lines, so
that no step pays for write-backs of the flush itself; the reported
ms_per_step is the mean step time, maximum over ranks.  A second pass of K
steps with an event between stages gives the per-stage times and the
roofline's kernel time.  With N > 1 (torchrun)
every rank runs an independent replica of the workload (weak scaling; the
path has no cross-rank step on a single-GPU-per-problem layout).
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("dispatch+combine tokens/s and HBM GB/s (% of 8 TB/s) at DeepSeek-V3 "
          "shape, 1 GB300")
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20  # twice the GB300's L2
# (t, k) pairs up to which the layout is one launch (kSmallLayoutPairs in
# combine_get_layout_gb300/csrc/ep_internal.h); used to count launches
SMALL_LAYOUT_PAIRS = 4096
SMALL_LAYOUT_CTAS = 152     # its CTAs (kSmallLayoutCtas)
SMALL_OWN_PAIRS = 64        # pairs a CTA may own to dispatch them (kSmallOwnPairs)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse_args():
    import workloads

    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(workloads.WORKLOADS), default="prefill")
    p.add_argument("--zero-padding", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-budget-s", type=float, default=12.0)
    p.add_argument("--bias", type=int, choices=[0, 1, 2], default=0,
                   help="combine epilogue: number of bf16 bias tensors")
    p.add_argument("--return-weights", action="store_true",
                   help="combine epilogue: also return the per-(t,k) gate weights")
    p.add_argument("--fp8-scales", choices=["row", "col"], default="row",
                   help="FP8 scale layout (col: column-major, TMA-aligned)")
    p.add_argument("--fp8-prequant", action="store_true",
                   help="FP8 dispatch of pre-quantised rows + scales (bit copies)")
    p.add_argument("--pass", dest="pass_", choices=["forward", "backward", "ranks"],
                   default="forward",
                   help="forward: layout, dispatch, combine; backward: layout, "
                        "combine backward (with gate gradients), dispatch backward; "
                        "ranks: layout, dispatch to ranks, expand, reduce to ranks, "
                        "combine over ranks (the non-expanded path)")
    p.add_argument("--e2e-chunks", type=int, default=0,
                   help="token chunks of the host-buffer entry points in the e2e leg "
                        "when they copy (copies of later chunks overlap the kernels of "
                        "earlier ones); 0 = chunks of about 48 MiB of rows, at least 2")
    p.add_argument("--e2e-depth", type=int, default=4,
                   help="batches in flight in the pipelined e2e leg (one stream and one "
                        "set of device buffers each)")
    p.add_argument("--e2e-graph", choices=["auto", "on", "off"], default="auto",
                   help="pipelined e2e leg: capture 64 consecutive steps' calls into one "
                        "CUDA graph and replay it (auto: when the kernels read and write the "
                        "host rows in place, i.e. small batches, where the host's per-step "
                        "calls would otherwise set the pace)")
    p.add_argument("--e2e-transfer", choices=["auto", "direct", "chunked", "copies"],
                   default="auto",
                   help="e2e leg: direct = the kernels read x from and write y to pinned "
                        "host memory in place (host-buffer entry points, 0 chunks); "
                        "chunked = the same entry points copying token chunks; copies = "
                        "whole-buffer copies on the stream around the device entry points; "
                        "auto = direct one step at a time, and for two batches in flight "
                        "chunked when a batch's rows span two 4 MiB chunks, else direct "
                        "(copies with the combine epilogue or FP8 input options, which have "
                        "device entry points only; those run one step at a time)")
    p.add_argument("--fused", action="store_true",
                   help="forward pass: layout and dispatch through ep_layout_and_dispatch "
                        "(one kernel for small inputs)")
    p.add_argument("--graph", action="store_true",
                   help="replay each step from one captured CUDA graph (removes host "
                        "launch overhead; for latency-bound sizes)")
    return p.parse_args()


# ---------------------------------------------------------------------------
# accounting
# ---------------------------------------------------------------------------

def algorithmic_bytes(wl, n_rows: int, nbias: int = 0, return_weights: bool = False,
                      prequant: bool = False) -> dict:
    """Bytes the method must move (each source row once, each destination row
    once, plus route metadata), per launch."""
    T, H, K, E, R = wl.num_tokens, wl.hidden, wl.num_topk, wl.num_experts, wl.num_ranks
    rowbytes = (H + 4 * (H // 128)) if wl.use_fp8_dispatch else 2 * H
    src_bytes = T * rowbytes if prequant else T * H * 2
    dispatch = src_bytes + n_rows * rowbytes + T * K * (4 + 4) + n_rows * 4
    combine = n_rows * H * 2 + T * H * 2 + T * K * (4 + 4) + nbias * T * H * 2
    if return_weights:
        combine += T * K * (4 + 4)
    layout = T * K * 8 + T * K * 4 + n_rows * 8 + T * R
    return {"dispatch": dispatch, "combine": combine, "layout": layout}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {
    "dispatch_bf16_kernel": "combine_get_layout_gb300/csrc/dispatch.cu",
    "dispatch_fp8_kernel": "combine_get_layout_gb300/csrc/dispatch.cu",
    "combine_kernel": "combine_get_layout_gb300/csrc/combine.cu",
    "combine_backward_kernel": "combine_get_layout_gb300/csrc/combine.cu",
    "dispatch_ranks_kernel": "combine_get_layout_gb300/csrc/ranks.cu",
    "expand_kernel": "combine_get_layout_gb300/csrc/ranks.cu",
    "reduce_ranks_kernel": "combine_get_layout_gb300/csrc/ranks.cu",
}


def source_sha(kernel: str) -> str:
    """First 16 hex digits of the SHA-256 of the kernel's .cu file followed by
    the shared headers it includes (csrc/*.cuh, csrc/*.h, in name order)."""
    h = hashlib.sha256()
    with open(os.path.join(ROOT, KERNEL_SOURCES[kernel]), "rb") as f:
        h.update(f.read())
    csrc = os.path.join(ROOT, "combine_get_layout_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """dram bytes per launch recorded from an ncu capture in profiles/, if the
    kernel's source is unchanged since (source hash recorded beside it)."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    if kernel not in KERNEL_SOURCES:
        return None
    want = source_sha(kernel)
    pat = re.compile(r"TRAFFIC kernel=(\S+) workload=(\S+) bytes_per_launch=(\d+) "
                     r"source_sha256=(\S+)")
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, fn)) as f:
            for line in f:
                m = pat.search(line)
                if m and m.group(1) == kernel and m.group(2) == workload and m.group(4) == want:
                    return int(m.group(3))
    return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", device_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as e:  # no nvidia-smi
            log(f"clock sampler unavailable: {e}")
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, smax = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            self.samples.append((time.perf_counter(), sm, smax, parts[4:8]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        if self.proc is None:
            return None
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        note = "samples inside the timed region"
        if not inside and self.samples:
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda s: abs(s[0] - mid))]
            note = "timed region shorter than the sampling period: nearest sample"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({n for s in inside for n, v in zip(self.NAMES, s[3])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "samples": len(inside), "note": note}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def job_throughput(tokens_per_rank: int, ms_local: float, world: int, device=None):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's step
    time.  Returns (value, ms_max)."""
    ms = reduce_max(ms_local, world, device)
    return tokens_per_rank * world / (ms / 1e3), ms


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline / reference arm)
# ---------------------------------------------------------------------------

def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_step_fn(wl, inp, nthreads=1):
    """One oracle step over the given inputs: layout -> dispatch -> combine
    (identity experts: combine reads the dispatched rows).  Output buffers are
    allocated once, outside the timing.  nthreads > 1: dispatch and combine
    run on token slices in that many threads (the oracle's own functions, same
    results); the layout stays sequential."""
    import numpy as np

    import oracle

    T, H, K = wl.num_tokens, wl.hidden, wl.num_topk
    cap = oracle.recv_capacity(T, K, wl.num_experts, wl.expert_alignment)
    recv_x = np.zeros((cap, H), np.uint16)
    recv_w = np.zeros(cap, np.float32)
    y = np.zeros((T, H), np.uint16)
    if wl.use_fp8_dispatch:
        recv_q = np.zeros((cap, H), np.uint8)
        recv_s = np.zeros((cap, H // 128), np.float32)

    def step():
        lay = oracle.layout(inp["topk_idx"], wl.num_experts, wl.num_ranks,
                            wl.expert_alignment, cap=cap)
        if wl.use_fp8_dispatch:
            # FP8 payload for the wire, bf16 rows for the experts' identity output
            oracle.dispatch_fp8(inp["x"], inp["topk_weights"], lay,
                                out=(recv_q, recv_s, recv_w), nthreads=nthreads)
        oracle.dispatch_bf16(inp["x"], inp["topk_weights"], lay, out=(recv_x, recv_w),
                             nthreads=nthreads)
        oracle.combine(recv_x, inp["topk_weights"], lay["slot_of"], out=y, nthreads=nthreads)
        return y

    return step


def time_oracle(wl, inp, budget_s, min_steps=1, max_steps=1000, nthreads=1):
    step = oracle_step_fn(wl, inp, nthreads)
    times = []
    t_start = time.perf_counter()
    while len(times) < max_steps:
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
        if len(times) >= min_steps and time.perf_counter() - t_start >= budget_s:
            break
    return times


def subsample(inp, wl, n_tokens):
    import workloads

    sub = {k: v[:n_tokens] for k, v in inp.items()}
    return sub, wl.with_(num_tokens=n_tokens)


def cpu_baseline(wl, inp, budget_s):
    """The oracle as it stands on a bounded sample: on all the host's cores
    (dispatch and combine on token slices, one thread a core; layout
    sequential), and single-threaded beside it."""
    n = wl.num_tokens
    cores = host_cores()
    mt = time_oracle(wl, inp, budget_s / 2, nthreads=cores)
    st = time_oracle(wl, inp, budget_s / 2)
    what = f"(T={n}; layout+dispatch+combine, identity experts)"
    return {"value": n * len(mt) / sum(mt), "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{len(mt)} full step(s) of the same workload {what}, "
                      f"{sum(mt):.1f} s wall on {cores} threads (dispatch and combine "
                      "split over tokens; layout sequential)",
            "single_thread": {"value": n * len(st) / sum(st), "unit": "tokens/s", "cores": 1,
                              "sample": f"{len(st)} full step(s) {what}, {sum(st):.1f} s "
                                        "on 1 thread"}}


def run_reference(args):
    """The oracle timed on the host cores: the reference arm of this path."""
    import numpy as np

    import workloads

    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    wl = workloads.WORKLOADS[args.workload]
    inp = workloads.make_inputs(wl, seed=0)
    cores = host_cores()
    # size each step's sample so that warm-up + timed steps take ~60 s at most
    cal_n = min(wl.num_tokens, 64 * cores)
    s_inp, s_wl = subsample(inp, wl, cal_n)
    t = time_oracle(s_wl, s_inp, 0.0, min_steps=2, max_steps=2, nthreads=cores)
    per_token = max(min(t) / cal_n, 1e-7)
    budget = 60.0 / max(1, args.steps + args.warmup)
    n = int(max(16, min(wl.num_tokens, budget / per_token)))
    s_inp, s_wl = subsample(inp, wl, n)
    step = oracle_step_fn(s_wl, s_inp, nthreads=cores)
    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = n / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": path_dtype(wl),
        "data": "synthetic (seeded router simulation)",
        "config": workload_config(wl, extra={"sample_tokens_per_step": n}),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {n} of {wl.num_tokens} tokens per step "
                                   "(same E/K/R/H), layout+dispatch+combine, identity experts; "
                                   f"dispatch and combine on {cores} threads (token slices), "
                                   "layout sequential"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def e2e_transfer(requested: str, device_entry_points_only: bool) -> str:
    """How the e2e leg moves x and y: "direct" (the host-buffer entry points
    with 0 chunks: the kernels read and write pinned host memory in place),
    "chunked" (the same entry points copying token chunks) or "copies"
    (whole-buffer copies around the device entry points).  "auto" is
    direct.  Options that only the device entry points offer (the combine
    epilogue, the FP8 input options) force copies."""
    if requested not in ("auto", "direct", "chunked", "copies"):
        raise ValueError(f"unknown e2e transfer {requested!r}")
    if device_entry_points_only:
        return "copies"
    return "direct" if requested == "auto" else requested


def pipelined_transfer(requested: str, device_entry_points_only: bool, row_bytes: int) -> str:
    """How the pipelined e2e leg (two batches in flight) moves x and y, or
    None where it does not run (options that only the device entry points
    offer).  "auto": the host-buffer entry points copying token chunks when
    a batch's rows span at least two 4 MiB chunks -- then one batch's rows
    going out and the next batch's coming in use the two copy engines at
    once -- else direct (small batches: the kernels read and write the host
    rows in place)."""
    if requested not in ("auto", "direct", "chunked", "copies"):
        raise ValueError(f"unknown e2e transfer {requested!r}")
    if device_entry_points_only:
        return None
    if requested != "auto":
        return requested
    return "chunked" if row_bytes >= 2 * (4 << 20) else "direct"


# steps of the pipelined e2e leg captured into one CUDA graph when it replays
E2E_GRAPH_STEPS = 64


def e2e_chunk_count(requested: int, row_bytes: int) -> int:
    """Token chunks for the copying host-buffer mode: `requested` when set,
    else chunks of about 48 MiB of x rows, 2 to 8 of them (measured on the
    pipelined leg: fewer, larger chunks win up to ~60 MB a chunk)."""
    if requested > 0:
        return requested
    return max(2, min(8, row_bytes // (48 << 20)))


def route_views(buf, T: int, K: int):
    """A step's routes (int64 [T, K]) followed by its gate weights (fp32
    [T, K]) in one uint8 buffer of T*K*12 bytes, so that one copy moves
    both.  Returns the two views."""
    import torch

    n = T * K
    return (buf[: n * 8].view(torch.int64).view(T, K),
            buf[n * 8: n * 12].view(torch.float32).view(T, K))


def e2e_headline(sequential: dict, pipelined) -> dict:
    """The e2e line's own figures: the faster way to drive the same calls
    (batches in flight -- graph-replayed for small batches -- or one step at
    a time), named in `mode`; the slower leg stays listed beside it."""
    best = (pipelined if pipelined is not None and pipelined["value"] >= sequential["value"]
            else sequential)
    return {"value": best["value"], "ms_per_step": best["ms_per_step"],
            "mode": "pipelined" if best is pipelined else "sequential",
            "transfer": best["transfer"], "pipelining": best.get("pipelining"),
            "launch": best.get("launch", "the calls of each step from the host"),
            "choice": "value and ms_per_step are the faster of the legs listed"}


def path_dtype(wl) -> str:
    """The arithmetic of the path: E4M3 rows (fp32 quantisation) or bf16 bit
    copies on dispatch; the combine folds bf16 rows in fp32 either way."""
    return "fp8_e4m3" if wl.use_fp8_dispatch else "bf16"


def pipelined_e2e(ep, ccfg, cfg, T, K, H, wl, device, stream, x_h, route_h, recv_x0, Y_d,
                  chunks, steps, warmup, world, y_want, copies=False, depth=2, graph_steps=0):
    """End to end with `depth` batches in flight, as a serving loop runs:
    step i goes on stream i % depth with its own device buffers and host
    output rows, so one step's combine (y over the host link to the host)
    overlaps later steps' layout and dispatch (x over the link to the
    device); a step waits only for the step `depth` before it.  Every
    step copies its routes and weights in (one packed copy), reads x from
    and writes y to pinned host memory through the host-buffer entry points
    (copies=True: copies x to the device and y back itself, on the step's
    stream, around ep_dispatch / ep_combine on device buffers, so that the
    two copy directions run on their own copy engines).  graph_steps > 0: the
    same calls for that many consecutive steps (rounded to a multiple of
    `depth`) are captured once into a CUDA graph, which is replayed, so the
    host enqueues one launch per graph instead of each step's calls.  No L2
    flush: a step touches far more HBM than L2 holds, or (small batches)
    the steps run back to back anyway.  Returns the throughput over at
    least `steps` steps (one event pair around all of them)."""
    import ctypes

    import torch

    p = lambda t: None if t is None else t.data_ptr()
    cap = cfg.capacity
    # no more slots than steps in either run, so that every slot's output is
    # written (and checked below)
    depth = max(1, min(depth, max(steps, warmup)))

    class Slot:
        pass

    slots = []
    for k in range(depth):
        sl = Slot()
        # (a captured step needs streams of its own: not the legacy default)
        sl.stream = stream if k == 0 and not graph_steps else torch.cuda.Stream(device)
        sl.sptr = ctypes.c_void_p(sl.stream.cuda_stream)
        sl.route = torch.empty_like(route_h, device=device)
        sl.idx, sl.w = route_views(sl.route, T, K)
        sl.L = ep.Layout(cfg, device=device)
        sl.rx = torch.empty((cap, H), dtype=torch.uint8 if wl.use_fp8_dispatch else torch.bfloat16,
                            device=device)
        sl.rs = (torch.empty((cap, H // 128), dtype=torch.float32, device=device)
                 if wl.use_fp8_dispatch else None)
        sl.rw = torch.empty(cap, dtype=torch.float32, device=device)
        staged = chunks or copies
        sl.x_d = torch.empty((T, H), dtype=torch.bfloat16, device=device) if staged else None
        sl.y_d = torch.empty((T, H), dtype=torch.bfloat16, device=device) if staged else None
        sl.y_h = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
        # experts: identity for bf16 rows, the seeded expert-output buffer for E4M3
        sl.ident = sl.rx if recv_x0 is not None else Y_d
        slots.append(sl)

    def step(sl):
        with torch.cuda.stream(sl.stream):
            if copies:
                sl.x_d.copy_(x_h, non_blocking=True)
            sl.route.copy_(route_h, non_blocking=True)
        st = ep.ep_get_layout(ccfg, T, p(sl.idx), sl.L.c, None, sl.sptr)
        assert st == 0, ep.ep_status_str(st)
        if copies:
            st = ep.ep_dispatch(ccfg, sl.L.c, p(sl.x_d), p(sl.w), p(sl.rx), p(sl.rs), p(sl.rw),
                                sl.sptr)
        else:
            st = ep.ep_dispatch_from_host(ccfg, sl.L.c, x_h.data_ptr(), p(sl.x_d), p(sl.w),
                                          p(sl.rx), p(sl.rs), p(sl.rw), chunks, sl.sptr)
        assert st == 0, ep.ep_status_str(st)
        if copies:
            st = ep.ep_combine(ccfg, sl.L.c, p(sl.ident), p(sl.w), p(sl.y_d), sl.sptr)
            assert st == 0, ep.ep_status_str(st)
            with torch.cuda.stream(sl.stream):
                sl.y_h.copy_(sl.y_d, non_blocking=True)
        else:
            st = ep.ep_combine_to_host(ccfg, sl.L.c, p(sl.ident), p(sl.w), p(sl.y_d),
                                       sl.y_h.data_ptr(), chunks, sl.sptr)
            assert st == 0, ep.ep_status_str(st)

    def run(n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(slots[0].stream)
        for sl in slots[1:]:
            sl.stream.wait_event(a)
        for i in range(n):
            step(slots[i % depth])
        for sl in slots[1:]:
            join = torch.cuda.Event()
            join.record(sl.stream)
            slots[0].stream.wait_event(join)
        b.record(slots[0].stream)
        return a, b, n

    launch = "the calls of each step from the host"
    if graph_steps > 0:
        G = depth * max(1, graph_steps // depth)
        run(depth)   # one-time set-up happens outside the capture
        torch.cuda.synchronize()
        cap_s = torch.cuda.Stream(device)
        cap_s.wait_stream(torch.cuda.current_stream(device))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap_s):
            fork = torch.cuda.Event()
            fork.record(cap_s)
            for sl in slots:
                sl.stream.wait_event(fork)
            for i in range(G):
                step(slots[i % depth])
            for sl in slots:
                join = torch.cuda.Event()
                join.record(sl.stream)
                cap_s.wait_event(join)
        torch.cuda.synchronize()
        launch = f"one CUDA graph of {G} steps (their calls captured once), replayed"

        def run(n):  # noqa: F811 -- whole replays covering at least n steps
            reps = max(1, -(-n // G))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(cap_s)
            with torch.cuda.stream(cap_s):
                for _ in range(reps):
                    graph.replay()
            b.record(cap_s)
            return a, b, reps * G

    run(warmup)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    a, b, done = run(steps)
    torch.cuda.synchronize()
    barrier(world)
    ms = reduce_max(a.elapsed_time(b) / done, world, device)
    for sl in slots:
        assert ep.ep_check_error(sl.L.c, sl.sptr) == 0
        # same inputs as the sequential leg: the same rows come back
        assert torch.equal(sl.y_h.view(torch.int16), y_want.view(torch.int16))
    return {"value": T * world / (ms / 1e3), "ms_per_step": ms, "steps_timed": done,
            "launch": launch,
            "pipelining": (f"{depth} batches in flight on {depth} streams (later steps' "
                           "layout and dispatch overlap a step's combine; each step still "
                           "moves its own x in and y out); one event pair around all steps, "
                           "no L2 flush")}


def workload_config(wl, extra=None):
    d = {
        "workload": f"{wl.name}: T={wl.num_tokens} H={wl.hidden} E={wl.num_experts} "
                    f"K={wl.num_topk} R={wl.num_ranks} A={wl.expert_alignment} "
                    f"{'fp8' if wl.use_fp8_dispatch else 'bf16'} dispatch, bf16 combine",
        "num_tokens": wl.num_tokens, "hidden": wl.hidden, "num_experts": wl.num_experts,
        "num_topk": wl.num_topk, "num_ranks": wl.num_ranks,
        "expert_alignment": wl.expert_alignment,
        "dispatch_format": "fp8_e4m3_1x128" if wl.use_fp8_dispatch else "bf16",
        "combine_accumulate": "f32",
    }
    if extra:
        d.update(extra)
    return d


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import ctypes

    import numpy as np
    import torch

    import workloads

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)
    if rank == 0:
        import importlib.util

        spec = importlib.util.spec_from_file_location(
            "ep_build_lib", os.path.join(ROOT, "combine_get_layout_gb300", "build_lib.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        if not mod.up_to_date():
            mod.build()
    barrier(world)
    import combine_get_layout_gb300 as ep

    wl = workloads.WORKLOADS[args.workload]
    inp = workloads.make_inputs(wl, seed=rank)
    n_rows = int((inp["topk_idx"] >= 0).sum())
    T, H, K = wl.num_tokens, wl.hidden, wl.num_topk
    cfg = ep.Config(T, H, K, wl.num_experts, wl.num_ranks, wl.expert_alignment,
                    wl.use_fp8_dispatch, args.zero_padding)
    cap = cfg.capacity
    ccfg = cfg.c()

    x_d = torch.from_numpy(inp["x"].view(np.int16)).to(device).view(torch.bfloat16)
    route_d = torch.empty(T * K * 12, dtype=torch.uint8, device=device)
    idx_d, w_d = route_views(route_d, T, K)
    idx_d.copy_(torch.from_numpy(inp["topk_idx"]))
    w_d.copy_(torch.from_numpy(inp["topk_weights"]))
    g = torch.Generator(device=device)
    g.manual_seed(1234 + rank)
    Y_d = torch.randn((cap, H), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    L = ep.Layout(cfg, device=device, with_ranks=args.pass_ == "ranks")
    rx_dtype = torch.uint8 if wl.use_fp8_dispatch else torch.bfloat16
    recv_x = torch.empty((cap, H), dtype=rx_dtype, device=device)
    recv_s = (torch.empty((cap, H // 128), dtype=torch.float32, device=device)
              if wl.use_fp8_dispatch else None)
    recv_w = torch.empty(cap, dtype=torch.float32, device=device)
    y_d = torch.empty((T, H), dtype=torch.bfloat16, device=device)
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def l2_flush():
        flush_w.zero_()
        flush_r.sum()
    stream = torch.cuda.current_stream(device)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    fn_stream = [sptr]  # the stream the library calls below launch on
    p = lambda t: None if t is None else t.data_ptr()

    def layout():
        st = ep.ep_get_layout(ccfg, T, p(idx_d), L.c, None, fn_stream[0])
        assert st == 0, ep.ep_status_str(st)

    fp8_opts = wl.use_fp8_dispatch and (args.fp8_scales == "col" or args.fp8_prequant)
    if fp8_opts and args.fp8_scales == "col":
        recv_s = torch.empty((H // 128, ep.ep_scale_ld(ccfg)), dtype=torch.float32,
                             device=device)
    xq_d = xs_d = None
    if wl.use_fp8_dispatch and args.fp8_prequant:  # synthetic E4M3 rows + scales
        xq_d = torch.randint(0, 0x7E, (T, H), generator=g, device=device,
                             dtype=torch.int32).to(torch.uint8)
        xs_d = torch.rand((T, H // 128), generator=g, device=device)
    epilogue = args.bias > 0 or args.return_weights
    biases = [torch.randn((T, H), generator=g, device=device).to(torch.bfloat16)
              for _ in range(args.bias)]
    comb_w = (torch.empty((T, K), dtype=torch.float32, device=device)
              if args.return_weights else None)

    def dispatch(xsrc):
        if fp8_opts:
            st = ep.ep_dispatch_fp8(ccfg, L.c, None if xq_d is not None else p(xsrc),
                                    p(xq_d), p(xs_d), p(w_d), p(recv_x), p(recv_s),
                                    args.fp8_scales == "col", p(recv_w), fn_stream[0])
        else:
            st = ep.ep_dispatch(ccfg, L.c, p(xsrc), p(w_d), p(recv_x), p(recv_s), p(recv_w),
                                fn_stream[0])
        assert st == 0, ep.ep_status_str(st)

    def combine(Y, out):
        if epilogue:
            b0 = p(biases[0]) if len(biases) > 0 else None
            b1 = p(biases[1]) if len(biases) > 1 else None
            st = ep.ep_combine_epilogue(ccfg, L.c, p(Y), p(w_d), b0, b1, p(recv_w),
                                        p(out), p(comb_w), fn_stream[0])
        else:
            st = ep.ep_combine(ccfg, L.c, p(Y), p(w_d), p(out), fn_stream[0])
        assert st == 0, ep.ep_status_str(st)

    # Stages of one step: (name, callable, kernels launched).  The layout is
    # one kernel for at most SMALL_LAYOUT_PAIRS (t, k) pairs, else count +
    # assign.
    lay_launches = 1 if T * K <= SMALL_LAYOUT_PAIRS else 2
    # one kernel for layout and dispatch (see ep_layout_and_dispatch)
    fused_small = (0 < T * K <= SMALL_LAYOUT_PAIRS
                   and -(-T // SMALL_LAYOUT_CTAS) * K <= SMALL_OWN_PAIRS)
    one = 1 if T > 0 else 0
    zp_extra = 1 if args.zero_padding else 0
    backward = args.pass_ == "backward"
    ranks_pass = args.pass_ == "ranks"
    if backward:
        dy_d = torch.randn((T, H), generator=g, device=device).to(torch.bfloat16)
        grad_rw = torch.randn(cap, generator=g, device=device)
        grad_Y = torch.empty((cap, H), dtype=torch.bfloat16, device=device)
        grad_w = torch.empty((T, K), dtype=torch.float32, device=device)
        grad_x = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        grad_w2 = torch.empty((T, K), dtype=torch.float32, device=device)

        def combine_bwd():
            st = ep.ep_combine_backward(ccfg, L.c, p(dy_d), p(w_d), p(Y_d), p(grad_Y),
                                        p(grad_w), fn_stream[0])
            assert st == 0, ep.ep_status_str(st)

        def dispatch_bwd():
            st = ep.ep_dispatch_backward(ccfg, L.c, p(grad_Y), p(grad_rw), p(grad_x),
                                         p(grad_w2), fn_stream[0])
            assert st == 0, ep.ep_status_str(st)

        stages = [("layout", layout, lay_launches),
                  ("combine_backward", combine_bwd, one + zp_extra),
                  ("dispatch_backward", dispatch_bwd, one)]
    elif ranks_pass:
        nrows = ep.ep_rank_rows_capacity(ccfg)
        rank_x = torch.empty((nrows, H), dtype=torch.bfloat16, device=device)
        rank_idx = torch.empty((nrows, K), dtype=torch.int32, device=device)
        rank_w = torch.empty((nrows, K), dtype=torch.float32, device=device)
        rank_y = torch.empty((nrows, H), dtype=torch.bfloat16, device=device)

        def dispatch_ranks():
            st = ep.ep_dispatch_ranks(ccfg, L.c, p(x_d), p(idx_d), p(w_d), p(rank_x),
                                      p(rank_idx), p(rank_w), fn_stream[0])
            assert st == 0, ep.ep_status_str(st)

        def expand():
            st = ep.ep_expand(ccfg, L.c, p(idx_d), p(rank_x), p(rank_w), p(recv_x),
                              p(recv_w), fn_stream[0])
            assert st == 0, ep.ep_status_str(st)

        def reduce_ranks():
            st = ep.ep_reduce_ranks(ccfg, L.c, p(idx_d), p(Y_d), p(w_d), p(rank_y),
                                    fn_stream[0])
            assert st == 0, ep.ep_status_str(st)

        def combine_ranks():
            st = ep.ep_combine_ranks(ccfg, L.c, p(rank_y), p(y_d), fn_stream[0])
            assert st == 0, ep.ep_status_str(st)

        stages = [("layout", layout, lay_launches),
                  ("dispatch_ranks", dispatch_ranks, one),
                  ("expand", expand, one + zp_extra),
                  ("reduce_ranks", reduce_ranks, one),
                  ("combine_ranks", combine_ranks, one)]
    elif args.fused:
        if fp8_opts:
            raise SystemExit("--fused takes no FP8 scale-layout or pre-quantised options")

        def layout_dispatch():
            st = ep.ep_layout_and_dispatch(ccfg, T, p(idx_d), L.c, p(x_d), p(w_d), p(recv_x),
                                           p(recv_s), p(recv_w), fn_stream[0])
            assert st == 0, ep.ep_status_str(st)

        stages = [("layout_dispatch", layout_dispatch,
                   (1 if fused_small else lay_launches + one) + zp_extra),
                  ("combine", lambda: combine(Y_d, y_d), one)]
    else:
        stages = [("layout", layout, lay_launches),
                  ("dispatch", lambda: dispatch(x_d), one + zp_extra),
                  ("combine", lambda: combine(Y_d, y_d), one)]
    launches_per_step = sum(n for _, _, n in stages)
    runners = [fn for _, fn, _ in stages]
    step_runners = runners   # what one timed step runs, in order
    if args.graph:
        # warm up (one-time per-device set-up happens outside any capture)
        for fn in runners:
            fn()
        torch.cuda.synchronize()

        def capture(fns):
            g_ = torch.cuda.CUDAGraph()
            cap_stream = torch.cuda.Stream(device)
            cap_stream.wait_stream(stream)
            with torch.cuda.graph(g_, stream=cap_stream):
                fn_stream[0] = ctypes.c_void_p(cap_stream.cuda_stream)
                for fn in fns:
                    fn()
                fn_stream[0] = sptr
            return g_

        # one graph per step for the timed steps; one per stage for the
        # stage-time pass (which needs events between stages)
        graphs = [capture([fn]) for fn in runners]
        step_graph = capture(runners)
        torch.cuda.synchronize()
        runners = [g_.replay for g_ in graphs]
        step_runners = [step_graph.replay]

    # ---- device-resident timing ---------------------------------------------
    dev_id = str(local)
    try:
        dev_id = "GPU-" + str(torch.cuda.get_device_properties(device).uuid).replace("GPU-", "")
    except Exception:
        pass
    sampler = ClockSampler(dev_id)
    for _ in range(args.warmup):
        l2_flush()
        for fn in step_runners:
            fn()
    torch.cuda.synchronize()
    assert ep.ep_check_error(L.c, sptr) == 0
    ns = len(runners)
    # The timed steps carry events only around the whole step, so that the
    # library's kernels chain from stage to stage as a caller's would.
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
           for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        l2_flush()
        sev[i][0].record(stream)
        for fn in step_runners:
            fn()
        sev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    # Stage times from a second pass with an event between stages (an event
    # there breaks the chaining, so its stages add up to more than a step).
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(ns + 1)]
          for _ in range(args.steps)]
    for i in range(args.steps):
        l2_flush()
        e = ev[i]
        for j, fn in enumerate(runners):
            e[j].record(stream)
            fn()
        e[ns].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    # What the layout adds to the chained step: the same steps with the layout
    # left out (dispatch and combine reuse the layout computed above), events
    # around each step as in the timed pass.
    hoisted_ms = None
    if stages[0][0] == "layout":
        hev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
               for _ in range(args.steps)]
        for i in range(args.steps):
            l2_flush()
            hev[i][0].record(stream)
            for fn in runners[1:]:
                fn()
            hev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        hoisted_ms = statistics.mean(a.elapsed_time(b_) for a, b_ in hev)
    # Steady state: the same steps back to back with no flush between them,
    # one event pair around all K, so that each step's write-back of the
    # lines it left dirty in L2 lands inside the timing (of the next step).
    for _ in range(args.warmup):
        for fn in step_runners:
            fn()
    torch.cuda.synchronize()
    barrier(world)
    ss = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ss[0].record(stream)
    for i in range(args.steps):
        for fn in step_runners:
            fn()
    ss[1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.perf_counter()
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    stage_ms = {name: [e[j].elapsed_time(e[j + 1]) for e in ev]
                for j, (name, _, _) in enumerate(stages)}
    step_ms = [a.elapsed_time(b_) for a, b_ in sev]
    ms_local = statistics.mean(step_ms)
    value, ms = job_throughput(T, ms_local, world, device)

    peak, peak_src = load_peaks()
    n_rank_rows = int(L.tokens_per_rank.sum()) if ranks_pass else 0
    if backward:
        b = {"combine_backward": T * H * 2 + 2 * n_rows * H * 2 + T * K * (4 + 4 + 4),
             "dispatch_backward": n_rows * H * 2 + T * H * 2 + T * K * (4 + 4 + 4)}
        kernels = {"combine_backward": "combine_backward_kernel",
                   "dispatch_backward": "combine_kernel"}
    elif ranks_pass:
        b = {"dispatch_ranks": T * H * 2 + n_rank_rows * (H * 2 + K * 8) + T * K * 12,
             "expand": n_rank_rows * H * 2 + n_rows * (H * 2 + 4) + T * K * 16,
             "reduce_ranks": n_rows * H * 2 + n_rank_rows * H * 2 + T * K * 16,
             "combine_ranks": n_rank_rows * H * 2 + T * H * 2 + T * wl.num_ranks * 4}
        kernels = {"dispatch_ranks": "dispatch_ranks_kernel", "expand": "expand_kernel",
                   "reduce_ranks": "reduce_ranks_kernel", "combine_ranks": "combine_kernel"}
    else:
        b = algorithmic_bytes(wl, n_rows, args.bias, args.return_weights,
                              wl.use_fp8_dispatch and args.fp8_prequant)
        kernels = {"dispatch": "dispatch_fp8_kernel" if wl.use_fp8_dispatch
                   else "dispatch_bf16_kernel", "combine": "combine_kernel"}
        if args.fused:
            b["layout_dispatch"] = b["dispatch"]
            kernels["layout_dispatch"] = ("layout_small_kernel" if fused_small
                                          else kernels["dispatch"])
    streaming = [name for name, _, _ in stages if name != "layout"]
    avg = {n: statistics.mean(stage_ms[n]) for n in streaming}
    med = {n: statistics.median(stage_ms[n]) for n in streaming}
    gbs = {n: b[n] / (avg[n] * 1e-3) / 1e9 for n in streaming}
    dom = max(streaming, key=lambda n: avg[n])
    dom_kernel = kernels[dom]
    achieved = gbs[dom]
    # the profile key names the pass when it is not the forward one
    traffic = profiled_traffic(dom_kernel, wl.name if args.pass_ == "forward"
                               else f"{wl.name}:{args.pass_}")
    roofline = {"bound": "hbm", "kernel": dom_kernel, "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)" if peak_src == "measured"
                else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": b[dom]}
    ss_value, ss_ms = job_throughput(T, ss[0].elapsed_time(ss[1]) / args.steps, world, device)
    touched = sum(b[n] for n in streaming)
    steady = {"value": ss_value, "unit": "tokens/s", "ms_per_step": ss_ms,
              "timing": (f"{args.steps} steps back to back, no L2 flush between them, one "
                         "event pair around all of them (each step's L2 write-back lands "
                         "inside the timing)"),
              "fits_in_l2": touched < 126 * 2**20}
    if steady["fits_in_l2"]:
        steady["note"] = ("the bytes one step touches fit in L2: later steps find their "
                          "inputs cached, so this is not a DRAM-bound figure")
    stream_ms = sum(avg.values())
    breakdown = {"layout_us": (1e3 * statistics.mean(stage_ms["layout"]) if "layout" in stage_ms
                               else None)}
    if hoisted_ms is not None:
        breakdown.update({
            "step_without_layout_us": 1e3 * hoisted_ms,
            "layout_in_step_us": 1e3 * (ms_local - hoisted_ms),
            "layout_in_step_note": ("step time minus the same step with the layout left "
                                    "out: the layout's cost on the chained critical path"),
        })
    for n in streaming:
        breakdown.update({f"{n}_us": 1e3 * avg[n], f"{n}_median_us": 1e3 * med[n],
                          f"{n}_tokens_per_s": T * world / (avg[n] * 1e-3),
                          f"{n}_gbs": gbs[n], f"{n}_pct_of_8tbs": 100 * gbs[n] / NOMINAL_HBM_GBS,
                          f"{n}_frac_of_measured": gbs[n] / peak})
    breakdown.update({
        "streaming_stages_tokens_per_s": T * world / (stream_ms / 1e3),
        "streaming_stages_gbs": sum(b[n] for n in streaming) / (stream_ms * 1e-3) / 1e9,
        "rows_dispatched": n_rows, "capacity_rows": cap,
        "wall_s_timed_region": t1 - t0,
    })
    if ranks_pass:
        breakdown["rank_rows"] = n_rank_rows
    if args.zero_padding and not (backward or ranks_pass):
        # the dispatch stage also clears the alignment gap rows: their bytes,
        # counted apart from the algorithmic bytes above
        used = int(L.expert_start[-1])
        rowbytes = (H + 4 * (H // 128)) if wl.use_fp8_dispatch else 2 * H
        pad_rows = used - n_rows
        pad_bytes = pad_rows * (rowbytes + 4)
        dname = "layout_dispatch" if args.fused else "dispatch"
        breakdown.update({
            "zero_padding_rows": pad_rows, "zero_padding_bytes": pad_bytes,
            f"{dname}_gbs_note": ("excludes the zero-padding bytes; the stage time "
                                  "includes clearing them"),
            f"{dname}_gbs_incl_padding": (b[dname] + pad_bytes) / (avg[dname] * 1e-3) / 1e9,
        })

    # ---- end to end through the API, host buffers ----------------------------
    e2e = None
    if not args.no_e2e and args.pass_ == "forward":
        x_h = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
        # routes and gate weights side by side in one pinned buffer: one copy
        route_h = torch.empty(T * K * 12, dtype=torch.uint8).pin_memory()
        for v, a in zip(route_views(route_h, T, K), (inp["topk_idx"], inp["topk_weights"])):
            v.copy_(torch.from_numpy(a))
        y_h = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
        # Experts: identity for bf16 rows (combine reads the dispatched rows);
        # for E4M3 rows, whose bf16 values no kernel of the path produces, the
        # experts' output is the device leg's seeded expert-output buffer,
        # already in HBM as a real expert's output would be.
        ident = recv_x if not wl.use_fp8_dispatch else Y_d
        # The host-buffer entry points either let the kernels read x and write
        # y in pinned host memory in place (direct: each byte crosses the host
        # link once, no staging) or move the rows in token chunks overlapped
        # with the kernels, which pays off when the rows span two chunks of at
        # least 4 MiB (below that, copying everything first and launching the
        # kernels back to back is faster).  The epilogue and FP8 input options
        # have device entry points only, so with those the rows are copied
        # whole.
        transfer = e2e_transfer(args.e2e_transfer, bool(epilogue or fp8_opts))
        host_io = transfer != "copies"
        chunks = 0 if transfer == "direct" else e2e_chunk_count(args.e2e_chunks, T * H * 2)

        def e2e_step():
            if not host_io:
                x_d.copy_(x_h, non_blocking=True)
            route_d.copy_(route_h, non_blocking=True)
            layout()
            if host_io:
                st = ep.ep_dispatch_from_host(ccfg, L.c, x_h.data_ptr(),
                                              None if chunks == 0 else p(x_d), p(w_d),
                                              p(recv_x), p(recv_s), p(recv_w), chunks, sptr)
                assert st == 0, ep.ep_status_str(st)
            else:
                dispatch(x_d)
            if host_io:
                st = ep.ep_combine_to_host(ccfg, L.c, p(ident), p(w_d),
                                           None if chunks == 0 else p(y_d), y_h.data_ptr(),
                                           chunks, sptr)
                assert st == 0, ep.ep_status_str(st)
            else:
                combine(ident, y_d)
                y_h.copy_(y_d, non_blocking=True)

        for _ in range(args.warmup):
            l2_flush()
            e2e_step()
        torch.cuda.synchronize()
        eev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize()
        for i in range(args.steps):
            l2_flush()
            eev[i][0].record(stream)
            e2e_step()
            eev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e_ms = reduce_max(statistics.mean(a.elapsed_time(b_) for a, b_ in eev), world, device)
        assert ep.ep_check_error(L.c, sptr) == 0
        sequential = {"value": T * world / (e_ms / 1e3), "unit": "tokens/s", "ms_per_step": e_ms,
                      "timing": "one step at a time, L2 flushed before each, events around "
                                "each step"}
        p_mode = pipelined_transfer(args.e2e_transfer, bool(epilogue or fp8_opts), T * H * 2)
        p_chunks = e2e_chunk_count(args.e2e_chunks, T * H * 2) if p_mode == "chunked" else 0
        p_graph = (E2E_GRAPH_STEPS if args.e2e_graph == "on" or
                   (args.e2e_graph == "auto" and p_mode == "direct") else 0)
        pipelined = (pipelined_e2e(ep, ccfg, cfg, T, K, H, wl, device, stream, x_h, route_h,
                                   None if wl.use_fp8_dispatch else recv_x, Y_d, p_chunks,
                                   args.steps, args.warmup, world, y_h,
                                   copies=(p_mode == "copies"), depth=args.e2e_depth,
                                   graph_steps=p_graph)
                     if p_mode is not None else None)
        sequential["transfer"] = (
            "ep_dispatch_from_host / ep_combine_to_host, direct (the kernels read x and write "
            "y in pinned host memory)" if transfer == "direct" else
            f"ep_dispatch_from_host / ep_combine_to_host, {chunks} token chunks (copies "
            "overlap the kernels)" if host_io else "whole-buffer copies on the stream")
        e2e = {"unit": "tokens/s",
               "h2d_bytes_per_step": x_h.numel() * 2 + route_h.numel(),
               "d2h_bytes_per_step": y_h.numel() * 2,
               "experts": ("identity (combine reads the dispatched bf16 rows)"
                           if not wl.use_fp8_dispatch else
                           "combine reads the device leg's seeded expert-output buffer"),
               "sequential": sequential}
        if pipelined is not None:
            pipelined["unit"] = "tokens/s"
            pipelined["transfer"] = (
                "ep_dispatch_from_host / ep_combine_to_host, direct (the kernels read x and "
                "write y in pinned host memory)" if p_mode == "direct" else
                f"ep_dispatch_from_host / ep_combine_to_host, {p_chunks} token chunks on the "
                "library's copy streams (one a direction)" if p_mode == "chunked" else
                "whole-buffer copies on each step's stream around ep_dispatch / ep_combine")
            e2e["pipelined"] = pipelined
        e2e.update(e2e_headline(sequential, pipelined))

    # ---- CPU baseline (rank 0, N = 1) ----------------------------------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.pass_ == "forward":
        cpu = cpu_baseline(wl, inp, args.cpu_budget_s)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": path_dtype(wl),
            "data": "synthetic (seeded router simulation, PCG64; no dataset)",
            "config": workload_config(wl, extra={
                "l2": "flushed before every step (256 MiB write, then 256 MiB read), outside the step events",
                "timing": ("step: events around each whole step; stage times and the roofline "
                           "from a second pass of the same steps with events between stages"),
                "step": " + ".join(name for name, _, _ in stages) +
                        ("; seeded N(0,1) dy and expert rows" if backward else
                         "; combine reads a device-resident seeded N(0,1) expert-output buffer"),
                "parallelism": f"{world} independent replica(s)",
                "launch": ("CUDA graph replay: one graph per step (stage times: one per stage)"
                           if args.graph else "direct C-ABI calls (host-launched)"),
                "zero_padding": bool(args.zero_padding),
                "combine_bias_tensors": args.bias,
                "combine_returns_weights": bool(args.return_weights),
                "fp8_scales": (args.fp8_scales if wl.use_fp8_dispatch else None),
                "fp8_prequantised_input": bool(wl.use_fp8_dispatch and args.fp8_prequant),
                "layout_and_dispatch": ("one call, one kernel" if args.fused and fused_small
                                        else "one call" if args.fused else "separate calls")}),
            "roofline": roofline,
            "steady_state": steady,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "breakdown": breakdown,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
