"""Benchmark of one paged E5M2-KV GQA decode step on GB300.

A step is one full xqa_decode (planner + split-KV partial + combine) over one
layer's decode batch. The default workload is 16 sequences with ragged contexts
drawn uniformly from [16384, 19200] (32 q / 4 kv heads, head_dim 128, 16-token
pages) — the "B16 ragged 17.8K" workload of the page "[Kernel][SM70] Pipeline
batched E5M2 XQA decode" (section "Starting bottleneck").

Metric: decode-attention µs/step and KV GB/s (algorithmic KV bytes =
sum_b ctx_b * Hkv * D * 2 per step, divided by the step time), and the
partial kernel's fraction of the measured HBM copy bandwidth.

Timing: steps are CUDA-graph replays on one stream, timed with CUDA events;
the KV cache rotates over several independent pools whose total exceeds the
129 MB L2 several times, so no step starts with its KV in L2.

``--impl reference`` times the float64 CPU oracle instead, on the same workload,
each step a bounded sample (one kv head of one sequence over a context prefix).

Under torchrun (N>1) every rank runs its own replica of the workload (weak
scaling, no collective on the data path); the step time is the maximum over
ranks.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/step and KV GB/s (% of GB300 HBM peak), B16 ragged ~17.8K ctx"
DEFAULT_WORKLOAD = "b16_ragged_ctx16384_19200"
FALLBACK_HBM_GBS = 6800.0
REPEATS = 5  # runs of the timed region for the per-step spread
NOMINAL_HBM_GBS = 8000.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "partial_kernel_b16_ragged.md")
KERNEL_SOURCES = ("paged_fp8_kv_gqa_gb300/csrc/partial.cu", "paged_fp8_kv_gqa_gb300/csrc/xqa_device.cuh")


# --------------------------------------------------------------------------
# distributed helpers (host scalars only; no collective on the data path)
# --------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int):
    if world <= 1:
        return None
    import torch.distributed as dist

    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend="gloo")
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def reduce_max(dist, x: float) -> float:
    """Max of a host scalar over ranks (identity without torch.distributed)."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / max_seconds


# --------------------------------------------------------------------------
# clocks, peaks, profile traffic
# --------------------------------------------------------------------------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampled every 100 ms while the timed region runs."""

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        return summarize_clocks(rows)


def summarize_clocks(rows):
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for r in rows:
        try:
            sm.append(float(r[1]))
            mx.append(float(r[2]))
        except ValueError:
            continue
        for name, val in zip(names, r[5:9]):
            if val.strip().lower() == "active":
                reasons.add(name)
    if not sm:
        return None
    sm.sort()
    return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "samples": len(sm),
            "reasons": sorted(reasons)}


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C/C++/CUDA source with comments removed and whitespace runs collapsed,
    so that editing a comment does not mark a profile as stale. String and
    character literals are kept as written."""
    out, i, n = [], 0, len(text)
    while i < n:
        ch = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif ch in "\"'":
            j = i + 1
            while j < n and text[j] != ch:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(ch)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the partial kernel's code (comments and layout ignored)."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per partial-kernel launch from the committed ncu summary, if it
    was taken on the current kernel source; else None."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    src = traffic = None
    for line in text.splitlines():
        line = line.strip().strip("`")
        if line.startswith("kernel_source_sha256:"):
            src = line.split(":", 1)[1].strip()
        elif line.startswith("dram_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    if src != kernel_source_hash() or traffic is None:
        return None
    return traffic


# --------------------------------------------------------------------------
# CPU oracle baseline
# --------------------------------------------------------------------------

ORACLE_SNIPPET = r"""
import json, os, sys, time
sys.path.insert(0, {root!r})
import numpy as np
from paged_fp8_kv_gqa_gb300 import workloads
from oracle import attention
w = workloads.make_workload({name!r})
budget, t_used, n, times = {budget!r}, 0.0, 0, []
while t_used < budget or n < 1:
    t0 = time.perf_counter()
    attention.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables,
                                     w.context_lens, w.k_scale, w.v_scale)
    dt = time.perf_counter() - t0
    times.append(dt); t_used += dt; n += 1
times.sort()
print(json.dumps({{"median_s": times[len(times)//2], "runs": n, "kv_bytes": w.kv_bytes}}))
"""


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, else implementer/part)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read().splitlines()
    except OSError:
        return "unknown"
    for key in ("model name", "Model name"):
        for line in info:
            if line.startswith(key):
                return line.split(":", 1)[1].strip()
    fields = {}
    for line in info:
        if ":" in line:
            k, v = (x.strip() for x in line.split(":", 1))
            fields.setdefault(k, v)
    if "CPU implementer" in fields:
        return f"implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    return "unknown"


def cpu_baseline(name: str, budget_s: float = 12.0):
    """The float64 oracle on the whole workload as it stands, in a fresh process,
    with numpy's BLAS on every core the process may use."""
    cores = _threads_note()
    code = ORACLE_SNIPPET.format(root=ROOT, name=name, budget=budget_s)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         timeout=900)
    if res.returncode != 0:
        return {"value": None, "unit": "GB/s", "cores": cores, "kind": "oracle",
                "sample": "failed: " + res.stderr.strip().splitlines()[-1][:200]}
    r = json.loads(res.stdout.strip().splitlines()[-1])
    return {"value": r["kv_bytes"] / r["median_s"] / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"whole {name} step (every sequence and kv head), float64 numpy, "
                      f"default BLAS threads on {cores} cores ({cpu_model()}), "
                      f"median of {r['runs']} runs, {r['median_s']:.2f} s/step"}


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def _device_workload(args, dev, xqa):
    """The workload of the command line on the device: (w, q, block tables,
    context lengths, [(K pool, V pool)] * pools, shape, workspace, out)."""
    import numpy as np
    import torch

    from paged_fp8_kv_gqa_gb300 import workloads

    if args.contexts:  # a custom length mix with the same recipe (not the headline)
        hq, hkv = (int(x) for x in args.heads.split(","))
        w = workloads.make_custom([int(c) for c in args.contexts.split(",")], hq, hkv, seed=7,
                                  kv_dtype=args.kv_dtype, q_len=args.q_len)
        args.workload = f"custom contexts {args.contexts}, {hq}/{hkv} heads"
    else:
        w = workloads.make_workload(args.workload, kv_dtype=args.kv_dtype, q_len=args.q_len)
    if args.kv_layout == "nhd":
        w = workloads.to_nhd(w)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    q, bt, lens = up(w.q), up(w.block_tables), up(w.context_lens)
    k0, v0 = up(w.k_cache), up(w.v_cache)
    pools = [(k0, v0)] + [(k0.clone(), v0.clone()) for _ in range(args.pools - 1)]
    shape = xqa.make_shape(q, k0, bt, min_pages_per_cta=args.min_pages,
                           merge_mode=args.merge_mode, kv_dtype=args.kv_dtype,
                           kv_layout=args.kv_layout)
    ws = xqa.alloc_workspace(shape, dev)
    out = torch.empty_like(q)
    return w, q, bt, lens, pools, shape, ws, out


def run_gpu(args, world, rank, local, dist):
    import numpy as np
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import paged_fp8_kv_gqa_gb300 as xqa

    if args.lib:  # a differently built libxqa.so with the same ABI (A/B comparisons)
        xqa._lib = None  # build() above loaded the in-tree library
        xqa.LIB_PATH = os.path.abspath(args.lib)
        xqa.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w, q, bt, lens, pools, shape, ws, out = _device_workload(args, dev, xqa)
    k0, v0 = pools[0]
    kv_bytes = w.kv_bytes
    stream = torch.cuda.Stream(device=dev)
    launches_per_step = xqa.xqa_kernels_per_call(shape)

    def step(i):
        # one step = the public decode call on the next KV pool of the rotation
        k, v = pools[i % len(pools)]
        xqa.xqa_decode(q, k, v, bt, lens, w.k_scale, w.v_scale, out=out, workspace=ws,
                       shape=shape, stream=stream)

    # eager warm-up (also sets kernel attributes before any capture)
    with torch.cuda.stream(stream):
        for i in range(max(3, min(args.warmup, 50))):
            step(i)
    stream.synchronize()
    assert xqa.xqa_read_status(ws, stream) == xqa.XQA_OK

    def capture(nsteps, first=0):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(nsteps):
                    step(first + i)
        return g

    # The timed graphs hold the decode calls and nothing else (no event nodes).
    C = max(1, min(args.steps, args.graph_steps))
    g_main = capture(C)
    rem = args.steps % C
    g_tail = capture(rem, C) if rem else None
    nrep = args.steps // C

    # graph warm-up: at least W steps, and about a second so clocks settle
    with torch.cuda.stream(stream):
        t_end = time.time() + args.warm_seconds
        done = 0
        while done < args.warmup or time.time() < t_end:
            g_main.replay()
            done += C
            if done % (C * 20) == 0:
                stream.synchronize()
    stream.synchronize()

    # ~100 us of GPU spin ahead of the start event, so that the host has the
    # first graph launch queued before the GPU reaches the event: the timed
    # region then holds device work only, not the host's launch latency
    spin_cycles = int(2e5)

    def timed_region():
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier(dist)
        with torch.cuda.stream(stream):  # graph replays launch on the current stream
            torch.cuda._sleep(spin_cycles)
            t0.record(stream)
            for _ in range(nrep):
                g_main.replay()
            if g_tail is not None:
                g_tail.replay()
            t1.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        barrier(dist)
        return t0.elapsed_time(t1)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler is not None:
        time.sleep(0.3)
    # the timed region (exactly K steps); then the same region again for the spread
    ms_total = timed_region()
    rep_ms = [ms_total] + [timed_region() for _ in range(max(0, args.repeats - 1))]
    clocks = sampler.stop() if sampler is not None else None
    ms_total_max = reduce_max(dist, ms_total)
    ms_per_step = ms_total_max / args.steps
    repeats = None
    if len(rep_ms) >= 2:
        per_step_us = sorted(m * 1e3 / args.steps for m in rep_ms)
        repeats = {"n": len(rep_ms), "steps_each": args.steps,
                   "median_us": _quantile(per_step_us, 0.5),
                   "p10_us": _quantile(per_step_us, 0.1), "p90_us": _quantile(per_step_us, 0.9),
                   "note": "the K-step timed region run again, same graphs; the headline "
                           "is the first run"}

    # The dominant kernel on its own: a separate graph whose every step is
    # bracketed by event nodes. An event node makes the next launch wait for
    # the previous one, so this time also holds the launch and prologue the
    # timed graph overlaps with the previous step: an upper bound per launch.
    kernel_us = None
    try:
        evs = [(torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True)) for _ in range(C)]
        g_ev = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g_ev, stream=stream):
                for i in range(C):
                    evs[i][0].record(stream)
                    step(i)
                    evs[i][1].record(stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g_ev.replay()
        stream.synchronize()
        kernel_us = sum(a.elapsed_time(b) for a, b in evs) / len(evs) * 1e3
    except TypeError:  # no external events in this torch
        pass
    status = xqa.xqa_read_status(ws, stream)

    # end to end through the public call, host buffers, copies inside the timed region
    e2e = None
    if args.e2e_steps > 0:
        hq = torch.from_numpy(w.q).pin_memory()
        hk = torch.from_numpy(w.k_cache).pin_memory()
        hv = torch.from_numpy(w.v_cache).pin_memory()
        hbt = torch.from_numpy(w.block_tables).pin_memory()
        hl = torch.from_numpy(w.context_lens).pin_memory()
        hout = torch.empty(tuple(w.q.shape), dtype=torch.float16).pin_memory()
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k0), torch.empty_like(v0)
        dbt, dl, dout = torch.empty_like(bt), torch.empty_like(lens), torch.empty_like(out)
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hbt, hl))
        d2h = hout.numel() * hout.element_size()

        def e2e_step():
            with torch.cuda.stream(stream):
                for d, h in ((dq, hq), (dk, hk), (dv, hv), (dbt, hbt), (dl, hl)):
                    d.copy_(h, non_blocking=True)
                xqa.xqa_decode(dq, dk, dv, dbt, dl, w.k_scale, w.v_scale, out=dout, workspace=ws,
                               shape=shape, stream=stream)  # shape carries format and layout
                hout.copy_(dout, non_blocking=True)
            stream.synchronize()

        for _ in range(2):
            e2e_step()
        barrier(dist)
        t_a = time.perf_counter()
        for _ in range(args.e2e_steps):
            e2e_step()
        t_e = reduce_max(dist, time.perf_counter() - t_a)
        e2e = {"value": aggregate_throughput(kv_bytes * args.e2e_steps, world, t_e) / 1e9,
               "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": args.e2e_steps,
               "us_per_step": t_e / args.e2e_steps * 1e6,
               "note": "pinned host q, K/V pools, block tables and lengths copied in, "
                       "output copied out, stream synchronised, every step"}

    if rank != 0:
        return None
    peak, peak_kind = hbm_peak()
    # The partial kernel's rate on the step's own clock: its launches take at
    # most the whole step (they are the step when the step is one launch), so
    # KV bytes per launch over the step time is a lower bound on its rate.
    achieved = kv_bytes / (ms_per_step * 1e-3) / 1e9
    basis = ("whole step: one partial-kernel launch per step, so the step time is the "
             "kernel's average launch duration over the timed region"
             if launches_per_step == 1 else
             f"whole step ({launches_per_step} launches per step): the partial kernel's "
             "average launch duration is at most the step time")
    # the committed capture is of the default configuration only
    profiled_config = (not args.contexts and args.workload == DEFAULT_WORKLOAD
                       and args.kv_dtype == "e5m2" and args.kv_layout == "hnd"
                       and args.q_len == 1 and args.merge_mode == 0 and args.min_pages == 0)
    traffic = profiled_traffic() if profiled_config else None
    value = aggregate_throughput(kv_bytes * args.steps, world, ms_total_max * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "us_per_step": ms_per_step * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": f"f16 mma / f32 acc ({args.kv_dtype} kv)",
        "data": "synthetic",
        "config": {
            "workload": args.workload,
            "batch": w.batch, "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "block_size": w.block_size,
            "total_context_tokens": int(w.context_lens.sum()),
            "kv_bytes_per_step": kv_bytes,
            "l2": f"inputs larger than L2: {len(pools)} rotating KV pools of "
                  f"{2 * w.k_cache.nbytes / 1e6:.0f} MB",
            "timing": f"CUDA graph replays of {C} steps on one stream (no event nodes inside), "
                      "CUDA events on the stream around exactly K steps",
            "launches_per_step": launches_per_step,
            "merge_mode": shape.merge_mode,
            "min_pages_per_cta": shape.min_pages_per_cta,
            "kv_dtype": args.kv_dtype,
            "kv_layout": args.kv_layout,
            "q_len": args.q_len,
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "pct_of_nominal_8tbs": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
        "roofline": {
            "bound": "hbm",
            "kernel": "xqa::partial_kernel",
            "achieved": round(achieved, 2),
            "peak": peak,
            "peak_kind": f"{peak_kind} (STREAM-style copy)",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": kv_bytes,
            "avg_launch_us": ms_per_step * 1e3,
            "basis": basis,
            "kernel_alone_us": kernel_us,
            "kernel_alone_note": "separate graph, event nodes around every launch (no overlap "
                                 "with the previous launch): an upper bound per launch",
        },
        "repeats": repeats,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "device_status": status,
    }
    if world == 1 and not args.no_cpu_baseline and not args.contexts:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    return line


# --------------------------------------------------------------------------
# phase breakdown from the diagnostic (timestamped) build
# --------------------------------------------------------------------------

STAMP_NAMES = ("entry", "inputs_readable", "range_known", "first_pages", "pages_done",
               "merges_buffered", "tickets_taken", "exit")
STAMPS_PER_CTA = 18  # the eight times above, pages, segments, eight more times
EXTRA_STAMPS = {10: "lengths_loaded", 11: "block_ids_loaded", 12: "all_warps_past_wait",
                13: "plan_done", 14: "page_loop_entered", 15: "first_search_done",
                16: "merge_range_known", 17: "merge_loads_in"}


def stamp_breakdown(st, page_bytes: int):
    """Phases of one launch from its per-CTA stamps (int [ctas, >= 10]: eight
    %globaltimer values in ns, then the CTA's pages and segments). Times in
    us, relative to the moment the launch could read its inputs (the first
    CTA past the wait for the previous kernels)."""
    import numpy as np

    st = np.asarray(st, dtype=np.int64)
    work = st[:, 8] > 0
    start = st[:, 1][st[:, 1] > 0].min()
    rel = (st[:, :8] - start) / 1e3
    w = rel[work]
    stream_us = w[:, 4] - w[:, 3]
    pages = st[work, 8]
    med = lambda a: float(np.median(a))
    return {
        "ctas_with_work": int(work.sum()),
        "entry_before_inputs_us": -med(rel[:, 0]),
        "range_known_us": med(w[:, 2]),
        "first_pages_us": med(w[:, 3]),
        "first_pages_last_cta_us": float(w[:, 3].max()),
        "pages_done_median_us": med(w[:, 4]),
        "pages_done_last_us": float(w[:, 4].max()),
        "exit_last_us": float(rel[:, 7].max()),
        "end_of_range_median_us": med(w[:, 7] - w[:, 4]),
        "steady_gbs": float((pages * page_bytes / (stream_us * 1e3)).sum()),
        "median_cta_stream_us": med(stream_us),
        "pages_per_cta_min_max": [int(pages.min()), int(pages.max())],
    }


def stamp_columns(st):
    """Per-CTA columns of one launch's stamps: pages, segments, and every
    stamped time in us from the first CTA past the wait (NaN where unset)."""
    import numpy as np

    st = np.asarray(st, dtype=np.int64)
    t0 = st[:, 1][st[:, 1] > 0].min()
    names = {**dict(enumerate(STAMP_NAMES)), **EXTRA_STAMPS}
    cols = {"pages": st[:, 8].astype(float), "segments": st[:, 9].astype(float)}
    for i, name in names.items():
        if i < st.shape[1]:
            cols[name] = np.where(st[:, i] > 0, (st[:, i] - t0) / 1e3, np.nan)
    return cols


def run_stamps(args):
    """Phase breakdown of the partial kernel from the timestamped diagnostic
    build (never the headline: its numbers come from the library as built).
    A CUDA graph of two decode steps is replayed; the stamps of the second
    step, which overlaps the first as steps do in the timed run, are read
    after each replay."""
    import ctypes

    import numpy as np
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import paged_fp8_kv_gqa_gb300 as xqa
    from paged_fp8_kv_gqa_gb300 import build as _build

    xqa._lib = None
    # a differently built stamped library with the same ABI (A/B of phases), else this tree's
    xqa.LIB_PATH = os.path.abspath(args.lib) if args.lib else _build.build(variant="stamps")
    lib = xqa.load_library()
    lib.xqa_diag_read_stamps.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    lib.xqa_diag_read_stamps.restype = ctypes.c_int
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    w, q, bt, lens, pools, shape, ws, out = _device_workload(args, dev, xqa)
    stream = torch.cuda.Stream(device=dev)
    n_ctas = shape.max_ctas or torch.cuda.get_device_properties(0).multi_processor_count

    def step(i):
        k, v = pools[i % len(pools)]
        xqa.xqa_decode(q, k, v, bt, lens, w.k_scale, w.v_scale, out=out, workspace=ws,
                       shape=shape, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(3):
            step(i)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            step(0)
            step(1)
    per, raw = [], []
    buf = np.zeros((n_ctas, STAMPS_PER_CTA), np.uint64)
    for r in range(args.stamp_samples + 5):
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        rc = lib.xqa_diag_read_stamps(buf.ctypes.data, n_ctas, int(stream.cuda_stream))
        if rc != 0:
            raise RuntimeError(f"xqa_diag_read_stamps: status {rc}")
        if r >= 5:
            per.append(stamp_breakdown(buf.copy(), 2 * w.head_dim * w.block_size))
            raw.append(stamp_columns(buf))
    keys = [k for k in per[0] if isinstance(per[0][k], float)]
    summary = {k: float(np.median([d[k] for d in per])) for k in keys}
    summary["ctas_with_work"] = per[0]["ctas_with_work"]
    summary["pages_per_cta_min_max"] = per[0]["pages_per_cta_min_max"]
    line = {"stamps": summary, "samples": len(per), "workload": args.workload,
            "kv_bytes_per_step": w.kv_bytes,
            "note": "medians over samples; times in us from the first CTA past the wait for "
                    "the previous kernels; steady_gbs = sum over CTAs of pages x 4096 B over "
                    "(pages done - first pages)"}
    # the CTA that exits last in each sample: its index, pages, segments and phase times
    last = []
    for cols in raw:
        i = int(np.nanargmax(cols["exit"]))
        last.append({k: float(v[i]) for k, v in cols.items()} | {"cta": i})
    line["last_exit"] = {k: float(np.median([d[k] for d in last])) for k in last[0]}
    line["last_exit"]["ctas_seen"] = sorted({d["cta"] for d in last})[:20]
    if args.stamps_per_cta:  # per CTA, median over samples: pages, segments, phase times (us)
        line["per_cta"] = {k: np.nanmedian(np.stack([d[k] for d in raw]), axis=0).round(3).tolist()
                           for k in raw[0]}
    return line


# --------------------------------------------------------------------------
# reference arm: the CPU oracle
# --------------------------------------------------------------------------

def run_reference(args, world, rank):
    import numpy as np

    from oracle import attention
    from paged_fp8_kv_gqa_gb300 import workloads

    if rank != 0:
        return None
    w = workloads.make_workload(args.workload)
    nseg = w.batch * w.num_kv_heads
    budget = args.reference_seconds
    # calibrate: one whole segment, then size a context prefix so all steps fit the budget
    t0 = time.perf_counter()
    sub = _segment_prefix(w, 0, int(w.context_lens[0]))
    attention.paged_decode_attention(*sub)
    per_token = (time.perf_counter() - t0) / int(w.context_lens[0])
    per_step = budget / max(1, args.steps + args.warmup)
    tokens = int(max(16, min(int(w.context_lens.min()), per_step / max(per_token, 1e-12))))
    samples = []
    for i in range(args.warmup + args.steps):
        s = i % nseg
        args_i = _segment_prefix(w, s, tokens)
        t = time.perf_counter()
        attention.paged_decode_attention(*args_i)
        dt = time.perf_counter() - t
        if i >= args.warmup:
            samples.append(dt)
    total = sum(samples)
    bytes_per_step = tokens * w.head_dim * 2
    value = bytes_per_step * len(samples) / total / 1e9
    sample = (f"one kv head of one sequence per step (rotating over the {nseg} (sequence, kv head) "
              f"pairs), first {tokens} context tokens; float64 numpy oracle")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total / len(samples) * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {
            "workload": args.workload,
            "batch": w.batch, "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "block_size": w.block_size,
            "total_context_tokens": int(w.context_lens.sum()),
            "kv_bytes_per_step": int(w.context_lens.sum()) * w.num_kv_heads * w.head_dim * 2,
            "sample_kv_bytes_per_step": bytes_per_step,
            "kv_dtype": w.kv_dtype, "kv_layout": w.kv_layout, "q_len": 1,
            "parallelism": "single process (rank 0)",
        },
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": _threads_note(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def _quantile(sorted_vals, q):
    """Linear-interpolated quantile of an ascending list."""
    x = q * (len(sorted_vals) - 1)
    i = int(x)
    j = min(i + 1, len(sorted_vals) - 1)
    return sorted_vals[i] + (sorted_vals[j] - sorted_vals[i]) * (x - i)


def _threads_note():
    try:
        return int(os.environ.get("OMP_NUM_THREADS") or 0) or len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def _segment_prefix(w, s, tokens):
    """Oracle arguments for kv head (s % Hkv) of sequence (s // Hkv) over its first tokens."""
    import numpy as np

    b, g = divmod(s, w.num_kv_heads)
    G = w.num_q_heads // w.num_kv_heads
    n = min(tokens, int(w.context_lens[b]))
    npg = (n + 15) // 16
    q = w.q[b:b + 1, g * G:(g + 1) * G]
    kc = w.k_cache[:, g:g + 1]
    vc = w.v_cache[:, g:g + 1]
    bt = w.block_tables[b:b + 1, :npg]
    lens = np.array([n], np.int32)
    return q, kc, vc, bt, lens, w.k_scale, w.v_scale


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=("xqa", "reference"), default="xqa")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--contexts", default="",
                    help="comma-separated context lengths of a custom workload (with --heads)")
    ap.add_argument("--heads", default="32,4", help="q heads,kv heads of a custom workload")
    ap.add_argument("--pools", type=int, default=4)
    ap.add_argument("--graph-steps", type=int, default=50)
    ap.add_argument("--repeats", type=int, default=REPEATS,
                    help="runs of the K-step timed region (the first is the headline; all "
                         "give the spread)")
    ap.add_argument("--kv-dtype", choices=("e5m2", "e4m3"), default="e5m2")
    ap.add_argument("--kv-layout", choices=("hnd", "nhd"), default="hnd")
    ap.add_argument("--q-len", type=int, default=1, help="new tokens per sequence")
    ap.add_argument("--min-pages", type=int, default=0,
                    help="minimum pages per CTA of the split rule (0: the library default)")
    ap.add_argument("--merge-mode", type=int, choices=(0, 1), default=0,
                    help="0: split segments merged inside the partial kernel; 1: combine kernel")
    ap.add_argument("--warm-seconds", type=float, default=1.0)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--reference-seconds", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--lib", default="", help="path of an alternative libxqa.so build")
    ap.add_argument("--stamps", action="store_true",
                    help="print the partial kernel's phase breakdown from the timestamped "
                         "diagnostic build instead of a bench line")
    ap.add_argument("--stamp-samples", type=int, default=50)
    ap.add_argument("--stamps-per-cta", action="store_true",
                    help="with --stamps: also print every CTA's pages and phase times")
    args = ap.parse_args(argv)
    if args.steps < 1 or args.warmup < 0:
        raise SystemExit("--steps must be >= 1 and --warmup >= 0")
    world, rank, local = dist_env()
    if args.stamps:
        print(json.dumps(run_stamps(args)), flush=True)
        return
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        dist = init_dist(world)
        line = run_gpu(args, world, rank, local, dist)
        if dist is not None:
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
