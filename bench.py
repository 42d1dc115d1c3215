#!/usr/bin/env python3
"""Benchmark of the paged KV cache decode step on GB300.

One step = copy_blocks of the workload's copy-on-write pairs (when it has
any) + paged_kv_append of the step's new tokens + paged_attention_decode over
every sequence; a step that appends one token per sequence at its last
position is the single fused call paged_attention_append_decode.

The default workload is the Llama-3.1-70B-class long-context layer (8
sequences of 131072 tokens, 64 query / 8 KV heads, bf16, block 32: 4 GiB of
K/V per step), the largest configuration on one GPU; the Llama-3-8B-class
layer (64 sequences, 32 query / 8 KV heads, bf16, block 16, contexts uniform
in [512, 4096]) is measured after it in the same run and reported under
``per_workload``.  ``--workload`` selects another main workload and
``--extra`` the others.

Metric: K/V bytes of the attended contexts per second (GB/s) and sequences per
second; the roofline object reports paged_attention_decode's algorithmic
bytes per launch over its CUDA-event time against the measured HBM peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME] [--extra A,B]

Under torchrun (N > 1) every rank runs its own batch (different seed) with no
data exchange; timing is the max over ranks and value aggregates all ranks.
``--impl reference`` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak); sequences/s per step"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = ROOT / "profiles" / "traffic_per_launch.txt"
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal
WARM_GPU_S = 0.5      # GPU time of warm-up steps run right before each timed region
STAT_MIN_STEPS = 50   # per-step timings behind the median / p10 / p90


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama70b_long")
    ap.add_argument("--extra", default=None,
                    help="comma-separated workloads measured after the main one and reported under per_workload "
                         "(default: llama8b when the main workload is llama70b_long, else none)")
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-seqs", type=int, default=0, help="0: the whole batch")
    ap.add_argument("--unfused", action="store_true", help="separate block-write and decode launches")
    ap.add_argument("--ungrouped", action="store_true",
                    help="shared-prefix workloads: plain paged_attention_decode instead of the grouped call")
    ap.add_argument("--warm-ms", type=float, default=WARM_GPU_S * 1e3,
                    help="GPU time of extra warm-up steps run right before each timed region (0: none, e.g. under "
                         "a profiler)")
    ap.add_argument("--stat-steps", type=int, default=STAT_MIN_STEPS,
                    help="steps of the per-step statistics run (at least --steps; 0: skip it)")
    ap.add_argument("--flush-l2", action="store_true",
                    help="write a 256 MB buffer before every step (outside the step's timing) so that no step "
                         "finds the previous one's K/V in L2")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- distributed plumbing
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws: int, backend: str):
    if ws <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_seed(base: int, rank: int) -> int:
    return base ^ (0x1000193 * rank) if rank else base


# ---------------------------------------------------------------- peaks, clocks, traffic
def measured_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return json.loads(p.read_text())
        except Exception:
            pass
    return {}


def _code_only(text: str) -> str:
    """C++ source without its comments and blank lines (no string literal in
    these sources holds a comment marker)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", line).rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def decode_source_hash(grouped: bool = False) -> str:
    """sha256[:16] over the code (comments dropped) of the sources the decode
    kernel is built from, plus the shared-prefix kernel's for a grouped call
    (whose traffic figure is the sum over its two kernels)."""
    import hashlib
    h = hashlib.sha256()
    names = ("decode.cu", "decode_common.cuh", "pkv_internal.cuh") + (("group_prefix.cu",) if grouped else ())
    for name in names:
        h.update(_code_only((ROOT / "paged_kv_cache_11_gb300" / "csrc" / name).read_text()).encode())
    return h.hexdigest()[:16]


def traffic_per_launch(workload: str):
    """dram read+write bytes per decode call from the committed ncu summary, if it
    still describes the current kernels (same source hash).  A grouped call's
    entry is named <workload>_grouped."""
    if not TRAFFIC_FILE.exists():
        return None
    h = decode_source_hash(grouped=workload.endswith("_grouped"))
    for line in TRAFFIC_FILE.read_text().splitlines():
        parts = line.split()
        if len(parts) >= 3 and parts[0] == workload and parts[1] == h:
            return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms; the
    summary covers the samples taken inside the marked intervals (each
    workload's warm-up, timed region and per-step statistics run)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.samples = []
        self.proc = None
        self.spans = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.spans.append([time.time(), None])
        elif self.spans:
            self.spans[-1][1] = time.time()

    @staticmethod
    def summarise(rows) -> dict | None:
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        spans = [(a, b if b is not None else time.time()) for a, b in self.spans]
        rows = [s for t, s in self.samples if any(a <= t <= b for a, b in spans)]
        if not rows:  # intervals shorter than the sampling period: the nearest samples
            rows = [s for t, s in self.samples if any(a - 0.15 <= t <= b + 0.15 for a, b in spans)]
        return self.summarise(rows)


# ---------------------------------------------------------------- workload description
def describe(wl) -> dict:
    s = wl.spec
    d = {"workload": s.name, "num_seqs": wl.num_seqs, "num_q_heads": s.num_q_heads,
         "num_kv_heads": s.num_kv_heads, "head_dim": s.head_dim, "block_size": s.block_size, "dtype": s.dtype,
         "context_lens": {"min": int(wl.context_lens.min()), "max": int(wl.context_lens.max()),
                          "mean": float(wl.context_lens.mean())},
         "pool_blocks": wl.num_blocks, "appended_tokens": int(len(wl.slot_mapping)),
         "cow_pairs": int(len(wl.cow_pairs)), "kv_bytes_per_step": wl.kv_bytes()}
    if s.groups:
        d["unique_kv_bytes_per_step"] = wl.unique_kv_bytes()
    return d


def decode_algorithmic_bytes(wl, fused: bool = False, groups=None) -> int:
    """Bytes paged_attention_decode must move: the attended K/V, q, the block-table
    entries it reads, context_lens and the fp32 output; the fused call also reads
    each new K/V row and its slot and writes the row into the cache.  The grouped
    call (groups = (group_starts, prefix_lens)) must read each shared block once:
    the distinct K/V slots, plus each group's shared table entries once, the
    prefix lengths and the group starts."""
    bs = wl.block_size
    blocks = int(((wl.context_lens.astype(np.int64) + bs - 1) // bs).sum())
    q = wl.num_seqs * wl.num_q_heads * wl.head_dim * 2
    out = wl.num_seqs * wl.num_q_heads * wl.head_dim * 4
    extra = 0
    if fused:
        extra = wl.num_seqs * (2 * 2 * wl.num_kv_heads * wl.head_dim * 2 + 8)
    if groups is not None:
        gs, pl = groups
        shared = int(pl.sum()) // bs - sum(int(pl[a]) // bs for a in gs[:-1] if a < len(pl))
        return wl.unique_kv_bytes() + q + out + (blocks - shared) * 4 + wl.num_seqs * 8 + len(gs) * 4 + extra
    return wl.kv_bytes() + q + out + blocks * 4 + wl.num_seqs * 4 + extra


# ---------------------------------------------------------------- CPU oracle timing
def time_oracle(wl, nseq: int, threads: int):
    """One oracle step (copy + append + decode) over the first nseq sequences; returns
    (seconds, kv_bytes, sequences, outputs [B, Hq, D] float64 with those sequences filled)."""
    import oracle
    nseq = min(nseq or wl.num_seqs, wl.num_seqs)
    sel = [(s, h) for s in range(nseq) for h in range(wl.num_q_heads)]
    kc, vc = wl.k_cache, wl.v_cache  # the oracle writes the same bytes the GPU step writes
    t0 = time.perf_counter()
    if len(wl.cow_pairs):
        oracle.copy_blocks(kc, vc, wl.cow_pairs)
    if len(wl.slot_mapping):
        m = wl.append_seq < nseq
        oracle.append(np.ascontiguousarray(wl.new_k[m]), np.ascontiguousarray(wl.new_v[m]), wl.slot_mapping[m], kc, vc)
    out, _ = oracle.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale, wl.dtype, select=sel,
                           threads=threads)
    dt = time.perf_counter() - t0
    kvb = int(wl.context_lens[:nseq].astype(np.int64).sum()) * 2 * wl.num_kv_heads * wl.head_dim * 2
    return dt, kvb, nseq, out


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from paged_kv_cache_11_gb300 import _build, workload as W
    import oracle
    _build.build_generator()
    oracle.build()
    wl = W.make_workload(args.workload)
    threads = host_threads()
    nseq = args.cpu_sample_seqs
    if not nseq:
        # size each step's sample so that warmup + steps take about a minute
        t1 = time_oracle(wl, 1, threads)[0]
        per_step = 60.0 / max(1, args.steps + args.warmup)
        nseq = int(max(1, min(wl.num_seqs, 8, per_step // max(t1, 1e-6))))
    for _ in range(max(0, args.warmup)):
        time_oracle(wl, nseq, threads)
    tot, kvb, seqs = 0.0, 0, 0
    for _ in range(args.steps):
        dt, b, n, _ = time_oracle(wl, nseq, threads)
        tot += dt
        kvb += b
        seqs += n
    gbs = kvb / tot / 1e9
    sample = f"first {nseq} of {wl.num_seqs} sequences per step (all their query heads), {args.steps} steps"
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": describe(wl), "seq_per_s": seqs / tot,
        "cpu_baseline": {"value": gbs, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": gbs, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- our arm
def percentiles(xs) -> dict:
    a = np.sort(np.asarray(xs, dtype=np.float64))
    return {"median_ms": float(np.median(a)), "p10_ms": float(np.percentile(a, 10)),
            "p90_ms": float(np.percentile(a, 90)), "n": int(len(a))}


class Device:
    """What every workload's measurement shares: the device, the stream, the
    process group and the clock sampler."""

    def __init__(self, torch, pkv, dev, rank, ws, dist, clocks):
        self.torch, self.pkv, self.dev, self.rank, self.ws, self.dist, self.clocks = \
            torch, pkv, dev, rank, ws, dist, clocks
        self.stream = torch.cuda.current_stream()


def measure(name: str, args, d: Device, cpu_seconds: float, single_thread: bool) -> dict:
    """One workload: warm-up, exactly args.steps timed steps, per-step
    statistics, the end-to-end run through host buffers, and (rank 0 of a
    one-process run) the oracle on the host cores over the same inputs, whose
    outputs also give the maximum error of the GPU result."""
    torch, pkv, dev, stream, dist = d.torch, d.pkv, d.dev, d.stream, d.dist
    from paged_kv_cache_11_gb300 import workload as W

    spec = W.SPECS[name]
    wl = W.make_workload(name, seed=rank_seed(W.default_seed(spec), d.rank))
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}[wl.dtype]

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(dt)

    kc, vc = up(wl.k_cache), up(wl.v_cache)
    q, nk, nv = up(wl.q), up(wl.new_k), up(wl.new_v)
    sm = torch.from_numpy(wl.slot_mapping).to(dev)
    bt = torch.from_numpy(wl.block_tables).to(dev)
    cl = torch.from_numpy(wl.context_lens).to(dev)
    cow = torch.from_numpy(wl.cow_pairs).to(dev) if len(wl.cow_pairs) else None
    out = torch.empty((wl.num_seqs, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device=dev)
    mcl = wl.max_context_len

    # A decode step that appends one token per sequence, at its last position,
    # runs the block write inside the decode call (paged_attention_append_decode,
    # or its grouped form when the batch holds forked groups), after the step's
    # copy-on-write copies if it has any; other steps run copy_blocks,
    # paged_kv_append and the decode call.
    fused = (not args.unfused) and np.array_equal(wl.append_seq, np.arange(wl.num_seqs))
    grouped = bool(spec.groups) and not args.ungrouped
    one_call = fused and cow is None  # the step is the decode call alone
    g_starts = g_plen = gs_d = pl_d = None
    if grouped:
        g_starts, g_plen, g_max = W.prefix_groups(wl)
        g_mpl = int(g_plen.max())
        gs_d, pl_d = torch.from_numpy(g_starts).to(dev), torch.from_numpy(g_plen).to(dev)
        need = pkv.paged_attention_grouped_workspace_bytes(wl.num_seqs, wl.num_q_heads, wl.head_dim, mcl, g_mpl,
                                                           args.partition_size)
    else:
        need = pkv.paged_attention_workspace_bytes(wl.num_seqs, wl.num_q_heads, wl.head_dim, mcl,
                                                   args.partition_size)
    wsp = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

    def decode(q_, bt_, cl_, out_, ws_, gs_=None, pl_=None, nk_=None, nv_=None, sm_=None):
        """The decode call (with the block write inside it when fused)."""
        kw = dict(out=out_, max_context_len=mcl, partition_size=args.partition_size, workspace=ws_)
        if grouped and fused:
            pkv.paged_attention_append_decode_grouped(q_, nk_, nv_, sm_, kc, vc, bt_, cl_, gs_, pl_, wl.scale,
                                                      max_group_size=g_max, max_prefix_len=g_mpl, **kw)
        elif grouped:
            pkv.paged_attention_decode_grouped(q_, kc, vc, bt_, cl_, gs_, pl_, wl.scale, max_group_size=g_max,
                                               max_prefix_len=g_mpl, **kw)
        elif fused:
            pkv.paged_attention_append_decode(q_, nk_, nv_, sm_, kc, vc, bt_, cl_, wl.scale, **kw)
        else:
            pkv.paged_attention_decode(q_, kc, vc, bt_, cl_, wl.scale, **kw)

    def step(ev=None):
        """One step; ev = (start, end) events bracket its decode call."""
        if cow is not None:
            pkv.copy_blocks(kc, vc, cow)
        if len(wl.slot_mapping) and not fused:
            pkv.paged_kv_append(nk, nv, sm, kc, vc)
        if ev is not None:
            ev[0].record(stream)
        decode(q, bt, cl, out, wsp, gs_d, pl_d, nk, nv, sm)
        if ev is not None:
            ev[1].record(stream)

    def event_pair():
        return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    if d.clocks:
        d.clocks.mark(True)
    # ---- warm-up: the requested steps, then more until WARM_GPU_S of GPU
    # time has run, so that the clocks and the memory system are at their
    # working state when the timed region starts (the GPU is never left idle
    # in between; the only gap is the barrier and synchronisation).
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert pkv.check_device_error() == 0, "device error during warm-up"
    warm_ms, batch = 0.0, 8
    while warm_ms < args.warm_ms:
        a, b = event_pair()
        a.record(stream)
        for _ in range(batch):
            step()
        b.record(stream)
        b.synchronize()
        ms = a.elapsed_time(b)
        warm_ms += ms
        batch = int(min(4096, max(batch, batch * args.warm_ms / max(ms, 1e-3) / 4)))

    # ---- the timed region: exactly args.steps steps.  A step that is one
    # launch (the fused decode) runs back to back between two events, so
    # consecutive launches overlap as they do in a serving loop and that
    # launch's duration is the step's.  A step of several launches also
    # brackets its decode call with events.
    evs = [event_pair() for _ in range(args.steps)] if (not one_call or args.flush_l2) else [None] * args.steps
    # --flush-l2: each step is bracketed by its own events and the flush runs
    # between steps, outside them
    step_evs = [event_pair() for _ in range(args.steps)] if args.flush_l2 else None
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if args.flush_l2 else None
    t_start, t_end = event_pair()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    l0 = pkv.launch_count()
    t_start.record(stream)
    for i in range(args.steps):
        if flush_buf is not None:
            flush_buf.zero_()
            step_evs[i][0].record(stream)
        step(evs[i])
        if flush_buf is not None:
            step_evs[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = pkv.launch_count() - l0
    if dist:
        dist.barrier()
    ms_total = t_start.elapsed_time(t_end)
    if step_evs is not None:
        ms_total = sum(a.elapsed_time(b) for a, b in step_evs)  # the steps alone, without the flushes
    if one_call and step_evs is None:
        dec_avg_ms = ms_total / args.steps
    else:
        dec_avg_ms = sum(a.elapsed_time(b) for a, b in evs) / len(evs)
    assert pkv.check_device_error() == 0, "device error in the timed region"

    # ---- per-step statistics: every step of a separate run of
    # max(STAT_MIN_STEPS, steps) steps bracketed by its own events (which also
    # bracket the decode call of a multi-launch step).  An event between two
    # launches keeps the next one from starting while the previous one
    # drains, so these times run slightly above the timed region's mean.
    n_stat = max(args.stat_steps, args.steps) if args.stat_steps > 0 else 0
    st_evs = [event_pair() for _ in range(n_stat)]
    dec_evs = [event_pair() for _ in range(n_stat)] if not one_call else None
    for i in range(n_stat):
        st_evs[i][0].record(stream)
        step(dec_evs[i] if dec_evs else None)
        st_evs[i][1].record(stream)
    torch.cuda.synchronize()
    if d.clocks:
        d.clocks.mark(False)
    stats = None
    if n_stat:
        stats = percentiles([a.elapsed_time(b) for a, b in st_evs])
        stats["how"] = ("each of %d steps bracketed by its own CUDA events on the launching stream (run after "
                        "the timed region; the events keep consecutive launches from overlapping)" % n_stat)
        if dec_evs:
            stats["decode_call"] = percentiles([a.elapsed_time(b) for a, b in dec_evs])
    assert pkv.check_device_error() == 0

    # ---- end to end: host buffers in, result out, through the public API.
    # Each step's inputs (q, new K/V, slot mapping, block tables, context
    # lengths, copy-on-write pairs) are packed in one pinned host buffer and
    # copied with one host->device copy; the output comes back with one
    # device->host copy.  Two device buffer sets let step i+1's inputs (and
    # step i-1's output) move on a copy stream while step i computes.
    host_parts = [("q", wl.q, dt), ("nk", wl.new_k, dt), ("nv", wl.new_v, dt),
                  ("sm", wl.slot_mapping, torch.int64), ("bt", wl.block_tables, torch.int32),
                  ("cl", wl.context_lens, torch.int32)]
    if cow is not None:
        host_parts.append(("cow", wl.cow_pairs, torch.int64))
    if grouped:
        host_parts += [("gs", g_starts, torch.int32), ("pl", g_plen, torch.int32)]
    offs, off = {}, 0
    for pname, arr, _ in host_parts:
        offs[pname] = off
        off += (arr.nbytes + 255) // 256 * 256
    h2d = off
    h_in = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    for pname, arr, _ in host_parts:
        h_in[offs[pname]:offs[pname] + arr.nbytes].copy_(
            torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).ravel()))
    d_in = [torch.empty(h2d, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_out = [torch.empty_like(out) for _ in range(2)]
    h_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    d2h = out.numel() * out.element_size()

    def views(buf):
        v = {}
        for pname, arr, tdt in host_parts:
            v[pname] = buf[offs[pname]:offs[pname] + arr.nbytes].view(tdt).view(arr.shape)
        return v

    dviews = [views(b) for b in d_in]
    wsp2 = [torch.empty_like(wsp) for _ in range(2)]
    cs, xs = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]

    def h2d_copy(i):
        b = i % 2
        with torch.cuda.stream(xs):
            xs.wait_event(comp_done[b])      # buffer b was last used by step i - 2
            d_in[b].copy_(h_in, non_blocking=True)
            h2d_done[b].record(xs)

    def e2e_compute(i):
        b = i % 2
        v = dviews[b]
        with torch.cuda.stream(cs):
            cs.wait_event(h2d_done[b])
            if cow is not None:
                pkv.copy_blocks(kc, vc, v["cow"])
            if len(wl.slot_mapping) and not fused:
                pkv.paged_kv_append(v["nk"], v["nv"], v["sm"], kc, vc)
            decode(v["q"], v["bt"], v["cl"], d_out[b], wsp2[b], v.get("gs"), v.get("pl"), v["nk"], v["nv"], v["sm"])
            comp_done[b].record(cs)

    def d2h_copy(i):
        b = i % 2
        with torch.cuda.stream(xs):
            xs.wait_event(comp_done[b])
            h_out[b].copy_(d_out[b], non_blocking=True)

    def e2e_run(n):
        h2d_copy(0)
        for i in range(n):
            if i + 1 < n:
                h2d_copy(i + 1)
            e2e_compute(i)
            d2h_copy(i)

    e2e_steps = max(1, min(args.steps, 1000))
    torch.cuda.synchronize()
    e2e_run(3)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = event_pair()
    torch.cuda.synchronize()
    e0.record(xs)
    e2e_run(e2e_steps)
    with torch.cuda.stream(xs):
        xs.wait_event(comp_done[(e2e_steps - 1) % 2])
        e1.record(xs)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    assert pkv.check_device_error() == 0
    out_host = out.cpu()
    assert torch.equal(h_out[(e2e_steps - 1) % 2], out_host), "end-to-end output differs from the resident run"

    # ---- aggregate over ranks
    kvb = float(wl.kv_bytes())
    ms_max = max_over_ranks(dist, ms_total, dev)
    e2e_max = max_over_ranks(dist, e2e_ms, dev)
    kv_all = sum_over_ranks(dist, kvb, dev)
    seqs_all = sum_over_ranks(dist, float(wl.num_seqs), dev)
    launches_all = int(sum_over_ranks(dist, float(launches), dev))

    peaks = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    steps = args.steps
    value = kv_all * steps / (ms_max / 1e3) / 1e9
    dec_bytes = decode_algorithmic_bytes(wl, fused, (g_starts, g_plen) if grouped else None)
    achieved = dec_bytes / (dec_avg_ms / 1e3) / 1e9
    traffic = traffic_per_launch(name + ("_grouped" if grouped else ""))
    dec_api = ("paged_attention_append_decode_grouped" if grouped and fused else
               "paged_attention_decode_grouped" if grouped else
               "paged_attention_append_decode" if fused else "paged_attention_decode")

    # ---- the oracle on the host cores (rank 0 of a one-process run): the
    # CPU baseline, and the maximum error of the GPU output against it
    cpu = None
    if d.ws == 1 and not args.no_cpu_baseline:
        threads = host_threads()
        t = b = reps = 0
        ref = None
        while reps == 0 or t < cpu_seconds:  # whole oracle steps, about cpu_seconds of CPU time
            dt1, b1, n, ref = time_oracle(wl, args.cpu_sample_seqs, threads)
            t, b, reps = t + dt1, b + b1, reps + 1
        gpu_out = out_host.numpy().astype(np.float64)[:n]
        err = float(np.abs(gpu_out - ref[:n]).max())
        cpu = {"value": b / t / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{reps} oracle step(s) over the first {n} of {wl.num_seqs} sequences (all query "
                         f"heads), {t:.1f} s on {threads} host threads",
               "max_abs_err": err, "max_abs_err_over": f"{n * wl.num_q_heads * wl.head_dim} outputs "
                                                       f"({n} sequences x {wl.num_q_heads} heads x {wl.head_dim})"}
        if single_thread:
            # the same oracle on one thread, over fewer sequences (about 3 s)
            n1 = max(1, int(n * min(1.0, 3.0 / max(threads * t / reps, 1e-9))))
            dt1, b1, n1, _ = time_oracle(wl, n1, 1)
            cpu["single_thread"] = {"value": b1 / dt1 / 1e9, "unit": UNIT, "cores": 1,
                                    "sample": f"one oracle step over the first {n1} of {wl.num_seqs} sequences, "
                                              f"{dt1:.1f} s on 1 host thread"}

    res = {
        "value": value, "ms_per_step": ms_max / steps, "seq_per_s": seqs_all * steps / (ms_max / 1e3),
        "pct_of_hbm_peak": 100.0 * value / peak,
        "pct_of_nominal_hbm": 100.0 * value / NOMINAL_HBM_GBS,  # the part's nominal 8 TB/s, for context
        "config": {**describe(wl), "parallelism": f"replicas x{d.ws}" if d.ws > 1 else "single GPU",
                   "l2": ("256 MB written before every step, outside the step's timing" if args.flush_l2 else
                          f"no flush ({wl.kv_bytes() / 1e6:.0f} MB of K/V per step vs 129 MB of L2)"),
                   "api": " + ".join((["copy_blocks"] if cow is not None else []) +
                                     (["paged_kv_append"] if len(wl.slot_mapping) and not fused else []) + [dec_api]),
                   "partition_size": pkv.paged_attention_partition_size(
                       wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, mcl, args.partition_size),
                   "warmup_gpu_ms": warm_ms},
        "roofline": {"kernel": dec_api + (" (shared-prefix kernel + decode kernel + merge; bytes: each distinct "
                                          "K/V slot once)" if grouped else " (decode kernel + split-K merge)"),
                     "bound": "hbm",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_src, "traffic": traffic,
                     "algorithmic_bytes_per_launch": dec_bytes, "avg_launch_ms": dec_avg_ms},
        "stats": stats,
        "max_abs_err": cpu["max_abs_err"] if cpu else None,
        "e2e": {"value": kv_all * e2e_steps / (e2e_max / 1e3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "how": "one packed pinned-host->device copy of the step's inputs and one device->pinned-host copy "
                       "of its output per step, double-buffered on a copy stream; the K/V pool stays resident"},
        "gpu_launches": launches_all,
        "cpu_baseline": cpu,
        "dtype": wl.dtype,
    }
    del kc, vc, wsp, wsp2, d_in, d_out
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import torch

    import paged_kv_cache_11_gb300 as pkv
    from paged_kv_cache_11_gb300 import _build

    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(ws, "nccl")
    _build.build_all()
    pkv.binding._lib()

    extra = ([w for w in args.extra.split(",") if w] if args.extra is not None else
             (["llama8b"] if args.workload == "llama70b_long" else []))
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    d = Device(torch, pkv, dev, rank, ws, dist, clocks)
    main = measure(args.workload, args, d, cpu_seconds=10.0, single_thread=True)
    others = {w: measure(w, args, d, cpu_seconds=3.0, single_thread=False) for w in extra if w != args.workload}
    clk = clocks.stop() if clocks else None
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    line = {
        "metric": METRIC, "value": main["value"], "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": main["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": main["dtype"], "data": "synthetic",
        "config": main["config"], "seq_per_s": main["seq_per_s"],
        "pct_of_hbm_peak": main["pct_of_hbm_peak"], "pct_of_nominal_hbm": main["pct_of_nominal_hbm"],
        "roofline": main["roofline"], "stats": main["stats"], "max_abs_err": main["max_abs_err"],
        "e2e": main["e2e"], "gpu_launches": main["gpu_launches"], "clocks": clk,
        "cpu_baseline": main["cpu_baseline"],
    }
    if others:
        line["per_workload"] = {w: {k: v for k, v in r.items() if k != "dtype"} for w, r in others.items()}
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------- swap / compaction rows
def _timed(fn, steps, stream):
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_data_movement(args):
    """--workload swap: every block of the llama8b batch swapped out to a
    page-locked host pool and back in (swap_blocks), against one contiguous
    cudaMemcpyAsync of the same bytes each way.  --workload compact: each
    llama8b sequence keeps every other token, rewritten into fresh target
    blocks (compact_tokens), against the measured HBM copy peak."""
    import torch

    import paged_kv_cache_11_gb300 as pkv
    from paged_kv_cache_11_gb300 import _build, workload as W

    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build_all()
    pkv.binding._lib()
    wl = W.make_workload("llama8b")
    up = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)
    kc, vc = up(wl.k_cache), up(wl.v_cache)
    stream = torch.cuda.current_stream()
    bs = wl.block_size
    used = np.concatenate([wl.block_tables[s, :(int(L) + bs - 1) // bs] for s, L in enumerate(wl.context_lens)])
    block_bytes = 2 * wl.num_kv_heads * bs * wl.head_dim * 2
    peaks = measured_peaks()
    steps = max(1, min(args.steps, 50))
    l0 = pkv.launch_count()
    if args.workload == "swap":
        n = len(used)
        hk = torch.empty((n,) + tuple(kc.shape[1:]), dtype=kc.dtype).pin_memory()
        hv = torch.empty_like(hk).pin_memory()
        out_pairs = torch.from_numpy(np.stack([used, np.arange(n)], 1).astype(np.int64)).to(dev)
        in_pairs = torch.from_numpy(np.stack([np.arange(n), used], 1).astype(np.int64)).to(dev)
        for _ in range(3):
            pkv.swap_blocks(kc, vc, hk, hv, out_pairs)
            pkv.swap_blocks(hk, hv, kc, vc, in_pairs)
        t_out = _timed(lambda: pkv.swap_blocks(kc, vc, hk, hv, out_pairs), steps, stream)
        t_in = _timed(lambda: pkv.swap_blocks(hk, hv, kc, vc, in_pairs), steps, stream)
        nbytes = n * block_bytes
        flat_d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        flat_h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        m_out = _timed(lambda: flat_h.copy_(flat_d, non_blocking=True), steps, stream)
        m_in = _timed(lambda: flat_d.copy_(flat_h, non_blocking=True), steps, stream)
        assert pkv.check_device_error() == 0
        out_gbs, in_gbs = nbytes / t_out / 1e6, nbytes / t_in / 1e6
        line = {"metric": "swap_blocks GB/s (GPU pool <-> page-locked host pool)", "value": min(out_gbs, in_gbs),
                "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": 3, "higher_is_better": True,
                "dtype": "bf16", "data": "synthetic",
                "config": {"workload": "swap", "blocks": n, "bytes_each_way": nbytes, "block_bytes": block_bytes,
                           "source": "every block of the llama8b batch"},
                "swap_out_gbs": out_gbs, "swap_in_gbs": in_gbs,
                "roofline": {"bound": "c2c", "unit": "GB/s",
                             "peak_out": nbytes / m_out / 1e6, "peak_in": nbytes / m_in / 1e6,
                             "frac_out": out_gbs / (nbytes / m_out / 1e6), "frac_in": in_gbs / (nbytes / m_in / 1e6),
                             "peak_source": "one contiguous cudaMemcpyAsync of the same bytes, measured here"},
                "gpu_launches": pkv.launch_count() - l0}
    else:
        srcs, dsts = [], []
        base = wl.num_blocks  # targets in a second pool half, so no target is a source
        for s, L in enumerate(wl.context_lens):
            keep = np.arange(0, int(L), 2)
            t0 = len(dsts)
            srcs += [int(wl.block_tables[s, p // bs]) * bs + int(p) % bs for p in keep]
            dsts += [(base + (t0 + i) // bs) * bs + (t0 + i) % bs for i in range(len(keep))]
        kc2 = torch.cat([kc, torch.empty_like(kc)])
        vc2 = torch.cat([vc, torch.empty_like(vc)])
        a = torch.tensor(srcs, dtype=torch.int64, device=dev)
        b = torch.tensor(dsts, dtype=torch.int64, device=dev)
        for _ in range(3):
            pkv.compact_tokens(a, b, kc2, vc2)
        t = _timed(lambda: pkv.compact_tokens(a, b, kc2, vc2), steps, stream)
        assert pkv.check_device_error() == 0
        nbytes = len(srcs) * 2 * wl.num_kv_heads * wl.head_dim * 2 * 2 + 2 * 8 * len(srcs)  # read+write K,V + slots
        gbs = nbytes / t / 1e6
        peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
        line = {"metric": "compact_tokens GB/s (token rows moved into fresh target blocks)", "value": gbs,
                "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": 3, "higher_is_better": True,
                "dtype": "bf16", "data": "synthetic",
                "config": {"workload": "compact", "tokens": len(srcs), "kept": "every other token of each "
                           "llama8b sequence"},
                "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                             "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": t},
                "gpu_launches": pkv.launch_count() - l0}
    print(json.dumps(line))
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.workload in ("swap", "compact"):
        return run_data_movement(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
