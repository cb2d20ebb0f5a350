#!/usr/bin/env python3
"""Benchmark of paged GQA split-KV decode attention on GB300.

A step is the whole hot path over one batch: the new token's RoPE + K/V
append, the split-KV decode and the merge of the split partials, as one
paged_decode_step call (split count from the library's planner).

Headline workload: the largest single-GPU configuration, the serving mix at
B=128 (Hq=64, Hkv=8, D=128, page_size=16, lognormal lengths, a quarter of the
rows padding at seq_len 0).  Its K+V (598 MB) is several times the L2, so its
steps run back to back inside CUDA-graph replays with no flush: a step finds
none of the previous step's K/V in L2.  The timed region holds exactly
--steps steps, in at least 10 replays of `inner` steps; the line reports the
region's mean per step and the replays' median, min and max.

``value`` is the KV-read throughput: the bytes of K and V the attention must
read (every token of every row, every kv head) divided by the step time,
summed over ranks.

Every other seeded configuration is measured in the same run (``configs``):
tiny, gqa_1b, ragged_b32, long_32k and the serving mix at B=1..64.  Inputs of
at least twice the L2 run back to back as above; smaller ones are timed two
ways: "rotation" (consecutive steps each read their own copy of the pools, as
consecutive layers of a model do, the copies holding at least 3x L2) and
"flushed" (one step per replay, the L2 flushed before it, outside the events).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--configs all|none|NAME,...] [--impl pkv|reference]

``--impl reference`` times the fp64 CPU oracle on the host cores instead (a
bounded sample of the same workload each step).  Under torchrun (N > 1)
each rank runs an independent replica on its own GPU (replicas only: the
path has no exchange step); timings are max-reduced over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged GQA decode attn: µs/call and KV-read GB/s (% of GB300 HBM peak)"
FALLBACK_HBM_GBS = 6800.0
HEADLINE = "serving_b128"
# layers of the pages' 1.2B model: the calls of one decode step in a replay
LAYERS = 24
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fused_decode_traffic.json")
DECODE_SRC = os.path.join(ROOT, "paged_kv_gqa_16_gb300", "csrc", "pkv_fused.cu")


def config_names():
    from paged_kv_gqa_16_gb300 import workloads as wl
    return ["tiny", "gqa_1b", "ragged_b32", "long_32k"] + [f"serving_b{B}"
                                                          for B in wl.SERVING_BATCHES]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--configs", default="all",
                    help="the per-configuration map: all, none, or a comma list of names")
    ap.add_argument("--splits", type=int, default=0, help="override the planner's split count")
    ap.add_argument("--pool-pages", type=int, default=0,
                    help="pool size of the headline workload (smaller pools for profiling)")
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layout", choices=["paged", "contig"], default="paged",
                    help="contig: the same rows in a contiguous cache [B, max_seq_len, Hkv, D] "
                         "through decode_attn_contig")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the prefill leg (paged_prefill_attn on three shapes)")
    ap.add_argument("--only-prefill", default=None,
                    choices=["all", "prefill_b32_512", "prefill_b4_4096", "extend_b16"],
                    help="run only the prefill leg on one shape (or all) and print its line")
    ap.add_argument("--no-loop", action="store_true",
                    help="skip the decode-loop leg (paged_kv_advance + step per graph)")
    ap.add_argument("--no-flush", action="store_true", help="skip the L2 flush (not for reporting)")
    ap.add_argument("--no-plan", action="store_true",
                    help="the unplanned calls (each computes the partition itself)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the all-core oracle baseline sample")
    ap.add_argument("--cpu-seconds-1t", type=float, default=6.0,
                    help="target CPU time of the one-thread oracle baseline sample")
    return ap.parse_args(argv)


def config_of(w, gpus: int, layout: str = "paged") -> dict:
    """The workload as the JSON line names it (the same for both arms)."""
    return {"workload": w.name + ("" if layout == "paged" else " (contiguous cache)"),
            "layout": layout, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
            "page_size": w.page_size, "num_pages": w.num_pages, "tokens": w.total_tokens,
            "live_rows": int((w.seq_lens > 0).sum()), "kv_bytes": w.kv_bytes(),
            "max_seq_len": w.max_seq_len, "parallelism": f"replicas x{gpus}"}


def alg_bytes_of(w) -> int:
    """Algorithmic bytes of one step: K and V of every token, q in and the
    output, the new token's K/V read and written to its slot, and the page
    tables (kv_indices, kv_indptr, seq_lens)."""
    n_idx = int(w.kv_indices.numel())
    return (w.kv_bytes() + w.B * w.Hq * w.D * 2 * 2 + w.B * w.Hkv * w.D * 2 * 2 * 2
            + 4 * n_idx + 8 * w.B)


# --------------------------------------------------------------------------
def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world <= 1:
        return
    import torch.distributed as dist
    if device is not None and dist.get_backend() == "nccl":
        dist.barrier(device_ids=[device.index])
    else:
        dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def load_bf16_peak() -> float:
    """Measured dense bf16 TFLOP/s (burst), else the fallback 1900."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def cached_traffic(workload: str, splits: int):
    """DRAM bytes per launch of the fused decode kernel from a committed ncu
    summary, valid only while the kernel source is unchanged (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            j = json.load(f)
        src_hash = hashlib.sha256(open(DECODE_SRC, "rb").read()).hexdigest()
        if j.get("source_sha256") != src_hash:
            return None
        e = j.get("workloads", {}).get(workload)
        if e is None or (e.get("splits") not in (None, splits)):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


def measure_read_peak(dev, stream, reps=10):
    """GB/s of a plain streaming read on this GPU: torch.sum over a 4 GiB
    float32 buffer (32x L2), median of `reps` timed with events."""
    import torch
    buf = torch.ones(1 << 30, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    for _ in range(3):
        torch.sum(buf, dim=0, out=sink)
    ms = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        torch.sum(buf, dim=0, out=sink)
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms.append(a.elapsed_time(b))
    del buf
    return buf_bytes_gbs(1 << 32, statistics.median(ms))


def buf_bytes_gbs(nbytes, ms):
    return nbytes / (ms * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self, t0=None, t1=None):
        """Median SM clock and active throttle reasons over the samples read
        inside [t0, t1] (host perf_counter times)."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if t0 is not None and not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_sample(w, target_s: float, max_reps: int = 1000, threads: int | None = None):
    """Time the fp64 oracle's step (append + decode) on the host cores over a
    bounded sample of the workload: whole rows, taken in order until their
    estimated cost reaches the target, repeated while time remains."""
    import numpy as np
    import oracle

    cores = cpu_cores() if threads is None else threads
    oracle.set_threads(cores)
    kp, vp, idx = w.compact_host()
    lens = w.seq_lens.numpy()
    ptr = w.kv_indptr.numpy()

    def run(rows):
        b0, b1 = rows
        sub_ptr = (ptr[b0:b1 + 1] - ptr[b0]).astype(np.int32)
        p0, p1 = int(ptr[b0]), int(ptr[b1])
        sl = lens[b0:b1].astype(np.int32)
        q2, kp2, vp2 = oracle.append(w.host("q")[b0:b1], w.host("k_new")[b0:b1],
                                     w.host("v_new")[b0:b1], kp[p0:p1], vp[p0:p1],
                                     np.arange(p1 - p0, dtype=np.int32), sub_ptr, sl,
                                     rope_base=w.rope_base, rope_q=True)
        oracle.decode(q2, kp2, vp2, np.arange(p1 - p0, dtype=np.int32), sub_ptr, sl, w.scale)
        return int(sl.sum())

    # calibrate on the first row
    t0 = time.perf_counter()
    tok1 = run((0, 1))
    dt1 = max(time.perf_counter() - t0, 1e-6)
    per_tok = dt1 / max(tok1, 1)
    budget_tok = target_s / per_tok
    b1 = 1
    while b1 < w.B and lens[:b1 + 1].sum() <= budget_tok:
        b1 += 1
    tokens = 0
    t0 = time.perf_counter()
    reps = 0
    while True:
        tokens += run((0, b1))
        reps += 1
        el = time.perf_counter() - t0
        if el >= target_s or reps >= max_reps:
            break
    el = time.perf_counter() - t0
    bytes_kv = tokens * w.Hkv * w.D * 2 * 2
    return {"seconds": el, "tokens": tokens, "rows": b1, "reps": reps, "cores": cores,
            "gbs": bytes_kv / el / 1e9}


# --------------------------------------------------------------------------
def run_reference(args):
    """The oracle, timed as the reference arm: each step is a bounded sample
    of the workload on the host cores."""
    rank, world, _ = dist_info()
    if rank != 0:
        return 0
    from paged_kv_gqa_16_gb300 import workloads as wl
    import oracle
    oracle.build()
    w = wl.make(args.workload)
    steps, warm = max(1, args.steps), max(0, args.warmup)
    # keep the whole run within a few minutes: per-step sample ~ budget/(steps+warm)
    per_step = max(0.05, min(2.0, 120.0 / (steps + warm)))
    for _ in range(min(warm, 3)):
        oracle_sample(w, per_step, max_reps=1)
    tot_s, tot_tok = 0.0, 0
    res = None
    for _ in range(steps):
        res = oracle_sample(w, per_step, max_reps=1)
        tot_s += res["seconds"]
        tot_tok += res["tokens"]
    gbs = tot_tok * w.Hkv * w.D * 4 / tot_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": warm,
        "ms_per_step": round(1e3 * tot_s / steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args.gpus, args.layout),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": res["cores"],
                         "kind": "oracle",
                         "sample": f"fp64 oracle append+decode on rows 0..{res['rows'] - 1} of "
                                   f"{w.name} per step"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def prefill_leg(pkv, wl, dev, stream, flush_l2, rank, names, reps=20):
    """paged_prefill_attn_ws (the prefill with its key-split workspace) on each
    named shape: one call per graph replay, the L2 flushed before each,
    median of `reps`; tensor roofline against the measured dense bf16 peak
    (burst: each call runs alone)."""
    import torch
    tf_peak = load_bf16_peak()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out_rows = []
    for name in names:
        label, kw = wl.PREFILL_SHAPES[name]
        c = wl.prefill_shape(name, seed=rank)
        pt = c.w.to_device(dev)
        pd = pkv.dims(c.w.B, c.w.Hq, c.w.Hkv, c.w.D, c.w.page_size, pt["k_pool"].shape[0],
                      int(c.w.kv_indices.numel()), c.w.max_seq_len, c.w.scale)
        pq, pqo = c.q.to(dev), c.qo_indptr.to(dev)
        pout = torch.empty(c.total_q, c.w.Hq, c.w.D, dtype=torch.bfloat16, device=dev)
        pst = torch.zeros(1, dtype=torch.int32, device=dev)
        max_q = max(kw["q_lens"])
        pws = torch.empty(pkv.prefill_workspace_bytes(c.w.D, sms), dtype=torch.uint8,
                          device=dev)

        def prun():
            pkv.paged_prefill_attn(pd, pq, pqo, pt["k_pool"], pt["v_pool"], pt["kv_indices"],
                                   pt["kv_indptr"], pt["seq_lens"], pout, status=pst,
                                   max_q_len=max_q, workspace=pws)

        for _ in range(3):
            prun()
        pg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(pg):
            prun()
        ms = []
        for _ in range(reps + 3):
            flush_l2()
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            pg.replay()
            e.record(stream)
            torch.cuda.synchronize(dev)
            ms.append(a.elapsed_time(e))
        if int(pst.item()) != 0:
            raise SystemExit(f"prefill status {int(pst.item()):#x}")
        us = 1e3 * statistics.median(ms[3:])
        tf = c.flops() / (us * 1e-6) / 1e12
        out_rows.append({"shape": label, "us": round(us, 1), "tflops": round(tf, 1),
                         "roofline": {"bound": "tensor", "achieved": round(tf, 1),
                                      "peak": tf_peak, "unit": "TFLOP/s",
                                      "frac": round(tf / tf_peak, 4)},
                         "flops": c.flops()})
        del pt, pg, pws
    return out_rows


def run_prefill_only(args):
    """--only-prefill: the prefill leg alone, one JSON line (for profiling)."""
    import torch
    from paged_kv_gqa_16_gb300 import build as pkv_build
    from paged_kv_gqa_16_gb300 import pkv
    from paged_kv_gqa_16_gb300 import workloads as wl
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pkv_build.build()
    pkv.lib()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device=dev)
    sink = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=sink)

    names = list(wl.PREFILL_SHAPES) if args.only_prefill == "all" else [args.only_prefill]
    rows = prefill_leg(pkv, wl, dev, torch.cuda.current_stream(dev), flush_l2, 0, names,
                       reps=max(1, args.steps))
    print(json.dumps({"metric": "paged prefill / extend attention TFLOP/s", "unit": "TFLOP/s",
                      "n_gpus": 1, "prefill": rows}), flush=True)
    return 0


# --------------------------------------------------------------------------
class StepState:
    """Device state of one workload for timing paged_decode_step: ``copies``
    pairs of K/V pools (the layers of one decode step: each its own pools,
    all named by one page table), the shared q / new K/V / lengths / table,
    the workspace (which holds the step's plan), the RoPE table and the
    output.  A decode step's first call computes the block partition and
    leaves it in the workspace as the plan; with ``planned`` the step's later
    calls (its other layers) run on that plan."""

    def __init__(self, pkv, w, dev, copies: int = 1, pool_pages: int = 0, splits: int = 0,
                 planned: bool = True):
        import torch
        P = pool_pages or w.num_pages
        self.w, self.dev, self.copies, self.P, self.planned = w, dev, copies, P, planned
        shape = (P, w.page_size, w.Hkv, w.D)
        idx = w.kv_indices.to(device=dev, dtype=torch.long)
        self.k_pools, self.v_pools = [], []
        kpg = w.k_pages.to(dev) if idx.numel() else None
        vpg = w.v_pages.to(dev) if idx.numel() else None
        for _ in range(copies):
            kp = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=dev)
            vp = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=dev)
            if idx.numel():
                kp[idx] = kpg
                vp[idx] = vpg
            self.k_pools.append(kp)
            self.v_pools.append(vp)
        del kpg, vpg
        self.k_pool, self.v_pool = self.k_pools[0], self.v_pools[0]
        self.kv_indices = w.kv_indices.to(dev)
        self.q = w.q.to(dev).contiguous()
        self.k_new = w.k_new.to(dev).contiguous()
        self.v_new = w.v_new.to(dev).contiguous()
        self.kv_indptr = w.kv_indptr.to(dev)
        self.seq_lens = w.seq_lens.to(dev)
        self.d = pkv.dims(w.B, w.Hq, w.Hkv, w.D, w.page_size, P, int(w.kv_indices.numel()),
                          w.max_seq_len, w.scale)
        self.S = splits or pkv.plan(self.d)[0]
        self.ws = pkv.alloc_workspace(self.d, self.S, dev)
        self.rope_rows = max(w.max_seq_len, 1)
        self.rope = torch.empty(self.rope_rows, w.D // 2, 2, dtype=torch.float32, device=dev)
        pkv.rope_table(self.rope, self.rope_rows, w.D, w.rope_base or 10000.0)
        self.out = torch.empty(w.B, w.Hq, w.D, dtype=torch.bfloat16, device=dev)
        self.pkv = pkv

    def plan(self, args=None):
        """The step's plan (once per decode step, for every layer's call)."""
        if not self.planned:
            return
        kv_indices, kv_indptr, seq_lens = args or (self.kv_indices, self.kv_indptr,
                                                   self.seq_lens)
        self.pkv.paged_decode_plan(self.d, kv_indices, kv_indptr, seq_lens, self.S, self.ws)

    def step(self, i: int = 0, args=None, planned: bool = False, out=None):
        """paged_decode_step on layer i's pools (or on the given device
        inputs, into the given output); planned: on the plan the step's first
        call left behind."""
        q, k_new, v_new, kv_indices, kv_indptr, seq_lens = args or (
            self.q, self.k_new, self.v_new, self.kv_indices, self.kv_indptr, self.seq_lens)
        fn = (self.pkv.paged_decode_step_planned if planned and self.planned
              else self.pkv.paged_decode_step)
        fn(self.d, q, k_new, v_new, self.k_pools[i], self.v_pools[i], kv_indices, kv_indptr,
           seq_lens, self.rope, self.rope_rows, self.S, self.ws,
           self.out if out is None else out)

    def decode(self, i: int = 0, planned: bool = False):
        fn = (self.pkv.paged_decode_attn_planned if planned and self.planned
              else self.pkv.paged_decode_attn)
        fn(self.d, self.q, self.k_pools[i], self.v_pools[i], self.kv_indices, self.kv_indptr,
           self.seq_lens, self.S, self.ws, self.out)

    def check_status(self, what: str):
        s = self.pkv.status_word(self.ws)
        if s != 0:
            raise SystemExit(f"device status {s:#x} {what}")


def capture(fn, n: int, first=None):
    """One CUDA graph holding first() (if given) and then n calls of fn(k),
    k = 0..n-1."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        if first is not None:
            first()
        for k in range(n):
            fn(k)
    return g


def replay_times(graph, reps: int, stream, dev, flush=None):
    """Milliseconds of each of `reps` replays (events on the replay stream),
    with `flush` run before each replay, outside the events."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for a, b in evs:
        if flush is not None:
            flush()
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    return [a.elapsed_time(b) for a, b in evs]


def rotation_copies(kv_bytes: int, l2: int) -> int:
    """Copies of the pools whose K+V together hold at least 3x L2 (2..64)."""
    return max(2, min(64, -(-3 * l2 // max(kv_bytes, 1))))


def measure_config(pkv, w, dev, stream, l2, flush_l2, peak, splits=0):
    """µs per paged_decode_step of one workload, with KV GB/s and the
    fraction of the HBM peak, timed as the module docstring describes: in
    each replay the first call computes the partition and leaves it as the
    plan, the later calls (the step's other layers) run on it; every call
    unplanned is timed the same way for reference."""
    import torch
    kv = w.kv_bytes()
    alg = alg_bytes_of(w)
    b2b = kv >= 2 * l2
    copies = 1 if b2b else rotation_copies(kv, l2)
    st = StepState(pkv, w, dev, copies=copies, splits=splits)
    st.plan()
    for i in range(copies):
        st.step(i)
    torch.cuda.synchronize(dev)
    st.check_status(f"after warm-up of {w.name}")

    def line(ms, mode, extra=None):
        r = {"us_per_call": round(1e3 * ms, 2),
             "kv_gbs": round(kv / (ms * 1e-3) / 1e9, 1),
             "pct_hbm": round(100.0 * kv / (ms * 1e-3) / 1e9 / peak, 1),
             "roofline_frac": round(alg / (ms * 1e-3) / 1e9 / peak, 4),
             "l2": mode}
        r.update(extra or {})
        return r

    def per_step(n, planned, flush=None, reps=15):
        # the step's first call writes the plan, its later calls run on it
        st.planned = planned
        g = capture(lambda k: st.step(k % copies, planned=k > 0), n)
        replay_times(g, 3, stream, dev, flush)
        ms = [t / n for t in replay_times(g, reps, stream, dev, flush)]
        del g
        return statistics.median(ms)

    out = {"splits": st.S, "kv_bytes": kv, "alg_bytes": alg, "tokens": w.total_tokens}
    # a replay is one decode step of a 24-layer model (the pages' 1.2B model)
    if b2b:
        n = LAYERS
        mode = (f"back to back, {n} steps per replay (the first leaves the plan), "
                f"K+V = {kv / l2:.1f} x L2, no flush")
    else:
        n = -(-LAYERS // copies) * copies
        mode = (f"rotation over {copies} layers' pools ({copies * kv / l2:.1f} x L2 of K+V), "
                f"{n} steps per replay (the first leaves the plan)")
    out.update(line(per_step(n, True), mode, {"replays": 15}))
    out["unplanned_us"] = round(1e3 * per_step(n, False), 2)
    if not b2b:
        out["flushed"] = line(per_step(1, True, flush_l2, 30),
                              "one (unplanned) step per replay, L2 flushed before it "
                              "(outside the events)", {"replays": 30})
    # paged_decode_plan alone (for callers that plan ahead of a step)
    st.planned = True
    gp = capture(lambda k: st.plan(), 1)
    replay_times(gp, 3, stream, dev)
    out["plan_us"] = round(1e3 * statistics.median(replay_times(gp, 20, stream, dev)), 2)
    torch.cuda.synchronize(dev)
    st.check_status(f"after timing {w.name}")
    del gp, st
    torch.cuda.empty_cache()
    return out


def pick_inner(K: int) -> int:
    """Steps per timed replay: the largest divisor of K that is at most
    min(20, K // 10), so the K timed steps form at least 10 replays."""
    cap = max(1, min(20, K // 10))
    for d in range(cap, 0, -1):
        if K % d == 0:
            return d
    return 1


def run_pkv(args):
    import numpy as np
    import torch
    from paged_kv_gqa_16_gb300 import build as pkv_build
    from paged_kv_gqa_16_gb300 import pkv
    from paged_kv_gqa_16_gb300 import workloads as wl

    rank, world, local = dist_info()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    if rank == 0:
        pkv_build.build()
    barrier(world, dev)
    pkv.lib()
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = load_peaks()

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2():
        """Evict the L2: write a buffer of twice its size, then read another
        of the same size so the lines left behind are clean (a dirty L2 would
        charge its write-back to the next timed kernel)."""
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_sink)

    # ---- the headline workload: each rank an independent replica (own seed)
    kw = {"num_pages": args.pool_pages} if args.pool_pages else {}
    w = wl.make(args.workload, seed=rank, **kw)
    st = StepState(pkv, w, dev, copies=1, splits=args.splits, planned=not args.no_plan)
    d, S = st.d, st.S
    step = st.step
    decode = st.decode
    plan = st.plan
    if args.layout == "contig":
        # the same rows in a contiguous cache: slot b holds row b's tokens in
        # order (gathered from its pages), NaN past them
        cache_len = w.max_seq_len
        ck = torch.full((w.B, cache_len, w.Hkv, w.D), float("nan"), dtype=torch.bfloat16,
                        device=dev)
        cv = torch.full_like(ck, float("nan"))
        ptr_h = w.kv_indptr.tolist()
        for b in range(w.B):
            L = int(w.seq_lens[b])
            if L == 0:
                continue
            pages = st.kv_indices[ptr_h[b]:ptr_h[b + 1]].long()
            ck[b, :L] = st.k_pool[pages].reshape(-1, w.Hkv, w.D)[:L]
            cv[b, :L] = st.v_pool[pages].reshape(-1, w.Hkv, w.D)[:L]
        del st.k_pool, st.v_pool, st.k_pools, st.v_pools
        torch.cuda.empty_cache()
        cd = pkv.dims(w.B, w.Hq, w.Hkv, w.D, cache_len, w.B, w.B, cache_len, w.scale)
        cws = pkv.alloc_workspace(cd, S, dev)
        st.ws = cws

        use_plan = not args.no_plan

        def step(i=0, a=None, planned=False):
            pkv.decode_attn_contig(cd, st.q, ck, cv, st.seq_lens, S, cws, st.out,
                                   k_new=st.k_new, v_new=st.v_new, rope_cos_sin=st.rope,
                                   rope_max_pos=st.rope_rows, planned=planned and use_plan)

        def decode(i=0, planned=False):
            pkv.decode_attn_contig(cd, st.q, ck, cv, st.seq_lens, S, cws, st.out,
                                   planned=planned and use_plan)

        args.no_e2e = True
        args.no_loop = True
        args.configs = "none"

    # (a contiguous cache adds its table launch to a step's first call only)
    launches_per_step = (1 if S == 1 else 2)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    st.check_status("after warm-up")

    kv_bytes = w.kv_bytes()
    alg_bytes = alg_bytes_of(w)
    back_to_back = kv_bytes >= 2 * l2
    K = max(1, args.steps)
    inner = pick_inner(K)
    reps = K // inner
    # each replay: `inner` steps of one decode step's metadata; the first
    # leaves the plan, the others run on it (unless --no-plan)
    g_step = capture(lambda k: step(0, None, k > 0), inner)
    replay_times(g_step, 3, stream, dev)
    est_ms = statistics.median(replay_times(g_step, 3, stream, dev))
    flush = None if (back_to_back or args.no_flush) else flush_l2

    # Timed region: exactly K steps in `reps` replays.  The clock sampler
    # runs across an untimed burst of the same replays just before it (the
    # region itself can be a few milliseconds, shorter than the sampling
    # period) and across the region.
    with ClockSampler(dev.index) as clk:
        time.sleep(0.3)              # let the sampler start
        t_clk0 = time.perf_counter()
        n_burst = max(1, int(0.8 / max(est_ms * 1e-3, 1e-6)))
        for _ in range(n_burst):
            if flush is not None:
                flush()
            g_step.replay()
        barrier(world, dev)
        torch.cuda.synchronize(dev)
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        wall0 = time.perf_counter()
        e_start.record(stream)
        for a, b in evs:
            if flush is not None:
                flush()
            a.record(stream)
            g_step.replay()
            b.record(stream)
        e_end.record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
        barrier(world, dev)
        t_clk1 = time.perf_counter()
        time.sleep(0.1)
    per_step = [a.elapsed_time(b) / inner for a, b in evs]
    # with flushes inside the region, its span includes them: use the replays
    ms_region = (e_start.elapsed_time(e_end) / K) if flush is None else statistics.mean(per_step)
    ms_step_max = reduce_max(ms_region, world, dev)
    st.check_status("after the timed run")
    clocks = clk.summary(t_clk0, t_clk1)
    clocks["window"] = (f"{n_burst} untimed replays just before the timed region, "
                        "then the timed region")

    total_bytes = kv_bytes * world
    value = total_bytes / (ms_step_max * 1e-3) / 1e9

    # decode-only and a cold single step (L2 flushed before it) on the same rows
    g_dec = capture(lambda k: decode(0, k > 0), inner)
    replay_times(g_dec, 3, stream, dev)
    ms_dec = statistics.median(t / inner for t in replay_times(g_dec, max(10, reps), stream,
                                                              dev, flush))
    g_one = capture(lambda k: step(), 1)
    replay_times(g_one, 3, stream, dev, flush_l2)
    ms_cold = statistics.median(replay_times(g_one, 30, stream, dev, flush_l2))
    ms_dec_max = reduce_max(ms_dec, world, dev)
    ms_cold_max = reduce_max(ms_cold, world, dev)
    del g_dec, g_one

    # e2e: host (pinned) inputs copied in, the step, the output copied back,
    # for every step.  A step's inputs sit in one pinned host block (each at a
    # 256-byte aligned offset), copied with one H2D copy into a device block
    # the step reads through views; its output is copied back with one D2H
    # copy.  As a serving loop does, the copies are double-buffered on two
    # copy streams: the next step's inputs come in while a step computes, and
    # the previous step's output goes out meanwhile.  E_STEPS steps (each an
    # unplanned call: a new decode step's inputs) are captured in one CUDA
    # graph; the per-step time is a replay's time over E_STEPS, so the first
    # copy in and the last copy out of each replay are counted.
    e2e = None
    if not args.no_e2e and args.layout == "paged":
        E_STEPS = 10
        names = ("q", "k_new", "v_new", "kv_indices", "kv_indptr", "seq_lens")
        srcs = {k: getattr(w, k).contiguous() for k in names}
        offs, blk_bytes = {}, 0
        for k in names:
            offs[k] = blk_bytes
            blk_bytes += (srcs[k].numel() * srcs[k].element_size() + 255) // 256 * 256

        def blk_view(blk, k):
            nb = srcs[k].numel() * srcs[k].element_size()
            return blk[offs[k]:offs[k] + nb].view(srcs[k].dtype).view(srcs[k].shape)

        host_blk = torch.zeros(blk_bytes, dtype=torch.uint8).pin_memory()
        for k in names:
            blk_view(host_blk, k).copy_(srcs[k])
        dev_blks = [torch.empty(blk_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
        e_args = [tuple(blk_view(bk, k) for k in names) for bk in dev_blks]
        outs = [torch.empty_like(st.out) for _ in range(2)]
        out_hosts = [torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
                     for _ in range(2)]
        h2d = blk_bytes
        d2h = out_hosts[0].numel() * out_hosts[0].element_size()
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e):
            main = torch.cuda.current_stream(dev)
            s_in.wait_stream(main)
            s_out.wait_stream(main)
            ev_step, ev_out = [], []
            for i in range(E_STEPS):
                b = i % 2
                ev_in = torch.cuda.Event()
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_step[i - 2])    # the block's last reader
                    dev_blks[b].copy_(host_blk, non_blocking=True)
                    ev_in.record(s_in)
                main.wait_event(ev_in)
                if i >= 2:
                    main.wait_event(ev_out[i - 2])         # the output's last copy out
                step(0, e_args[b], False, outs[b])
                e_s = torch.cuda.Event()
                e_s.record(main)
                ev_step.append(e_s)
                e_o = torch.cuda.Event()
                with torch.cuda.stream(s_out):
                    s_out.wait_event(e_s)
                    out_hosts[b].copy_(outs[b], non_blocking=True)
                    e_o.record(s_out)
                ev_out.append(e_o)
            main.wait_stream(s_in)
            main.wait_stream(s_out)
        replay_times(g_e2e, 3, stream, dev)
        Ke = max(10, min(K // E_STEPS, 50))
        e_ms = statistics.mean(replay_times(g_e2e, Ke, stream, dev, flush)) / E_STEPS
        e_ms = reduce_max(e_ms, world, dev)
        torch.cuda.synchronize(dev)
        if not torch.equal(out_hosts[(E_STEPS - 1) % 2].view(torch.int16),
                           outs[(E_STEPS - 1) % 2].cpu().view(torch.int16)):
            raise SystemExit("e2e: the output copied back differs from the device output")
        e2e = {"value": round(total_bytes / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(e_ms, 5), "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h,
               "path": (f"per step: pinned host block -> one H2D copy, the step "
                        f"(paged_decode_step), one D2H copy of the output; copies "
                        f"double-buffered on two copy streams, overlapping the neighbouring "
                        f"steps; {E_STEPS} steps per CUDA graph replay")}
        del g_e2e, dev_blks
        st.check_status("after the e2e leg")

    plan_us = None
    if st.planned:
        gp = capture(lambda k: plan(), 1)
        replay_times(gp, 3, stream, dev)
        plan_us = round(1e3 * statistics.median(replay_times(gp, 20, stream, dev)), 2)
        del gp
    achieved = alg_bytes / (ms_region * 1e-3) / 1e9
    read_peak = measure_read_peak(dev, stream)
    traffic = cached_traffic(w.name, S) if args.layout == "paged" else None
    del g_step
    planned = st.planned
    st_config = config_of(w, world, args.layout)
    del st
    torch.cuda.empty_cache()

    # ---- every seeded configuration -------------------------------------
    configs = {}
    ragged = None
    if args.configs != "none":
        names_c = config_names() if args.configs == "all" else args.configs.split(",")
        for name in names_c:
            wc = wl.make(name, seed=rank)
            configs[name] = measure_config(pkv, wc, dev, stream, l2, flush_l2, peak)
            if name == "ragged_b32":
                ragged = wc
            del wc

    # decode loop: the ragged rows as a loop whose table grows on the device.
    # LOOP steps per graph, each paged_kv_advance + paged_decode_step (the
    # step's new token at the advanced length), against the same graph
    # without the advance; the small state is reset between replays, outside
    # the events, and nothing is flushed (consecutive steps, as in serving).
    loop = None
    if not args.no_loop:
        wr = ragged if ragged is not None else wl.make("ragged_b32", seed=rank)
        LOOP, lreps = 20, 20
        before = (wr.seq_lens - 1).clamp(min=0).tolist()     # cached tokens before a step
        held_max = max(-(-L // wr.page_size) for L in before)
        cap = held_max + -(-LOOP // wr.page_size) + 2
        need = sum(-(-L // wr.page_size) for L in before) + wr.B * (-(-LOOP // wr.page_size) + 1)
        ls = wl.decode_loop(B=wr.B, Hq=wr.Hq, Hkv=wr.Hkv, D=wr.D, page_size=wr.page_size,
                            seq_lens=before, steps=LOOP, cap=cap, num_pages=need + 64,
                            seed=1000 + rank)

        def t16(a):
            return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(dev)

        ld = pkv.dims(wr.B, wr.Hq, wr.Hkv, wr.D, wr.page_size, ls.num_pages, len(ls.kv_indices),
                      ls.max_seq_len, wr.scale)
        lS = args.splits or pkv.plan(ld)[0]
        lws = pkv.alloc_workspace(ld, lS, dev)
        lq, lkn, lvn = t16(ls.q), t16(ls.k_new), t16(ls.v_new)
        lkp, lvp = t16(ls.k_pool), t16(ls.v_pool)
        lrope = torch.empty(ls.max_seq_len, wr.D // 2, 2, dtype=torch.float32, device=dev)
        pkv.rope_table(lrope, ls.max_seq_len, wr.D, wr.rope_base or 10000.0)
        lsl0 = torch.from_numpy(ls.seq_lens).to(dev)
        lind0 = torch.from_numpy(ls.kv_indices).to(dev)
        lsl, lind = lsl0.clone(), lind0.clone()
        lptr = torch.from_numpy(ls.kv_indptr).to(dev)
        lfree = torch.from_numpy(ls.free_pages).to(dev)
        lhead = torch.zeros(1, dtype=torch.int32, device=dev)
        lout = torch.empty(wr.B, wr.Hq, wr.D, dtype=torch.bfloat16, device=dev)

        def one(stp, adv):
            if adv == "fused":
                # the loop opens with one advance; each step then advances
                # for the next inside its own combine launch
                if stp == 0:
                    pkv.paged_kv_advance(ld, lsl, lptr, lind, lfree, lhead, status=lws)
                pkv.paged_decode_step_advance(ld, lq, lkn[stp], lvn[stp], lkp, lvp, lind, lptr,
                                              lsl, lrope, ls.max_seq_len, lS, lws, lout,
                                              lfree, lhead)
                return
            if adv:
                pkv.paged_kv_advance(ld, lsl, lptr, lind, lfree, lhead, status=lws)
            pkv.paged_decode_step(ld, lq, lkn[stp], lvn[stp], lkp, lvp, lind, lptr, lsl, lrope,
                                  ls.max_seq_len, lS, lws, lout)

        def reset():
            lsl.copy_(lsl0)
            lind.copy_(lind0)
            lhead.zero_()

        def loop_graph(adv):
            reset()
            for stp in range(LOOP):
                one(stp, adv)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for stp in range(LOOP):
                    one(stp, adv)
            return g

        def loop_timed(g):
            ms = []
            for _ in range(lreps + 3):
                reset()
                ms.append(replay_times(g, 1, stream, dev)[0] / LOOP)
            return statistics.median(ms[3:])

        g_adv, g_noadv, g_fused = loop_graph(True), loop_graph(False), loop_graph("fused")
        ms_adv = loop_timed(g_adv)
        pages_taken = int(lhead.item())
        ms_fused = loop_timed(g_fused)
        ms_noadv = loop_timed(g_noadv)
        if pkv.status_word(lws) != 0:
            raise SystemExit(f"device status {pkv.status_word(lws):#x} after the loop leg")
        loop = {"workload": wr.name, "steps_per_graph": LOOP, "replays": lreps,
                "us_per_step": round(1e3 * ms_adv, 2),
                "us_per_step_without_advance": round(1e3 * ms_noadv, 2),
                "advance_us": round(1e3 * (ms_adv - ms_noadv), 2),
                "us_per_step_fused_advance": round(1e3 * ms_fused, 2),
                "fused_advance_us": round(1e3 * (ms_fused - ms_noadv), 2),
                "pages_taken_per_replay": pages_taken,
                "note": "same rows; table strided with room to grow; steps back to back, "
                        "no flush; fused: paged_decode_step_advance (its graph holds one "
                        "extra advance launch, counted in its per-step time)"}
        del lkp, lvp, lkn, lvn, g_adv, g_noadv, g_fused

    # prefill / extend: paged_prefill_attn on three shapes (see prefill_leg)
    prefill = None
    if not args.no_prefill and args.layout == "paged":
        prefill = prefill_leg(pkv, wl, dev, stream, flush_l2, rank, list(wl.PREFILL_SHAPES))

    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline:
        res = oracle_sample(w, args.cpu_seconds)
        one_t = oracle_sample(w, args.cpu_seconds_1t, threads=1)
        cpu = {"value": round(res["gbs"], 4), "unit": "GB/s", "cores": res["cores"],
               "kind": "oracle",
               "sample": f"fp64 oracle append+decode, rows 0..{res['rows'] - 1} of {w.name} "
                         f"x{res['reps']} ({res['seconds']:.1f} s, OpenMP over (row, head))",
               "single_thread": {"value": round(one_t["gbs"], 4), "unit": "GB/s", "cores": 1,
                                 "sample": f"rows 0..{one_t['rows'] - 1} of {w.name} "
                                           f"x{one_t['reps']} ({one_t['seconds']:.1f} s)"}}
    spread = {"replays": reps, "steps_per_replay": inner,
              "median_us": round(1e3 * statistics.median(per_step), 2),
              "min_us": round(1e3 * min(per_step), 2),
              "max_us": round(1e3 * max(per_step), 2)}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": max(3, args.warmup), "ms_per_step": round(ms_step_max, 5),
        "timing": (f"CUDA graph replay, {inner} steps per replay x {reps} replays = the K "
                   "timed steps; events on the replay stream around the region and each "
                   "replay; ms_per_step = region / K"),
        "spread": spread,
        "us_per_call": round(1e3 * ms_step_max, 2),
        "pct_hbm_peak": round(100.0 * value / world / peak, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": st_config,
        "plan": {"num_splits": S, "chunk": pkv.split_chunk(d, S), "planned": planned,
                 "plan_us": plan_us,
                 "note": "in each replay the first step (paged_decode_step) leaves its "
                         "partition as the plan; the replay's other steps "
                         "(paged_decode_step_planned) run on it, as a decode step's later "
                         "layers would; plan_us: paged_decode_plan alone, for reference"},
        "l2": (f"inputs larger than L2 (K+V = {kv_bytes / l2:.1f} x L2): steps back to back "
               "inside each replay, no flush" if back_to_back else
               "flushed before every replay (2x L2 written, then 2x L2 read), outside the "
               "events") if not args.no_flush else "warm",
        "roofline": {"bound": "hbm",
                     "kernel": "fused_decode_kernel (paged_decode_step; its piece combine "
                               "is inside the timed call)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_kind} (copy bandwidth)",
                     "us_per_launch": round(1e3 * ms_region, 2),
                     "alg_bytes_per_launch": alg_bytes,
                     "read_peak": {"gbs": round(read_peak, 1),
                                   "frac": round(achieved / read_peak, 4),
                                   "how": "torch.sum over a 4 GiB float32 buffer on this GPU, "
                                          "median of 10 (a plain streaming read)"}},
        "configs": configs or None,
        "cold_single_step": {"us": round(1e3 * ms_cold_max, 2),
                             "kv_read_gbs": round(total_bytes / (ms_cold_max * 1e-3) / 1e9, 1),
                             "note": "one step per replay, L2 flushed before it; includes the "
                                     "event/launch floor of an isolated call"},
        "decode_only": {"call": "paged_decode_attn", "us": round(1e3 * ms_dec_max, 2),
                        "kv_read_gbs": round(kv_bytes / (ms_dec_max * 1e-3) / 1e9, 1)},
        "gpu_launches": K * launches_per_step + (
            0 if args.layout != "contig" else (reps if planned else K)),
        "clocks": clocks,
        "wall_s_timed": round(wall, 4),
        "e2e": e2e,
        "decode_loop": loop,
        "prefill": prefill,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.only_prefill:
        return run_prefill_only(args)
    return run_pkv(args)


if __name__ == "__main__":
    sys.exit(main())
