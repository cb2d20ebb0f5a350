#!/usr/bin/env python3
"""Benchmark of one decode step of paged GQA attention on GB300.

A step is the whole hot path over one batch: fused RoPE + K/V append, the
split-KV decode kernel and the combine (the split count comes from the
library's planner).  The default workload is the batched ragged decode
(B=32, Hq=32, Hkv=8, D=128, page_size=16, seq_lens uniform in [512, 4096],
pages scattered over a 65536-page pool).

Printed: one JSON line.  ``value`` is the KV-read throughput of the step:
the bytes of K and V the attention must read (every token of every row,
every kv head) divided by the step time, summed over ranks.  The L2 is
flushed (a 2x-L2 write) between timed steps, outside the timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--splits S] [--pool-pages P] [--impl pkv|reference]

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
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fused_decode_traffic.json")
DECODE_SRC = os.path.join(ROOT, "paged_kv_gqa_16_gb300", "csrc", "pkv_fused.cu")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="ragged_b32")
    ap.add_argument("--splits", type=int, default=0, help="override the planner's split count")
    ap.add_argument("--pool-pages", type=int, default=0,
                    help="pool size of the ragged workload (smaller pools for profiling)")
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
    ap.add_argument("--flush-always", action="store_true",
                    help="flush the L2 before every step even when the inputs exceed it")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args(argv)


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


def oracle_sample(w, target_s: float, max_reps: int = 1000):
    """Time the fp64 oracle's step (append + decode) on the host cores over a
    bounded sample of the workload: whole rows, taken in order until their
    estimated cost reaches the target, repeated while time remains."""
    import numpy as np
    import oracle
    from paged_kv_gqa_16_gb300 import workloads as wl

    cores = cpu_cores()
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
        "config": {"workload": w.name + ("" if args.layout == "paged" else " (contiguous cache)"),
                   "layout": args.layout, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "page_size": w.page_size, "num_pages": w.num_pages},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": res["cores"],
                         "kind": "oracle",
                         "sample": f"fp64 oracle append+decode on rows 0..{res['rows'] - 1} of "
                                   f"{w.name} per step"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0



# Prefill / extend shapes: the pages' 512-token prompts at the 1B-class head
# shape, a long prefill, and an extend of 256 new tokens on 2,048-token rows.
PREFILL_SHAPES = {
    "prefill_b32_512": ("prefill B=32 x 512 (Hq 32, Hkv 8, D 64)",
                        dict(B=32, Hq=32, Hkv=8, D=64, page_size=16, seq_lens=[512] * 32,
                             q_lens=[512] * 32)),
    "prefill_b4_4096": ("prefill B=4 x 4096 (Hq 32, Hkv 8, D 128)",
                        dict(B=4, Hq=32, Hkv=8, D=128, page_size=16, seq_lens=[4096] * 4,
                             q_lens=[4096] * 4)),
    "extend_b16": ("extend B=16, 256 new of 2048 (Hq 32, Hkv 8, D 128)",
                   dict(B=16, Hq=32, Hkv=8, D=128, page_size=16, seq_lens=[2048] * 16,
                        q_lens=[256] * 16)),
}


def prefill_leg(pkv, wl, dev, stream, flush_l2, rank, names, reps=20):
    """paged_prefill_attn on each named shape: one call per graph replay, the
    L2 flushed before each, median of `reps`; tensor roofline against the
    measured dense bf16 peak (burst: each call runs alone)."""
    import torch
    tf_peak = load_bf16_peak()
    out_rows = []
    for name in names:
        label, kw = PREFILL_SHAPES[name]
        c = wl.prefill("prefill", seed=rank, **kw)
        pt = c.w.to_device(dev)
        pd = pkv.dims(c.w.B, c.w.Hq, c.w.Hkv, c.w.D, c.w.page_size, pt["k_pool"].shape[0],
                      int(c.w.kv_indices.numel()), c.w.max_seq_len, c.w.scale)
        pq, pqo = c.q.to(dev), c.qo_indptr.to(dev)
        pout = torch.empty(c.total_q, c.w.Hq, c.w.D, dtype=torch.bfloat16, device=dev)
        pst = torch.zeros(1, dtype=torch.int32, device=dev)
        max_q = max(kw["q_lens"])

        def prun():
            pkv.paged_prefill_attn(pd, pq, pqo, pt["k_pool"], pt["v_pool"], pt["kv_indices"],
                                   pt["kv_indptr"], pt["seq_lens"], pout, status=pst,
                                   max_q_len=max_q)

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
        del pt, pg
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

    names = list(PREFILL_SHAPES) if args.only_prefill == "all" else [args.only_prefill]
    rows = prefill_leg(pkv, wl, dev, torch.cuda.current_stream(dev), flush_l2, 0, names,
                       reps=max(1, args.steps))
    print(json.dumps({"metric": "paged prefill / extend attention TFLOP/s", "unit": "TFLOP/s",
                      "n_gpus": 1, "prefill": rows}), flush=True)
    return 0


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

    # each rank: an independent replica of the workload (own seed)
    kw = {"num_pages": args.pool_pages} if args.pool_pages else {}
    w = wl.make(args.workload, seed=rank, **kw)
    t = w.to_device(dev)
    P = t["k_pool"].shape[0]
    d = pkv.dims(w.B, w.Hq, w.Hkv, w.D, w.page_size, P, int(w.kv_indices.numel()),
                 w.max_seq_len, w.scale)
    S = args.splits or pkv.plan(d)[0]
    ws = pkv.alloc_workspace(d, S, dev)
    rope_rows = max(w.max_seq_len, 1)
    rope = torch.empty(rope_rows, w.D // 2, 2, dtype=torch.float32, device=dev)
    pkv.rope_table(rope, rope_rows, w.D, w.rope_base or 10000.0)
    out = torch.empty(w.B, w.Hq, w.D, dtype=torch.bfloat16, device=dev)
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

    def step(q, k_new, v_new, kv_indices, kv_indptr, seq_lens):
        """One pass of the hot path on the current stream: the new token's
        RoPE + append, the split decode and the combine (paged_decode_step)."""
        pkv.paged_decode_step(d, q, k_new, v_new, t["k_pool"], t["v_pool"], kv_indices,
                              kv_indptr, seq_lens, rope, rope_rows, S, ws, out)

    def decode(q, kv_indices, kv_indptr, seq_lens):
        pkv.paged_decode_attn(d, q, t["k_pool"], t["v_pool"], kv_indices, kv_indptr,
                              seq_lens, S, ws, out)

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
            pages = t["kv_indices"][ptr_h[b]:ptr_h[b + 1]].long()
            ck[b, :L] = t["k_pool"][pages].reshape(-1, w.Hkv, w.D)[:L]
            cv[b, :L] = t["v_pool"][pages].reshape(-1, w.Hkv, w.D)[:L]
        del t["k_pool"], t["v_pool"]
        torch.cuda.empty_cache()
        d = pkv.dims(w.B, w.Hq, w.Hkv, w.D, cache_len, w.B, w.B, cache_len, w.scale)
        ws = pkv.alloc_workspace(d, S, dev)

        def step(q, k_new, v_new, kv_indices, kv_indptr, seq_lens):
            pkv.decode_attn_contig(d, q, ck, cv, seq_lens, S, ws, out, k_new=k_new, v_new=v_new,
                                   rope_cos_sin=rope, rope_max_pos=rope_rows)

        def decode(q, kv_indices, kv_indptr, seq_lens):
            pkv.decode_attn_contig(d, q, ck, cv, seq_lens, S, ws, out)

        args.no_e2e = True
        args.no_loop = True

    launches_per_step = (1 if S == 1 else 2) + (1 if args.layout == "contig" else 0)
    dev_args = (t["q"], t["k_new"], t["v_new"], t["kv_indices"], t["kv_indptr"], t["seq_lens"])

    for _ in range(max(3, args.warmup)):
        step(*dev_args)
    torch.cuda.synchronize(dev)
    if pkv.status_word(ws) != 0:
        raise SystemExit(f"device status {pkv.status_word(ws):#x} after warm-up")

    # Timing.  Inputs at least twice the L2 size are streamed back to back:
    # INNER consecutive steps are captured in one CUDA graph (each step's
    # kernels chained to the previous ones, as in a decode loop) and replayed
    # between one pair of events; a step's K/V are evicted by the time the
    # next step reads them.  Smaller inputs: one step per graph, the L2
    # flushed before every step outside the events.
    kv_bytes = w.kv_bytes()
    back_to_back = kv_bytes >= 2 * l2 and not args.flush_always
    inner = 20 if back_to_back else 1

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(inner):
                fn()
        return g

    g_step = capture(lambda: step(*dev_args))
    g_dec = capture(lambda: decode(t["q"], t["kv_indices"], t["kv_indptr"], t["seq_lens"]))
    g_one = torch.cuda.CUDAGraph()                  # one flushed step, for the cold figure
    with torch.cuda.graph(g_one):
        step(*dev_args)
    for _ in range(3):
        g_step.replay()
        g_dec.replay()
        g_one.replay()
    stream = torch.cuda.current_stream(dev)

    def timed(graph, K, flush_each):
        """Per-step milliseconds: events around each replay / steps per replay."""
        reps = max(1, -(-K // inner)) if not flush_each else K
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for k in range(reps):
            if flush_each and not args.no_flush:
                flush_l2()
            evs[k][0].record(stream)
            graph.replay()
            evs[k][1].record(stream)
        torch.cuda.synchronize(dev)
        per = 1 if flush_each else inner
        return [a.elapsed_time(b) / per for a, b in evs]

    K = args.steps
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        time.sleep(0.4)              # let the sampler start before the timed region
        wall0 = time.perf_counter()
        step_ms = timed(g_step, K, not back_to_back)
        wall = time.perf_counter() - wall0
    barrier(world, dev)
    dec_ms = timed(g_dec, max(50, min(K, 2000)), not back_to_back)
    cold_ms = timed(g_one, max(20, min(K // 10, 500)), True)
    ms_step = statistics.mean(step_ms)
    ms_dec = statistics.mean(dec_ms)
    ms_step_max = reduce_max(ms_step, world, dev)
    ms_dec_max = reduce_max(ms_dec, world, dev)
    ms_cold_max = reduce_max(statistics.mean(cold_ms), world, dev)

    total_bytes = kv_bytes * world
    value = total_bytes / (ms_step_max * 1e-3) / 1e9

    # e2e: host (pinned) inputs copied in, the step, the output copied back.
    # The step's inputs sit in one pinned host block (each at a 256-byte
    # aligned offset) copied with one H2D copy into one device block the step
    # reads through views; the copy in, the step and the copy of the output
    # back are captured in one CUDA graph, replayed once per step.
    e2e = None
    if not args.no_e2e:
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
        dev_blk = torch.empty(blk_bytes, dtype=torch.uint8, device=dev)
        e_args = tuple(blk_view(dev_blk, k) for k in names)
        out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = blk_bytes
        d2h = out_host.numel() * out_host.element_size()
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e):
            dev_blk.copy_(host_blk, non_blocking=True)
            step(*e_args)
            out_host.copy_(out, non_blocking=True)
        for _ in range(3):
            g_e2e.replay()
        Ke = max(10, min(K, 500))
        e_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(Ke)]
        torch.cuda.synchronize(dev)
        for k in range(Ke):
            if not args.no_flush and not back_to_back:
                flush_l2()
            e_evs[k][0].record(stream)
            g_e2e.replay()
            e_evs[k][1].record(stream)
        torch.cuda.synchronize(dev)
        e_ms = statistics.mean(a.elapsed_time(b) for a, b in e_evs)
        e_ms = reduce_max(e_ms, world, dev)
        e2e = {"value": round(total_bytes / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(e_ms, 5), "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h,
               "path": "pinned host block -> one H2D copy, the step, one D2H copy of the "
                       "output, captured in one CUDA graph per step"}
        del g_e2e, dev_blk

    status = pkv.status_word(ws)
    if status != 0:
        raise SystemExit(f"device status {status:#x} after the timed run")

    # decode loop: the same rows as a loop whose table grows on the device.
    # LOOP steps per graph, each paged_kv_advance + paged_decode_step (the
    # step's new token at the advanced length), against the same graph
    # without the advance; the small state is reset between replays, outside
    # the events, and nothing is flushed (consecutive steps, as in serving).
    loop = None
    if not args.no_loop:
        LOOP, reps = 20, 20
        before = (w.seq_lens - 1).clamp(min=0).tolist()     # cached tokens before a step
        held_max = max(-(-L // w.page_size) for L in before)
        cap = held_max + -(-LOOP // w.page_size) + 2
        need = sum(-(-L // w.page_size) for L in before) + w.B * (-(-LOOP // w.page_size) + 1)
        ls = wl.decode_loop(B=w.B, Hq=w.Hq, Hkv=w.Hkv, D=w.D, page_size=w.page_size,
                            seq_lens=before, steps=LOOP, cap=cap, num_pages=need + 64,
                            seed=1000 + rank)

        def t16(a):
            return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(dev)

        ld = pkv.dims(w.B, w.Hq, w.Hkv, w.D, w.page_size, ls.num_pages, len(ls.kv_indices),
                      ls.max_seq_len, w.scale)
        lS = args.splits or pkv.plan(ld)[0]
        lws = pkv.alloc_workspace(ld, lS, dev)
        lq, lkn, lvn = t16(ls.q), t16(ls.k_new), t16(ls.v_new)
        lkp, lvp = t16(ls.k_pool), t16(ls.v_pool)
        lrope = torch.empty(ls.max_seq_len, w.D // 2, 2, dtype=torch.float32, device=dev)
        pkv.rope_table(lrope, ls.max_seq_len, w.D, w.rope_base or 10000.0)
        lsl0 = torch.from_numpy(ls.seq_lens).to(dev)
        lind0 = torch.from_numpy(ls.kv_indices).to(dev)
        lsl, lind = lsl0.clone(), lind0.clone()
        lptr = torch.from_numpy(ls.kv_indptr).to(dev)
        lfree = torch.from_numpy(ls.free_pages).to(dev)
        lhead = torch.zeros(1, dtype=torch.int32, device=dev)
        lout = torch.empty(w.B, w.Hq, w.D, dtype=torch.bfloat16, device=dev)

        def one(st, adv):
            if adv == "fused":
                # the loop opens with one advance; each step then advances
                # for the next inside its own combine launch
                if st == 0:
                    pkv.paged_kv_advance(ld, lsl, lptr, lind, lfree, lhead, status=lws)
                pkv.paged_decode_step_advance(ld, lq, lkn[st], lvn[st], lkp, lvp, lind, lptr,
                                              lsl, lrope, ls.max_seq_len, lS, lws, lout,
                                              lfree, lhead)
                return
            if adv:
                pkv.paged_kv_advance(ld, lsl, lptr, lind, lfree, lhead, status=lws)
            pkv.paged_decode_step(ld, lq, lkn[st], lvn[st], lkp, lvp, lind, lptr, lsl, lrope,
                                  ls.max_seq_len, lS, lws, lout)

        def reset():
            lsl.copy_(lsl0)
            lind.copy_(lind0)
            lhead.zero_()

        def loop_graph(adv):
            reset()
            for st in range(LOOP):
                one(st, adv)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for st in range(LOOP):
                    one(st, adv)
            return g

        def loop_timed(g):
            ms = []
            for _ in range(reps + 3):
                reset()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g.replay()
                b.record(stream)
                torch.cuda.synchronize(dev)
                ms.append(a.elapsed_time(b) / LOOP)
            return statistics.median(ms[3:])

        g_adv, g_noadv, g_fused = loop_graph(True), loop_graph(False), loop_graph("fused")
        ms_adv = loop_timed(g_adv)
        pages_taken = int(lhead.item())
        ms_fused = loop_timed(g_fused)
        ms_noadv = loop_timed(g_noadv)
        if pkv.status_word(lws) != 0:
            raise SystemExit(f"device status {pkv.status_word(lws):#x} after the loop leg")
        loop = {"steps_per_graph": LOOP, "replays": reps,
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
        prefill = prefill_leg(pkv, wl, dev, stream, flush_l2, rank, list(PREFILL_SHAPES))

    # roofline of the dominant kernel, the fused step kernel (its launch is
    # timed as the step call, so the small piece combine is included).
    # Algorithmic bytes per call: K and V of every token, q, the new token's
    # K/V read and written to its slot, the output, and the page tables.
    n_idx = int(w.kv_indices.numel())
    io_bytes = (w.B * w.Hq * w.D * 2 * 2            # q in, out
                + w.B * w.Hkv * w.D * 2 * 2 * 2     # k_new/v_new in, slot writes
                + 4 * n_idx + 8 * w.B)              # kv_indices, kv_indptr, seq_lens
    alg_bytes = kv_bytes + io_bytes
    dec_bytes = kv_bytes + w.B * w.Hq * w.D * 2 * 2 + 4 * n_idx + 8 * w.B
    peak, peak_kind = load_peaks()
    achieved = alg_bytes / (ms_step * 1e-3) / 1e9
    read_peak = measure_read_peak(dev, stream)
    traffic = cached_traffic(w.name, S) if args.layout == "paged" else None
    clocks = clk.summary(wall0, wall0 + wall)

    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline:
        res = oracle_sample(w, args.cpu_seconds)
        cpu = {"value": round(res["gbs"], 4), "unit": "GB/s", "cores": res["cores"],
               "kind": "oracle",
               "sample": f"fp64 oracle append+decode, rows 0..{res['rows'] - 1} of {w.name} "
                         f"x{res['reps']} ({res['seconds']:.1f} s)"}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": max(3, args.warmup), "ms_per_step": round(ms_step_max, 5),
        "timing": "CUDA graph replay; events on the replay stream around each replay",
        "us_per_call": round(1e3 * ms_step_max, 2),
        "pct_hbm_peak": round(100.0 * value / world / peak, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "page_size": w.page_size, "num_pages": P, "tokens": w.total_tokens,
                   "kv_bytes": kv_bytes, "num_splits": S, "chunk": pkv.split_chunk(d, S),
                   "l2": (f"inputs larger than L2 (K+V = {kv_bytes / l2:.1f} x L2): {inner} steps "
                         "back to back per graph replay, no flush" if back_to_back else
                         "flushed between steps (2x L2 written, then 2x L2 read), outside "
                         "the timed events") if not args.no_flush else "warm",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm",
                     "kernel": "fused_decode_kernel (paged_decode_step; its piece combine "
                               "is inside the timed call)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_kind} (copy bandwidth)",
                     "us_per_launch": round(1e3 * ms_step, 2),
                     "alg_bytes_per_launch": alg_bytes,
                     "read_peak": {"gbs": round(read_peak, 1),
                                   "frac": round(achieved / read_peak, 4),
                                   "how": "torch.sum over a 4 GiB float32 buffer on this GPU, "
                                          "median of 10 (a plain streaming read)"}},
        "cold_single_step": {"us": round(1e3 * ms_cold_max, 2),
                             "kv_read_gbs": round(total_bytes / (ms_cold_max * 1e-3) / 1e9, 1),
                             "note": "one step per replay, L2 flushed before it; includes the "
                                     "~6 us event/launch floor of an isolated call"},
        "decode_only": {"call": "paged_decode_attn", "us": round(1e3 * ms_dec_max, 2),
                        "kv_read_gbs": round(kv_bytes / (ms_dec_max * 1e-3) / 1e9, 1),
                        "alg_gbs": round(dec_bytes / (ms_dec_max * 1e-3) / 1e9, 1)},
        "gpu_launches": len(step_ms) * (1 if not back_to_back else inner) * launches_per_step,
        "clocks": clocks,
        "wall_s_timed": round(wall, 3),
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
