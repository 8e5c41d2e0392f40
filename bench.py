#!/usr/bin/env python
"""Throughput of the FP4 indexer decode step on GB300.

One step = the whole hot path over one decode batch: K store of each sequence's
newest compressed token, Q quant, schedule, paged-MQA logits, top-k.  Default
workload: 64 sequences x 1 query row, context lengths ~U[8192, 32768] compressed
tokens, pages from a permuted 40,960-page pool, 64 heads x 128, k = 2,048.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fp4idx|reference]

Prints one JSON line (rank 0).  On one GPU the default line also carries
`per_config`: the tiny decode, the draft batch (256 x 6 rows), the 8,192-row prefill
chunk and the 65,536-row K store, each measured the same way with a bounded number of
steps, with its own roofline object and a bounded oracle sample (--no-per-config leaves
them out).  --impl reference times the CPU oracle on this host's cores on the same
workload (rows sampled per step).  Under torchrun each rank runs its own replica of the
batch (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP4 indexer decode: K-cache GB/s vs HBM peak; query rows/s (logits+top-k)"
UNIT = "query rows/s"
L2_FLUSH_BYTES = 256 << 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "logits_mxf4_traffic.json")
LOGITS_SRC = os.path.join(ROOT, "sparse_attention_fp4_gb300", "csrc", "logits_mxf4.cu")

WORKLOADS = {
    "decode_b64": ("decode_batch64", 1001, {}),
    "tiny": ("tiny_decode", 1000, {}),
    "draft_b256": ("draft_batch256", 1002, {}),
    "prefill": ("prefill_chunk", 1003, {}),
    # the last 1,024 rows of the prefill chunk (for profiling captures)
    "prefill_1024": ("prefill_chunk", 1003, {"rows": 1024}),
}


# ------------------------------------------------------------------ distributed plumbing (timing only)
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def dist_init(backend):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def dist_barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def dist_reduce(value: float, op: str, device=None) -> float:
    """max or sum of a host scalar over ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(rows_this_rank: int, seconds_this_rank: float, device=None):
    """Whole-job throughput: all ranks' rows over the slowest rank's time."""
    total_rows = dist_reduce(rows_this_rank, "sum", device)
    slowest = dist_reduce(seconds_this_rank, "max", device)
    return total_rows / slowest, slowest


# ------------------------------------------------------------------ workload
def make_batch(name):
    from sparse_attention_fp4_gb300 import workloads as wl
    fn, seed, kw = WORKLOADS[name]
    return getattr(wl, fn)(seed, **kw)


def newest_rows(b):
    """Per sequence with stored tokens: (sequence id, index of its newest K row).  The
    K rows are stored sequence by sequence in token order."""
    toks = b.seq_tokens.astype(np.int64)
    ends = np.cumsum(toks) - 1
    seqs = np.nonzero(toks > 0)[0]
    return seqs, ends[seqs]


def algorithmic_bytes(b):
    """Bytes the logits pass must move from HBM at minimum: the K cache of every token a
    sequence's rows see (64 B payload + 4 B scale, once per sequence), the packed
    queries (4,352 B/row), head weights (256 B/row), page ids and row metadata; top-k
    output 4 B/index."""
    L = b.context_lens.astype(np.int64)
    T = b.n_rows
    # the K cache of a sequence is needed once, up to its longest row's context
    seq_max = np.zeros(int(b.row_seq.max()) + 1 if T else 0, np.int64)
    np.maximum.at(seq_max, b.row_seq.astype(np.int64), L)
    pages = np.ceil(seq_max / 64.0).sum()
    kbytes = 68.0 * seq_max.sum()
    logits_pass = kbytes + 4352.0 * T + 256.0 * T + 4.0 * pages + 8.0 * T
    return dict(k_cache=kbytes, logits_pass=logits_pass, topk_out=4.0 * T * b.topk)


LOGITS_DEPS = ("logits_mxf4.cu", "ptx.cuh", "schedule.cuh", "fp4idx_internal.cuh", "select.cuh", "pipeline.cuh")


def source_hash(deps):
    """Hash of a kernel's sources: a stored DRAM traffic figure is reported only while the
    kernel it was measured on is unchanged."""
    h = hashlib.sha256()
    for f in deps:
        with open(os.path.join(os.path.dirname(LOGITS_SRC), f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def kernel_source_hash():
    return source_hash(LOGITS_DEPS)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# Nominal dense FP4 (e2m1, block-scaled) over dense bf16 tensor throughput on GB300:
# 13.5 / 2.25 PFLOP/s.  The FP4 peak is the measured bf16 peak times this ratio.
FP4_OVER_BF16 = 6.0


def measured_fp4_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]) * FP4_OVER_BF16, "measured bf16 burst x nominal fp4/bf16 ratio 6"
    return 1900.0 * FP4_OVER_BF16, "fallback bf16 x nominal fp4/bf16 ratio 6"


def logits_flops(b):
    """Tensor work of the logits contraction: 2 * 64 heads * 128 dims per visible (row,
    token) pair."""
    return 2.0 * 64 * 128 * float(b.context_lens.astype(np.int64).sum())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = os.path.join("/tmp", "fp4idx_clocks_%d.csv" % os.getpid())

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-i", self.gpu_id, "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx.append(float(p[2]))
                    power.append(float(p[3]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def gpu_id_for(device_index):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(device_index)


# ------------------------------------------------------------------ the GPU arm
class DecodeStep:
    """Device-resident inputs of one decode batch and the five launches of a step."""

    def __init__(self, b, device, fused=False, prep="one"):
        import torch

        from sparse_attention_fp4_gb300 import fp4idx
        from sparse_attention_fp4_gb300 import workloads as wl
        self.fp4idx = fp4idx
        self.b = b
        self.device = device

        def bf16(a):
            return torch.from_numpy(np.array(a, copy=True).view(np.int16)).to(device).view(torch.bfloat16)

        def dev(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(device)

        ks = b.kstore
        self.cs = bf16(wl.rope_cos_sin_table())
        self.payload, self.scale = fp4idx.alloc_cache(b.num_pages, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        # fill the cache (setup, untimed)
        chunk = 1 << 20
        nw = bf16(ks.norm_w)
        for r0 in range(0, ks.n_rows, chunk):
            r1 = min(ks.n_rows, r0 + chunk)
            fp4idx.store_k(bf16(ks.k_rows[r0:r1]), dev(ks.positions[r0:r1]), dev(ks.slots[r0:r1]), nw, ks.eps,
                           self.cs, self.payload, self.scale, status=self.status)
        _, idx = newest_rows(b)
        self.h_new = dict(k=np.ascontiguousarray(ks.k_rows[idx]), pos=np.ascontiguousarray(ks.positions[idx]),
                          slots=np.ascontiguousarray(ks.slots[idx]))
        self.new_k = bf16(self.h_new["k"])
        self.new_pos = dev(self.h_new["pos"])
        self.new_slots = dev(self.h_new["slots"])
        self.norm_w = nw
        self.eps = ks.eps
        self.q = bf16(b.q)
        self.qpos = dev(b.q_positions)
        self.w = dev(b.w)
        self.pt = dev(b.page_table)
        self.rs = dev(b.row_seq)
        self.cl = dev(b.context_lens)
        self.T = b.n_rows
        self.k = b.topk
        self.max_ctx = int(max(1, b.context_lens.max()))
        self.qp, self.qs = fp4idx.alloc_query(self.T, device=device)
        self.sched = torch.empty(fp4idx.schedule_workspace_bytes(self.T), dtype=torch.uint8, device=device)
        self.logits = torch.empty((self.T, (self.max_ctx + 3) // 4 * 4), dtype=torch.float32, device=device)
        self.topk = torch.empty((self.T, self.k), dtype=torch.int32, device=device)
        self.topk_ws = torch.empty(fp4idx.topk_workspace_bytes(self.T, self.max_ctx), dtype=torch.uint8,
                                   device=device)
        self.fused_ws = torch.empty(fp4idx.logits_workspace_bytes(self.T, self.max_ctx, self.k), dtype=torch.uint8,
                                    device=device)
        self.fused = fused  # False: fp4idx_logits_topk (two launches); True: fp4idx_logits_topk_fused
        self.prep = prep  # "one": fp4idx_prepare_step; "three": schedule, K store and Q quant calls
        torch.cuda.synchronize(device)

    def calls(self):
        """The launches of a step, in order, as (name, callable): the step preparation
        (fp4idx_prepare_step: schedule, K store of the newest rows, Q quant, one launch),
        then the read side -- the logits launch and the top-k launch of
        fp4idx_logits_topk, or with `fused` the one launch of fp4idx_logits_topk_fused."""
        f = self.fp4idx
        if self.prep == "one":
            base = [("prepare_step", lambda: f.prepare_step(
                self.new_k, self.new_pos, self.new_slots, self.norm_w, self.eps, self.q, self.qpos, self.cs,
                self.payload, self.scale, self.qp, self.qs, self.cl, self.rs, self.sched, status=self.status))]
        else:  # the three calls fp4idx_prepare_step stands for, one after another
            base = [
                ("build_schedule", lambda: f.build_schedule(self.cl, self.rs, self.sched)),
                ("store_k", lambda: f.store_k(self.new_k, self.new_pos, self.new_slots, self.norm_w, self.eps,
                                              self.cs, self.payload, self.scale, status=self.status)),
                ("quant_q", lambda: f.quant_q(self.q, self.qpos, self.cs, self.qp, self.qs, status=self.status)),
            ]
        if self.fused:
            return base + [("logits_topk_fused", self.logits_topk)]
        return base + [
            ("logits", lambda: f.logits(self.qp, self.qs, self.w, self.payload, self.scale, self.pt, self.rs, self.cl,
                                        self.max_ctx, self.sched, self.logits, status=self.status)),
            ("topk", lambda: f.topk(self.logits, self.cl, self.max_ctx, self.k, self.topk_ws, self.topk,
                                    status=self.status)),
        ]

    def logits_topk(self):
        """The read side's entry point as a caller uses it: fp4idx_logits_topk (or, with
        `fused`, fp4idx_logits_topk_fused)."""
        self.fp4idx.logits_topk(self.qp, self.qs, self.w, self.payload, self.scale, self.pt, self.rs, self.cl,
                                self.max_ctx, self.k, self.sched, self.fused_ws, self.topk, status=self.status,
                                fused=self.fused)

    def launch(self):
        for _, fn in self.calls():
            fn()

    def launch_step(self, marks=None):
        """The step as a caller issues it on one stream: fp4idx_prepare_step, then the read
        side's call (the form captured into the step's graph).  With `marks` (timing
        events, one more than the read side's launches) the read side's launches are
        issued one by one with a mark before each and after the last."""
        import torch
        calls = self.calls()
        n = self.n_prep()
        for _, fn in calls[:n]:
            fn()
        if marks:
            cur = torch.cuda.current_stream()
            for i, (_, fn) in enumerate(calls[n:]):
                marks[i].record(cur)
                fn()
            marks[len(calls) - n].record(cur)
        else:
            self.logits_topk()

    def read_side_names(self):
        return [n for n, _ in self.calls()[self.n_prep():]]

    def n_prep(self):
        return 1 if self.prep == "one" else 3


def make_flush(device):
    """L2 flush between timed launches: a 256 MiB write and a 256 MiB read (twice the L2)."""
    import torch
    flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def flush_l2():
        flush_w.zero_()
        _ = flush_r.sum()
    return flush_l2


SPIN_CYCLES = int(2e5)  # ~0.1 ms at GB300 clocks: covers the host's enqueue of the next step


def stored_traffic(workload):
    """DRAM bytes per logits launch from an ncu capture of this workload, or None when no
    capture exists or the kernel's sources changed since it was taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        tr = json.load(f)
    if tr.get("kernel_source_hash") != kernel_source_hash():
        return None
    w = tr.get("workloads", {}).get(workload)
    return w.get("dram_bytes_per_launch") if w else None


def time_step(st, steps, warmup, flush_l2, device, live_n=500, alone_n=200):
    """Times the step of `st` as one CUDA graph replay per step (L2 flushed and a spin
    kernel ahead of each, outside the events), then the read side's launches inside an
    instrumented copy of the graph, then every launch captured and replayed alone."""
    import torch
    for _ in range(max(3, warmup)):  # warm-up (also sets kernel attributes before capture)
        st.launch()
    torch.cuda.synchronize()
    assert st.fp4idx.read_status(st.status) == 0, "device status after warm-up"

    # the step as one CUDA graph (decode steps replay captured graphs)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        st.launch()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        st.launch_step()
    # an instrumented copy of the step: event-record nodes around each launch of the read
    # side (the marks slow a step a little, so the timed loop replays the plain graph)
    names = st.read_side_names()
    try:
        marks = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(names) + 1)]
        gm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gm):
            st.launch_step(marks)
    except TypeError:
        marks, gm = None, None
    for _ in range(max(3, warmup)):
        g.replay()
    torch.cuda.synchronize()

    K = steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(gpu_id_for(device.index)).start()
    time.sleep(0.3)
    dist_barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for i in range(K):
        flush_l2()
        torch.cuda._sleep(SPIN_CYCLES)
        starts[i].record()
        g.replay()
        ends[i].record()
    torch.cuda.synchronize()
    dist_barrier()
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    step_ms = [starts[i].elapsed_time(ends[i]) for i in range(K)]

    # kernel times inside the step, from the instrumented graph (same flush and spin); a
    # fixed number of replays whatever K: event timestamps are coarse, so the mean needs
    # many of them
    live = {n: [] for n in names}
    if marks:
        for i in range(live_n):
            flush_l2()
            torch.cuda._sleep(SPIN_CYCLES)
            gm.replay()
            marks[-1].synchronize()  # every replay re-records the marks: read them now
            for j, n in enumerate(names):
                live[n].append(marks[j].elapsed_time(marks[j + 1]) * 1e3)

    # per-kernel breakdown: each launch captured in its own graph and replayed alone
    subs = []
    for name, fn in st.calls():
        sg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(sg):
            fn()
        subs.append((name, sg))
    per_times = {name: [] for name, _ in subs}
    for i in range(alone_n):
        for name, sg in subs:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            flush_l2()
            torch.cuda._sleep(SPIN_CYCLES)
            e0.record()
            sg.replay()
            e1.record()
            per_times[name].append((e0, e1))
    torch.cuda.synchronize()
    per = {n: statistics.mean([a.elapsed_time(b) for a, b in v]) * 1e3 for n, v in per_times.items()}
    main = names[0]  # the logits launch (with the selection, for fp4idx_logits_topk_fused)
    if marks:
        logits_us = statistics.mean(live[main])
        live_us = {n: {"mean": round(statistics.mean(v), 2), "median": round(statistics.median(v), 2)}
                   for n, v in live.items()}
        timing_src = ("event-record nodes around the launch inside an instrumented copy of the step graph, "
                      "mean over %d replays (L2 flushed before each)" % len(live[main]))
    else:
        logits_us = statistics.mean([a.elapsed_time(b) for a, b in per_times[main]]) * 1e3
        live_us = None
        timing_src = "the launch captured alone in a graph (includes the graph launch), mean"
    return dict(total_s=sum(step_ms) / 1e3, t_wall=t_wall, clocks=clocks, live_us=live_us,
                alone_us={k: round(v, 2) for k, v in per.items()}, logits_us=logits_us, timing_src=timing_src,
                status=st.fp4idx.read_status(st.status))


def roofline_for(b, workload, st, logits_us, timing_src):
    """Roofline object of the logits launch: HBM-bound against the measured copy
    bandwidth, except for the prefill chunk, whose one sequence's K stays in L2 and which is
    measured against the FP4 tensor peak."""
    ab = algorithmic_bytes(b)
    traffic = stored_traffic(workload)
    kname = "logits_mxf4_kernel" + (" (with the fused top-k selection)" if st.fused else "")
    if workload.startswith("prefill"):
        fl = logits_flops(b)
        tpk, tpk_src = measured_fp4_tflops()
        tach = fl / (logits_us * 1e-6) / 1e12
        return {"bound": "tensor", "achieved": round(tach, 1), "peak": round(tpk, 1), "unit": "TFLOP/s",
                "frac": round(tach / tpk, 4), "traffic": traffic, "kernel": kname, "algorithmic_flops": fl,
                "avg_launch_us": round(logits_us, 2), "launch_timing": timing_src, "peak_source": tpk_src}
    peak, peak_kind = measured_peaks()
    # the fused launch also writes the selection (4 B an index)
    main_bytes = ab["logits_pass"] + (ab["topk_out"] if st.fused else 0.0)
    achieved = main_bytes / (logits_us * 1e-6) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": kname,
            "algorithmic_bytes": main_bytes, "avg_launch_us": round(logits_us, 2), "launch_timing": timing_src,
            "peak_source": "%s copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" % peak_kind}


def step_description(st):
    return "%s + %s, one CUDA graph replay" % (
        "fp4idx_prepare_step (schedule + K store of the newest token per sequence + Q quant, one launch)"
        if st.prep == "one" else "fp4idx_build_schedule, fp4idx_store_k, fp4idx_quant_q",
        "fp4idx_logits_topk_fused (logits and selection in one launch)" if st.fused else
        "fp4idx_logits_topk (logits launch, top-k launch)")


# the other configurations the default line carries: (workload, timed steps, CPU seconds)
PER_CONFIG = (("tiny", 2000, 3.0), ("draft_b256", 200, 5.0), ("prefill", 50, 5.0))


def measure_config(workload, steps, cpu_seconds, args, device, flush_l2):
    """One of the other configurations, measured the way the headline is (step graph, L2
    flushed between steps) with a bounded number of steps, and its oracle on the host
    cores for a bounded sample."""
    import torch
    b = make_batch(workload)
    st = DecodeStep(b, device, fused=args.fused, prep=args.prep)
    r = time_step(st, steps, args.warmup, flush_l2, device, live_n=min(steps, 200), alone_n=min(steps, 50))
    value = st.T * steps / r["total_s"]
    out = {"workload": b.name, "rows": b.n_rows, "topk": b.topk, "context_tokens": int(b.context_lens.sum()),
           "value": round(value, 1), "unit": UNIT, "steps": steps, "ms_per_step": round(r["total_s"] / steps * 1e3, 5),
           "kernel_us_in_step": r["live_us"], "kernel_us_alone": r["alone_us"],
           "roofline": roofline_for(b, workload, st, r["logits_us"], r["timing_src"]),
           "clocks": r["clocks"], "device_status": r["status"], "gpu_launches": len(st.calls()) * steps}
    del st
    torch.cuda.empty_cache()
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(b, cpu_seconds)
    return out


def run_gpu(args):
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init("nccl")
    b = make_batch(args.workload)
    st = DecodeStep(b, device, fused=args.fused, prep=args.prep)
    flush_l2 = make_flush(device)

    K = args.steps
    r = time_step(st, K, args.warmup, flush_l2, device)
    value, slowest = aggregate(st.T * K, r["total_s"], device)
    ms_per_step = slowest / K * 1e3
    ab = algorithmic_bytes(b)
    roofline = roofline_for(b, args.workload, st, r["logits_us"], r["timing_src"])

    desc = step_description(st)
    launches = len(st.calls()) * K
    e2e = run_e2e(st, args, flush_l2) if not args.no_e2e else None
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(b, args.cpu_seconds)
    per_config = None
    if world == 1 and args.workload == "decode_b64" and not args.no_per_config:
        del st
        torch.cuda.empty_cache()
        per_config = {w: measure_config(w, n, c, args, device, flush_l2) for w, n, c in PER_CONFIG}
        per_config["kstore"] = measure_kstore(args, device)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp4(e2m1,ue8m0)->f32", "data": "synthetic",
            "config": {"workload": b.name, "rows": b.n_rows, "heads": 64, "head_dim": 128, "topk": b.topk,
                       "context_tokens": int(b.context_lens.sum()), "cache_pages": b.num_pages,
                       "step": desc,
                       "l2": "flushed between steps (256 MiB write + 256 MiB read, untimed)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "kcache_gbs": round(ab["k_cache"] / (r["logits_us"] * 1e-6) / 1e9, 1),
            "kernel_us_in_step": r["live_us"],
            "kernel_us_alone": r["alone_us"],
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": r["clocks"],
            "wall_s_timed_region": round(r["t_wall"], 3),
            "device_status": r["status"],
        }
        if per_config is not None:
            line["per_config"] = per_config
        print(json.dumps(line), flush=True)


def run_e2e(st, args, flush_l2):
    """Same metric through the C ABI with host buffers: every step copies its inputs from
    pinned host memory, makes the two calls a caller makes (fp4idx_prepare_step, then the
    logits + top-k call) and reads the selection back."""
    import torch
    b = st.b
    # the step's inputs, each as a 256-byte aligned slice of one pinned staging buffer and
    # of one device buffer that the calls read: a step moves them with one copy
    srcs = [("new_k", st.h_new["k"]), ("new_pos", st.h_new["pos"]), ("new_slots", st.h_new["slots"]),
            ("q", b.q), ("qpos", b.q_positions), ("w", b.w), ("pt", b.page_table), ("rs", b.row_seq),
            ("cl", b.context_lens)]
    offs, total = [], 0
    for name, arr in srcs:
        offs.append(total)
        total += (np.ascontiguousarray(arr).nbytes + 255) // 256 * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    hv = host.numpy()
    dev_in = torch.empty(total, dtype=torch.uint8, device=st.device)
    for (name, arr), off in zip(srcs, offs):
        raw = np.ascontiguousarray(arr).view(np.uint8).reshape(-1)
        hv[off:off + raw.size] = raw
        t = getattr(st, name)
        assert raw.size == t.numel() * t.element_size(), name
        setattr(st, name, dev_in[off:off + raw.size].view(t.dtype).view(t.shape))
    out = torch.empty((st.T, st.k), dtype=torch.int32).pin_memory()
    h2d = total
    d2h = out.numel() * out.element_size()
    K = min(args.steps, 200)

    def step():
        dev_in.copy_(host, non_blocking=True)
        st.launch_step()
        out.copy_(st.topk, non_blocking=True)

    # the step as a serving loop replays it: one CUDA graph holding the copies in from
    # pinned host memory, the four calls and the copy of the selection back
    s = torch.cuda.Stream(st.device)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    times = []
    for i in range(K + 3):
        flush_l2()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1) / 1e3)
    ok = np.array_equal(out.numpy(), st.topk.cpu().numpy())
    value, _ = aggregate(st.T * K, sum(times), st.device)
    return {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": K, "ms_per_step": round(sum(times) / K * 1e3, 4),
            "how": "one CUDA graph replay per step: one host-to-device copy of the step's inputs (packed in one "
                   "pinned buffer), the step-preparation call and the logits/top-k call, device-to-host copy of "
                   "the selection",
            "selection_read_back_matches": bool(ok)}


# ------------------------------------------------------------------ the CPU oracle (baseline / reference arm)
class OracleStep:
    def __init__(self, b):
        import oracle
        from sparse_attention_fp4_gb300 import workloads as wl
        self.oracle = oracle
        self.b = b
        self.cs = wl.rope_cos_sin_table()
        self.payload, self.scale, st = oracle.store_k(b.kstore, self.cs)  # cache fill: setup, untimed
        assert st == 0
        self.new_seqs, idx = newest_rows(b)
        ks = b.kstore
        from sparse_attention_fp4_gb300.workloads import KStoreInputs
        self.new = KStoreInputs(ks.k_rows[idx], ks.positions[idx], ks.slots[idx], ks.norm_w, ks.eps, ks.num_pages)

    def run(self, rows):
        """The step for a sample of query rows: K store of the newest rows of their
        sequences, Q quant, logits and top-k of those rows.  Returns seconds."""
        o = self.oracle
        b = self.b
        t0 = time.perf_counter()
        seqs = set(int(s) for s in b.row_seq[rows])
        sel = [i for i, s in enumerate(self.new_seqs) if int(s) in seqs]
        from sparse_attention_fp4_gb300.workloads import KStoreInputs
        new = KStoreInputs(self.new.k_rows[sel], self.new.positions[sel], self.new.slots[sel], self.new.norm_w,
                           self.new.eps, self.new.num_pages)
        o.store_k(new, self.cs, self.payload, self.scale)
        qp, qs, _ = o.quant_q(b.q[rows], b.q_positions[rows], self.cs)
        lg, _, _ = o.logits(qp, qs, b.w[rows], self.payload, self.scale, b.page_table, b.row_seq[rows],
                            b.context_lens[rows], with_bound=False)
        for i, t in enumerate(rows):
            o.topk(lg[i], int(b.context_lens[t]), b.topk)
        return time.perf_counter() - t0


def cpu_baseline(b, seconds):
    import oracle
    cores = oracle.max_threads()
    step = OracleStep(b)
    rows_per = 8
    done, secs, i = 0, 0.0, 0
    while secs < seconds and done < max(b.n_rows * 4, 64):
        rows = np.arange(i, i + rows_per) % b.n_rows
        secs += step.run(rows)
        done += rows_per
        i += rows_per
    return {"value": round(done / secs, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d query rows (%d per call, full contexts) of the same workload incl. K store of their "
                      "newest tokens, Q quant, binary64 logits and top-k; %.1f s" % (done, rows_per, secs)}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    b = make_batch(args.workload)
    step = OracleStep(b)
    cores = oracle.max_threads()
    rows_per = 8
    warm = 0.0
    for i in range(max(3, args.warmup)):  # warm-up: page in the oracle and its inputs
        warm += step.run(np.arange(i * rows_per, (i + 1) * rows_per) % b.n_rows)
    # a bounded sample: about a minute for the K timed steps, 1 to 8 rows each
    rate = rows_per * max(3, args.warmup) / max(warm, 1e-9)
    rows_per = int(max(1, min(8, rate * 60.0 / max(1, args.steps))))
    secs = 0.0
    for i in range(args.steps):
        secs += step.run(np.arange(i * rows_per, (i + 1) * rows_per) % b.n_rows)
    value = rows_per * args.steps / secs
    sample = "%d query rows per step (full contexts), %d steps" % (rows_per, args.steps)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(secs / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": b.name, "rows_sampled_per_step": rows_per, "topk": b.topk},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


KSTORE_DEPS = ("store_quant.cu", "schedule_build.cuh", "schedule.cuh", "launchers.cuh", "fp4idx_internal.cuh")
KSTORE_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "store_k_traffic.json")


def stored_kstore_traffic():
    """DRAM bytes per launch of store_k_kernel on the 65,536-row workload, from an ncu
    capture, while the kernel's sources are unchanged since it was taken."""
    if not os.path.exists(KSTORE_TRAFFIC_FILE):
        return None
    with open(KSTORE_TRAFFIC_FILE) as f:
        tr = json.load(f)
    return tr.get("dram_bytes_per_launch") if tr.get("kernel_source_hash") == source_hash(KSTORE_DEPS) else None


def measure_kstore(args, device):
    """The K-store configuration alone: 65,536 bf16 index-K rows through RMSNorm, RoPE,
    Hadamard and FP4 quantisation into scattered slots of a 2,048-page split cache (and the
    same rows into the 132 B/token FP8 layout), timed as captured graphs with the L2
    flushed before every launch."""
    import torch
    from sparse_attention_fp4_gb300 import fp4idx
    from sparse_attention_fp4_gb300 import workloads as wl
    ks = wl.kstore_65536()
    bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    k = bf16(ks.k_rows)
    pos = torch.from_numpy(ks.positions).to(device)
    slots = torch.from_numpy(ks.slots).to(device)
    nw = bf16(ks.norm_w)
    cs = bf16(wl.rope_cos_sin_table())
    payload, scale = fp4idx.alloc_cache(ks.num_pages, device=device)
    fp8 = torch.zeros((ks.num_pages, fp4idx.FP8_PAGE_BYTES), dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    calls = {"fp4": lambda: fp4idx.store_k(k, pos, slots, nw, ks.eps, cs, payload, scale, status=status),
             "fp8": lambda: fp4idx.store_k_fp8(k, pos, slots, nw, ks.eps, cs, fp8, status=status)}
    res = {}
    n_timed = min(args.steps, 200)
    sampler = ClockSampler(gpu_id_for(device.index)).start()
    for name, fn in calls.items():
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        # event-record nodes inside the graph, around the launch: the interval holds the
        # kernel, not the graph's own launch
        e0 = torch.cuda.Event(enable_timing=True, external=True)
        e1 = torch.cuda.Event(enable_timing=True, external=True)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            e0.record()
            fn()
            e1.record()
        ts = []
        for _ in range(n_timed):
            flush.zero_()
            torch.cuda._sleep(SPIN_CYCLES)
            g.replay()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        # the mean: event timestamps are coarse (steps of about 1 us were seen on GB300), so
        # a median snaps to a step while the mean of many launches does not
        us = statistics.mean(ts)
        out_b = 68 if name == "fp4" else 132
        nbytes = len(ks.positions) * (256 + 128 + 8 + out_b)  # row + cos/sin + position/slot + written entry
        res[name] = {"us": round(us, 2), "us_median": round(statistics.median(ts), 2),
                     "rows_per_s": round(len(ks.positions) / (us * 1e-6), 1),
                     "algorithmic_bytes": nbytes, "algorithmic_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "bytes_per_token": out_b}
    clocks = sampler.stop()
    assert fp4idx.read_status(status) == 0
    cpu = None
    if not args.no_cpu_baseline:
        # the oracle's K store on a bounded slice of the same rows (host cores)
        import dataclasses
        import oracle
        cs_np = wl.rope_cos_sin_table()
        n, secs, done = 4096, 0.0, 0
        while secs < min(args.cpu_seconds, 5.0) and done < len(ks.positions):
            sub = dataclasses.replace(ks, k_rows=ks.k_rows[done:done + n], positions=ks.positions[done:done + n],
                                      slots=ks.slots[done:done + n])
            t0 = time.perf_counter()
            oracle.store_k(sub, cs_np)
            secs += time.perf_counter() - t0
            done += len(sub.positions)
        cpu = {"value": round(done / secs, 1), "unit": "rows/s", "cores": oracle.max_threads(), "kind": "oracle",
               "sample": "%d rows of the same workload in slices of %d; %.3f s" % (done, n, secs)}
    peak, peak_kind = measured_peaks()
    fp4 = res["fp4"]
    roofline = {"bound": "hbm", "achieved": fp4["algorithmic_gbs"], "peak": peak, "unit": "GB/s",
                "frac": round(fp4["algorithmic_gbs"] / peak, 4), "traffic": stored_kstore_traffic(),
                "kernel": "store_k_kernel", "algorithmic_bytes": fp4["algorithmic_bytes"], "avg_launch_us": fp4["us"],
                "launch_timing": "event-record nodes around the launch inside its graph, mean of %d replays (L2 "
                                 "flushed before each)" % n_timed,
                "peak_source": "%s copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" % peak_kind}
    return {"workload": "kstore_65536", "rows": len(ks.positions), "cache_pages": ks.num_pages,
            "value": fp4["rows_per_s"], "unit": "rows/s", "steps": n_timed, "ms_per_step": round(fp4["us"] / 1e3, 5),
            "fp4": fp4, "fp8_132B": res["fp8"], "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks,
            "gpu_launches": 2 * n_timed}


def run_kstore(args):
    import torch
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    r = measure_kstore(args, device)
    line = {"metric": "K store rows/s (65,536 rows, split FP4 cache)", "value": r["value"], "unit": "rows/s",
            "n_gpus": 1, "steps": r["steps"], "warmup": max(3, args.warmup), "ms_per_step": r["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16->e2m1,ue8m0",
            "data": "synthetic",
            "config": {"workload": "kstore_65536", "rows": r["rows"], "cache_pages": r["cache_pages"],
                       "l2": "flushed before every launch"}}
    line.update({k: r[k] for k in ("fp4", "fp8_132B", "roofline", "cpu_baseline", "clocks", "gpu_launches")})
    print(json.dumps(line), flush=True)


def run_pages(args):
    """Whole-page access to the split cache on the decode pool (40,960 pages): export of
    every page in a random order to page rows, import back, and dequantisation of 8,192
    pages to fp32, each timed as a captured graph with the L2 flushed before every launch.
    Bytes counted: payload + scale read and written (4,352 B each way per page); for the
    dequantisation 4,352 B read and 32,768 B written per page."""
    import torch
    from sparse_attention_fp4_gb300 import fp4idx
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    P, n_deq = 40960, 8192
    gen = torch.Generator(device=device)
    gen.manual_seed(1005)
    payload = torch.randint(0, 256, (P, 4, 64, 16), dtype=torch.uint8, device=device, generator=gen)
    scale = torch.randint(100, 154, (P, 4, 64), dtype=torch.uint8, device=device, generator=gen)
    ids = torch.randperm(P, device=device, generator=gen).to(torch.int32)
    rows_p = torch.empty((P, 4096), dtype=torch.uint8, device=device)
    rows_s = torch.empty((P, 256), dtype=torch.uint8, device=device)
    out = torch.empty((n_deq, 64, 128), dtype=torch.float32, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    before = payload.clone(), scale.clone()
    calls = {"export": (lambda: fp4idx.export_pages(payload, scale, ids, rows_p, rows_s, status=status),
                        P * 4352 * 2),
             "import": (lambda: fp4idx.import_pages(rows_p, rows_s, ids, payload, scale, status=status),
                        P * 4352 * 2),
             "dequant": (lambda: fp4idx.dequant_pages(payload, scale, ids[:n_deq], out, status=status),
                         n_deq * (4352 + 32768))}
    peak, _ = measured_peaks()
    res = {}
    for name, (fn, nbytes) in calls.items():
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        ts = []
        for _ in range(min(args.steps, 200)):
            flush.zero_()
            torch.cuda._sleep(200000)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        us = statistics.median(ts)
        gbs = nbytes / (us * 1e-6) / 1e9
        res[name] = {"us": round(us, 2), "gbs": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak, 4)}
    assert fp4idx.read_status(status) == 0
    # export then import at the same ids restores the cache byte for byte
    assert torch.equal(payload, before[0]) and torch.equal(scale, before[1])
    print(json.dumps({"metric": "split-cache page export GB/s (40,960 pages, random order)",
                      "value": res["export"]["gbs"], "unit": "GB/s", "n_gpus": 1, "higher_is_better": True,
                      "data": "synthetic (random cache bytes)",
                      "config": {"workload": "pages_40960", "cache_pages": P, "dequant_pages": n_deq,
                                 "l2": "flushed before every launch"},
                      "export": res["export"], "import": res["import"], "dequant": res["dequant"]}), flush=True)


def run_cp_merge(args):
    """The exchange step of a context-parallel indexer on one GPU: 64 rows of the decode
    shape (contexts U[8192, 32768] compressed tokens), each split over 4 shards of equal
    token ranges; per shard the top-2048 (value, global position) candidates, chosen on
    the host from N(0,1) logits; fp4idx_topk_merge selects each row's top-2048 from the
    8,192 candidates.  Timed as a captured graph with the L2 flushed before each launch."""
    import torch
    from sparse_attention_fp4_gb300 import fp4idx
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    rng = np.random.default_rng(1006)
    T, S, k, span = 64, 4, 2048, 32768
    lens = rng.integers(8192, 32769, size=T)
    width = span // S
    cv = np.zeros((T, S, k), np.float32)
    ci = np.full((T, S, k), -1, np.int32)
    for t in range(T):
        row = rng.standard_normal(int(lens[t])).astype(np.float32)
        for s in range(S):
            lo = s * width
            part = row[lo:lo + width]
            if part.size == 0:
                continue
            order = np.lexsort((np.arange(part.size), -part.astype(np.float64)))[:k]
            sel = np.sort(order)
            ci[t, s, :sel.size] = sel + lo
            cv[t, s, :sel.size] = part[sel]
    d_cv = torch.from_numpy(cv).to(device)
    d_ci = torch.from_numpy(ci).to(device)
    out = torch.empty((T, k), dtype=torch.int32, device=device)
    ws = torch.empty(fp4idx.topk_merge_workspace_bytes(T, S, k), dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    fn = lambda: fp4idx.topk_merge(d_cv, d_ci, ws, out, status=status)
    for _ in range(max(3, args.warmup)):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    ts = []
    for _ in range(min(args.steps, 500)):
        flush.zero_()
        torch.cuda._sleep(200000)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    us = statistics.median(ts)
    assert fp4idx.read_status(status) == 0
    print(json.dumps({"metric": "context-parallel top-k merge, query rows/s (4 shards x 2,048 candidates)",
                      "value": round(T / (us * 1e-6), 1), "unit": "query rows/s", "n_gpus": 1,
                      "higher_is_better": True, "data": "synthetic",
                      "config": {"workload": "cp_merge_64x4x2048", "rows": T, "shards": S, "topk": k,
                                 "l2": "flushed before every launch"},
                      "merge_us": round(us, 2),
                      "candidate_bytes": int(T * S * k * 8)}), flush=True)


def run_qpack(args):
    """Q pack + head weights in one launch for the decode batch (64 rows, 64 heads x 128) with
    a hidden size of 7,168 (a reading: the pages give none), against the Q quant alone;
    graph replays with the L2 flushed before each launch.  Bytes counted: Q in (16 KB/row),
    packed Q out (4,352 B/row), hidden in (14 KB/row), the projection (917 KB, once), head
    weights out (256 B/row)."""
    import torch
    from sparse_attention_fp4_gb300 import fp4idx
    from sparse_attention_fp4_gb300 import workloads as wl
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    rng = np.random.default_rng(1007)
    T, D = 64, 7168
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    q = bf(wl.f32_to_bf16_bits(rng.standard_normal((T, 64, 128)).astype(np.float32)))
    qpos = torch.from_numpy(rng.integers(0, 131072, size=T).astype(np.int32)).to(device)
    hidden = bf(wl.f32_to_bf16_bits(rng.standard_normal((T, D)).astype(np.float32)))
    w_proj = bf(wl.f32_to_bf16_bits((rng.standard_normal((64, D)) / np.sqrt(D)).astype(np.float32)))
    cs = bf(wl.rope_cos_sin_table())
    qp, qs = fp4idx.alloc_query(T)
    w_out = torch.empty((T, 64), dtype=torch.float32, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    calls = {"quant_q_w": (lambda: fp4idx.quant_q_w(q, qpos, cs, hidden, w_proj, 0.125, qp, qs, w_out,
                                                    status=status),
                           T * (16384 + 4352 + 2 * D + 256) + 64 * D * 2),
             "quant_q": (lambda: fp4idx.quant_q(q, qpos, cs, qp, qs, status=status), T * (16384 + 4352))}
    peak, _ = measured_peaks()
    res = {}
    for name, (fn, nbytes) in calls.items():
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        ts = []
        for _ in range(min(args.steps, 500)):
            flush.zero_()
            torch.cuda._sleep(200000)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        us = statistics.median(ts)
        res[name] = {"us": round(us, 2), "algorithmic_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "frac_of_measured_hbm": round(nbytes / (us * 1e-6) / 1e9 / peak, 4)}
    assert fp4idx.read_status(status) == 0
    print(json.dumps({"metric": "Q pack + head weights, query rows/s (64 rows, hidden 7,168)",
                      "value": round(T / (res["quant_q_w"]["us"] * 1e-6), 1), "unit": "query rows/s", "n_gpus": 1,
                      "higher_is_better": True, "data": "synthetic",
                      "config": {"workload": "qpack_64x7168", "rows": T, "hidden_dim": D,
                                 "l2": "flushed before every launch"},
                      "quant_q_w": res["quant_q_w"], "quant_q_alone": res["quant_q"]}), flush=True)


def run_fp8_compare(args):
    """The same-box FP4/FP8 comparison on the decode batch (64 rows, contexts 8k-32k tokens):
    the logits launch over the split FP4 cache (68 B/token) and over the fused FP8 cache
    (132 B/token), each captured alone in a graph and replayed with the L2 flushed before
    every launch.  Bytes counted per launch: the K cache of every visible token once per
    sequence, the packed queries (FP4 4,352 B/row; FP8 8,192 B + 256 B of scales), head
    weights, page ids and row metadata."""
    import torch
    from sparse_attention_fp4_gb300 import fp4idx
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    b = make_batch("decode_b64")
    st = DecodeStep(b, device)
    ks = b.kstore
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    pages = torch.zeros((b.num_pages, fp4idx.FP8_PAGE_BYTES), dtype=torch.uint8, device=device)
    chunk = 1 << 20
    for r0 in range(0, ks.n_rows, chunk):
        r1 = min(ks.n_rows, r0 + chunk)
        fp4idx.store_k_fp8(bf(ks.k_rows[r0:r1]), torch.from_numpy(ks.positions[r0:r1]).to(device),
                           torch.from_numpy(ks.slots[r0:r1]).to(device), st.norm_w, ks.eps, st.cs, pages,
                           status=st.status)
    T = st.T
    q8 = torch.empty((T, 8, 64, 16), dtype=torch.uint8, device=device)
    s8 = torch.empty((T, 64), dtype=torch.float32, device=device)
    st.launch()  # FP4 queries and the schedule
    fp4idx.quant_q_fp8(st.q, st.qpos, st.cs, q8, s8, status=st.status)
    lg8 = torch.empty_like(st.logits)
    calls = dict(st.calls())
    L = b.context_lens.astype(np.int64)
    seq_max = np.zeros(int(b.row_seq.max()) + 1, np.int64)
    np.maximum.at(seq_max, b.row_seq.astype(np.int64), L)
    meta = 256.0 * T + 4.0 * np.ceil(seq_max / 64.0).sum() + 8.0 * T
    runs = {"fp4": (calls["logits"], 68.0 * seq_max.sum() + 4352.0 * T + meta, 68.0 * seq_max.sum()),
            "fp8": (lambda: fp4idx.logits_fp8(q8, s8, st.w, pages, st.pt, st.rs, st.cl, st.max_ctx, st.sched, lg8,
                                              status=st.status),
                    132.0 * seq_max.sum() + 8448.0 * T + meta, 132.0 * seq_max.sum())}
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    peak, peak_kind = measured_peaks()
    res = {}
    for name, (fn, nbytes, kbytes) in runs.items():
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        ts = []
        for _ in range(min(args.steps, 500)):
            flush.zero_()
            torch.cuda._sleep(200000)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        us = statistics.median(ts)
        res[name] = {"us": round(us, 2), "query_rows_per_s": round(T / (us * 1e-6), 1),
                     "kcache_gbs": round(kbytes / (us * 1e-6) / 1e9, 1),
                     "algorithmic_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "frac_of_%s_hbm" % peak_kind: round(nbytes / (us * 1e-6) / 1e9 / peak, 4),
                     "algorithmic_bytes": nbytes}
    assert fp4idx.read_status(st.status) == 0
    print(json.dumps({"metric": "paged logits, FP8 132 B/token vs FP4 68 B/token cache, query rows/s",
                      "value": res["fp8"]["query_rows_per_s"], "unit": "query rows/s", "n_gpus": 1,
                      "higher_is_better": True, "dtype": "e4m3->f32 (fp8) / e2m1,ue8m0->f32 (fp4)",
                      "data": "synthetic",
                      "config": {"workload": b.name, "rows": T, "context_tokens": int(L.sum()),
                                 "l2": "flushed before every launch", "timing": "median of graph replays"},
                      "fp8": res["fp8"], "fp4": res["fp4"],
                      "fp8_over_fp4_time": round(res["fp8"]["us"] / res["fp4"]["us"], 3)}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["fp4idx", "reference"], default="fp4idx")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + ["kstore", "pages", "cp_merge", "qpack", "fp8_compare"], default="decode_b64")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="leave out the other configurations (tiny, draft, prefill, K store) of the default line")
    ap.add_argument("--prep", choices=["one", "three"], default="one",
                    help="step preparation as fp4idx_prepare_step (one launch) or as its three calls")
    ap.add_argument("--fused", action="store_true",
                    help="read side through fp4idx_logits_topk_fused (one launch) instead of fp4idx_logits_topk")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "kstore":
        run_kstore(args)
    elif args.workload == "pages":
        run_pages(args)
    elif args.workload == "cp_merge":
        run_cp_merge(args)
    elif args.workload == "qpack":
        run_qpack(args)
    elif args.workload == "fp8_compare":
        run_fp8_compare(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
