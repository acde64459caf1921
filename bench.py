#!/usr/bin/env python
"""Benchmark of libnorm's normalization hot path on GB300.

One step = every row of the hot path, forward then backward, through the C ABI,
on the full-size synthetic workloads:
  * LayerNorm fp32 [64, 256]     (the small case: latency-bound, a few µs per call)
  * RMSNorm   bf16 [16384, 4096] (LLaMA-style, 8 outlier columns x20)
  * LayerNorm fp16 [25216, 768]  (ViT-B tokens)
  * BatchNorm2d fp32 [256, 64, 56, 56] + residual + ReLU, training (ResNet)
  * BatchNorm2d fp16 [128, 512, 7, 7] + GELU(erf), training
  * BatchNorm2d fp32 [256, 64, 56, 56] + residual + ReLU, eval (running statistics)
L2 is flushed before every call: a 512 MB write, then a read of another 512 MB
buffer, so the call starts with none of its data in L2 and without the flush's
dirty lines (whose write-back would otherwise land inside the timed call); each
call is timed with CUDA events on the stream it is launched on.  value = algorithmic bytes of the step
(every input read once, every output written once, saved statistics, ReLU mask
bits) / summed device time, in GB/s.  Per-call times, GB/s and fraction of the
measured HBM copy bandwidth are reported per workload.  Beside the step, and
outside its value, extra_rows times the channels-first LayerNorm on fp16
[128, 96, 56, 56] (ConvNeXt-T's 96 channels of 56x56) and GELU with fused
dropout (p = 0.1) on fp16 [25216, 3072] (ViT-B MLP hidden activations) and the
ViT-B LayerNorm fp16 [25216, 768] with its output kept in fp32, the same way.

--impl reference times the CPU oracle (plain double-precision C) on a bounded
sample of the same workloads (a quarter of the rows or channels of each), on all
host cores: each thread runs the unchanged oracle on its own share of the rows
or channels.  The GPU run's cpu_baseline reports the same on all cores and on
one core.

Multi-GPU: one process per GPU (torchrun); each rank runs the same step on its
own GPU (independent replicas, no collective on the data path); value sums
the bytes of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fwd+bwd achieved HBM GB/s and % of GB300 peak per norm config; µs per call"
UNIT = "GB/s"
WORKLOAD = ("norm suite fwd+bwd: LayerNorm f32 [64,256] + RMSNorm bf16 [16384,4096] + LayerNorm f16 [25216,768] + "
            "BatchNorm2d f32 [256,64,56,56]+res+ReLU train + BatchNorm2d f16 [128,512,7,7]+GELU "
            "train + BatchNorm2d f32 [256,64,56,56]+res+ReLU eval")
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 512 << 20
SAMPLE_FRACTION = 4   # the CPU oracle runs on 1/4 of the rows / channels of each workload


# ---------------------------------------------------------------------------
# multi-process plumbing (also exercised by the CPU tests with gloo)
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(value: float) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate(local_ms: float, local_bytes: float, world: int) -> tuple[float, float]:
    """(slowest rank's time in ms, whole-job GB/s) for weak scaling: every rank
    moved local_bytes in its own time."""
    slowest = reduce_max(local_ms)
    return slowest, world * local_bytes / (slowest * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# peaks, clocks, ncu traffic
# ---------------------------------------------------------------------------

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines: list[str] = []
        self.first = 0  # samples before this index were taken before the load began
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_live(self, timeout_s: float = 3.0):
        """Returns once the first sample has arrived (or after `timeout_s`) and
        marks the samples so far as taken before the load."""
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < timeout_s:
            time.sleep(0.01)
        self.first = len(self.lines)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sms, maxs, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        # the samples taken under load; all of them if none landed in that window
        window = self.lines[self.first:] or self.lines
        for ln in window:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxs.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxs),
                "reasons": sorted(reasons), "samples": len(sms)}


def ncu_traffic(kernel: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if the
    sources that kernel is built from are unchanged since the capture (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    from normalization_layernorm_rmsnorm_gb300.build import source_digest
    e = d.get(kernel)
    if not e or e.get("source_digest") != source_digest(e.get("sources")):
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# the GPU workload
# ---------------------------------------------------------------------------

def run_gpu(args, world, rank, local):
    import torch

    import normalization_layernorm_rmsnorm_gb300 as nrm
    from normalization_layernorm_rmsnorm_gb300 import workloads

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    nrm.load()
    calls = workloads.build_calls(dev)
    extra = workloads.build_extra_calls(dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_rd = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sum = torch.empty(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def one_step(record, which=calls):
        for c in which:
            flush.fill_(1.0)
            torch.sum(flush_rd, dim=0, keepdim=True, out=flush_sum)  # L2 left clean
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record(stream)
            c.fn()
            e.record(stream)
            if record is not None:
                record.append((c, s, e))

    # clocks are sampled from the first warm-up step to the end of the timed steps
    clocks = ClockSampler(local)
    clocks.start()
    clocks.wait_live()
    for _ in range(args.warmup):
        one_step(None)
    nrm.nrm_sync_status()
    torch.cuda.synchronize()

    barrier()
    torch.cuda.synchronize()
    recs = []
    for _ in range(args.steps):
        one_step(recs)
    torch.cuda.synchronize()
    barrier()
    clock_info = clocks.stop()
    nrm.nrm_sync_status()
    for c, s, e in recs:
        c.times_ms.append(s.elapsed_time(e))
    # the operations built beyond the step, timed the same way after it
    for _ in range(args.warmup):
        one_step(None, extra)
    recs = []
    for _ in range(args.steps):
        one_step(recs, extra)
    torch.cuda.synchronize()
    nrm.nrm_sync_status()
    for c, s, e in recs:
        c.times_ms.append(s.elapsed_time(e))

    step_ms_local = sum(statistics.mean(c.times_ms) for c in calls)
    step_bytes = sum(c.bytes for c in calls)
    step_ms, value = aggregate(step_ms_local, step_bytes, world)

    peak, peak_src = hbm_peak()
    per = per_workload(calls, peak)
    extra_rows = per_workload(extra, peak)

    dom = max(calls, key=lambda c: statistics.mean(c.times_ms) / c.launches)
    dom_t = statistics.mean(dom.times_ms)
    achieved = dom.bytes / (dom_t * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic(dom.kernel),
                "kernel": dom.kernel, "workload": dom.workload + " " + dom.phase,
                "bytes_per_launch": dom.bytes, "launch_us": round(dom_t * 1e3, 2),
                "peak_source": peak_src}

    e2e = run_e2e([calls, workloads.build_calls(dev)], args, stream, step_bytes, world)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded counter-based generator; shapes of the articles' models)",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}",
                   "l2": "flushed before every call (512 MB write, then 512 MB read: no call data, no dirty lines)",
                   "timing": "CUDA events around each call on its stream; step = sum of calls"},
        "roofline": roofline,
        "gpu_launches": sum(c.launches for c in calls) * args.steps,
        "e2e": e2e,
        "clocks": clock_info,
        "per_config": per,
        "extra_rows": extra_rows,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    return line


def per_workload(calls, peak):
    """Per workload and phase: mean and median device time, bytes, GB/s and
    fraction of the measured HBM bandwidth."""
    per = {}
    for c in calls:
        t = statistics.mean(c.times_ms)
        gbs = c.bytes / (t * 1e-3) / 1e9
        d = per.setdefault(c.workload, {})
        d[f"{c.phase}_us"] = round(t * 1e3, 2)
        d[f"{c.phase}_us_median"] = round(statistics.median(c.times_ms) * 1e3, 2)
        d[f"{c.phase}_bytes"] = c.bytes
        d[f"{c.phase}_gbs"] = round(gbs, 1)
        d[f"{c.phase}_frac"] = round(gbs / peak, 4)
    for d in per.values():
        if "fwd_us" in d and "bwd_us" in d:
            t = (d["fwd_us"] + d["bwd_us"]) * 1e-6
            d["fwd_bwd_us"] = round(d["fwd_us"] + d["bwd_us"], 2)
            d["fwd_bwd_gbs"] = round((d["fwd_bytes"] + d["bwd_bytes"]) / t / 1e9, 1)
            d["fwd_bwd_frac"] = round((d["fwd_bytes"] + d["bwd_bytes"]) / t / 1e9 / peak, 4)
    return per


def e2e_plan(calls):
    """The copies of one end-to-end step: {call index: tensors to upload before
    it} and {call index: tensors to download after it}.  An input is uploaded
    before the call that first reads it unless an earlier call of the step
    writes it (saved statistics, the ReLU mask stay on the device); an output
    is downloaded after the call that last writes it."""
    import collections
    first_read, last_write, written = {}, {}, set()
    for i, c in enumerate(calls):
        for t in c.inputs:
            if id(t) not in written:
                first_read.setdefault(id(t), (i, t))
        for t in c.outputs:
            written.add(id(t))
            last_write[id(t)] = (i, t)
    up = collections.defaultdict(list)
    down = collections.defaultdict(list)
    for i, t in first_read.values():
        up[i].append(t)
    for i, t in last_write.values():
        down[i].append(t)
    return up, down


def run_e2e(call_sets, args, stream, step_bytes, world):
    """Same step through host buffers, inside the timed region: every input
    uploaded from pinned host memory before the call that first reads it,
    every output downloaded after the call that last writes it.  Uploads and
    downloads run on their own streams, so they overlap each other and the
    other calls' kernels.  Two sets of device buffers alternate between steps:
    a step's uploads wait only for the kernels of the step two before (which
    read the same buffers) and its kernels only for that step's downloads, so
    the host link carries both directions at once throughout.  The pinned
    host buffers are shared by the two sets (uploads only read them; the
    downloads into them are ordered on one stream)."""
    import torch

    plans = [e2e_plan(calls) for calls in call_sets]
    up0, down0 = plans[0]
    host_up = {i: [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu()) for t in lst]
               for i, lst in up0.items()}
    host_down = {i: [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in lst] for i, lst in down0.items()}
    for up, down in plans[1:]:  # the sets are built alike: the same tensors in the same order
        assert {i: [t.shape for t in l] for i, l in up.items()} == {i: [t.shape for t in l] for i, l in up0.items()}
        assert {i: [t.shape for t in l] for i, l in down.items()} == {i: [t.shape for t in l] for i, l in down0.items()}
    h2d = sum(t.numel() * t.element_size() for lst in host_up.values() for t in lst)
    d2h = sum(t.numel() * t.element_size() for lst in host_down.values() for t in lst)
    steps = max(2, min(args.steps, 10))
    h2d_s = torch.cuda.Stream()
    d2h_s = torch.cuda.Stream()

    def step(k, prev):
        calls = call_sets[k % len(call_sets)]
        up, down = plans[k % len(call_sets)]
        if prev is not None:  # the last step on the same device buffers
            h2d_s.wait_event(prev[0])
            stream.wait_event(prev[1])
        up_done = []
        with torch.cuda.stream(h2d_s):
            for i in range(len(calls)):
                for d, h in zip(up[i], host_up.get(i, [])):
                    d.copy_(h, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(h2d_s)
                up_done.append(ev)
        for i, c in enumerate(calls):
            stream.wait_event(up_done[i])
            with torch.cuda.stream(stream):
                c.fn()
            if down[i]:
                ev = torch.cuda.Event()
                ev.record(stream)
                d2h_s.wait_event(ev)
                with torch.cuda.stream(d2h_s):
                    for d, h in zip(down[i], host_down[i]):
                        h.copy_(d, non_blocking=True)
        kernels_done = torch.cuda.Event()
        kernels_done.record(stream)
        copies_done = torch.cuda.Event()
        copies_done.record(d2h_s)
        return kernels_done, copies_done

    torch.cuda.synchronize()
    for k in range(len(call_sets)):
        step(k, None)
    torch.cuda.synchronize()
    barrier()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    h2d_s.wait_event(s)
    d2h_s.wait_event(s)
    prev = [None] * len(call_sets)
    last = None
    for k in range(steps):
        last = prev[k % len(call_sets)] = step(k, prev[k % len(call_sets)])
    stream.wait_event(last[1])  # the last downloads are inside the timed region
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    ms, gbs = aggregate(ms, step_bytes, world)
    return {"value": round(gbs, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3), "steps": steps,
            "overlap": "uploads, kernels and downloads on three streams, ordered per tensor; "
                       "two sets of device buffers alternate between steps"}


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def oracle_sample():
    """A bounded sample of each workload: the first 1/SAMPLE_FRACTION of the
    rows (row norms) or channels (BatchNorm), as float64 arrays, with the
    algorithmic bytes the same calls would move at the workload's dtypes."""
    from normalization_layernorm_rmsnorm_gb300 import synth
    items = []
    for name in ("ln_f32_64x256", "rms_bf16_16384x4096", "ln_f16_25216x768"):
        cfg = synth.CONFIGS[name]
        rows = cfg.rows // SAMPLE_FRACTION
        inp = synth.row_inputs(cfg, rows=rows)
        es = 2 if cfg.dtype != "f32" else 4
        a = {k: v.f64() for k, v in inp.items()}
        if cfg.kind == "rmsnorm":
            b = (2 * rows * cfg.cols * es + cfg.cols * es + rows * 4
                 + 3 * rows * cfg.cols * es + rows * 4 + 2 * cfg.cols * es)
        else:
            b = (2 * rows * cfg.cols * es + 2 * cfg.cols * es + 2 * rows * 4
                 + 3 * rows * cfg.cols * es + 2 * rows * 4 + 3 * cfg.cols * es)
        items.append((name, cfg, a, b, f"first {rows} of {cfg.rows} rows"))
    for name, training in (("bn_f32_256x64x56x56_res_relu", True), ("bn_f16_128x512x7x7_gelu", True),
                           ("bn_f32_256x64x56x56_res_relu", False)):
        cfg = synth.CONFIGS[name]
        ch = cfg.c // SAMPLE_FRACTION
        inp = synth.bn_inputs(cfg, channels=ch)
        a = {k: v.f64() for k, v in inp.items()}
        es = 2 if cfg.dtype != "f32" else 4
        m = cfg.n * ch * cfg.l
        words = cfg.n * ch * ((cfg.l + 31) // 32) * 4 if cfg.act == "relu" else 0
        acts = 3 if cfg.residual else 2          # fwd: x, (res), y
        bacts = 5 if cfg.residual else 3         # bwd: dy, x, dx, (dres)
        if not cfg.residual:
            bacts = 3
        b = (acts * m * es + words + 8 * ch * 4) + (bacts * m * es + words + 6 * ch * 4)
        tag = name + ("" if training else "_eval")
        items.append((tag, cfg, a, b, f"first {ch} of {cfg.c} channels"))
    return items


def oracle_step(orc, items):
    import oracle
    acts = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu": oracle.ACT_GELU}
    for tag, cfg, a, _, _ in items:
        if hasattr(cfg, "kind"):
            if cfg.kind == "rmsnorm":
                orc.rmsnorm_fwd(a["x"], a["w"], cfg.eps)
                orc.rmsnorm_bwd(a["dy"], a["x"], a["w"], cfg.eps)
            else:
                orc.layernorm_fwd(a["x"], a["w"], a["b"], cfg.eps)
                orc.layernorm_bwd(a["dy"], a["x"], a["w"], cfg.eps)
        else:
            training = not tag.endswith("_eval")
            res = a.get("res")
            f = orc.batchnorm_fwd(a["x"], res, a["w"], a["b"], cfg.eps, cfg.momentum, training,
                                  acts[cfg.act], a["running_mean"], a["running_var"],
                                  want_mask=cfg.act == "relu")
            orc.batchnorm_bwd(a["dy"], a["x"], res, a["w"], a["b"], a["running_mean"],
                              a["running_var"], cfg.eps, training, acts[cfg.act], mask=f["mask"])


def host_cores() -> int:
    """Cores this process may run on (the host's hardware concurrency unless
    an affinity mask narrows it)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_parts(items, parts):
    """Splits each sampled workload into `parts` pieces along its rows (row
    norms) or channels (BatchNorm), as contiguous float64 arrays: the oracle's
    results for the pieces are its results for the whole, row by row or channel
    by channel, and each thread runs the unchanged oracle on its own pieces."""
    import numpy as np
    out = [[] for _ in range(parts)]
    for tag, cfg, a, b, desc in items:
        row_norm = hasattr(cfg, "kind")
        extent = a["x"].shape[0] if row_norm else a["x"].shape[1]
        for i in range(parts):
            lo, hi = extent * i // parts, extent * (i + 1) // parts
            if hi <= lo:
                continue
            piece = {}
            for k, v in a.items():
                if row_norm:
                    piece[k] = np.ascontiguousarray(v[lo:hi]) if v.ndim == 2 else v
                else:
                    piece[k] = np.ascontiguousarray(v[:, lo:hi, :] if v.ndim == 3 else v[lo:hi])
            out[i].append((tag, cfg, piece, 0, desc))
    return [p for p in out if p]


def oracle_parallel(orc, parts):
    """One oracle step over all pieces, one thread per piece list (the oracle
    is a C library called through ctypes, which releases the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=len(parts)) as ex:
        for f in [ex.submit(oracle_step, orc, p) for p in parts]:
            f.result()


def cpu_baseline(reps_one=8, reps_all=48):
    """The oracle on the bounded sample: on one core (`reps_one` steps), then on
    every host core (`reps_all` steps); value = the all-cores figure."""
    import oracle
    orc = oracle.get()
    items = oracle_sample()
    total = sum(i[3] for i in items)
    t0 = time.perf_counter()
    for _ in range(reps_one):
        oracle_step(orc, items)
    dt1 = time.perf_counter() - t0
    cores = host_cores()
    parts = oracle_parts(items, cores)
    oracle_parallel(orc, parts)  # warm-up: page the pieces in
    t0 = time.perf_counter()
    for _ in range(reps_all):
        oracle_parallel(orc, parts)
    dtn = time.perf_counter() - t0
    sample = "; ".join(f"{i[0]}: {i[4]}" for i in items) + " (fwd+bwd each, C, fp64)"
    return {"value": round(total * reps_all / dtn / 1e9, 4), "unit": UNIT, "cores": len(parts),
            "kind": "oracle", "host_cores": cores, "seconds": round(dtn, 2),
            "threads": f"{len(parts)} threads, each running the oracle on its share of the rows or channels",
            "single_core": {"value": round(total * reps_one / dt1 / 1e9, 4), "unit": UNIT, "cores": 1,
                            "seconds": round(dt1, 2)},
            "sample": sample}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    import oracle
    orc = oracle.get()
    items = oracle_sample()
    total = sum(i[3] for i in items)
    cores = host_cores()
    parts = oracle_parts(items, cores)
    for _ in range(args.warmup):
        oracle_parallel(orc, parts)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_parallel(orc, parts)
        times.append(time.perf_counter() - t0)
    ms = statistics.mean(times) * 1e3
    value = total / (ms * 1e-3) / 1e9
    sample = ("; ".join(f"{i[0]}: {i[4]}" for i in items)
              + f" (fwd+bwd each, C, fp64, {len(parts)} threads on {cores} host cores)")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded counter-based generator; shapes of the articles' models)",
        "config": {"workload": WORKLOAD, "sample": f"1/{SAMPLE_FRACTION} of each workload"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": len(parts), "kind": "oracle",
                         "host_cores": cores, "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("libnorm", "reference"), default="libnorm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    import torch
    import torch.distributed as dist
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        line = run_gpu(args, world, rank, local)
    finally:
        if world > 1 and dist.is_initialized():
            dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
