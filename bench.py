#!/usr/bin/env python3
"""Benchmark of the fused attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-per-workload]

A step is one pass of the whole hot path over one batch of synthetic input:
the block-mask build (tile classification + work order) and the fused
forward kernel, through the C ABI, on inputs already resident in HBM.

Metric: useful TFLOPS = 4 * D * (visible (query, key) pairs) / time, so the
two GEMMs are counted only on unmasked pairs; softmax work is not counted.
The headline workload is dense B=4 H=16 S=4096 D=128; the other named
workloads are reported per mask type under "per_workload", each with the
forward kernel's median / p10 / p90 duration, the block-mask rebuild's time,
the backward's time (attn_bwd) and its TFLOPS at 2.5x the forward's FLOPs,
and the CTA-pair forward for D = 128.  The launch-bound tiny workload is
also timed from cold L2 and replayed from a CUDA graph.

One JSON line is printed by rank 0.  With N > 1 (torchrun, one process per
GPU) every rank runs an independent replica of the workload ("scaling":
"weak"): the path has no exchange step, so no collective is used.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

def visible_pairs(w: workloads.Workload, doc_ids=None, prefix_len=None) -> int:
    """Exact number of visible (query, key) pairs summed over batch and heads."""
    total = 0
    for b in range(w.B):
        i = np.arange(w.S_q, dtype=np.int64)
        qpos = i + w.q_offset
        lo = np.zeros(w.S_q, dtype=np.int64)
        hi = np.full(w.S_q, w.S_k - 1, dtype=np.int64)
        if w.causal:
            hi = np.minimum(hi, qpos)
        if w.window:
            lo = np.maximum(lo, qpos - w.window + 1)
            hi = np.minimum(hi, qpos)
        if prefix_len is not None:
            hi = np.minimum(hi, np.maximum(qpos, int(prefix_len[b]) - 1))
        if doc_ids is not None:
            ids = np.asarray(doc_ids[b])
            # packed documents: row i sees the keys of its own document
            starts = np.searchsorted(ids, ids, side="left")
            ends = np.searchsorted(ids, ids, side="right") - 1
            lo = np.maximum(lo, starts[:w.S_q])
            hi = np.minimum(hi, ends[:w.S_q])
        total += int(np.clip(hi - lo + 1, 0, None).sum())
    return total * w.H


def useful_flops(w, pairs):
    return 4.0 * w.D * pairs


def algorithmic_bytes(w):
    """Q, K, V read once; O and LSE written once."""
    return (2 * (w.B * w.H * w.S_q * w.D) * 2 + 2 * (w.B * w.H_kv * w.S_k * w.D) * 2
            + 4 * w.B * w.H * w.S_q)


KERNEL_SOURCES = ("attention_attn_fwd_04_gb300/csrc/attn_fwd_sm103.cu",
                  "attention_attn_fwd_04_gb300/csrc/sm103_ptx.cuh",
                  "attention_attn_fwd_04_gb300/csrc/attn_internal.h")


def kernel_source_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the forward kernel from the committed ncu
    summary of this workload, or None when there is none or the kernel
    source changed since it was captured."""
    import re
    path = os.path.join(ROOT, "profiles", "attn_fwd_kernel_%s.md" % workload)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        text = f.read()
    m = re.search(r"kernel source sha256\[:16\]: `([0-9a-f]+)`", text)
    b = re.search(r"dram bytes per launch \(read \+ write\): (\d+)", text)
    if not m or not b or m.group(1) != kernel_source_sha():
        return None
    return int(b.group(1))


# Nominal dense bf16 tensor peak of one GB300 (no sparsity), TFLOP/s, and
# its L2 size.
NOMINAL_BF16_TFLOPS = 2250.0
L2_BYTES = 129 * 2**20


def load_peaks():
    """The measured peaks (the generated MEASURED_PEAKS.json), else the
    fallback figures of an earlier GB300 measurement; says which."""
    fallback = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            if float(d["bf16_tflops"]) > 0:
                return d, "measured"
        except (OSError, ValueError, KeyError, TypeError):
            pass
    return fallback, "fallback"


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in (self.out or "").splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        # the median over every sample taken while the timed region ran
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def mods_of(w, inp, dev):
    kw = {}
    if w.causal:
        kw["causal"] = True
    if w.window:
        kw["window"] = w.window
    if w.document:
        kw["doc_ids"] = inp["doc_ids"].to(dev)
    if w.prefix_lm:
        kw["prefix_len"] = inp["prefix_len"].to(dev)
    if w.alibi:
        kw["alibi"] = True
    if w.softcap:
        kw["softcap"] = w.softcap
    if w.q_offset:
        kw["q_offset"] = w.q_offset
    return kw


def quantile(xs, f):
    """The f-quantile of xs by linear interpolation between order statistics."""
    ys = sorted(xs)
    x = f * (len(ys) - 1)
    i = int(x)
    return ys[i] if i + 1 >= len(ys) else ys[i] + (x - i) * (ys[i + 1] - ys[i])


def time_workload(attn, w, inp, dev, steps, warmup, flush_l2=False):
    """Device timing of `steps` whole steps (block mask + forward) on resident
    inputs, with the forward kernel's and the block-mask rebuild's own
    durations per step (CUDA events on the launching stream).

    flush_l2 writes a 256 MB buffer (larger than the 129 MB L2) before each
    step, outside the events, so every forward starts from cold L2; the
    step total then counts only the events' spans."""
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    kw = mods_of(w, inp, dev)
    mask_kw = {n: kw[n] for n in ("causal", "window", "doc_ids", "prefix_len", "q_offset") if n in kw}
    score_kw = {n: kw[n] for n in ("alibi", "softcap") if n in kw}
    o = torch.empty((w.B, w.H, w.S_q, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.S_q), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    bm = attn.build_block_mask(w.B, w.H, w.S_q, w.S_k, device=dev, **mask_kw)
    scrub = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush_l2 else None

    def step(ev=None):
        if scrub is not None:
            scrub.fill_(1)
        if ev is not None:
            ev[0].record(stream)
        bm.rebuild(stream)  # a1: tile classes + work order, into the same buffer
        if ev is not None:
            ev[1].record(stream)
        attn.attn_fwd_into(q, k, v, o, lse, scale=w.scale, block_mask=bm, stream=stream,
                           **mask_kw, **score_kw)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    start.record(stream)
    for e in evs:
        step(e)
    end.record(stream)
    torch.cuda.synchronize(dev)
    kern_ms = [e[1].elapsed_time(e[2]) for e in evs]
    mask_ms = [e[0].elapsed_time(e[1]) for e in evs]
    if flush_l2:
        total_ms = sum(e[0].elapsed_time(e[2]) for e in evs)
    else:
        total_ms = start.elapsed_time(end)
    st = attn.get_device_status(device=dev)
    if st != 0:
        raise RuntimeError("device status %s" % attn.status_string(st))
    return {"ms_step": total_ms / steps, "kernel_ms_mean": statistics.mean(kern_ms),
            "kernel_ms_median": statistics.median(kern_ms),
            "kernel_ms_p10": quantile(kern_ms, 0.1), "kernel_ms_p90": quantile(kern_ms, 0.9),
            "mask_build_ms": statistics.mean(mask_ms)}


def time_graph(attn, w, inp, dev, steps, warmup):
    """A launch-bound workload's step (block-mask rebuild + forward, the
    same C ABI calls) captured once in a CUDA graph and replayed: the
    device-side cost of the step once host and Python launch overhead no
    longer paces the GPU.  CUDA events around every replay."""
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    kw = mods_of(w, inp, dev)
    mask_kw = {n: kw[n] for n in ("causal", "window", "doc_ids", "prefix_len", "q_offset") if n in kw}
    score_kw = {n: kw[n] for n in ("alibi", "softcap") if n in kw}
    o = torch.empty((w.B, w.H, w.S_q, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.S_q), dtype=torch.float32, device=dev)
    bm = attn.build_block_mask(w.B, w.H, w.S_q, w.S_k, device=dev, **mask_kw)

    def step(stream):
        bm.rebuild(stream)
        attn.attn_fwd_into(q, k, v, o, lse, scale=w.scale, block_mask=bm, stream=stream,
                           **mask_kw, **score_kw)

    for _ in range(warmup):
        step(torch.cuda.current_stream(dev))
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        step(torch.cuda.current_stream(dev))
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    st = attn.get_device_status(device=dev)
    if st != 0:
        raise RuntimeError("device status %s" % attn.status_string(st))
    ms = [a.elapsed_time(b) for a, b in evs]
    return {"ms_per_step_graph": statistics.median(ms), "ms_per_step_graph_p10": quantile(ms, 0.1),
            "ms_per_step_graph_p90": quantile(ms, 0.9)}


def time_pair(attn, w, inp, dev, steps, warmup, flops, peak):
    """The same steps with the CTA-pair forward (option cta_pair; D = 128):
    its step time and the pair kernel's own throughput."""
    attn.set_option("cta_pair", 1)
    try:
        t = time_workload(attn, w, inp, dev, steps, warmup)
        ms, kms = t["ms_step"], t["kernel_ms_mean"]
    finally:
        attn.set_option("cta_pair", 0)
    kt = flops / (kms * 1e-3) / 1e12
    return {"pair_ms_per_step": ms, "pair_kernel_ms": kms, "pair_kernel_tflops": kt,
            "pair_frac": kt / peak}


def time_backward(attn, w, inp, dev, steps, warmup):
    """Device time of one attn_bwd call (block masks, row statistics, dQ and
    dK/dV kernels) on resident inputs, after the forward produced O and LSE."""
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    kw = mods_of(w, inp, dev)
    o, lse = attn.attn_fwd(q, k, v, scale=w.scale, **kw)
    g = torch.Generator(device=dev).manual_seed(7)
    do = torch.randn(o.shape, device=dev, generator=g).to(torch.bfloat16)
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        attn.attn_bwd(q, k, v, o, lse, do, scale=w.scale, stream=stream, **kw)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        attn.attn_bwd(q, k, v, o, lse, do, scale=w.scale, stream=stream, **kw)
    end.record(stream)
    torch.cuda.synchronize(dev)
    st = attn.get_device_status(device=dev)
    if st != 0:
        raise RuntimeError("device status %s" % attn.status_string(st))
    return start.elapsed_time(end) / steps


def time_mods3(attn, w, inp, dev, steps, warmup, R=256, p_open=0.5, seed=11):
    """The headline shape with the two descriptor mods of the next-step row:
    a seeded block map opening about half of the 128 x 128 tiles
    (block-sparse attention) and a relative-position bias table with R = 256.
    Returns (visible pairs, forward ms, backward ms)."""
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    g = torch.Generator().manual_seed(seed)
    nq, nk = -(-w.S_q // 128), -(-w.S_k // 128)
    blocks = (torch.rand((1, nq, nk), generator=g) < p_open).to(torch.uint8)
    rel = (torch.randn((w.H, 2 * R + 1), generator=g) * 0.5).to(torch.float32)
    kw = dict(blocks=blocks.to(dev), rel_bias=rel.to(dev))
    pairs = w.B * w.H * int(blocks.sum()) * 128 * 128  # S is a multiple of 128 here
    stream = torch.cuda.current_stream(dev)
    o, lse = attn.attn_fwd(q, k, v, scale=w.scale, **kw)
    do = torch.randn(o.shape, device=dev, generator=torch.Generator(device=dev).manual_seed(3))
    do = do.to(torch.bfloat16)

    def timed(fn, n):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / n

    fwd_ms = timed(lambda: attn.attn_fwd_into(q, k, v, o, lse, scale=w.scale, stream=stream, **kw),
                   steps)
    bwd_ms = timed(lambda: attn.attn_bwd(q, k, v, o, lse, do, scale=w.scale, stream=stream, **kw),
                   max(3, steps // 10))
    st = attn.get_device_status(device=dev)
    if st != 0:
        raise RuntimeError("device status %s" % attn.status_string(st))
    return pairs, fwd_ms, bwd_ms


def time_e2e(attn, w, inp, dev, steps, warmup):
    """Same metric through the public host-memory entry point
    (attn_fwd_host): every step copies Q, K, V (+ mask arrays) in from
    page-locked host memory and O, LSE back out.  The library overlaps one
    step's input copy with the previous step's compute and the output copy
    of the one before; the timed region still holds every step's copies."""
    hq, hk, hv = (inp[n].pin_memory() for n in ("q", "k", "v"))
    extra = {n: inp[n].pin_memory() for n in ("doc_ids", "prefix_len") if n in inp}
    ho = torch.empty((w.B, w.H, w.S_q, w.D), dtype=torch.bfloat16).pin_memory()
    hl = torch.empty((w.B, w.H, w.S_q), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream(dev)
    kw = mods_of(w, extra, torch.device("cpu"))

    def step():
        attn.attn_fwd_host(hq, hk, hv, out=ho, lse=hl, scale=w.scale, device=dev, stream=stream,
                           **kw)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        step()
    end.record(stream)
    torch.cuda.synchronize(dev)
    st = attn.get_device_status(device=dev)
    if st != 0:
        raise RuntimeError("device status %s" % attn.status_string(st))
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, *extra.values()))
    d2h = ho.numel() * 2 + hl.numel() * 4
    return start.elapsed_time(end) / steps, h2d, d2h


def oracle_sample(w, inp, target_s=15.0, seed=5):
    """Time the fp64 oracle on a bounded row sample; returns (TFLOPS, rows,
    secs, cores, visible pairs in the sample)."""
    import oracle
    cores = oracle.num_threads()
    g = torch.Generator().manual_seed(seed)
    N = w.B * w.H * w.S_q
    # calibrate on a few rows, then size the sample to ~target_s seconds
    probe = torch.randperm(N, generator=g)[:max(cores, 16)].numpy()
    t0 = time.perf_counter()
    oracle.attn_workload_rows(w, inp, rows=probe)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(min(N, max(len(probe), len(probe) * target_s / dt)))
    rows = torch.randperm(N, generator=g)[:n].numpy()
    t0 = time.perf_counter()
    oracle.attn_workload_rows(w, inp, rows=rows)
    secs = time.perf_counter() - t0
    # useful pairs in the sample: each sampled row contributes its visible keys
    pairs_per_row = visible_pairs(w, inp.get("doc_ids"), inp.get("prefix_len")) / N
    flops = useful_flops(w, pairs_per_row * n)
    return flops / secs / 1e12, n, secs, cores, pairs_per_row * n


def run_reference(args, world, rank):
    """Reference arm: the fp64 CPU oracle, as it stands, on the host cores.

    Each step times a seeded row sample of the workload; the sample size is
    set once from a calibration so that the whole --warmup + --steps run
    stays within about two minutes of CPU time."""
    if rank != 0:
        return
    import oracle
    w = workloads.get(args.workload)
    inp = workloads.generate(w)
    cores = oracle.num_threads()
    N = w.B * w.H * w.S_q
    g = torch.Generator().manual_seed(5)
    probe = torch.randperm(N, generator=g)[:max(cores, 16)].numpy()
    t0 = time.perf_counter()
    oracle.attn_workload_rows(w, inp, rows=probe)
    per_row = max(time.perf_counter() - t0, 1e-4) / len(probe)
    budget = min(args.ref_seconds, 120.0 / max(1, args.steps + args.warmup))
    n = int(min(N, max(cores, budget / per_row)))
    pairs_per_row = visible_pairs(w, inp.get("doc_ids"), inp.get("prefix_len")) / N
    vals, step_s = [], []
    for i in range(args.warmup + args.steps):
        rows = torch.randperm(N, generator=torch.Generator().manual_seed(100 + i))[:n].numpy()
        t0 = time.perf_counter()
        oracle.attn_workload_rows(w, inp, rows=rows)
        secs = time.perf_counter() - t0
        if i >= args.warmup:
            vals.append(useful_flops(w, pairs_per_row * n) / secs / 1e12)
            step_s.append(secs)
    value = statistics.mean(vals)
    pairs = visible_pairs(w, inp.get("doc_ids"), inp.get("prefix_len"))
    line = {
        "impl": "reference", "metric": "attention fwd useful TFLOPS (%s)" % w.name,
        "value": value, "unit": "TFLOPS", "n_gpus": 1, "steps": args.steps,
        # a step is the bounded row sample, timed as it ran; the whole
        # workload's time at the same rate is reported apart, labelled
        "warmup": args.warmup, "ms_per_step": statistics.mean(step_s) * 1e3,
        "ms_per_step_extrapolated": False,
        "full_workload_ms_extrapolated": useful_flops(w, pairs) / (value * 1e12) * 1e3,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": run_config(w, 1, False, useful_flops(w, pairs), pairs),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": "%d seeded query rows per step of %s (of %d rows)"
                                   % (n, w.name, N)},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_config(w, world, cta_pair, flops, pairs):
    """The workload keys of a bench line, the same for both arms."""
    return {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.H_kv, "S": w.S_q, "D": w.D,
            "parallelism": "replicas" if world > 1 else "single", "cta_pair": cta_pair,
            "l2": ("inputs larger than L2 (%d MB of Q/K/V)" % (algorithmic_bytes(w) // 2**20)
                   if algorithmic_bytes(w) > L2_BYTES else
                   "inputs fit in L2 (%d KB); timed warm, the cold-L2 time is reported apart"
                   % (algorithmic_bytes(w) // 1024)),
            "useful_flops": flops, "visible_pairs": pairs}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=workloads.HEADLINE, choices=list(workloads.WORKLOADS))
    ap.add_argument("--no-per-workload", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=8.0)
    ap.add_argument("--cta-pair", action="store_true",
                    help="run the timed forward on CTA pairs (option cta_pair, D = 128)")
    args = ap.parse_args()
    world, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import attention_attn_fwd_04_gb300 as attn
    if args.cta_pair:
        attn.set_option("cta_pair", 1)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peak_kind = load_peaks()

    w = workloads.get(args.workload)
    inp = workloads.generate(w)
    pairs = visible_pairs(w, inp.get("doc_ids"), inp.get("prefix_len"))
    flops = useful_flops(w, pairs)

    barrier(world)
    with ClockSampler(local) as clk:
        tw = time_workload(attn, w, inp, dev, args.steps, args.warmup)
    ms_step, kern_ms_mean = tw["ms_step"], tw["kernel_ms_mean"]
    clocks = clk.summary()
    ms_step_max = max_over_ranks(ms_step, world)
    value = world * flops / (ms_step_max * 1e-3) / 1e12

    # The burst cuBLAS figure: this kernel stays at full SM clock (see
    # "clocks"), so the power-capped sustained figure would flatter it.
    peak = peaks["bf16_tflops"]
    achieved = flops / (kern_ms_mean * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": profiled_traffic(w.name),
                "algorithmic_bytes": algorithmic_bytes(w),
                "kernel": "attn_fwd_kernel", "kernel_ms_mean": kern_ms_mean,
                "kernel_ms_median": tw["kernel_ms_median"],
                "kernel_ms_p10": tw["kernel_ms_p10"], "kernel_ms_p90": tw["kernel_ms_p90"],
                "peak_kind": "%s burst bf16 (cuBLAS)" % peak_kind,
                # the same kernel against the nominal dense bf16 tensor peak
                "nominal_peak": NOMINAL_BF16_TFLOPS,
                "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS}

    e2e = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h = time_e2e(attn, w, inp, dev, min(max(3, args.steps // 10), 200),
                                    args.warmup)
        e2e_ms = max_over_ranks(e2e_ms, world)
        e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    per = {}
    if not args.no_per_workload:
        for name, wx in workloads.WORKLOADS.items():
            bsteps = min(max(3, args.steps // 100), 20)
            if name == w.name:
                per[name] = {"tflops": value / world, "kernel_tflops": achieved,
                             "ms_per_step": ms_step, "frac": achieved / peak,
                             "kernel_ms_median": tw["kernel_ms_median"],
                             "kernel_ms_p10": tw["kernel_ms_p10"],
                             "kernel_ms_p90": tw["kernel_ms_p90"],
                             "mask_build_ms": tw["mask_build_ms"]}
                bms = time_backward(attn, w, inp, dev, bsteps, 3)
                per[name].update(bwd_ms=bms, bwd_tflops=2.5 * flops / (bms * 1e-3) / 1e12)
                if w.D == 128:
                    per[name].update(time_pair(attn, w, inp, dev, min(max(5, args.steps // 4), 500),
                                               3, flops, peak))
                continue
            ix = workloads.generate(wx)
            px = visible_pairs(wx, ix.get("doc_ids"), ix.get("prefix_len"))
            fx = useful_flops(wx, px)
            tx = time_workload(attn, wx, ix, dev, min(max(5, args.steps // 4), 500), 3)
            msx, kx = tx["ms_step"], tx["kernel_ms_mean"]
            per[name] = {"tflops": fx / (msx * 1e-3) / 1e12,
                         "kernel_tflops": fx / (kx * 1e-3) / 1e12,
                         "ms_per_step": msx, "kernel_ms": kx,
                         "kernel_ms_median": tx["kernel_ms_median"],
                         "kernel_ms_p10": tx["kernel_ms_p10"],
                         "kernel_ms_p90": tx["kernel_ms_p90"],
                         "mask_build_ms": tx["mask_build_ms"],
                         "frac": fx / (kx * 1e-3) / 1e12 / peak,
                         "hbm_gbs": algorithmic_bytes(wx) / (kx * 1e-3) / 1e9}
            if wx.S_q * wx.B * wx.H <= 4096:
                # the launch-bound tiny case, again from cold L2 each step
                tc = time_workload(attn, wx, ix, dev, min(max(5, args.steps // 20), 100), 3,
                                   flush_l2=True)
                per[name].update(kernel_ms_l2_flushed=tc["kernel_ms_median"],
                                 ms_per_step_l2_flushed=tc["ms_step"])
            # backward: 2.5x the forward's useful FLOPs (dQ, dK, dV and the
            # recomputed S and dP over the visible pairs, the usual count)
            bms = time_backward(attn, wx, ix, dev, bsteps, 3)
            per[name].update(bwd_ms=bms, bwd_tflops=2.5 * fx / (bms * 1e-3) / 1e12)
            if wx.D == 128:
                per[name].update(time_pair(attn, wx, ix, dev, min(max(5, args.steps // 4), 500), 3,
                                           fx, peak))
            del ix
        # the descriptor mods of the next-step row on the headline shape
        pm, fm, bmm = time_mods3(attn, w, inp, dev, min(max(5, args.steps // 4), 200), 3)
        fm_flops = 4.0 * w.D * pm
        per["blocks50_relbias256_" + w.name.split("_", 1)[1]] = {
            "tflops": fm_flops / (fm * 1e-3) / 1e12, "ms_per_step": fm,
            "frac": fm_flops / (fm * 1e-3) / 1e12 / peak, "visible_pairs": pm,
            "bwd_ms": bmm, "bwd_tflops": 2.5 * fm_flops / (bmm * 1e-3) / 1e12}

    # last, so that a failed capture cannot disturb the numbers above: the
    # launch-bound tiny workload replayed from a CUDA graph
    if not args.no_per_workload:
        for name, wx in workloads.WORKLOADS.items():
            if wx.S_q * wx.B * wx.H > 4096 or name not in per:
                continue
            try:
                per[name].update(time_graph(attn, wx, workloads.generate(wx), dev,
                                            min(max(20, args.steps // 10), 200), 5))
            except Exception as e:  # reported, not fatal
                per[name]["graph_error"] = str(e)[:200]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, n, secs, cores, spairs = oracle_sample(w, inp, target_s=15.0)
        cpu = {"value": tf, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
               "sample": "%d seeded query rows of %s (%.1f s)" % (n, w.name, secs),
               "rows_per_s": n / secs, "visible_pairs_per_s": spairs / secs,
               # labelled extrapolation: the sample's rate over every visible pair
               "extrapolated_full_workload_s": secs * pairs / spairs}

    if rank == 0:
        line = {
            "metric": "attention fwd useful TFLOPS (%s)" % w.name,
            "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": run_config(w, world, bool(args.cta_pair), flops, pairs),
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clocks,
            "gpu_launches": 3 * args.steps,
            "per_workload": per,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
