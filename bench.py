#!/usr/bin/env python3
"""Benchmark of the exact tiled attention hot path on GB300.

One step is one pass over both halves of the hot path, each on its
full-size synthetic workload, with inputs resident in HBM:
  prefill  attn_fwd, bf16, causal, B=1, H=32, Hkv=8, N=8192, d=128
  decode   attn_decode_paged, bf16, 64 sequences x 1 token, H=32, Hkv=8, d=128,
           KV lengths uniform in [512, 32768], page size 16, pages at a random
           permutation of the pool (split kernel + merge kernel)
``value`` is the prefill throughput in TFLOP/s (4 N^2 d B H / 2 for causal),
the decode throughput is reported in GB/s beside it, each with its roofline.
``configs`` adds every workload of the suite timed on its own (fp32 N=256 d=64
with Q x1 and x30; bf16 B=4 H=12 N=2048 d=64 causal and non-causal; bf16
B=2 H=16 N=16384 d=128 causal with Q x1 and x40; the step's two halves), each
with its roofline fraction, the SM clock across its launches and the float64
oracle's host time on a sample of the same inputs.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
With --gpus N > 1 it runs under torch.distributed.run, one independent replica
per GPU (the path has no exchange step), and reports the aggregate.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill attention TFLOP/s & split-KV decode HBM GB/s on 1 GB300 (% roofline)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))


def reduce_max(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ peaks and clocks

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        for line in self.out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return None
        loaded = [r for r in rows if r[2] > 200.0] or rows   # samples drawing real power
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


def probe_mhz(p):
    """Average SM clock between two attn_clock_probe records (None unless both landed on one SM)."""
    t0, c0, sm0, ok0, t1, c1, sm1, ok1 = p
    if ok0 != 1 or ok1 != 1 or sm0 != sm1 or t1 <= t0:
        return None
    return round(1000.0 * (c1 - c0) / (t1 - t0), 1)


def smi_index(local_rank: int) -> str:
    """nvidia-smi's name for this rank's GPU (CUDA_VISIBLE_DEVICES entries are physical ids or UUIDs)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# ------------------------------------------------------------------ ncu traffic records

def kernel_source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "exact_tiled_attention_11_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "prefill_bf16": ["prefill_bf16.cu", "tc05.cuh", "common.cuh"],
    "decode_split": ["decode.cu", "common.cuh"],
    "prefill_fp8": ["prefill_fp8.cu", "tc05.cuh", "common.cuh"],
    "fp8_quantize": ["fp8_quantize.cu", "common.cuh"],
}


def recorded_traffic(name):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(name)
    if not rec or rec.get("source_sha") != kernel_source_sha(KERNEL_SOURCES[name]):
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ workload

def make_inputs(dev, seed=0):
    import torch
    from exact_tiled_attention_11_gb300 import workloads as W
    q, k, v = W.prefill_inputs_for(W.C3, seed=seed)
    kv = W.decode_inputs_for(W.C4, seed=seed)
    host = {"q": q, "k": k, "v": v, "dq": kv.q, "page_table": kv.page_table, "kv_lens": kv.kv_lens}
    d = {
        "q": q.to(dev), "k": k.to(dev), "v": v.to(dev),
        "dq": kv.q.to(dev), "k_pages": kv.k_pages.to(dev), "v_pages": kv.v_pages.to(dev),
        "page_table": kv.page_table.to(dev), "kv_lens": kv.kv_lens.to(dev),
    }
    d["o"] = torch.empty_like(d["q"])
    d["lse"] = torch.empty(W.C3.B, W.C3.H, W.C3.N, dtype=torch.float32, device=dev)
    d["do"] = torch.empty(W.C4.B, W.C4.H, W.C4.d, dtype=torch.bfloat16, device=dev)
    d["dlse"] = torch.empty(W.C4.B, W.C4.H, dtype=torch.float32, device=dev)
    return host, d, kv


def decode_bytes(kv):
    """Algorithmic bytes of one decode: K/V of the attended tokens, q, page table
    entries used, kv_lens, O (bf16) and LSE written."""
    import torch
    B, H, d = kv.q.shape
    pages_used = int(((kv.kv_lens.to(torch.int64) + kv.page_size - 1) // kv.page_size).sum())
    return kv.kv_bytes() + kv.q.numel() * 2 + pages_used * 4 + B * 4 + B * H * d * 2 + B * H * 4


# ------------------------------------------------------------------ the FP8 variant of the prefill

def fp8_variant(dev, d, t_peak, hbm_peak, reps=10):
    """attn_fp8_quantize + attn_fwd_fp8 on the benchmark's prefill inputs (B=1, H=32,
    Hkv=8, N=8192, d=128, causal), timed apart from the step: each launch between
    its own pair of CUDA events, with a 256 MiB write between launches so that no
    input is served from L2 and a device delay after it (device time only).  The fp8 tensor peak is the measured bf16 peak times
    the nominal fp8/bf16 ratio (2)."""
    import torch
    import exact_tiled_attention_11_gb300 as lib
    from exact_tiled_attention_11_gb300 import workloads as W
    stream = torch.cuda.current_stream(dev)
    signs = W.fp8_signs(128).to(dev)
    x = lib.attn_fp8_quantize(d["q"], d["k"], d["v"], signs)
    o = torch.empty_like(d["o"])
    lse = torch.empty_like(d["lse"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(fn):
        for _ in range(3):
            fn()
        tot = 0.0
        for _ in range(reps):
            flush.fill_(1)
            device_delay(stream, 100.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            tot += e0.elapsed_time(e1)
        return tot / reps

    q_ms = timed(lambda: lib.attn_fp8_quantize(d["q"], d["k"], d["v"], signs, x))
    a_ms = timed(lambda: lib.attn_fwd_fp8(x, o, lse, causal=True, scale=W.C3.scale))
    if lib.attn_device_error() != 0:
        raise SystemExit("a kernel recorded a device error in the FP8 measurement")
    flops = W.C3.flops(causal=True)
    n_in = d["q"].numel() + d["k"].numel() + d["v"].numel()
    q_bytes = n_in * 2 + n_in + 4 * (x.q_scale.numel() + x.k_scale.numel() + x.v_scale.numel())
    tf = flops / (a_ms * 1e-3) / 1e12
    gbs = q_bytes / (q_ms * 1e-3) / 1e9
    fp8_peak = 2.0 * t_peak
    return {
        "attention": {"kernel": "prefill_fp8_kernel", "value": tf, "unit": "TFLOP/s", "ms_per_call": a_ms,
                      "roofline": {"bound": "tensor", "achieved": tf, "peak": fp8_peak, "unit": "TFLOP/s",
                                   "frac": tf / fp8_peak, "traffic": recorded_traffic("prefill_fp8"),
                                   "peak_source": "2 x measured bf16_tflops (nominal fp8/bf16 ratio)"}},
        "quantize": {"kernel": "fp8_quantize_kernel", "value": gbs, "unit": "GB/s", "ms_per_call": q_ms,
                     "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                                  "frac": gbs / hbm_peak, "traffic": recorded_traffic("fp8_quantize"),
                                  "algorithmic_bytes_per_launch": q_bytes}},
        "l2": "256 MiB write between launches",
    }


# ------------------------------------------------------------------ launch overhead (eager vs CUDA graph)

def launch_overhead(dev, calls=20, reps=20):
    """Wall time per attn_decode_paged call on a launch-bound problem (one sequence of
    16 tokens, H=32, Hkv=8): issued eagerly through the binding, and replayed from a
    CUDA graph that captured `calls` back-to-back calls (one decode step of a
    `calls`-layer model).  Measured apart from the benchmark's timed region."""
    import torch
    import exact_tiled_attention_11_gb300 as lib
    from exact_tiled_attention_11_gb300 import workloads as W
    kv = W.decode_inputs(1, 32, 8, 128, 16, 16, 16, seed=5)
    t = [x.to(dev) for x in (kv.q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens)]
    S = lib.attn_decode_max_splits(1, 32, 8, kv.max_pages)
    ws = torch.empty(lib.attn_decode_workspace_size(1, 32, 128, S), dtype=torch.uint8, device=dev)
    o = torch.empty(1, 32, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(1, 32, dtype=torch.float32, device=dev)

    def call():
        lib.attn_decode_paged(*t, o, lse, num_splits=S, workspace=ws)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(5):
            call()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(calls * reps):
        call()
    torch.cuda.synchronize(dev)
    eager_us = (time.perf_counter() - t0) / (calls * reps) * 1e6
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(calls):
            call()
    graph.replay()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(reps):
        graph.replay()
    torch.cuda.synchronize(dev)
    graph_us = (time.perf_counter() - t0) / (calls * reps) * 1e6
    return {"workload": "attn_decode_paged, 1 sequence x 16 tokens, H=32 Hkv=8 d=128 (2 kernels per call)",
            "eager_us_per_call": eager_us, "graph_us_per_call": graph_us, "calls_per_graph": calls}


# ------------------------------------------------------------------ every workload, timed alone

def device_delay(stream, us):
    """Keep ``stream`` busy for about ``us`` microseconds with a spin kernel, so that the
    work queued behind it is already enqueued when it ends: an event-timed region that
    starts after it measures device time, not the host's time to enqueue the launch
    (host costs are in the end-to-end measurement)."""
    import torch
    sleep = getattr(torch.cuda, "_sleep", None)  # PyTorch's spin kernel (clock cycles)
    if sleep is None:
        return
    with torch.cuda.stream(stream):
        sleep(int(us * 2.1e3))  # cycles at up to 2.1 GHz


def time_launches(stream, fn, flush, reps, warmup=5):
    """Event-timed launches of ``fn`` on ``stream``: each between its own pair of CUDA
    events, an L2-sized write and a 100 us device delay between launches (outside the
    events).  Returns the sorted per-launch milliseconds."""
    import torch
    for _ in range(warmup):
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for e0, e1 in ev:
        flush.fill_(1)
        device_delay(stream, 100.0)
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return sorted(e0.elapsed_time(e1) for e0, e1 in ev)


def _timing(ms):
    return {"ms": statistics.median(ms), "ms_min": ms[0], "ms_max": ms[-1], "n": len(ms)}


def oracle_rows_sample(q, k, v, planes, rows, causal, scale):
    """Time the float64 oracle on sampled query rows of (batch, head) planes; return (flops, seconds)."""
    import numpy as np
    import oracle
    d = q.shape[-1]
    N, Nk = q.shape[2], k.shape[2]
    t0 = time.perf_counter()
    flops = 0.0
    for b, h in planes:
        oracle.attention_rows(q, k, v, b, h, rows, causal=causal, scale=scale)
        keys = np.minimum(rows + 1 + (Nk - N), Nk) if causal else np.full(len(rows), Nk)
        flops += float(np.sum(4.0 * keys * d))
    return flops, time.perf_counter() - t0


def per_config(dev, stream, t_peak, peak_src, step, baseline, reps=20, with_oracle=True):
    """Every workload of the benchmark suite on its own: TFLOP/s (4 N^2 d B H, halved
    for causal) or GB/s, the fraction of the measured roofline, the average SM clock
    across the timed launches (two on-device clock probes), and the float64 oracle's
    host time on a bounded sample of the same inputs, extrapolated to the whole
    workload by its FLOP count.  The long causal prefill (N=8192) and the paged
    decode come from the benchmark step itself."""
    import numpy as np
    import torch
    import exact_tiled_attention_11_gb300 as lib
    from exact_tiled_attention_11_gb300 import workloads as W

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    probe = torch.zeros(8, dtype=torch.int64, device=dev)
    rng = np.random.default_rng(1)
    out = {}

    def timed(fn):
        lib.attn_clock_probe(probe[:4], stream=stream)
        ms = time_launches(stream, fn, flush, reps)
        lib.attn_clock_probe(probe[4:], match=probe[:4], stream=stream)
        torch.cuda.synchronize()
        return ms, probe_mhz(probe.cpu().tolist())

    def oracle_leg(host, cfg, causal, n_planes, n_rows):
        if not with_oracle:
            return None
        planes = [(int(rng.integers(cfg.B)), int(rng.integers(cfg.H))) for _ in range(n_planes)]
        rows = np.sort(rng.choice(cfg.N, min(n_rows, cfg.N), replace=False))
        fl, dt = oracle_rows_sample(*host, planes, rows, causal, cfg.scale)
        rate = fl / dt
        return {"value": rate / 1e12, "unit": "TFLOP/s", "seconds": dt, "cores": host_cores(), "kind": "oracle",
                "est_seconds_whole_workload": cfg.flops(causal) / rate,
                "sample": f"{n_planes} (batch, head) planes x {len(rows)} random query rows ({fl:.3g} FLOP)"}

    # ---- the latency floor: one launch of a kernel that does no work (the clock probe)
    floor = time_launches(stream, lambda: lib.attn_clock_probe(probe[:4], stream=stream), flush, reps)
    floor_us = 1e3 * statistics.median(floor)

    # ---- fp32 exact attention, B=1 H=1 N=256 d=64, non-causal, Q x1 and x30
    for mult in W.C1.q_mults:
        host = W.prefill_inputs_for(W.C1, q_mult=mult)
        q, k, v = (t.to(dev) for t in host)
        o, lse = torch.empty_like(q), torch.empty(1, 1, W.C1.N, dtype=torch.float32, device=dev)
        ms, mhz = timed(lambda: lib.attn_fwd(q, k, v, o, lse, causal=False, scale=W.C1.scale))
        t = _timing(ms)
        tf = W.C1.flops(False) / (t["ms"] * 1e-3) / 1e12
        out[f"C1 fp32 x{mult:g}"] = {
            "workload": f"{W.C1.name}, non-causal, Q x{mult:g}", "dtype": "f32", **t, "value": tf,
            "unit": "TFLOP/s", "bound": "latency", "latency_floor_us": floor_us, "frac": floor_us / (1e3 * t["ms"]),
            "frac_of": "launch latency floor (event-timed launch of an empty kernel) / this launch",
            "sm_mhz": mhz, "oracle": oracle_leg(host, W.C1, False, 1, W.C1.N)}

    # ---- bf16 d=64, B=4 H=12 N=2048, causal and non-causal
    host = W.prefill_inputs_for(W.C2)
    q, k, v = (t.to(dev) for t in host)
    o, lse = torch.empty_like(q), torch.empty(W.C2.B, W.C2.H, W.C2.N, dtype=torch.float32, device=dev)
    for causal in (False, True):
        ms, mhz = timed(lambda: lib.attn_fwd(q, k, v, o, lse, causal=causal, scale=W.C2.scale))
        t = _timing(ms)
        tf = W.C2.flops(causal) / (t["ms"] * 1e-3) / 1e12
        out[f"C2 bf16 d64 {'causal' if causal else 'non-causal'}"] = {
            "workload": f"{W.C2.name}, {'causal' if causal else 'non-causal'}", "dtype": "bf16", **t,
            "value": tf, "unit": "TFLOP/s", "bound": "tensor", "kernel": "prefill_bf16_kernel<64>",
            "peak": t_peak, "frac": tf / t_peak, "peak_source": f"{peak_src} bf16_tflops (burst)",
            "sm_mhz": mhz, "oracle": oracle_leg(host, W.C2, causal, 2, 256)}
    del q, k, v, o, lse

    # ---- the step's own prefill (N=8192 causal GQA) and decode
    out["C3 bf16 N8192 causal GQA (step)"] = {
        "workload": W.C3.name, "dtype": "bf16", **_timing(sorted(step["pre_ms"])),
        "value": step["pre_tflops_median"], "unit": "TFLOP/s", "bound": "tensor",
        "kernel": "prefill_bf16_kernel<128>", "peak": t_peak, "frac": step["pre_tflops_median"] / t_peak,
        "sm_mhz": step["mhz"], "note": "inside the benchmark step, after the decode has streamed 4.1 GB",
        "oracle": baseline.get("prefill") if baseline else None}
    out["C4 paged decode (step)"] = {
        "workload": W.C4.name, "dtype": "bf16", **_timing(sorted(step["dec_ms"])),
        "value": step["dec_gbs_median"], "unit": "GB/s", "bound": "hbm", "peak": step["hbm_peak"],
        "frac": step["dec_gbs_median"] / step["hbm_peak"], "sm_mhz": step["mhz"],
        "oracle": baseline.get("decode") if baseline else None}

    # ---- bf16 d=128, B=2 H=16 N=16384 causal, Q x1 and x40
    kv_dev = None
    for mult in W.C5.q_mults:
        host = W.prefill_inputs_for(W.C5, q_mult=mult)
        q = host[0].to(dev)
        if kv_dev is None:
            kv_dev = (host[1].to(dev), host[2].to(dev))
        k, v = kv_dev
        o, lse = torch.empty_like(q), torch.empty(W.C5.B, W.C5.H, W.C5.N, dtype=torch.float32, device=dev)
        ms, mhz = timed(lambda: lib.attn_fwd(q, k, v, o, lse, causal=True, scale=W.C5.scale))
        t = _timing(ms)
        tf = W.C5.flops(True) / (t["ms"] * 1e-3) / 1e12
        out[f"C5 bf16 N16384 causal x{mult:g}"] = {
            "workload": f"{W.C5.name}, Q x{mult:g}", "dtype": "bf16", **t, "value": tf, "unit": "TFLOP/s",
            "bound": "tensor", "kernel": "prefill_bf16_kernel<128>", "peak": t_peak, "frac": tf / t_peak,
            "peak_source": f"{peak_src} bf16_tflops (burst)", "sm_mhz": mhz,
            "oracle": oracle_leg(host, W.C5, True, 1, 128)}
        del q, o, lse
    if lib.attn_device_error() != 0:
        raise SystemExit("a kernel recorded a device error in the per-workload measurements")
    return {"timing": (f"each launch between its own CUDA events on the launching stream, {reps} launches after "
                       f"5 warm-up, median reported; a 256 MiB write between launches (L2 flush)"),
            "runs": out}


# ------------------------------------------------------------------ CPU oracle legs

def oracle_prefill_sample(q, k, v, heads, rows, scale):
    """Time the float64 oracle on sampled (head, rows) of the long causal workload; return (flops, seconds)."""
    import numpy as np
    import oracle
    t0 = time.perf_counter()
    flops = 0.0
    d = q.shape[-1]
    for h in heads:
        oracle.attention_rows(q, k, v, 0, h, rows, causal=True, scale=scale)
        flops += float(np.sum(4.0 * (rows + 1) * d))    # causal: row r attends r + 1 keys
    return flops, time.perf_counter() - t0


def oracle_decode_sample(kv, seqs, scale):
    import oracle
    t0 = time.perf_counter()
    oracle.decode_paged(kv.q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens, scale=scale, seqs=seqs)
    dt = time.perf_counter() - t0
    Hkv, d = kv.k_pages.shape[1], kv.k_pages.shape[3]
    nbytes = sum(int(kv.kv_lens[b]) for b in seqs) * Hkv * d * 2 * 2
    return nbytes, dt


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


PREFILL_SAMPLE = {"heads": [0, 4, 9, 13, 18, 22, 27, 31], "rows": 4096}
DECODE_SAMPLE_SEQS = [0, 7, 21, 42]


def cpu_baseline(host, kv):
    import numpy as np
    from exact_tiled_attention_11_gb300 import workloads as W
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(W.C3.N, PREFILL_SAMPLE["rows"], replace=False))
    fl, dt = oracle_prefill_sample(host["q"], host["k"], host["v"], PREFILL_SAMPLE["heads"], rows, W.C3.scale)
    nb, ddt = oracle_decode_sample(kv, DECODE_SAMPLE_SEQS, W.C4.scale)
    pre_sample = (f"{len(PREFILL_SAMPLE['heads'])} heads x {len(rows)} random query rows of the N=8192 causal "
                  f"workload ({fl:.3g} algorithmic FLOP)")
    dec_sample = f"{len(DECODE_SAMPLE_SEQS)} of 64 sequences ({nb / 1e9:.3f} GB of K/V)"
    return {
        "value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
        "sample": (f"float64 NumPy oracle, prefill: {pre_sample} in {dt:.2f} s; decode: {dec_sample} in "
                   f"{ddt:.2f} s"),
        "prefill": {"value": fl / dt / 1e12, "unit": "TFLOP/s", "seconds": dt, "cores": host_cores(),
                    "kind": "oracle", "est_seconds_whole_workload": W.C3.flops(True) / (fl / dt),
                    "sample": pre_sample},
        "decode": {"value": nb / ddt / 1e9, "unit": "GB/s", "seconds": ddt, "cores": host_cores(), "kind": "oracle",
                   "est_seconds_whole_workload": kv.kv_bytes() / (nb / ddt), "sample": dec_sample},
    }


# ------------------------------------------------------------------ the reference arm: the oracle on the host

def bench_config(world, decode_desc):
    from exact_tiled_attention_11_gb300 import workloads as W
    return {
        "workload": f"{W.C3.name} + {W.C4.name}",
        "prefill": "attn_fwd bf16 causal B=1 H=32 Hkv=8 N=8192 d=128 scale=1/sqrt(128)",
        "decode": decode_desc,
        "l2": "no flush; every input set is larger than L2 (prefill 160 MiB touched, decode streams 4.1 GB per step)",
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, on bounded samples of the same workload."""
    if rank != 0:
        return 0
    import numpy as np
    from exact_tiled_attention_11_gb300 import workloads as W
    q, k, v = W.prefill_inputs_for(W.C3)
    kv = W.decode_inputs_for(W.C4)
    rng = np.random.default_rng(0)
    per_step_rows = 1024
    times, flops, dtimes, dbytes = [], [], [], []
    for i in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(W.C3.N, per_step_rows, replace=False))
        fl, dt = oracle_prefill_sample(q, k, v, [i % W.C3.H], rows, W.C3.scale)
        nb, ddt = oracle_decode_sample(kv, [i % W.C4.B], W.C4.scale)
        if i >= args.warmup:
            times.append(dt)
            flops.append(fl)
            dtimes.append(ddt)
            dbytes.append(nb)
    value = sum(flops) / sum(times) / 1e12
    ms = 1e3 * (sum(times) + sum(dtimes)) / len(times)
    sample = (f"each step: float64 NumPy oracle on {per_step_rows} random query rows of one head of the "
              f"N=8192 causal prefill workload (heads cycle per step) and on one of the 64 decode sequences")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(world, "attn_decode_paged workload, oracle gather + attention per sequence"),
        "decode": {"value": sum(dbytes) / sum(dtimes) / 1e9, "unit": "GB/s"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm

def run_ours(args, rank, local_rank, world):
    import torch
    import exact_tiled_attention_11_gb300 as lib
    from exact_tiled_attention_11_gb300 import workloads as W

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib.load_library()
    stream = torch.cuda.current_stream(dev)

    host, d, kv = make_inputs(dev)
    pre_flops = W.C3.flops(causal=True)
    dec_bytes = decode_bytes(kv)
    splits = lib.attn_decode_max_splits(W.C4.B, W.C4.H, W.C4.Hkv, kv.max_pages)
    ws = torch.empty(lib.attn_decode_workspace_size(W.C4.B, W.C4.H, W.C4.d, splits), dtype=torch.uint8, device=dev)

    def prefill():
        lib.attn_fwd(d["q"], d["k"], d["v"], d["o"], d["lse"], causal=True, scale=W.C3.scale)

    def decode():
        lib.attn_decode_paged(d["dq"], d["k_pages"], d["v_pages"], d["page_table"], d["kv_lens"], d["do"],
                              d["dlse"], scale=W.C4.scale, num_splits=0, workspace=ws)

    for _ in range(max(args.warmup, 3)):
        prefill()
        decode()
    torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    probe = torch.zeros(8, dtype=torch.int64, device=dev)  # two clock probes around the timed region
    with ClockSampler(smi_index(local_rank)) as clk:
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        lib.attn_clock_probe(probe[:4], stream=stream)
        # the first step's launches are enqueued while this delay runs (device time only)
        device_delay(stream, 300.0)
        start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            prefill()
            ev[i][1].record(stream)
            decode()
            ev[i][2].record(stream)
        stop.record(stream)
        lib.attn_clock_probe(probe[4:], match=probe[:4], stream=stream)
        torch.cuda.synchronize()
    timed_mhz = probe_mhz(probe.cpu().tolist())
    barrier(world)
    elapsed_ms = start.elapsed_time(stop)
    pre_ms = [e[0].elapsed_time(e[1]) for e in ev]
    dec_ms = [e[1].elapsed_time(e[2]) for e in ev]
    if lib.attn_device_error() != 0:
        raise SystemExit("a kernel recorded a device error during the benchmark")

    elapsed_ms = reduce_max(elapsed_ms, world)
    pre_tot = reduce_max(sum(pre_ms), world)
    dec_tot = reduce_max(sum(dec_ms), world)
    ms_per_step = elapsed_ms / args.steps
    pre_tflops = world * pre_flops * args.steps / (pre_tot * 1e-3) / 1e12
    dec_gbs = world * dec_bytes * args.steps / (dec_tot * 1e-3) / 1e9

    # ---------------- end to end through the public API: pinned host buffers, copies inside the timed region
    e2e = None
    if rank == 0 or world > 1:
        pin = {n: host[n].pin_memory() for n in ("q", "k", "v", "dq", "page_table", "kv_lens")}
        out_o = torch.empty(d["o"].shape, dtype=d["o"].dtype).pin_memory()
        out_lse = torch.empty(d["lse"].shape, dtype=torch.float32).pin_memory()
        out_do = torch.empty(d["do"].shape, dtype=d["do"].dtype).pin_memory()
        out_dlse = torch.empty(d["dlse"].shape, dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = sum(t.numel() * t.element_size() for t in (out_o, out_lse, out_do, out_dlse))
        pre_h2d = sum(pin[n].numel() * pin[n].element_size() for n in ("q", "k", "v"))

        bufs = (d["q"], d["k"], d["v"], d["o"], d["lse"])

        def e2e_step(evs):
            evs[0].record(stream)
            # prefill through the host-buffer entry point: Q, K, V in and O, LSE out,
            # pipelined with the attention by groups of KV heads inside the call
            lib.attn_fwd_host(pin["q"], pin["k"], pin["v"], out_o, out_lse, buffers=bufs, causal=True,
                              scale=W.C3.scale, stream=stream)
            evs[1].record(stream)
            d["dq"].copy_(pin["dq"], non_blocking=True)
            d["page_table"].copy_(pin["page_table"], non_blocking=True)
            d["kv_lens"].copy_(pin["kv_lens"], non_blocking=True)
            decode()
            out_do.copy_(d["do"], non_blocking=True)
            out_dlse.copy_(d["dlse"], non_blocking=True)
            evs[2].record(stream)

        for _ in range(max(args.warmup, 3)):
            e2e_step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
        torch.cuda.synchronize()
        eev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        barrier(world)
        for i in range(args.steps):
            e2e_step(eev[i])
        torch.cuda.synchronize()
        barrier(world)
        e_pre = reduce_max(sum(e[0].elapsed_time(e[1]) for e in eev), world)
        e_dec = reduce_max(sum(e[1].elapsed_time(e[2]) for e in eev), world)
        e2e = {"value": world * pre_flops * args.steps / (e_pre * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "prefill_h2d_bytes_per_step": pre_h2d,
               "decode": {"value": world * dec_bytes * args.steps / (e_dec * 1e-3) / 1e9, "unit": "GB/s"},
               "ms_per_step": (e_pre + e_dec) / args.steps,
               "note": ("prefill through attn_fwd_host (host buffers; copies pipelined with the attention "
                        "inside the call); decode KV pool is device-resident cache state, per step only q, "
                        "page table and kv_lens go H2D")}

    if rank != 0:
        return 0

    peaks, peak_src = load_peaks()
    t_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    pre_avg_s = pre_tot / args.steps * 1e-3 / 1.0
    dec_avg_s = dec_tot / args.steps * 1e-3
    pre_launch_tflops = pre_flops / pre_avg_s / 1e12
    dec_launch_gbs = dec_bytes / dec_avg_s / 1e9
    roof_pre = {"bound": "tensor", "achieved": pre_launch_tflops, "peak": t_peak, "unit": "TFLOP/s",
                "frac": pre_launch_tflops / t_peak, "traffic": recorded_traffic("prefill_bf16"),
                "kernel": "prefill_bf16_kernel<128>", "peak_source": f"{peak_src} bf16_tflops (burst)",
                "algorithmic_flops_per_launch": pre_flops}
    roof_dec = {"bound": "hbm", "achieved": dec_launch_gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": dec_launch_gbs / hbm_peak, "traffic": recorded_traffic("decode_split"),
                "kernel": "decode_split_kernel + merge_kernel (one attn_decode_paged call)",
                "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes_per_launch": dec_bytes}
    dominant = roof_dec if dec_tot > pre_tot else roof_pre
    clocks = clk.summary()
    if clocks is not None or timed_mhz is not None:
        clocks = dict(clocks or {})
        # average SM clock across exactly the timed region, from the device's own counters
        clocks["sm_mhz_timed_region"] = timed_mhz

    line = {
        "metric": METRIC, "value": pre_tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(world, (f"attn_decode_paged bf16 B=64 H=32 Hkv=8 d=128 page=16 lengths "
                                       f"randint[512,32768] seed 0 (pool {kv.k_pages.shape[0]} pages), "
                                       f"auto split count {splits}")),
        "decode": {"value": dec_gbs, "unit": "GB/s", "frac_of_hbm": dec_gbs / hbm_peak,
                   "ms_per_call": dec_tot / args.steps},
        "prefill": {"value": pre_tflops, "unit": "TFLOP/s", "frac_of_bf16": pre_tflops / t_peak,
                    "ms_per_call": pre_tot / args.steps},
        "roofline": dominant,
        "rooflines": {"prefill": roof_pre, "decode": roof_dec},
        "e2e": e2e,
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    line["launch_overhead"] = launch_overhead(dev)
    line["fp8"] = fp8_variant(dev, d, t_peak, hbm_peak)
    with_oracle = world == 1 and not args.no_cpu_baseline
    if with_oracle:
        line["cpu_baseline"] = cpu_baseline(host, kv)
    step = {"pre_ms": pre_ms, "dec_ms": dec_ms, "mhz": timed_mhz, "hbm_peak": hbm_peak,
            "pre_tflops_median": pre_flops / (statistics.median(pre_ms) * 1e-3) / 1e12,
            "dec_gbs_median": dec_bytes / (statistics.median(dec_ms) * 1e-3) / 1e9}
    line["configs"] = per_config(dev, stream, t_peak, peak_src, step, line.get("cpu_baseline"),
                                 with_oracle=with_oracle)
    print(json.dumps(line), flush=True)
    return 0


def run_profile_case(args):
    """One kernel family alone, for ncu: W warm-up launches then one more launch.

    prefill: a prefill workload (--workload C3: B=1, H=32, Hkv=8, N=8192, d=128
             causal; C2: B=4, H=12, N=2048, d=64; C5: B=2, H=16, N=16384, d=128).
    fp8:     the same inputs through attn_fp8_quantize + attn_fwd_fp8.
    decode:  the paged decode workload restricted to its first --decode-batch
             sequences (same length distribution and page placement recipe).
    """
    import torch
    import exact_tiled_attention_11_gb300 as lib
    from exact_tiled_attention_11_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    lib.load_library()
    if args.profile == "prefill":
        cfg = {"C2": W.C2, "C3": W.C3, "C5": W.C5}[args.workload]
        causal = True if args.causal is None else bool(args.causal)
        q, k, v = (t.to(dev) for t in W.prefill_inputs_for(cfg, q_mult=args.q_mult))
        for _ in range(args.warmup + 1):
            lib.attn_fwd(q, k, v, causal=causal, scale=cfg.scale)
        print(f"prefill case: {cfg.name}, causal={causal}, Q x{args.q_mult:g}, {cfg.flops(causal):.4g} FLOP per call")
    elif args.profile == "fp8":
        q, k, v = (t.to(dev) for t in W.prefill_inputs_for(W.C3))
        signs = W.fp8_signs(128).to(dev)
        for _ in range(args.warmup + 1):
            x = lib.attn_fp8_quantize(q, k, v, signs)
            lib.attn_fwd_fp8(x, causal=True, scale=W.C3.scale)
    else:
        kv = W.decode_inputs_for(W.C4, B=args.decode_batch)
        t = [x.to(dev) for x in (kv.q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens)]
        for _ in range(args.warmup + 1):
            lib.attn_decode_paged(*t, scale=W.C4.scale, num_splits=0)
        print(f"decode case: {args.decode_batch} sequences, {decode_bytes(kv)} algorithmic bytes per call")
    torch.cuda.synchronize()
    assert lib.attn_device_error() == 0
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=["prefill", "decode", "fp8"], default=None,
                    help="run one kernel family alone (for ncu) instead of the benchmark")
    ap.add_argument("--decode-batch", type=int, default=16)
    ap.add_argument("--workload", choices=["C2", "C3", "C5"], default="C3",
                    help="--profile prefill: C2 (B4 H12 N2048 d64), C3 (B1 H32/8 N8192 d128), C5 (B2 H16 N16384 d128)")
    ap.add_argument("--causal", type=int, choices=[0, 1], default=None, help="--profile prefill: causal (default 1)")
    ap.add_argument("--q-mult", type=float, default=1.0, help="--profile prefill: Q multiplier (30 or 40 stress)")
    args = ap.parse_args(argv)
    if args.profile:
        return run_profile_case(args)
    args.warmup = max(args.warmup, 3)
    rank, local_rank, world = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" and torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world)
        return run_ours(args, rank, local_rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
