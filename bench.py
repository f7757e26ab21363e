#!/usr/bin/env python
"""Benchmark of the GB300 bf16 attention forward (one JSON line on rank 0).

Metric: attention forward TFLOPS = 4*B*H*Sq*Skv*d per call / time, and its fraction of the
measured GB300 dense bf16 peak.  Default workload: the largest single-GPU configuration, the
video-diffusion self-attention B=1, H=12, Sq=Skv=32760, d=128, BSHD, where one step runs its
two output rounding modes (RTNE, RTZ) back to back.  Inputs are seeded synthetic N(0,1) bf16
tensors already resident in HBM; where one input set is smaller than twice the 126 MB L2,
consecutive calls rotate over enough sets that their total exceeds it.

The roofline's kernel time is the attention kernel's duration from events recorded around it
in a second pass of the same calls, capped at the timed per-call time (an event between the
two kernels adds its own cost and serialises the combine's launch, so on a short call the raw
event time can run past the call); both are reported.

The `e2e` figure is the same metric through the public API with the data in pinned host
memory: every step copies its Q, K, V to the device and every output back, inside the timed
region, pipelined over two copy streams so that step i+1's inputs and step i's outputs move
while step i computes.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Causal workloads count 4*d flops per visible (query, key) pair and head, i.e. the masked
half of the score matrix is not counted as work.

--impl reference times the CPU oracle (fp64, OpenMP) on a bounded sample of the same
workload on the host cores.  Under torchrun (N > 1) each rank runs an independent replica
(no collective on the data path); value = all ranks' flops / max elapsed time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import itertools
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from workloads import WORKLOADS, make_qkv  # noqa: E402

METRIC = "attention fwd TFLOPS (4*B*H*Sq*Skv*d) and % of GB300 bf16 dense peak"
FALLBACK_PEAK_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
DEFAULT_STEPS = {"square": 1000, "cross": 1000, "video": 60, "stress": 1000, "tiny": 1000,
                 "causal_gqa": 200, "square_d64": 1000}
DEFAULT_WARMUP = {"square": 100, "cross": 100, "video": 5, "stress": 100, "tiny": 100,
                  "causal_gqa": 20, "square_d64": 100}
L2_BYTES = 126 * 2**20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--workload", default="video", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--op", default="fwd", choices=["fwd", "bwd", "varlen", "varlen_bwd", "paged", "paged_decode"],
                    help="bwd: time the attention backward (attn_bwd) instead of the forward; "
                         "varlen: the forward on a variable-length causal GQA prefill batch; "
                         "varlen_bwd: the backward on that batch; "
                         "paged: a chunked prefill over a paged K/V cache; "
                         "paged_decode: one query per sequence over a paged cache, heads packed")
    ap.add_argument("--no-pack", action="store_true",
                    help="with --op paged_decode: one query head per tile (no head packing)")
    ap.add_argument("--pack", action="store_true",
                    help="with --op varlen or paged: pack the query heads of each K/V head into one tile")
    ap.add_argument("--splits", type=int, default=0,
                    help="with --op varlen, paged or paged_decode: max_splits (>= 2: split the keys of "
                         "query blocks into up to that many parts when the items number fewer than the CTAs)")
    ap.add_argument("--decode-seqs", type=int, default=None,
                    help="with --op paged_decode: the number of sequences (default %d)" % 64)
    ap.add_argument("--paged-seqs", type=int, default=None,
                    help="with --op paged: the number of sequences (default %d)" % 16)
    ap.add_argument("--chunk", type=int, default=None,
                    help="with --op paged: the query chunk per sequence (default %d)" % 512)
    ap.add_argument("--deterministic", action="store_true",
                    help="with --op bwd: the deterministic backward (dQ summed in key-tile order)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device) -> float:
    """Largest value of x over all ranks (the job's elapsed time is its slowest rank's)."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flop_per_call: float, calls_per_rank: int, elapsed_ms: float) -> float:
    """Aggregate throughput: every rank runs the same replica workload (weak scaling)."""
    return world * flop_per_call * calls_per_rank / (elapsed_ms * 1e-3) / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0) or 0), \
            float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_PEAK_TFLOPS, 0.0, FALLBACK_HBM_GBS, "fallback"


def source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bf16_attention_forward_gb300", "csrc")
    for name in ("attn_fwd.cu", "ptx.cuh"):          # the forward kernel's sources
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str = "attn_fwd_kernel"):
    """DRAM bytes per launch of the attention kernel from the committed ncu summary, if it
    was taken on the current kernel source; otherwise None."""
    path = os.path.join(ROOT, "profiles", "%s_%s_traffic.md" % (kernel, workload))
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    kv = {}
    for ln in lines:
        if ln.startswith("- ") and ":" in ln:
            k_, v_ = ln[2:].split(":", 1)
            kv[k_.strip()] = v_.strip().strip("`")
    if kv.get("source_sha256_16") != source_hash():
        return None
    try:
        return int(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, enabled: bool = True):
        self.dev = device_index
        self.enabled = enabled
        self.proc = None
        self.path = None

    def __enter__(self):
        if not self.enabled:
            return self
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.enabled or self.proc is None or not self.path:
            return None
        rows = []
        for ln in open(self.path):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2])
                          if v.lower().startswith("active")})
        loaded = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def visible_keys(w, rows) -> int:
    """Keys that take part, summed over flat query rows (b*H + h)*Sq + i."""
    if not w.causal:
        return len(rows) * w.Skv
    off = w.Skv - w.Sq
    return sum(min(max(r % w.Sq + off + 1, 0), w.Skv) for r in rows)


def cpu_oracle_sample(w, qkv_cpu, mode: str, seconds: float, seed: int = 99):
    """Time the oracle on a seeded row sample sized to about `seconds` of host work."""
    import oracle
    q, k, v = qkv_cpu
    total = w.B * w.H * w.Sq
    threads = len(os.sched_getaffinity(0))
    g = torch.Generator().manual_seed(seed)
    probe = torch.randint(0, total, (8 * threads,), generator=g).tolist()
    oracle.attention(q, k, v, w.layout, mode, rows=probe[:threads], threads=threads,
                     causal=w.causal)   # warm-up
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.layout, mode, rows=probe, threads=threads, causal=w.causal)
    dt = max(time.perf_counter() - t0, 1e-4)
    n = int(max(threads, min(total, len(probe) * seconds / dt)))
    rows = torch.randint(0, total, (n,), generator=g).tolist()
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.layout, mode, rows=rows, threads=threads, causal=w.causal)
    dt = time.perf_counter() - t0
    flop = 4.0 * visible_keys(w, rows) * w.d
    return {"value": flop / dt / 1e12, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
            "sample": "%d of %d query rows (seeded), %s keys, mode %s, %.1f s"
                      % (n, total, "their visible" if w.causal else "all %d" % w.Skv, mode, dt)}


def run_reference(args, w, rank, world):
    if rank != 0:
        return 0
    steps = args.steps if args.steps is not None else DEFAULT_STEPS[w.name]
    warmup = args.warmup if args.warmup is not None else DEFAULT_WARMUP[w.name]
    import oracle
    q, k, v = make_qkv(w.B, w.H, w.Sq, w.Skv, w.d, w.layout, seed=w.seed, sigma=w.sigma,
                       nonfinite_frac=w.nonfinite_frac, Hkv=w.kv_heads)
    threads = len(os.sched_getaffinity(0))
    total = w.B * w.H * w.Sq
    budget = 150.0                           # seconds for the whole run
    g = torch.Generator().manual_seed(7)
    probe = torch.randint(0, total, (max(threads, 8),), generator=g).tolist()
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.layout, w.modes[0], rows=probe, threads=threads, causal=w.causal)
    per_row = max(time.perf_counter() - t0, 1e-4) / len(probe)
    rows_per_step = int(max(1, min(total, budget / (steps + warmup) / per_row)))
    samples = [torch.randint(0, total, (rows_per_step,), generator=g).tolist()
               for _ in range(min(steps + warmup, 8))]
    for i in range(warmup):
        oracle.attention(q, k, v, w.layout, w.modes[i % len(w.modes)],
                         rows=samples[i % len(samples)], threads=threads, causal=w.causal)
    t0 = time.perf_counter()
    for i in range(steps):
        oracle.attention(q, k, v, w.layout, w.modes[i % len(w.modes)],
                         rows=samples[i % len(samples)], threads=threads, causal=w.causal)
    dt = time.perf_counter() - t0
    flop = 4.0 * w.d * sum(visible_keys(w, samples[i % len(samples)]) for i in range(steps))
    val = flop / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOPS", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": dt * 1e3 / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,%g) bf16)" % w.sigma,
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.kv_heads, "Sq": w.Sq,
                   "Skv": w.Skv, "d": w.d, "causal": w.causal, "layout": w.layout,
                   "modes": list(w.modes),
                   "step": "oracle on %d seeded query rows (%s keys)"
                           % (rows_per_step, "visible" if w.causal else "all")},
        "cpu_baseline": {"value": val, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": "%d of %d query rows per step" % (rows_per_step, total)},
        "e2e": {"value": val, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_backward(args, w):
    """Time attn_bwd on resident inputs (the forward's output and LSE made beforehand).
    FLOP per call: five matrix products of 2*d per visible (query, key) pair and head."""
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    dev = torch.device("cuda", 0)
    import bf16_attention_forward_gb300 as attn
    attn.load()
    steps = args.steps if args.steps is not None else 100
    warmup = max(3, args.warmup if args.warmup is not None else 10)
    q, k, v = (t.to(dev) for t in make_qkv(w.B, w.H, w.Sq, w.Skv, w.d, w.layout, seed=w.seed,
                                               sigma=w.sigma, Hkv=w.kv_heads))
    g = make_qkv(w.B, w.H, w.Sq, 1, w.d, w.layout, seed=w.seed + 77)[0].to(dev)
    o, lse = attn.attn_fwd_ex(q, k, v, layout=w.layout, causal=w.causal, return_lse=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    a_ws = None

    def call():
        nonlocal a_ws
        attn.attn_bwd(q, k, v, o, g, lse, layout=w.layout, causal=w.causal, dq=dq, dk=dk, dv=dv,
                      workspace=a_ws, deterministic=args.deterministic)

    # size the workspace once, outside the timed region
    import ctypes
    a = attn.BwdArgs()
    a.B, a.H, a.Hkv, a.Sq, a.Skv, a.d = w.B, w.H, w.kv_heads, w.Sq, w.Skv, w.d
    a.layout, a.causal = attn.LAYOUTS[w.layout], int(w.causal)
    a.deterministic = int(args.deterministic)
    a_ws = torch.empty(max(int(attn.load().attn_bwd_workspace_size(ctypes.byref(a))), 16),
                       dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0, enabled=not args.no_clocks) as clocks:
        t0.record()
        for _ in range(steps):
            call()
        t1.record()
        torch.cuda.synchronize(dev)
    st, site = attn.bwd_device_status()
    assert st == 0, "backward device status %d at wait site %d" % (st, site)
    ms = t0.elapsed_time(t1) / steps
    flop = 10 * w.B * w.H * w.visible_pairs * w.d
    value = flop / (ms * 1e-3) / 1e12
    peak, peak_sust, _, peak_src = measured_peaks()
    line = {
        "metric": "attention bwd TFLOPS (10*B*H*Sq*Skv*d: five products per visible pair)",
        "value": value, "unit": "TFLOPS", "n_gpus": 1, "steps": steps, "warmup": warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic (seeded N(0,%g) bf16)" % w.sigma,
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.kv_heads, "Sq": w.Sq,
                   "Skv": w.Skv, "d": w.d, "causal": w.causal, "layout": w.layout,
                   "deterministic": bool(args.deterministic),
                   "step": ("one deterministic attn_bwd call: D/LSE preprocessing, the tcgen05 backward "
                            "kernel storing each key tile's dQ terms, and the ordered dQ sum and rounding "
                            "with any split units' dK/dV sums") if args.deterministic else
                           ("one attn_bwd call: D/LSE preprocessing with the dQ zeroing, the tcgen05 "
                            "backward kernel, and the dQ rounding with any split units' dK/dV sums")},
        "roofline": {"bound": "tensor", "achieved": value, "peak": peak, "unit": "TFLOP/s",
                     "frac": value / peak, "peak_source": peak_src + " burst bf16 (cuBLAS)",
                     "timed": "whole call"},
        "clocks": clocks.summary(),
        "gpu_launches": 3 * steps,
    }
    print(json.dumps(line), flush=True)
    return 0


# A variable-length prefill batch: 16 sequences with seeded lengths in [256, 8192], 32 query
# heads on 8 K/V heads, d = 128, causal, packed along the token axis (attn_fwd_varlen).
VARLEN_SEQS, VARLEN_H, VARLEN_HKV, VARLEN_D, VARLEN_SEED = 16, 32, 8, 128, 9


def varlen_lengths():
    import numpy as np
    return np.random.default_rng(VARLEN_SEED).integers(256, 8193, VARLEN_SEQS).tolist()


def run_varlen(args, backward=False):
    """Time attn_fwd_varlen (or, with ``backward``, attn_bwd_varlen on the forward's output
    and LSE) on resident inputs.  FLOP per call: 4*d (backward: 10*d, five products) per
    visible (query, key) pair and head, summed over the sequences (the causal mask's hidden
    half not counted)."""
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    dev = torch.device("cuda", 0)
    import bf16_attention_forward_gb300 as attn
    attn.load()
    steps = args.steps if args.steps is not None else 50
    warmup = max(3, args.warmup if args.warmup is not None else 10)
    lens = varlen_lengths()
    total = sum(lens)
    q, k, v = (t[0].to(dev) for t in make_qkv(1, VARLEN_H, total, total, VARLEN_D, "bshd", seed=VARLEN_SEED,
                                               Hkv=VARLEN_HKV))
    cu = torch.tensor([0] + list(itertools.accumulate(lens)), dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    import ctypes
    a = attn.VarlenArgs()
    a.B, a.H, a.Hkv, a.total_q, a.total_k, a.d = len(lens), VARLEN_H, VARLEN_HKV, total, total, VARLEN_D
    ws = torch.empty(int(attn.load().attn_fwd_varlen_workspace_size(ctypes.byref(a))), dtype=torch.uint8, device=dev)

    a.pack_heads = int(args.pack and not backward)
    a.max_splits = 0 if backward else args.splits
    ws = torch.empty(int(attn.load().attn_fwd_varlen_workspace_size(ctypes.byref(a))), dtype=torch.uint8, device=dev)

    def call():
        attn.attn_fwd_varlen(q, k, v, cu, cu, max_seqlen_q=max(lens), o=o, causal=True, workspace=ws,
                             pack_heads=args.pack, max_splits=args.splits)

    if backward:
        o, lse = attn.attn_fwd_varlen(q, k, v, cu, cu, causal=True, return_lse=True)
        g = make_qkv(1, VARLEN_H, total, 1, VARLEN_D, "bshd", seed=VARLEN_SEED + 77)[0][0].to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        b = attn.BwdVarlenArgs()
        b.B, b.H, b.Hkv, b.total_q, b.total_k, b.d = len(lens), VARLEN_H, VARLEN_HKV, total, total, VARLEN_D
        bws = torch.empty(int(attn.load().attn_bwd_varlen_workspace_size(ctypes.byref(b))), dtype=torch.uint8,
                          device=dev)

        def call():
            attn.attn_bwd_varlen(q, k, v, o, g, lse, cu, cu, causal=True, dq=dq, dk=dk, dv=dv, workspace=bws)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0, enabled=not args.no_clocks) as clocks:
        t0.record()
        for _ in range(steps):
            call()
        t1.record()
        torch.cuda.synchronize(dev)
    st, site = attn.device_status()
    assert st == 0, "device status %d at site %d" % (st, site)
    if backward:
        st, site = attn.bwd_device_status()
        assert st == 0, "backward device status %d at site %d" % (st, site)
    ms = t0.elapsed_time(t1) / steps
    pairs = sum(n * (n + 1) // 2 for n in lens)
    flop = (10 if backward else 4) * VARLEN_H * VARLEN_D * pairs
    value = flop / (ms * 1e-3) / 1e12
    peak, _, _, peak_src = measured_peaks()
    line = {
        "metric": ("attention bwd TFLOPS (10*d per visible pair and head, variable-length batch)" if backward else
                   "attention fwd TFLOPS (4*d per visible pair and head, variable-length batch)"),
        "value": value, "unit": "TFLOPS", "n_gpus": 1, "steps": steps, "warmup": warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": "varlen_prefill" + ("_bwd" if backward else ""), "sequences": len(lens), "lengths": lens,
                   "pack_heads": bool(args.pack and not backward),
                   "max_splits": 0 if backward else args.splits,
                   "total_tokens": total, "H": VARLEN_H, "Hkv": VARLEN_HKV, "d": VARLEN_D, "causal": True,
                   "layout": "packed tokens [T, H, d]", "modes": ["rtne"], "flop_per_call": flop,
                   "step": ("one attn_bwd_varlen call: planning (offsets, tensor maps, units), row "
                            "statistics with the dQ zeroing, the tcgen05 backward kernel, the dQ rounding")
                           if backward else ("one attn_fwd_varlen call: the offsets/tensor-map preprocessing "
                                             "kernel and the attention kernel"),
                   "l2": "inputs %.0f MB > 126 MB L2" % ((q.numel() + k.numel() + v.numel()) * 2 / 2**20)},
        "roofline": {"bound": "tensor", "achieved": value, "peak": peak, "unit": "TFLOP/s",
                     "frac": value / peak, "peak_source": peak_src + " burst bf16 (cuBLAS)",
                     "timed": "whole call"},
        "clocks": clocks.summary(),
        "gpu_launches": (4 if backward else (3 if args.splits > 1 else 2)) * steps,
    }
    print(json.dumps(line), flush=True)
    return 0


# Chunked prefill over a paged K/V cache: 16 sequences whose caches hold seeded lengths in
# [2048, 16384] tokens (256-slot pages in a shuffled order), each with its last 512 tokens as
# the new query chunk (causal, aligned at the end), 32 query heads on 8 K/V heads, d = 128.
PAGED_SEQS, PAGED_CHUNK, PAGED_PAGE, PAGED_SEED = 16, 512, 256, 10
# Decoding over a paged cache: 64 sequences with seeded cache lengths in [4096, 16384], one new
# query each (the last cache slot), query heads packed per K/V head unless --no-pack.
DECODE_SEQS, DECODE_SEED = 64, 11


def run_paged(args, decode=False):
    """Time attn_fwd_paged on resident inputs.  FLOP per call: 4*d per visible (query, key)
    pair and head.  Decoding is memory-bound: its line also reports the K/V bytes per second
    against the HBM peak."""
    import numpy as np
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    dev = torch.device("cuda", 0)
    import bf16_attention_forward_gb300 as attn
    attn.load()
    steps = args.steps if args.steps is not None else 50
    warmup = max(3, args.warmup if args.warmup is not None else 10)
    seqs, chunk = ((args.decode_seqs or DECODE_SEQS, 1) if decode
                   else (args.paged_seqs or PAGED_SEQS, args.chunk or PAGED_CHUNK))
    pack = (decode and not args.no_pack) or (not decode and args.pack)
    rng = np.random.default_rng(DECODE_SEED if decode else PAGED_SEED)
    lens_k = rng.integers(4096 if decode else 2048, 16385, seqs).tolist()
    need = [-(-n // PAGED_PAGE) for n in lens_k]
    n_pages = sum(need)
    H, Hkv, d = VARLEN_H, VARLEN_HKV, VARLEN_D
    g = torch.Generator(device="cpu").manual_seed(PAGED_SEED)
    kc = torch.randn((n_pages, PAGED_PAGE, Hkv, d), generator=g).to(torch.bfloat16).to(dev)
    vc = torch.randn((n_pages, PAGED_PAGE, Hkv, d), generator=g).to(torch.bfloat16).to(dev)
    order = rng.permutation(n_pages)
    table = np.zeros((seqs, max(need)), dtype=np.int32)
    nxt = 0
    for b, n in enumerate(need):
        table[b, :n] = order[nxt:nxt + n]
        nxt += n
    total_q = seqs * chunk
    q = torch.randn((total_q, H, d), generator=g).to(torch.bfloat16).to(dev)
    o = torch.empty_like(q)
    cu_q = torch.arange(0, total_q + 1, chunk, dtype=torch.int32, device=dev)
    seqlens = torch.tensor(lens_k, dtype=torch.int32, device=dev)
    bt = torch.as_tensor(table).to(dev)
    import ctypes
    a = attn.PagedArgs()
    a.B, a.H, a.Hkv, a.total_q, a.num_pages, a.page_size, a.max_pages, a.d = \
        seqs, H, Hkv, total_q, n_pages, PAGED_PAGE, table.shape[1], d
    a.pack_heads = int(pack)
    a.max_splits = args.splits
    ws = torch.empty(int(attn.load().attn_fwd_paged_workspace_size(ctypes.byref(a))), dtype=torch.uint8, device=dev)

    def call():
        attn.attn_fwd_paged(q, kc, vc, cu_q, seqlens, bt, max_seqlen_q=chunk, o=o, causal=True, workspace=ws,
                            pack_heads=pack, max_splits=args.splits)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0, enabled=not args.no_clocks) as clocks:
        t0.record()
        for _ in range(steps):
            call()
        t1.record()
        torch.cuda.synchronize(dev)
    st, site = attn.device_status()
    assert st == 0, "device status %d at site %d" % (st, site)
    ms = t0.elapsed_time(t1) / steps
    # query i of a chunk sits at position Sk - C + i and sees Sk - C + i + 1 keys
    pairs = sum(chunk * n - chunk * (chunk - 1) // 2 for n in lens_k)
    flop = 4 * H * d * pairs
    value = flop / (ms * 1e-3) / 1e12
    peak, _, hbm, peak_src = measured_peaks()
    kv_bytes = 2 * sum(lens_k) * Hkv * d * 2
    line = {
        "metric": ("attention fwd K/V GB/s (paged K/V decoding: each cache's keys and values read once)" if decode
                   else "attention fwd TFLOPS (4*d per visible pair and head, paged K/V chunked prefill)"),
        "value": kv_bytes / (ms * 1e-3) / 1e9 if decode else value, "unit": "GB/s" if decode else "TFLOPS",
        "n_gpus": 1, "steps": steps, "warmup": warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": "paged_decode" if decode else "paged_chunked_prefill", "sequences": seqs,
                   "cache_lengths": lens_k, "chunk": chunk, "page_size": PAGED_PAGE, "pages": n_pages, "H": H,
                   "Hkv": Hkv, "d": d, "causal": True, "pack_heads": pack, "max_splits": args.splits,
                   "modes": ["rtne"], "flop_per_call": flop,
                   "tflops": value, "kv_bytes_read": kv_bytes,
                   "step": "one attn_fwd_paged call: the offsets/table/tensor-map preprocessing kernel "
                           "and the attention kernel" + (" (and the merge of key parts)" if args.splits > 1 else ""),
                   "l2": "K/V cache %.0f MB > 126 MB L2" % (2 * kc.numel() * 2 / 2**20)},
        "roofline": ({"bound": "hbm", "achieved": kv_bytes / (ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                      "frac": kv_bytes / (ms * 1e-3) / 1e9 / hbm, "peak_source": peak_src + " HBM copy",
                      "timed": "whole call",
                      "traffic": (recorded_traffic("paged_decode")
                                  if seqs == DECODE_SEQS and pack and args.splits < 2 else None)} if decode else
                     {"bound": "tensor", "achieved": value, "peak": peak, "unit": "TFLOP/s",
                      "frac": value / peak, "peak_source": peak_src + " burst bf16 (cuBLAS)",
                      "timed": "whole call", "kv_gbs": kv_bytes / (ms * 1e-3) / 1e9, "hbm_peak_gbs": hbm}),
        "clocks": clocks.summary(),
        "gpu_launches": (3 if args.splits > 1 else 2) * steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    world, rank, local = dist_env()
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w, rank, world)
    if args.op == "bwd":
        return run_backward(args, w)
    if args.op in ("varlen", "varlen_bwd"):
        return run_varlen(args, backward=args.op == "varlen_bwd")
    if args.op == "paged":
        return run_paged(args)
    if args.op == "paged_decode":
        return run_paged(args, decode=True)

    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import bf16_attention_forward_gb300 as attn
    attn.load()

    steps = args.steps if args.steps is not None else DEFAULT_STEPS[w.name]
    warmup = max(3, args.warmup if args.warmup is not None else DEFAULT_WARMUP[w.name])
    modes = list(w.modes)
    set_bytes = w.min_bytes                                     # q, k, v, o
    nsets = max(1, -(-(2 * L2_BYTES) // set_bytes)) if set_bytes < 2 * L2_BYTES else 1
    cpu_sets = [make_qkv(w.B, w.H, w.Sq, w.Skv, w.d, w.layout, seed=w.seed + 1000 * i,
                         sigma=w.sigma, nonfinite_frac=w.nonfinite_frac, Hkv=w.kv_heads)
                for i in range(nsets)]
    sets = [tuple(t.to(dev) for t in s) for s in cpu_sets]
    outs = [torch.empty_like(s[0]) for s in sets]
    extended = w.causal or w.kv_heads != w.H
    plan = attn.plan_ex(w.B, w.H, w.Sq, w.Skv, Hkv=w.kv_heads, d=w.d, causal=w.causal,
                        num_sms=torch.cuda.get_device_properties(dev).multi_processor_count)
    split = plan["split_units"] > 0
    ws_bytes = attn.workspace_size_ex(*sets[0], layout=w.layout, causal=w.causal)
    workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    calls_per_step = len(modes)
    n_launch = steps * calls_per_step
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_launch)]
    for trio in ev:            # torch creates the CUDA event on its first record
        for e in trio:
            e.record(stream)

    def fwd(q, k, v, o, mode, events=None):
        if extended:
            attn.attn_fwd_ex(q, k, v, o, layout=w.layout, round=mode, causal=w.causal,
                             workspace=workspace, events=events)
        else:
            attn.attn_fwd(q, k, v, o, layout=w.layout, round=mode, workspace=workspace,
                          events=events)

    def call(i, mode, events=None):
        s = sets[i % nsets]
        fwd(s[0], s[1], s[2], outs[i % nsets], mode, events)

    for i in range(warmup * calls_per_step):
        call(i, modes[i % calls_per_step])
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local, enabled=not args.no_clocks) as clocks:
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        t_start.record(stream)
        for i in range(n_launch):
            call(i, modes[i % calls_per_step])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    # Per-kernel durations for the roofline, from a second pass of the same calls with events
    # recorded by the library around each kernel on the launching stream (kept out of the
    # timed region above: an event between the two kernels also serialises their launch).
    for i in range(n_launch):
        call(i, modes[i % calls_per_step], events=ev[i])
    torch.cuda.synchronize(dev)
    st, site = attn.device_status()
    assert st == 0, "device status %d at wait site %d" % (st, site)
    main_ms = [e[0].elapsed_time(e[1]) for e in ev]
    comb_ms = [e[1].elapsed_time(e[2]) for e in ev]
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    flop_call = w.flop
    value = whole_job_tflops(world, flop_call, n_launch, elapsed_ms)

    peak, peak_sust, hbm, peak_src = measured_peaks()
    # The attention kernel's time: its event-measured duration, capped at the timed per-call
    # time (events between the kernels add their own cost and serialise the combine's
    # programmatic launch, so on short calls the raw event time can exceed the call).
    call_ms = elapsed_ms / n_launch
    main_ev, comb_ev = statistics.mean(main_ms), statistics.mean(comb_ms)
    main_avg = min(main_ev, call_ms)
    share = main_avg / call_ms
    assert main_avg <= call_ms
    achieved = flop_call / (main_avg * 1e-3) / 1e12
    # the kernel that runs: one 128-row query tile per (b, h) takes the short-query kernel
    kernel = "attn_fwd_short_kernel" if w.Sq <= 128 else "attn_fwd_kernel"
    # the bound is the roofline the workload's arithmetic intensity (FLOP per algorithmic
    # byte) meets first: below the ridge (peak FLOP/s over HBM bytes/s) it is HBM
    intensity = flop_call / w.min_bytes
    ridge = peak * 1e12 / (hbm * 1e9)
    if intensity < ridge:
        achieved_gbs = w.min_bytes / (main_avg * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s",
                    "frac": achieved_gbs / hbm, "traffic": recorded_traffic(w.name, kernel),
                    "peak_source": peak_src + " HBM copy",
                    "tensor_tflops": achieved, "tensor_frac": achieved / peak}
    else:
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": recorded_traffic(w.name, kernel),
                    "peak_source": peak_src + " burst bf16 (cuBLAS)",
                    "frac_of_sustained": (achieved / peak_sust) if peak_sust else None}
    roofline.update({"kernel": kernel, "algorithmic_bytes": w.min_bytes, "flop_per_launch": flop_call,
                     "intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
                     "kernel_ms_avg": main_avg, "call_ms_avg": call_ms, "kernel_share_of_call": share,
                     "kernel_ms_events_avg": main_ev,
                     "kernel_ms_events_median": statistics.median(main_ms)})
    extra = {}
    if split:
        # workspace rows that hold real queries: 256 per split unit, Sq when that is fewer
        rows = plan["split_units"] * min(256, w.Sq)
        comb_bytes = rows * plan["splits"] * (w.d * 4 + 4) + min(rows, w.B * w.H * w.Sq) * 2 * w.d
        # the combine's own duration from its events; the part of it the call exposes
        # (it starts while the attention kernel's last CTAs run) is the rest of the call
        extra["combine"] = {"ms_events_avg": comb_ev, "exposed_ms": call_ms - main_avg,
                            "algorithmic_bytes": comb_bytes,
                            "achieved_gbs": comb_bytes / (comb_ev * 1e-3) / 1e9, "peak_gbs": hbm,
                            "frac": comb_bytes / (comb_ev * 1e-3) / 1e9 / hbm,
                            "traffic": recorded_traffic(w.name, "attn_combine_kernel")}

    # end to end through the public API with host buffers (pinned), copies timed.  Every step
    # copies its Q, K, V in from pinned host memory and every output back; the copies run on
    # two copy streams (one per direction) against two device copies of the inputs and
    # outputs, so step i+1's inputs and step i's outputs move while step i's calls run, in the
    # order a pipelined user would issue them.  Events order each copy with the calls that
    # read or overwrite its buffer.
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (t.pin_memory() for t in cpu_sets[0])
        ho = [torch.empty(hq.shape, dtype=hq.dtype).pin_memory() for _ in modes]
        dins = [tuple(torch.empty_like(t) for t in sets[0][:3]) for _ in range(2)]
        douts = [[torch.empty_like(sets[0][0]) for _ in modes] for _ in range(2)]
        h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_ready = [torch.cuda.Event() for _ in range(2)]
        in_free = [torch.cuda.Event() for _ in range(2)]
        out_ready = [[torch.cuda.Event() for _ in modes] for _ in range(2)]
        out_free = [[torch.cuda.Event() for _ in modes] for _ in range(2)]
        e2e_steps = max(3, min(steps, 50))

        def h2d(i):
            bset = i % 2
            h2d_s.wait_event(in_free[bset])
            with torch.cuda.stream(h2d_s):
                for t, h in zip(dins[bset], (hq, hk, hv)):
                    t.copy_(h, non_blocking=True)
            in_ready[bset].record(h2d_s)

        def compute(i):
            bset = i % 2
            stream.wait_event(in_ready[bset])
            for m, mode in enumerate(modes):
                stream.wait_event(out_free[bset][m])
                fwd(*dins[bset], douts[bset][m], mode)
                out_ready[bset][m].record(stream)
            in_free[bset].record(stream)

        def d2h(i):
            bset = i % 2
            for m in range(len(modes)):
                d2h_s.wait_event(out_ready[bset][m])
                with torch.cuda.stream(d2h_s):
                    ho[m].copy_(douts[bset][m], non_blocking=True)
                out_free[bset][m].record(d2h_s)

        def e2e_run(n, start=None):
            if start is not None:
                h2d_s.wait_event(start)
            h2d(0)
            for i in range(n):
                if i + 1 < n:
                    h2d(i + 1)
                compute(i)
                d2h(i)
            bset = (n - 1) % 2
            for m in range(len(modes)):
                stream.wait_event(out_free[bset][m])

        e2e_run(3)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_run(e2e_steps, start=a)
        b.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(a.elapsed_time(b), dev)
        h2d_bytes = sum(t.numel() * 2 for t in (hq, hk, hv))
        d2h_bytes = sum(t.numel() * 2 for t in ho)
        e2e = {"value": whole_job_tflops(world, flop_call, len(modes) * e2e_steps, e2e_ms),
               "unit": "TFLOPS", "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
               "steps": e2e_steps, "copies": "pipelined: two copy streams, two device buffer sets"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(w, cpu_sets[0], modes[0], seconds=12.0)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": steps, "warmup": warmup, "ms_per_step": elapsed_ms / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,%g) bf16%s)" % (
                w.sigma, ", %g non-finite K/V" % w.nonfinite_frac if w.nonfinite_frac else ""),
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.kv_heads, "Sq": w.Sq,
                       "Skv": w.Skv, "d": w.d, "causal": w.causal, "layout": w.layout,
                       "modes": modes, "flop_per_call": flop_call,
                       "step": "%d calls (one per rounding mode)" % calls_per_step,
                       "l2": ("rotating %d input sets, %.0f MB > 126 MB L2" % (nsets, nsets * set_bytes / 2**20))
                             if nsets > 1 else "inputs %.0f MB > 126 MB L2" % (set_bytes / 2**20),
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "plan": plan},
            "pct_of_peak": 100.0 * value / peak,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clocks.summary(),
            "gpu_launches": n_launch * (2 if split else 1),
            "source_sha256_16": source_hash(),
        }
        line.update(extra)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
