#!/usr/bin/env python3
"""Benchmark of the TurboQuant hot path on one GB300 (or N replicas).

A step is one decode step of a serving loop over the workload's cache:
  append   the step's new tokens per (sequence, kv-head) go into the cache:
           tokens leaving the residual window are quantized into the planes
           and the new tokens are written into the window ring (norm,
           rotation, code search, packing, window bookkeeping);
  decode   attention of every query head over the whole compressed context
           (query rotation, compressed-domain scoring, softmax, rotated V sum,
           split merge and inverse rotation).
Single-layer workloads run one tq_decode_step call (append of one token and the
decode: one launch when its plan fits one wave of the GPU, else an append
launch and a decode launch).  The 36-layer serving workload runs, for every
layer, tq_append_kv of its 64 new tokens per sequence and tq_decode_attention.
The headline value is context tokens attended per second (summed over layers).
Bulk quantize of the whole context (K and V) is measured separately and
reported in GB/s; the long-context workload also times its 4096-token
streaming chunk.

Inputs are seeded synthetic tensors shaped like the workload (see
kv_cache_quantization_random_gb300/workloads.py).  Caches larger than L2 are
read from HBM by cycling through R copies whose total is more than 4x the L2
size; a cache smaller than that (the single-head workload) is timed one step
at a time with L2 flushed before each step.  The timed region repeats the K
steps until at least a second has passed and reports the median per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     (the CPU oracle as the reference arm)
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn compressed KV tokens/s and HBM GB/s (% of peak); quantize GB/s"
# what the decode arithmetic runs in (scores: fp16 hi + lo split operands on
# the tensor cores, ~22 bits; V sum: fp16 operands; fp32 accumulation, softmax
# and merge); the quantize runs in fp32
DTYPE = "f16 hi/lo mma, f32 accumulate"
TOLERANCE = 2e-3


# ----------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# the files that define the decode kernel, its launch and its split plan
DECODE_SOURCES = ("tq_decode.cu", "tq_decode_g1.cu", "tq_decode_g2.cu", "tq_decode_g4.cu",
                  "tq_decode_g8.cu", "tq_decode_kernel.cuh", "tq_device.cuh", "tq_internal.h",
                  "tq_host.cpp")


def sources_digest() -> str:
    """sha256 of the concatenated decode sources (DECODE_SOURCES, in that order)."""
    import hashlib
    d = os.path.join(ROOT, "kv_cache_quantization_random_gb300", "csrc")
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(d, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def captured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel sources changed since that capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    digest = sources_digest()
    for ln in lines:
        parts = ln.split()
        if len(parts) != 4 or ln.startswith("#") or parts[:2] != [kernel, workload]:
            continue
        kv = dict(p.split("=", 1) for p in parts[2:])
        if kv.get("sources") == digest:
            return int(kv["dram_bytes_per_launch"])
    return None


def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over the ranks of the default process group (x
    itself without one); every rank gets the result."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def whole_job_rate(units_per_rank: float, ms_per_step: float, world: int) -> float:
    """Units per second of the whole job: every rank processes units_per_rank
    per step, and a step takes the slowest rank's time."""
    return world * units_per_rank / (ms_per_step * 1e-3)


def largest_divisor_at_most(n: int, cap: int) -> int:
    for s in range(min(n, cap), 0, -1):
        if n % s == 0:
            return s
    return 1


def median(xs):
    ys = sorted(xs)
    n = len(ys)
    return ys[n // 2] if n % 2 else 0.5 * (ys[n // 2 - 1] + ys[n // 2])


# --------------------------------------------------------------- workload
def layer_formats(w):
    """(k_bits, v_bits) of every layer: protected boundary layers at
    protect_bits ("윈도우용 터보퀀트(TurboQuant) 구현을 개선하다", finding 4)."""
    out = []
    for l in range(w.n_layers):
        prot = l < w.protect_first or l >= w.n_layers - w.protect_last
        out.append((w.protect_bits, w.protect_bits) if prot else (w.k_bits, w.v_bits))
    return out


def vector_bytes(w, kb=None, vb=None):
    """Bytes of one packed key and one packed value vector (codes + norms [+ residual sketch])."""
    d = w.head_dim
    kb = w.k_bits if kb is None else kb
    vb = w.v_bits if vb is None else vb
    kbytes = d * kb // 8 + 4 + ((w.qjl_m // 8 + 4) if w.k_qjl else 0) + \
        ((d // 8 + 4) if w.k_sign else 0)
    vbytes = d * vb // 8 + 4
    return kbytes, vbytes


def storage(w):
    """Real bytes per vector and the compression against bf16 (the write-up's
    52 B and 4.9x for a 3-bit vector: "윈도우용 터보퀀트(TurboQuant) 구현을
    개선하다", finding 3)."""
    fm = layer_formats(w)
    per_layer = [sum(vector_bytes(w, kb, vb)) for kb, vb in fm]
    kb, vb = vector_bytes(w)
    bf16 = 2 * w.head_dim * 2
    return {"k_bytes_per_vector": kb, "v_bytes_per_vector": vb,
            "bf16_bytes_per_kv_pair": bf16,
            "compression_vs_bf16": bf16 * len(per_layer) / sum(per_layer),
            "what": "packed codes + fp32 norm (+ 16 sign bytes + fp32 scale for residual-sketch "
                    "keys), averaged over layers; the window's bf16 tokens excluded"}


def decode_bytes(w, seq, kb=None, vb=None):
    """Bytes one decode launch must move: packed K and V of quantized tokens,
    bf16 window K and V, bf16 query in, fp32 output."""
    d, W = w.head_dim, w.window
    kbytes, vbytes = vector_bytes(w, kb, vb)
    total = 0
    for T in seq:
        nq = max(int(T) - W, 0)
        nw = int(T) - nq
        total += w.n_kv_heads * (nq * (kbytes + vbytes) + nw * d * 2 * 2)
    total += len(seq) * w.n_q_heads * d * (2 + 4)
    return total


def in_bytes_per_vector(w):
    return w.head_dim * (4 if w.in_dtype == "fp32" else 2)


def make_config(B, w, sparse_v=0):
    return B.Config(k_bits=w.k_bits, v_bits=w.v_bits, residual_window=w.window,
                    seed=w.codec_seed, n_layers=w.n_layers, n_protect_first=w.protect_first,
                    n_protect_last=w.protect_last, protect_bits=w.protect_bits,
                    k_mode=(B.TQ_MODE_MSE_QJL if w.k_qjl else
                            B.TQ_MODE_MSE_SIGN if w.k_sign else B.TQ_MODE_MSE),
                    qjl_m=w.qjl_m, sparse_v=sparse_v)


def graph_of(fn, n):
    """A CUDA graph of fn(0) .. fn(n-1), captured on a side stream."""
    import torch
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(n):
                fn(i)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def graph_ms(g, per_replay, min_seconds=0.2, min_reps=5):
    """Median CUDA-event time of one unit of a graph holding per_replay units,
    replayed until min_seconds have passed."""
    import torch
    g.replay()
    torch.cuda.synchronize()
    times, spent = [], 0.0
    while spent < min_seconds or len(times) < min_reps:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        times.append(ms / per_replay)
        spent += ms * 1e-3
    return median(times)


def timed_region(run_rep, K, device, local, min_seconds=1.0, flush=None):
    """The timed region: repetitions of exactly K steps, between a barrier and
    a synchronize on both sides, until min_seconds have passed (at least 3).
    run_rep() launches the K steps of one repetition; with flush (a callable
    that writes a buffer larger than L2), run_rep(i) launches step i alone and
    the flush runs before every step, outside its events.  Returns the median
    ms per step (max over ranks), the repetitions, the wall-clock seconds of
    the region and the clock record."""
    import torch
    barrier()
    torch.cuda.synchronize()
    per_step, reps = [], 0
    t_start = time.perf_counter()
    with ClockSampler(local) as clocks:
        while time.perf_counter() - t_start < min_seconds or reps < 3:
            if flush is None:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                run_rep()
                b.record()
                torch.cuda.synchronize()
                per_step.append(a.elapsed_time(b) / K)
            else:
                evs = []
                for i in range(K):
                    flush()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    run_rep(i)
                    b.record()
                    evs.append((a, b))
                torch.cuda.synchronize()
                per_step.extend(a.elapsed_time(b) for a, b in evs)
            reps += 1
    spent = time.perf_counter() - t_start
    torch.cuda.synchronize()
    barrier()
    return max_over_ranks(median(per_step), device), reps, spent, clocks.summary()


# ---------------------------------------------------------- single layer
def build_state(B, w, device, sparse_v=0):
    """Inputs, planes and window ring of a single-layer workload's context."""
    import torch
    from kv_cache_quantization_random_gb300 import workloads as WL
    T, Wn = w.context, w.window
    nq = T - Wn
    cfg = make_config(B, w, sparse_v)
    tables = B.device_tables(cfg, device)
    K, V = WL.make_kv(w, device=device)
    kp = B.Planes(cfg, 0, 0, w.batch, w.n_kv_heads, nq, device)
    vp = B.Planes(cfg, 0, 1, w.batch, w.n_kv_heads, nq, device)
    kw = vw = None
    if Wn:
        kw = torch.empty(w.batch, w.n_kv_heads, Wn, w.head_dim, dtype=torch.bfloat16, device=device)
        vw = torch.empty_like(kw)
    st = dict(cfg=cfg, tables=tables, K=K, V=V, kp=kp, vp=vp, kw=kw, vw=vw, nq=nq)
    reset_window(st, w)
    return st


def reset_window(st, w):
    """Window ring: token t in [T - W, T) in slot t mod W."""
    import torch
    T, Wn, nq = w.context, w.window, st["nq"]
    if Wn:
        idx = torch.arange(nq, T, device=st["K"].device)
        st["kw"][:, :, idx % Wn] = st["K"][:, :, nq:T].to(torch.bfloat16)
        st["vw"][:, :, idx % Wn] = st["V"][:, :, nq:T].to(torch.bfloat16)


def window_before_step(st, w, seq):
    """Window ring as it stands before a step appends token T-1: the slot of
    token T-1 still holds token T-1-W, which the step's append quantizes."""
    import torch
    Wn = w.window
    if not Wn:
        return
    for b, T in enumerate(seq):
        t = int(T) - 1 - Wn
        if t >= 0:
            st["kw"][b, :, t % Wn] = st["K"][b, :, t].to(torch.bfloat16)
            st["vw"][b, :, t % Wn] = st["V"][b, :, t].to(torch.bfloat16)


def run_single(args, w, rank, world, local):
    import numpy as np
    import torch

    from kv_cache_quantization_random_gb300 import binding as B
    from kv_cache_quantization_random_gb300 import workloads as WL

    B.load(build_if_missing=True)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])

    st = build_state(B, w, device, sparse_v=args.sparse_v)
    cfg, tables, kp, vp = st["cfg"], st["tables"], st["kp"], st["vp"]
    K, V, nq, Wn, T = st["K"], st["V"], st["nq"], w.window, w.context

    # ---- bulk quantize of the whole context (K and V), from a CUDA graph
    def quantize_all():
        B.tq_quantize_kv(cfg, tables, 0, 0, K[:, :, :nq], kp)
        B.tq_quantize_kv(cfg, tables, 0, 1, V[:, :, :nq], vp)

    for _ in range(3):
        quantize_all()
    torch.cuda.synchronize()
    qiters = 10
    q_ms = graph_ms(graph_of(lambda i: quantize_all(), qiters), qiters)
    # keys in MSE+QJL mode: the QJL kernel alone, and the rate of its
    # projection, 2 (hi, lo) x 2 x keys x m x d flops on the tensor cores
    qjl_proj = None
    if w.k_qjl:
        k_ms = graph_ms(graph_of(lambda i: B.tq_quantize_kv(cfg, tables, 0, 0, K[:, :, :nq], kp),
                                 qiters), qiters)
        n_keys = w.batch * w.n_kv_heads * nq
        flops = 2 * 2 * n_keys * w.qjl_m * w.head_dim
        tflops = flops / (k_ms * 1e-3) / 1e12
        bf16_peak = float(peaks["bf16_tflops"])
        qjl_proj = {"kernel": "tq::quantize_qjl_kernel", "ms": k_ms, "gflop": flops / 1e9,
                    "tflops": tflops, "bf16_peak_tflops": bf16_peak,
                    "frac_of_bf16_peak": tflops / bf16_peak, "peak_source": f"{peak_kind} bf16_tflops",
                    "note": "projection flops over the whole kernel's time (codes, norms and residuals "
                            "included); ncu's sm__pipe_tensor_cycles_active is in profiles/"}
    n_vec = w.batch * w.n_kv_heads * nq
    kbts, vbts = vector_bytes(w)
    q_bytes = n_vec * (2 * in_bytes_per_vector(w) + kbts + vbts)
    q_gbs = q_bytes / (q_ms * 1e-3) / 1e9
    if B.tq_get_device_error() != B.TQ_OK:
        raise RuntimeError("device error after quantize")

    # ---- L2: replicas of the compressed cache (more than 4x L2 in total), or
    # an L2 flush before every step when the cache is much smaller than L2
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    seq = WL.seq_lens(w)
    dec_bytes = decode_bytes(w, seq)
    cache_bytes = sum(t.numel() for t in (kp.codes, kp.norms, vp.codes, vp.norms)) + \
        (2 * st["kw"].numel() * 2 if Wn else 0)
    # replicas cover 4x L2 with at most 64 copies; a smaller cache (the
    # single-head workload) is timed one step at a time with L2 flushed
    R = max(2, math.ceil(4 * l2 / max(cache_bytes, 1)) + 1)
    flush_mode = R > 64
    R = 1 if flush_mode else R
    reps = []
    for r in range(R):
        if r == 0:
            reps.append((kp, vp, st["kw"], st["vw"]))
            continue
        kr = B.Planes(cfg, 0, 0, w.batch, w.n_kv_heads, nq, device)
        vr = B.Planes(cfg, 0, 1, w.batch, w.n_kv_heads, nq, device)
        for src, dst in ((kp, kr), (vp, vr)):
            dst.codes.copy_(src.codes)
            dst.norms.copy_(src.norms)
            if src.qjl_signs is not None:
                dst.qjl_signs.copy_(src.qjl_signs)
                dst.qjl_rnorm.copy_(src.qjl_rnorm)
        kwr = st["kw"].clone() if Wn else None
        vwr = st["vw"].clone() if Wn else None
        reps.append((kr, vr, kwr, vwr))
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=device) if flush_mode else None
    flush = (lambda: flush_buf.fill_(1)) if flush_mode else None

    # ---- step inputs: one new token per (sequence, kv-head), one query per head
    q = WL.make_q(w, device=device)
    knew = K[:, :, T - 1:T].contiguous()
    vnew = V[:, :, T - 1:T].contiguous()
    seq_before = torch.tensor(seq - 1, dtype=torch.int32, device=device)
    seq_t = torch.tensor(seq, dtype=torch.int32, device=device)
    Tmax = int(seq.max())
    out = torch.empty(w.batch, w.n_q_heads, w.head_dim, device=device)
    ws = B.new_workspace(cfg, w.batch, w.n_q_heads, w.n_kv_heads, Tmax, device)

    def append(r):
        kr, vr, kwr, vwr = reps[r]
        B.tq_append_kv(cfg, tables, 0, knew, vnew, seq_before, kwr, vwr, kr, vr)

    def decode(r):
        kr, vr, kwr, vwr = reps[r]
        B.tq_decode_attention(cfg, tables, 0, q, w.softmax_scale, kr, vr, seq_t, Tmax, out, ws,
                              k_win=kwr, v_win=vwr)

    def step(i):
        kr, vr, kwr, vwr = reps[i % R]
        B.tq_decode_step(cfg, tables, 0, q, w.softmax_scale, knew, vnew, seq_before, Tmax, kr, vr,
                         out, ws, k_win=kwr, v_win=vwr)

    # tq_decode_step: one launch (the decode kernel appends the token) when its
    # plan fits one wave, else an append launch and a decode launch
    launches_per_step = B.tq_decode_step_launches(cfg, 0, w.batch, w.n_q_heads, w.n_kv_heads,
                                                  int(seq.max()))

    # ---- warmup (direct launches), then graphs of S steps
    warm = max(args.warmup, 3)
    for i in range(warm):
        step(i)
    torch.cuda.synchronize()
    if B.tq_get_device_error() != B.TQ_OK:
        raise RuntimeError("device error during warmup")
    K_steps = args.steps
    S = 1 if flush_mode else largest_divisor_at_most(K_steps, 128)
    g_step = graph_of(step, S)
    g_dec = graph_of(lambda i: decode(i % R), S)
    g_app = graph_of(lambda i: append(i % R), S)

    # ---- timed region: repetitions of exactly K steps
    if flush_mode:
        ms_per_step, n_reps, spent, clocks = timed_region(
            lambda i: g_step.replay(), K_steps, device, local, args.min_seconds, flush=flush)
    else:
        def rep():
            for _ in range(K_steps // S):
                g_step.replay()
        ms_per_step, n_reps, spent, clocks = timed_region(rep, K_steps, device, local,
                                                          args.min_seconds)
    tokens_per_step = int(seq.sum())
    value = whole_job_rate(tokens_per_step, ms_per_step, world)

    # ---- per-kernel durations (decode-only and append-only graphs)
    if flush_mode:
        def per_launch_ms(g):
            ts = []
            for _ in range(max(50, min(K_steps, 500))):
                flush()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                b.record()
                ts.append((a, b))
            torch.cuda.synchronize()
            return median([a.elapsed_time(b) for a, b in ts])
        dec_ms, app_ms = per_launch_ms(g_dec), per_launch_ms(g_app)
    else:
        dec_ms, app_ms = graph_ms(g_dec, S), graph_ms(g_app, S)
    if B.tq_get_device_error() != B.TQ_OK:
        raise RuntimeError("device error during timed steps")
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9

    # ---- sparse V: the exact decode of the same cache for comparison, and an
    # upper bound of the share of 32-token chunks whose V sum the kernel may
    # skip (all weights of the chunk below 2^-sparse_v of the head's final
    # maximum; the kernel compares with the running maximum, which is lower,
    # so it skips at most this share), from the oracle's scores of kv-head 0
    sparse = None
    if args.sparse_v > 0:
        cfg_exact = make_config(B, w, 0)

        def decode_exact(r):
            kr, vr, kwr, vwr = reps[r]
            B.tq_decode_attention(cfg_exact, tables, 0, q, w.softmax_scale, kr, vr, seq_t, Tmax,
                                  out, ws, k_win=kwr, v_win=vwr)

        for i in range(3):
            decode_exact(i % R)
        ex_ms = graph_ms(graph_of(lambda i: decode_exact(i % R), S), S)
        sparse = {"sparse_v": args.sparse_v, "decode_ms": dec_ms, "exact_decode_ms": ex_ms,
                  "skippable_chunks_upper_bound": sparse_skip_bound(w, st, q, seq, args.sparse_v)}

    # ---- optional: several query tokens per sequence (speculative verify)
    multi = None
    if args.n_queries > 1:
        nQ = args.n_queries
        gq = torch.Generator(device=device)
        gq.manual_seed(w.data_seed * 7 + nQ)
        qm = torch.randn((w.batch, w.n_q_heads, nQ, w.head_dim), generator=gq, device=device,
                         dtype=torch.float32).to(torch.bfloat16)
        outm = torch.empty(w.batch, w.n_q_heads, nQ, w.head_dim, device=device)
        wsm = B.new_workspace(cfg, w.batch, w.n_q_heads * nQ, w.n_kv_heads, Tmax, device)

        def decode_multi(r):
            kr, vr, kwr, vwr = reps[r]
            B.tq_decode_attention_multi(cfg, tables, 0, qm, w.softmax_scale, kr, vr, seq_t, Tmax,
                                        outm, wsm, k_win=kwr, v_win=vwr)

        for i in range(3):
            decode_multi(i % R)
        mq_ms = graph_ms(graph_of(lambda i: decode_multi(i % R), S), S)
        mq_bytes = dec_bytes + len(seq) * w.n_q_heads * (nQ - 1) * w.head_dim * (2 + 4)
        multi = {"n_queries": nQ, "ms": mq_ms, "gbs": mq_bytes / (mq_ms * 1e-3) / 1e9,
                 "query_token_attends_per_s": nQ * tokens_per_step / (mq_ms * 1e-3),
                 "vs_single_query_ms": dec_ms}

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(B, w, cfg, tables, reps, R, q, knew, vnew, seq_before, Tmax, out, ws, S,
                  K_steps, device, tokens_per_step, world, flush)

    # ---- the long-context workload's streaming chunk: tq_append_kv of
    # new_tokens tokens per sequence at the end of the context
    chunk = None
    if w.new_tokens > 8:
        n_new = w.new_tokens
        nv = w.batch * w.n_kv_heads * n_new
        c_bytes = nv * (2 * in_bytes_per_vector(w) + kbts + vbts) + \
            w.batch * w.n_kv_heads * min(n_new, Wn) * w.head_dim * 2 * 2
        # chunk r appends tokens [T - (r+1) n_new, T - r n_new) at that position:
        # Rc distinct input slices and plane rows, more than 4x L2 in all, so
        # that consecutive appends find neither their inputs nor their
        # destination rows in L2
        Rc = max(1, min(int(math.ceil(4 * l2 / c_bytes)) + 1, (int(seq.min()) - Wn) // n_new - 1))
        chunks = []
        for r in range(Rc):
            t1 = T - r * n_new
            chunks.append((K[:, :, t1 - n_new:t1], V[:, :, t1 - n_new:t1],
                           torch.tensor(seq - (r + 1) * n_new, dtype=torch.int32, device=device)))

        def chunk_append(i):
            kch, vch, sb = chunks[i % Rc]
            B.tq_append_kv(cfg, tables, 0, kch, vch, sb, st["kw"], st["vw"], kp, vp)

        for i in range(3):
            chunk_append(i)
        c_ms = graph_ms(graph_of(chunk_append, Rc), Rc)
        chunk = {"new_tokens": n_new, "ms": c_ms, "bytes": c_bytes,
                 "gbs": c_bytes / (c_ms * 1e-3) / 1e9,
                 "frac_of_peak": c_bytes / (c_ms * 1e-3) / 1e9 / hbm_peak,
                 "l2": f"{Rc} chunks at distinct positions cycled ({Rc * c_bytes / 1e6:.0f} MB)",
                 "what": "tq_append_kv of one streaming chunk per (sequence, kv-head): quantize "
                         "of the tokens leaving the window (bf16 in, packed out) and the ring "
                         "update (bf16 out)"}
        if B.tq_get_device_error() != B.TQ_OK:
            raise RuntimeError("device error during the chunk appends")

    # ---- sampled parity at full size, in the launch configuration timed above
    parity = None
    if not args.no_parity and rank == 0:
        # the timed steps rewrote one row and one window slot of every replica
        # (and the chunk appends rewrote replica 0): restore replica 0 from the
        # inputs, as it stands before the step's append, and check one step
        quantize_all()
        reset_window(st, w)
        window_before_step(st, w, seq)
        parity = sampled_parity(B, w, st, q, out, reps[0], seq, step)

    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": K_steps, "warmup": warm, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
        "config": {
            "workload": w.name, "batch": w.batch, "q_heads": w.n_q_heads,
            "kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "context": int(seq.max()),
            "k_bits": w.k_bits, "v_bits": w.v_bits, "k_qjl": w.k_qjl, "k_sign": w.k_sign,
            "window": Wn, "kv_dist": w.dist, "new_tokens_per_step": 1,
            "parallelism": f"replicas x{world}", "sparse_v": args.sparse_v,
            "l2": (f"flushed before every step ({2 * l2 / 1e6:.0f} MB write outside the step's "
                   f"events; the cache is {cache_bytes / 1e6:.2f} MB)") if flush_mode else
                  (f"{R} cache replicas cycled ({R * cache_bytes / 1e6:.0f} MB > 4 x L2 "
                   f"{l2 / 1e6:.0f} MB)"),
            "graph_steps": S,
        },
        "timing": {"repetitions": n_reps, "seconds": spent, "statistic": "median of the "
                   "repetitions' ms per step" if not flush_mode else "median over single steps"},
        "roofline": {
            "kernel": "tq::decode_kernel", "bound": "hbm", "achieved": dec_gbs,
            "peak": hbm_peak, "unit": "GB/s", "frac": dec_gbs / hbm_peak,
            "peak_source": f"{peak_kind} hbm_gbs",
            "traffic": (args.decode_traffic if args.decode_traffic is not None
                        else captured_traffic("decode_kernel", w.name)),
            "bytes_per_launch": dec_bytes, "launch_ms": dec_ms,
            "note": "launch_ms = a CUDA graph of decode launches back to back, over cache replicas, "
                    "divided by the launches; a one-wave grid lets the next launch's CTAs build "
                    "their tables while its last CTAs merge",
        },
        "decode": {"ms": dec_ms, "gbs": dec_gbs, "frac_of_peak": dec_gbs / hbm_peak,
                   "tokens_per_s": tokens_per_step / (dec_ms * 1e-3), "bytes": dec_bytes},
        "append": {"ms": app_ms, "launches": 1,
                   "what": "tq_append_kv of the step's token alone (append-only graph)"},
        "quantize": {"ms": q_ms, "gbs": q_gbs, "frac_of_peak": q_gbs / hbm_peak,
                     "vectors": 2 * n_vec, "bytes": q_bytes, "what": "bulk quantize of the "
                     "context's K and V (input dtype in, packed planes out)"},
        "storage": storage(w),
        "e2e": e2e,
        "gpu_launches": K_steps * launches_per_step * n_reps,
        "clocks": clocks,
        "parity": parity,
    }
    if chunk is not None:
        res["chunk_quantize"] = chunk
    if sparse is not None:
        res["sparse_v"] = sparse
    if multi is not None:
        res["multi_query"] = multi
    if qjl_proj is not None:
        res["qjl_projection"] = qjl_proj
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    return res


def run_e2e(B, w, cfg, tables, reps, R, q, knew, vnew, seq_before, Tmax, out, ws, S, K_steps,
            device, tokens_per_step, world, flush=None):
    """End to end through the public API with host buffers: every step's
    inputs (query, new K and V token) start in pinned host memory and its
    output ends there.  Three ways, all CUDA graphs of S steps:
      host-mapped (the headline): tq_decode_step is given the pinned host
          buffers themselves; the kernel reads the inputs across the host link
          and writes the output into host memory, so the bytes cross every
          step with no copy engine in the chain of launches;
      copy engine, pipelined: step i's inputs go to the device by
          cudaMemcpyAsync on a copy-in stream while step i-1's kernels run,
          and its output back on a copy-out stream while step i+1's run, with
          double-buffered inputs and outputs and graph edges ordering every
          reuse of a buffer;
      copy engine, serial: each step's copy-in, kernels and copy-out one after
          another.
    With flush (a cache smaller than L2), each graph replay is one step,
    timed alone after an L2 flush."""
    import torch

    def timed(g):
        if flush is None:
            return graph_ms(g, S, min_seconds=0.5)
        ts = []
        for _ in range(max(50, min(K_steps, 500))):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            ts.append((a, b))
        torch.cuda.synchronize()
        return median([a.elapsed_time(b) for a, b in ts]) / S
    parts = [q, knew, vnew]
    nbytes = [t.numel() * t.element_size() for t in parts]
    offs = [0]
    for n in nbytes[:-1]:
        offs.append(offs[-1] + (n + 255) // 256 * 256)
    total_in = offs[-1] + nbytes[-1]
    hbuf = torch.empty(total_in, dtype=torch.uint8).pin_memory()
    for t, o, n in zip(parts, offs, nbytes):
        hbuf[o:o + n].copy_(t.contiguous().view(torch.uint8).view(-1).cpu())
    dbufs = [torch.empty(total_in, dtype=torch.uint8, device=device) for _ in range(2)]
    dviews = [tuple(d[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(parts, offs, nbytes))
              for d in dbufs]
    outs = [out, torch.empty_like(out)]
    ouths = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]

    def e2e_step(i):
        dbufs[0].copy_(hbuf, non_blocking=True)
        qd, kd, vd = dviews[0]
        kr, vr, kwr, vwr = reps[i % R]
        B.tq_decode_step(cfg, tables, 0, qd, w.softmax_scale, kd, vd, seq_before, Tmax, kr, vr,
                         outs[0], ws, k_win=kwr, v_win=vwr)
        ouths[0].copy_(outs[0], non_blocking=True)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    serial_ms = timed(graph_of(e2e_step, S))

    def capture_pipelined():
        g = torch.cuda.CUDAGraph()
        sc = torch.cuda.Stream()
        cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
        sc.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(sc):
            with torch.cuda.graph(g, stream=sc):
                cin.wait_stream(sc)
                cout.wait_stream(sc)
                ev_in, ev_done, ev_out = [], [], []
                for i in range(S):
                    j = i % 2
                    with torch.cuda.stream(cin):
                        if i >= 2:
                            cin.wait_event(ev_done[i - 2])      # step i-2 has read dbufs[j]
                        dbufs[j].copy_(hbuf, non_blocking=True)
                        ev_in.append(torch.cuda.Event())
                        ev_in[i].record(cin)
                    sc.wait_event(ev_in[i])
                    if i >= 2:
                        sc.wait_event(ev_out[i - 2])           # outs[j] has been read back
                    qd_, kd_, vd_ = dviews[j]
                    kr, vr, kwr, vwr = reps[i % R]
                    B.tq_decode_step(cfg, tables, 0, qd_, w.softmax_scale, kd_, vd_, seq_before, Tmax,
                                     kr, vr, outs[j], ws, k_win=kwr, v_win=vwr)
                    ev_done.append(torch.cuda.Event())
                    ev_done[i].record(sc)
                    with torch.cuda.stream(cout):
                        cout.wait_event(ev_done[i])
                        ouths[j].copy_(outs[j], non_blocking=True)
                        ev_out.append(torch.cuda.Event())
                        ev_out[i].record(cout)
                sc.wait_stream(cin)
                sc.wait_stream(cout)
        torch.cuda.current_stream().wait_stream(sc)
        torch.cuda.synchronize()
        return g

    pipe_ms = timed(capture_pipelined())
    if B.tq_get_device_error() != B.TQ_OK:
        raise RuntimeError("device error during the end-to-end steps")
    # the host copies hold what the last steps computed
    n_out = 2 if S >= 2 else 1
    for j in range(n_out):
        if not torch.equal(ouths[j], outs[j].cpu()):
            raise RuntimeError("end-to-end steps: host output differs from the device's")

    # host-mapped: the pinned host views of the same inputs, the output into
    # pinned host memory (double-buffered, as above)
    hviews = tuple(hbuf[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(parts, offs, nbytes))
    houts = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]

    def mapped_step(i):
        kr, vr, kwr, vwr = reps[i % R]
        B.tq_decode_step(cfg, tables, 0, hviews[0], w.softmax_scale, hviews[1], hviews[2],
                         seq_before, Tmax, kr, vr, houts[i % 2], ws, k_win=kwr, v_win=vwr)

    for i in range(3):
        mapped_step(i)
    torch.cuda.synchronize()
    mapped_ms = timed(graph_of(mapped_step, S))
    if B.tq_get_device_error() != B.TQ_OK:
        raise RuntimeError("device error during the host-mapped steps")
    # the host outputs equal the device path's for the same inputs and cache
    e2e_step(0)
    mapped_step(0)
    torch.cuda.synchronize()
    if not torch.equal(houts[0], ouths[0]):
        raise RuntimeError("host-mapped step: output differs from the device path's")
    mapped_ms = max_over_ranks(mapped_ms, device)
    pipe_ms = max_over_ranks(pipe_ms, device)
    serial_ms = max_over_ranks(serial_ms, device)
    return {"value": whole_job_rate(tokens_per_step, mapped_ms, world), "unit": "tokens/s",
            "ms_per_step": mapped_ms, "h2d_bytes_per_step": total_in,
            "d2h_bytes_per_step": ouths[0].numel() * ouths[0].element_size(),
            "what": "inputs read from and the output written to pinned host memory by the step's "
                    "kernels (host-mapped pointers through tq_decode_step)",
            "copy_engine_pipelined": {"value": whole_job_rate(tokens_per_step, pipe_ms, world),
                                      "ms_per_step": pipe_ms,
                                      "what": "cudaMemcpyAsync in and out on their own streams, "
                                              "overlapping the neighbouring steps' kernels"},
            "copy_engine_serial": {"value": whole_job_rate(tokens_per_step, serial_ms, world),
                                   "ms_per_step": serial_ms,
                                   "what": "each step's copy-in, kernels and copy-out one after "
                                           "another"}}


def append_launches(w, kb, vb, n_new):
    """Kernel launches of one tq_append_kv (the library's dispatch): one for at
    most 8 new tokens per sequence (the append kernel); above that one bulk
    launch for keys and values of one bit width (bf16 rows, keys not in QJL
    mode), else one per kind."""
    if n_new <= 8:
        return 1
    return 1 if kb == vb and not w.k_qjl else 2


# ------------------------------------------------------------ 36 layers
def run_layered(args, w, rank, world, local):
    """The serving workload: every step appends new_tokens tokens per
    sequence to every layer (tq_append_kv: quantize into the planes, W = 0)
    and decodes every layer (tq_decode_attention).  The cache of all layers
    is far larger than L2, so it streams from HBM without replicas."""
    import numpy as np
    import torch

    from kv_cache_quantization_random_gb300 import binding as B
    from kv_cache_quantization_random_gb300 import workloads as WL

    B.load(build_if_missing=True)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    cfg = make_config(B, w, args.sparse_v)
    tables = B.device_tables(cfg, device)
    seq = WL.seq_lens(w)
    Tmax = int(seq.max())
    n_new, L, H = w.new_tokens, w.n_layers, w.n_kv_heads
    fm = layer_formats(w)
    seq_t = torch.tensor(seq, dtype=torch.int32, device=device)
    seq_before = torch.tensor(seq - n_new, dtype=torch.int32, device=device)
    # per layer: planes holding every sequence's context, and the step's new
    # tokens (the last n_new tokens of each sequence, gathered)
    pos = torch.as_tensor(seq[:, None] - n_new + np.arange(n_new)[None, :], device=device,
                          dtype=torch.long)                                   # [B, n_new]
    layers = []
    q_ms_total, q_bytes_total = 0.0, 0
    for l in range(L):
        K, V = WL.make_kv(w, layer=l, device=device)
        kp = B.Planes(cfg, l, 0, w.batch, H, Tmax, device)
        vp = B.Planes(cfg, l, 1, w.batch, H, Tmax, device)
        B.tq_quantize_kv(cfg, tables, l, 0, K[:, :, :Tmax], kp)
        B.tq_quantize_kv(cfg, tables, l, 1, V[:, :, :Tmax], vp)
        idx = pos[:, None, :, None].expand(w.batch, H, n_new, w.head_dim)
        knew = torch.gather(K, 2, idx).contiguous()
        vnew = torch.gather(V, 2, idx).contiguous()
        layers.append(dict(kp=kp, vp=vp, knew=knew, vnew=vnew))
        del K, V
    torch.cuda.synchronize()
    if B.tq_get_device_error() != B.TQ_OK:
        raise RuntimeError("device error while filling the cache")
    q = WL.make_q(w, device=device)
    out = torch.empty(w.batch, w.n_q_heads, w.head_dim, device=device)
    ws = B.new_workspace(cfg, w.batch, w.n_q_heads, H, Tmax, device)

    def append(l):
        c = layers[l]
        B.tq_append_kv(cfg, tables, l, c["knew"], c["vnew"], seq_before, None, None, c["kp"],
                       c["vp"])

    def decode(l):
        c = layers[l]
        B.tq_decode_attention(cfg, tables, l, q, w.softmax_scale, c["kp"], c["vp"], seq_t, Tmax,
                              out, ws)

    def step(_):
        for l in range(L):
            append(l)
            decode(l)

    warm = max(args.warmup, 3)
    for i in range(warm):
        step(i)
    torch.cuda.synchronize()
    if B.tq_get_device_error() != B.TQ_OK:
        raise RuntimeError("device error during warmup")
    K_steps = args.steps
    g_step = graph_of(step, 1)

    def rep():
        for _ in range(K_steps):
            g_step.replay()

    ms_per_step, n_reps, spent, clocks = timed_region(rep, K_steps, device, local, args.min_seconds)
    tokens_per_step = L * int(seq.sum())
    value = whole_job_rate(tokens_per_step, ms_per_step, world)
    # per-kernel: all layers' decodes alone, all layers' appends alone
    dec_ms = graph_ms(graph_of(decode, L), 1)
    app_ms = graph_ms(graph_of(append, L), 1)
    dec_bytes = sum(decode_bytes(w, seq, kb, vb) for kb, vb in fm)
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    nv = w.batch * H * n_new
    app_bytes = sum(nv * (2 * in_bytes_per_vector(w) + sum(vector_bytes(w, kb, vb)))
                    for kb, vb in fm)
    app_gbs = app_bytes / (app_ms * 1e-3) / 1e9
    # per format: one protected and one K4/V2 layer decoded alone
    per_fmt = {}
    for l in sorted({0, w.protect_first}):
        kb, vb = fm[l]
        ms = graph_ms(graph_of(lambda i: decode(l), 16), 16)
        by = decode_bytes(w, seq, kb, vb)
        per_fmt[f"layer{l}_k{kb}v{vb}"] = {"ms": ms, "gbs": by / (ms * 1e-3) / 1e9,
                                           "frac_of_peak": by / (ms * 1e-3) / 1e9 / hbm_peak}
    if B.tq_get_device_error() != B.TQ_OK:
        raise RuntimeError("device error during timed steps")

    # e2e: the step's inputs (all layers' new K/V tokens and the query) come
    # from pinned host memory and the last layer's output goes back
    parts = [q] + [c[k] for c in layers for k in ("knew", "vnew")]
    nbytes = [t.numel() * t.element_size() for t in parts]
    total_in = sum(nbytes)
    hbuf = torch.empty(total_in, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(total_in, dtype=torch.uint8, device=device)
    o = 0
    for t, n in zip(parts, nbytes):
        hbuf[o:o + n].copy_(t.contiguous().view(torch.uint8).view(-1).cpu())
        o += n
    outh = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    # the query and every layer's new tokens become views of the device buffer
    # that one host-to-device copy fills each step
    dbuf.copy_(hbuf)
    views, oo = [], 0
    for t, n in zip(parts, nbytes):
        views.append(dbuf[oo:oo + n].view(t.dtype).view(t.shape))
        oo += n
    kept = [q] + [(c["knew"], c["vnew"]) for c in layers]   # the graphs above hold their pointers
    q = views[0]
    for l, c in enumerate(layers):
        c["knew"], c["vnew"] = views[1 + 2 * l], views[2 + 2 * l]

    def e2e_step(_):
        dbuf.copy_(hbuf, non_blocking=True)
        step(0)
        outh.copy_(out, non_blocking=True)

    e2e_step(0)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(graph_ms(graph_of(e2e_step, 1), 1, min_seconds=0.5), device)
    del kept

    parity = None
    if not args.no_parity and rank == 0:
        parity = layered_parity(B, w, cfg, tables, layers, q, seq, seq_t, Tmax, ws, device)

    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": K_steps, "warmup": warm, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
        "config": {
            "workload": w.name, "batch": w.batch, "q_heads": w.n_q_heads, "kv_heads": H,
            "head_dim": w.head_dim, "layers": L, "context": f"ragged {w.ragged[0]}-{w.ragged[1]}, "
            f"sum {int(seq.sum())}", "k_bits": w.k_bits, "v_bits": w.v_bits,
            "protected": f"layers 0-{w.protect_first - 1} and {L - w.protect_last}-{L - 1} at "
                         f"{w.protect_bits} bits", "window": w.window, "kv_dist": w.dist,
            "new_tokens_per_step": n_new, "parallelism": f"replicas x{world}",
            "l2": f"{L} layers' planes ({sum(c['kp'].codes.numel() + c['vp'].codes.numel() for c in layers) / 1e9:.1f} GB) "
                  "stream from HBM every step",
        },
        "timing": {"repetitions": n_reps, "seconds": spent,
                   "statistic": "median of the repetitions' ms per step"},
        "roofline": {
            "kernel": "tq::decode_kernel", "bound": "hbm", "achieved": dec_gbs, "peak": hbm_peak,
            "unit": "GB/s", "frac": dec_gbs / hbm_peak, "peak_source": f"{peak_kind} hbm_gbs",
            "traffic": (args.decode_traffic if args.decode_traffic is not None
                        else captured_traffic("decode_kernel", w.name)),
            "bytes_per_launch": dec_bytes / L, "launch_ms": dec_ms / L,
            "note": "all layers' decode launches back to back; per launch = their mean",
        },
        "decode": {"ms_all_layers": dec_ms, "gbs": dec_gbs, "frac_of_peak": dec_gbs / hbm_peak,
                   "bytes_all_layers": dec_bytes, "per_format": per_fmt},
        "append": {"ms_all_layers": app_ms, "gbs": app_gbs, "frac_of_peak": app_gbs / hbm_peak,
                   "bytes_all_layers": app_bytes,
                   "what": f"tq_append_kv of {n_new} new tokens per sequence into every layer"},
        "storage": storage(w),
        "e2e": {"value": whole_job_rate(tokens_per_step, e2e_ms, world), "unit": "tokens/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": total_in,
                "d2h_bytes_per_step": outh.numel() * outh.element_size(), "pipelined": False},
        "gpu_launches": K_steps * n_reps * sum(1 + append_launches(w, kb, vb, n_new) for kb, vb in fm),
        "clocks": clocks,
        "parity": parity,
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    return res


def layered_parity(B, w, cfg, tables, layers, q, seq, seq_t, Tmax, ws, device):
    """One step's decode of a protected and a K4/V2 layer against the oracle,
    on sequence 0 and two kv-heads, after the step's append."""
    import numpy as np
    import torch
    import oracle as O
    from kv_cache_quantization_random_gb300 import workloads as WL
    res = {}
    worst = 0.0
    heads = [0, w.n_kv_heads - 1]
    T = int(seq[0])
    for l in sorted({0, w.protect_first}):
        kb, vb, _ = B.tq_layer_spec_get(cfg, l)
        c = layers[l]
        # the step: append the new tokens, then decode
        B.tq_append_kv(cfg, tables, l, c["knew"], c["vnew"],
                       seq_t - w.new_tokens, None, None, c["kp"], c["vp"])
        out = torch.empty(w.batch, w.n_q_heads, w.head_dim, device=device)
        B.tq_decode_attention(cfg, tables, l, q, w.softmax_scale, c["kp"], c["vp"], seq_t, Tmax,
                              out, ws)
        torch.cuda.synchronize()
        K, V = WL.make_kv(w, layer=l, device=device)
        f64 = lambda t: t.float().cpu().numpy().astype(np.float64)
        Kh, Vh = f64(K[:1, heads, :T]), f64(V[:1, heads, :T])
        del K, V
        g = w.group
        qh = [h * g + j for h in heads for j in range(g)]
        qs = f64(q[:1, qh])
        ck, bk = O.codebook_fp32(kb, w.head_dim)
        cv, bv = O.codebook_fp32(vb, w.head_dim)
        sk = O.rotation_signs(w.codec_seed, l, 0, w.head_dim)
        sv = O.rotation_signs(w.codec_seed, l, 1, w.head_dim)
        qk = O.quantize_vectors(Kh, ck, bk, sk)
        qv = O.quantize_vectors(Vh, cv, bv, sv)
        ref = O.decode_attention(qs, qk["codes"], qk["norms"], qv["codes"], qv["norms"], ck, cv,
                                 sk, sv, [T], w.softmax_scale)
        mine = f64(out[:1, qh])
        rel = float((np.linalg.norm(mine - ref, axis=-1) / np.linalg.norm(ref, axis=-1)).max())
        gk = O.unpack_codes(c["kp"].codes_view()[:1, heads, :T].cpu().numpy(), kb, w.head_dim)
        band = O.near_boundary(qk["y"], bk, w.head_dim)
        res[f"layer{l}_k{kb}v{vb}"] = {
            "max_rel_l2": rel,
            "key_code_mismatches_outside_band": int(((gk != qk["codes"]) & ~band).sum())}
        worst = max(worst, rel)
    return {"max_rel_l2": worst, "tolerance": TOLERANCE, "pass": worst < TOLERANCE,
            "sequence_checked": 0, "kv_heads_checked": heads, "layers": res}


# ------------------------------------------------------------- parity (single layer)
def _oracle_inputs(w, st, q, heads):
    """fp64 copies of the inputs of kv-heads `heads` (sequence 0)."""
    import numpy as np
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)
    K = f64(st["K"][:1, heads])
    V = f64(st["V"][:1, heads])
    g = w.group
    qh = [h * g + j for h in heads for j in range(g)]
    return K, V, f64(q[:1, qh])


def _oracle_cache(w, K, V, T, layer=0, kb=None, vb=None):
    """The oracle's own compressed cache of K, V [B', H', >=T, d], plus window ring."""
    import numpy as np
    import oracle as O
    kb = w.k_bits if kb is None else kb
    vb = w.v_bits if vb is None else vb
    Wn = w.window
    nq = T - Wn
    ck, bk = O.codebook_fp32(kb, w.head_dim)
    cv, bv = O.codebook_fp32(vb, w.head_dim)
    sk = O.rotation_signs(w.codec_seed, layer, 0, w.head_dim)
    sv = O.rotation_signs(w.codec_seed, layer, 1, w.head_dim)
    qk = O.quantize_vectors(K[:, :, :nq], ck, bk, sk)
    qv = O.quantize_vectors(V[:, :, :nq], cv, bv, sv)
    qjl = None
    if w.k_qjl:
        S = O.qjl_matrix(w.codec_seed, layer, w.qjl_m, w.head_dim)
        r = O.qjl_residual(qk["y"], qk["codes"], qk["norm64"], ck)
        bits, gamma, _ = O.qjl_sketch(r, S)
        qjl = dict(bits=bits, gamma=gamma, S=S)
    dsign = None
    if w.k_sign:
        r = O.qjl_residual(qk["y"], qk["codes"], qk["norm64"], ck)
        bits, scale = O.direct_sign_sketch(r)
        dsign = dict(bits=bits, scale=scale)
    kw = vw = None
    if Wn:
        kw = np.zeros((K.shape[0], K.shape[1], Wn, w.head_dim))
        vw = np.zeros_like(kw)
        for t in range(nq, T):
            kw[:, :, t % Wn] = K[:, :, t]
            vw[:, :, t % Wn] = V[:, :, t]
    return dict(ck=ck, bk=bk, cv=cv, bv=bv, sk=sk, sv=sv, qk=qk, qv=qv, qjl=qjl, dsign=dsign,
                kw=kw, vw=vw)


def _oracle_decode(w, c, qs, seq):
    import oracle as O
    return O.decode_attention(qs, c["qk"]["codes"], c["qk"]["norms"], c["qv"]["codes"],
                              c["qv"]["norms"], c["ck"], c["cv"], c["sk"], c["sv"], seq,
                              w.softmax_scale, window=w.window, k_win=c["kw"], v_win=c["vw"],
                              qjl=c["qjl"], dsign=c["dsign"])


def score_quality(w, K, qs, c, T):
    """Attention-score fidelity of the compressed keys on the sampled heads
    (the write-up's quality figures: score similarity and top-1 agreement,
    "윈도우용 터보퀀트(TurboQuant) 구현을 개선하다", results): cosine
    similarity of the compressed-domain scores of the quantized tokens with
    the exact fp64 scores of the same bf16 keys, and how often their argmax
    agrees, over the sampled query heads."""
    import numpy as np
    import oracle as O
    nq = T - w.window
    g = w.group
    RK = O.rotation_matrix(c["sk"])
    sims, top1 = [], []
    for j, hk in enumerate(range(K.shape[1])):
        kc = c["qk"]["codes"][0, j, :nq]
        kn = c["qk"]["norms"][0, j, :nq].astype(np.float64)
        approx_keys = c["ck"].astype(np.float64)[kc]
        for i in range(g):
            qv = qs[0, j * g + i]
            exact = K[0, j, :nq] @ qv
            approx = kn * (approx_keys @ (RK @ qv))
            sims.append(float(exact @ approx / (np.linalg.norm(exact) * np.linalg.norm(approx))))
            top1.append(int(np.argmax(exact) == np.argmax(approx)))
    return {"score_cosine_similarity_mean": float(np.mean(sims)),
            "score_cosine_similarity_min": float(np.min(sims)),
            "top1_agreement": float(np.mean(top1)), "query_heads": len(sims),
            "what": "MSE codes only (no residual term); synthetic keys, not a model's"}


def sparse_skip_bound(w, st, q, seq, k):
    """Share of the 32-token chunks of kv-head 0 (sequence 0) whose softmax
    weights are all below 2^-k of each query head's final maximum, from the
    oracle's compressed-domain scores."""
    import numpy as np
    import oracle as O
    K, V, qs = _oracle_inputs(w, st, q, [0])
    T = int(seq[0])
    c = _oracle_cache(w, K, V, T)
    nq = T - w.window
    RK = O.rotation_matrix(c["sk"])
    keys = c["qk"]["norms"][0, 0, :nq].astype(np.float64)[:, None] * c["ck"].astype(np.float64)[c["qk"]["codes"][0, 0, :nq]]
    s = np.stack([keys @ (RK @ qs[0, j]) for j in range(w.group)]) * w.softmax_scale   # [G, nq]
    s2 = s / math.log(2.0)                                                              # log2 units
    below = s2 < (s2.max(axis=1, keepdims=True) - k)
    n = nq // 32
    chunks = below[:, :n * 32].reshape(w.group, n, 32).all(axis=(0, 2))
    return float(chunks.mean()) if n else 0.0


def sampled_parity(B, w, st, q, out, rep0, seq, step):
    """Oracle decode of a sample of kv-heads of sequence 0 at full context,
    against the CUDA output of the timed launch configuration."""
    import numpy as np
    import torch
    import oracle as O
    step(0)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    heads = [0] if w.context > 200000 or w.n_kv_heads == 1 else [0, w.n_kv_heads - 1]
    K, V, qs = _oracle_inputs(w, st, q, heads)
    T = int(seq[0])
    c = _oracle_cache(w, K, V, T)
    gk = O.unpack_codes(rep0[0].codes_view()[:1, heads].cpu().numpy(), w.k_bits, w.head_dim)
    nq = T - w.window
    band = O.near_boundary(c["qk"]["y"], c["bk"], w.head_dim)
    diff = gk[:, :, :nq] != c["qk"]["codes"]
    code_diff = int(diff.sum())
    outside = int((diff & ~band).sum())
    ref = _oracle_decode(w, c, qs, [T])
    g = w.group
    qh = [h * g + j for h in heads for j in range(g)]
    mine = got[:1, qh]
    rel = np.linalg.norm(mine - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
    return {"max_rel_l2": float(rel.max()), "tolerance": TOLERANCE,
            "pass": bool(rel.max() < TOLERANCE),
            "kv_heads_checked": heads, "query_heads_checked": len(qh),
            "key_code_mismatches_in_boundary_band": code_diff - outside,
            "key_code_mismatches_outside_band": outside,
            "quality": score_quality(w, K, qs, c, T)}


# ------------------------------------------------------- the oracle on the host
# The oracle's slice of each workload (the same slices as its parity checks):
# the single-head and Llama-shaped workloads whole; the batch-16 workloads 2
# sequences; the long-context workload one kv-head of 131,072 tokens; the
# serving workload 4 sequences x 3 layers (a protected one, a K4/V2 one and
# the last).
def oracle_slice(w):
    from kv_cache_quantization_random_gb300 import workloads as WL
    seq = WL.seq_lens(w)
    if w.name == "long_1m":
        return dict(batch=1, heads=[0], layers=[0], seq=[131072], frac_label="1 kv-head x 131,072 tokens")
    if w.n_layers > 1:
        return dict(batch=4, heads=list(range(w.n_kv_heads)),
                    layers=[0, w.protect_first, w.n_layers - 1], seq=[int(t) for t in seq[:4]],
                    frac_label="4 sequences x 3 layers (0, 4, 35), all kv-heads")
    if w.batch > 2:
        return dict(batch=2, heads=list(range(w.n_kv_heads)), layers=[0],
                    seq=[int(t) for t in seq[:2]], frac_label="2 sequences, all kv-heads")
    return dict(batch=w.batch, heads=list(range(w.n_kv_heads)), layers=[0],
                seq=[int(t) for t in seq], frac_label="whole step")


def oracle_slice_step(w, sl):
    """Prepare the oracle's compressed cache of the slice (CPU inputs drawn from
    the same seeded generators) and return (step, token_kvheads): step() runs
    one step of the slice (quantize of the appended tokens, then decode), and
    token_kvheads counts the (token, kv-head) pairs its decodes attend."""
    import numpy as np
    import oracle as O
    from kv_cache_quantization_random_gb300 import workloads as WL
    f64 = lambda t: t.float().numpy().astype(np.float64)
    Tmax = max(sl["seq"])
    n_new = w.new_tokens if w.n_layers > 1 else 1
    fm = layer_formats(w)
    caches = []
    for l in sl["layers"]:
        kb, vb = fm[l]
        K, V = WL.make_kv(w, layer=l, tokens=Tmax, batch=sl["batch"])
        K, V = f64(K[:, sl["heads"]]), f64(V[:, sl["heads"]])
        c = _oracle_cache(w, K, V, Tmax, layer=l, kb=kb, vb=vb)
        new = (K[:, :, Tmax - n_new:Tmax], V[:, :, Tmax - n_new:Tmax])
        caches.append((c, new))
    g = w.group
    qh = [h * g + j for h in sl["heads"] for j in range(g)]
    qs = f64(WL.make_q(w)[:sl["batch"], qh])

    def step():
        for c, (kn, vn) in caches:
            # append: quantize the step's tokens (those leaving the window;
            # with W = 0, the new ones)
            O.quantize_vectors(kn, c["ck"], c["bk"], c["sk"])
            O.quantize_vectors(vn, c["cv"], c["bv"], c["sv"])
            _oracle_decode(w, c, qs, sl["seq"])

    token_kvheads = len(sl["layers"]) * len(sl["heads"]) * sum(sl["seq"])
    return step, token_kvheads


def workload_token_kvheads(w):
    from kv_cache_quantization_random_gb300 import workloads as WL
    return w.n_layers * w.n_kv_heads * int(WL.seq_lens(w).sum())


def workload_tokens(w):
    from kv_cache_quantization_random_gb300 import workloads as WL
    return w.n_layers * int(WL.seq_lens(w).sum())


def oracle_timing_child(args):
    """Child process of cpu_baseline: time the oracle's slice with the thread
    count the parent pinned (BLAS/OpenMP threads from the environment, CPU
    affinity here), print one JSON line."""
    # the affinity first: threads that numpy's BLAS starts at import inherit it
    n = args.child_threads
    cpus = sorted(os.sched_getaffinity(0))[:n]
    os.sched_setaffinity(0, cpus)
    from kv_cache_quantization_random_gb300 import workloads as WL
    w = WL.get(args.workload)
    if args.llama_kv:
        w = WL.with_llama_kv(w)
    sl = oracle_slice(w)
    step, units = oracle_slice_step(w, sl)
    step()                                   # warm-up
    runs = 0
    t0 = time.perf_counter()
    while True:
        step()
        runs += 1
        el = time.perf_counter() - t0
        if el >= args.cpu_seconds or runs >= 1000:
            break
    s_per_step = el / runs
    print(json.dumps({"ns_per_token_kvhead": s_per_step / units * 1e9, "runs": runs,
                      "seconds": el, "threads": n, "slice": sl["frac_label"],
                      "slice_token_kvheads": units}), flush=True)


def oracle_timing(w, threads, seconds, llama_kv):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
              "NUMEXPR_NUM_THREADS"):
        env[k] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--impl", "oracle-child", "--workload",
           w.name, "--child-threads", str(threads), "--cpu-seconds", str(seconds)]
    if llama_kv:
        cmd.append("--llama-kv")
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(f"oracle timing child failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(w, seconds):
    """The oracle, as it stands, timed on this host's cores on its slice of the
    workload, with all cores and with one (BLAS/OpenMP threads pinned to the
    count), scaled to the workload's whole step."""
    cores = len(os.sched_getaffinity(0))
    llama_kv = w.dist == "llama" and w.name != "llama8b_32k"
    full = oracle_timing(w, cores, seconds, llama_kv)
    one = oracle_timing(w, 1, seconds, llama_kv)
    tk = workload_token_kvheads(w)
    tokens = workload_tokens(w)
    value = tokens / (full["ns_per_token_kvhead"] * 1e-9 * tk)
    return {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{full['slice']} ({full['slice_token_kvheads']} token-kvheads per step): "
                      f"{full['runs']} steps in {full['seconds']:.1f} s; scaled to the workload's "
                      f"{tk} token-kvheads per step",
            "ns_per_token_kvhead": full["ns_per_token_kvhead"],
            "one_core": {"ns_per_token_kvhead": one["ns_per_token_kvhead"],
                         "value": tokens / (one["ns_per_token_kvhead"] * 1e-9 * tk),
                         "runs": one["runs"], "seconds": one["seconds"]},
            "threads_pinned": "OMP/OpenBLAS/MKL threads = cores used; CPU affinity set"}


# ------------------------------------------------------------ reference arm
def run_reference(args, w, rank, world):
    """The CPU oracle timed as the reference implementation, on the same
    workload, metric and unit.  Each step is the oracle's slice of the
    workload's step (the whole step for the single-head and Llama-shaped
    workloads), measured as it runs; value counts the tokens the slice
    attends."""
    import numpy as np
    if rank != 0:
        return None
    cores = len(os.sched_getaffinity(0))
    sl = oracle_slice(w)
    step, units = oracle_slice_step(w, sl)
    warm = max(args.warmup, 3)
    for _ in range(warm):
        step()
    steps = max(1, min(args.steps, args.reference_max_steps))
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    el = time.perf_counter() - t0
    ms_per_step = el / steps * 1e3
    # tokens attended per step of the slice (summed over its layers, all
    # query heads of its kv-heads), in the workload's unit
    slice_tokens = units / w.n_kv_heads
    value = slice_tokens / (ms_per_step * 1e-3)
    tk = workload_token_kvheads(w)
    full_ms = ms_per_step * tk / units
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": steps, "warmup": warm, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "batch": w.batch, "q_heads": w.n_q_heads,
                       "kv_heads": w.n_kv_heads, "head_dim": w.head_dim,
                       "context": int(max(sl["seq"])), "k_bits": w.k_bits, "v_bits": w.v_bits,
                       "window": w.window, "parallelism": "host cores", "slice": sl["frac_label"]},
            "full_step_ms_estimate": full_ms,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: oracle append + decode over the slice "
                                       f"({sl['frac_label']}), {units} token-kvheads"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference", "oracle-child"], default="ours")
    ap.add_argument("--workload", default="llama8b_32k")
    ap.add_argument("--llama-kv", action="store_true",
                    help="Llama-shaped key/value distributions for the workloads that default "
                         "to the single-head workload's")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="repeat the K timed steps until this much time has passed")
    ap.add_argument("--no-parity", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--child-threads", type=int, default=1)
    ap.add_argument("--reference-max-steps", type=int, default=40)
    ap.add_argument("--n-queries", type=int, default=1,
                    help="also time decode of N query tokens per sequence (causal, in the window)")
    ap.add_argument("--sparse-v", type=int, default=0,
                    help="skip a 32-token chunk's V sum when all its softmax weights are below "
                         "2^-N of the running maximum (0: exact, the default)")
    ap.add_argument("--decode-traffic", type=float, default=None,
                    help="dram bytes per decode launch from an ncu capture of the current kernel")
    args = ap.parse_args()
    if args.impl == "oracle-child":
        oracle_timing_child(args)
        return

    from kv_cache_quantization_random_gb300 import workloads as WL
    w = WL.get(args.workload)
    if args.llama_kv:
        w = WL.with_llama_kv(w)
    rank, world, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, w, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    res = (run_layered if w.n_layers > 1 else run_single)(args, w, rank, world, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
