#!/usr/bin/env python3
"""Benchmark of the TurboQuant hot path on one GB300 (or N replicas).

A step is one decode step of a serving loop over the workload's cache, one
tq_decode_step call:
  append   one new token per (sequence, kv-head): the token leaving the
           residual window is quantized into the planes and the new token is
           written into the window ring (norm, rotation, code search, packing,
           window bookkeeping);
  decode   attention of every query head over the whole compressed context
           (query rotation, compressed-domain scoring, softmax, rotated V sum,
           split merge and inverse rotation), launched so that it overlaps the
           append.
The headline value is context tokens attended per second.  Bulk quantize of
the whole context (K and V) is measured separately and reported in GB/s.

Inputs are seeded synthetic tensors shaped like the workload (see
kv_cache_quantization_random_gb300/workloads.py).  Timed steps cycle through R
copies of the compressed cache whose total is more than 4x the L2 cache, so
every step streams its cache from HBM.

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


def whole_job_rate(units_per_rank: float, ms_per_step: float, world: int) -> float:
    """Units per second of the whole job: every rank processes units_per_rank
    per step, and a step takes the slowest rank's time."""
    return world * units_per_rank / (ms_per_step * 1e-3)


def largest_divisor_at_most(n: int, cap: int) -> int:
    for s in range(min(n, cap), 0, -1):
        if n % s == 0:
            return s
    return 1


# --------------------------------------------------------------- workload
def packed_bytes(w):
    """Bytes of one packed key and one packed value vector (codes + norms [+ QJL])."""
    d = w.head_dim
    kbytes = d * w.k_bits // 8 + 4 + ((w.qjl_m // 8 + 4) if w.k_qjl else 0) + \
        ((d // 8 + 4) if w.k_sign else 0)
    vbytes = d * w.v_bits // 8 + 4
    return kbytes, vbytes


def algorithmic_bytes(w, seq, W):
    """Bytes decode attention must move: packed K and V of quantized tokens,
    bf16 window K and V, bf16 query in, fp32 output."""
    d = w.head_dim
    kbytes, vbytes = packed_bytes(w)
    total = 0
    for T in seq:
        nq = max(int(T) - W, 0)
        nw = int(T) - nq
        total += w.n_kv_heads * (nq * (kbytes + vbytes) + nw * d * 2 * 2)
    total += len(seq) * w.n_q_heads * d * (2 + 4)
    return total


def build_state(B, w, device, layer=0, sparse_v=0):
    """Inputs, planes and window ring of the workload's context (not yet quantized)."""
    import torch
    from kv_cache_quantization_random_gb300 import workloads as WL
    T, Wn = w.context, w.window
    nq = T - Wn
    cfg = B.Config(k_bits=w.k_bits, v_bits=w.v_bits, residual_window=Wn, seed=w.codec_seed,
                   k_mode=(B.TQ_MODE_MSE_QJL if w.k_qjl else
                           B.TQ_MODE_MSE_SIGN if w.k_sign else B.TQ_MODE_MSE), qjl_m=w.qjl_m,
                   sparse_v=sparse_v)
    tables = B.device_tables(cfg, device)
    K, V = WL.make_kv(w, layer=layer, device=device)
    kp = B.Planes(cfg, layer, 0, w.batch, w.n_kv_heads, nq, device)
    vp = B.Planes(cfg, layer, 1, w.batch, w.n_kv_heads, nq, device)
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
        st["kw"][:, :, idx % Wn] = st["K"][:, :, nq:T]
        st["vw"][:, :, idx % Wn] = st["V"][:, :, nq:T]


def window_before_step(st, w, seq):
    """Window ring as it stands before a step appends token T-1: the slot of
    token T-1 still holds token T-1-W, which the step's append quantizes."""
    Wn = w.window
    if not Wn:
        return
    for b, T in enumerate(seq):
        t = int(T) - 1 - Wn
        if t >= 0:
            st["kw"][b, :, t % Wn] = st["K"][b, :, t]
            st["vw"][b, :, t % Wn] = st["V"][b, :, t]


def run_ours(args, w, rank, world, local):
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

    # ---- bulk quantize of the whole context (K and V), timed separately
    def quantize_all():
        B.tq_quantize_kv(cfg, tables, 0, 0, K[:, :, :nq], kp)
        B.tq_quantize_kv(cfg, tables, 0, 1, V[:, :, :nq], vp)

    for _ in range(3):
        quantize_all()
    torch.cuda.synchronize()
    # device time of the launches, without the host's per-call overhead:
    # qiters calls replayed from one CUDA graph, best of 5 replays
    qiters = 10

    def graph_ms(fn):
        gq = torch.cuda.CUDAGraph()
        sq = torch.cuda.Stream()
        sq.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(sq):
            with torch.cuda.graph(gq, stream=sq):
                for _ in range(qiters):
                    fn()
        torch.cuda.current_stream().wait_stream(sq)
        gq.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        best = float("inf")
        for _ in range(5):
            e0.record()
            gq.replay()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) / qiters)
        return best

    q_ms = graph_ms(quantize_all)
    # keys in MSE+QJL mode: the QJL kernel alone, and the rate of its
    # projection, 2 (hi, lo) x 2 x keys x m x d flops on the tensor cores
    qjl_proj = None
    if w.k_qjl:
        k_ms = graph_ms(lambda: B.tq_quantize_kv(cfg, tables, 0, 0, K[:, :, :nq], kp))
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
    in_b = w.head_dim * (4 if w.in_dtype == "fp32" else 2)
    kbts, vbts = packed_bytes(w)
    q_bytes = n_vec * (2 * in_b + kbts + vbts)
    q_gbs = q_bytes / (q_ms * 1e-3) / 1e9
    if B.tq_get_device_error() != B.TQ_OK:
        raise RuntimeError("device error after quantize")

    # ---- replicas of the compressed cache (more than 4x L2 in total)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    seq = WL.seq_lens(w)
    dec_bytes = algorithmic_bytes(w, seq, Wn)
    cache_bytes = sum(t.numel() for t in (kp.codes, kp.norms, vp.codes, vp.norms)) + \
        (2 * st["kw"].numel() * 2 if Wn else 0)
    R = max(2, min(64, math.ceil(4 * l2 / max(cache_bytes, 1)) + 1))
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
        # tq_decode_step: the append and the decode that overlaps it
        kr, vr, kwr, vwr = reps[i % R]
        B.tq_decode_step(cfg, tables, 0, q, w.softmax_scale, knew, vnew, seq_before, Tmax, kr, vr,
                         out, ws, k_win=kwr, v_win=vwr)

    # one append launch (one new token per sequence) + one decode launch
    launches_per_step = 2

    # ---- warmup (direct launches), then capture graphs of S steps
    warm = max(args.warmup, 3)
    for i in range(warm):
        step(i)
    torch.cuda.synchronize()
    if B.tq_get_device_error() != B.TQ_OK:
        raise RuntimeError("device error during warmup")
    K_steps = args.steps
    S = largest_divisor_at_most(K_steps, 128)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(S):
                    fn(i)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        return g

    g_step = capture(step)
    g_dec = capture(lambda i: decode(i % R))
    g_app = capture(lambda i: append(i % R))
    for g in (g_step, g_dec, g_app):
        g.replay()
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(K_steps // S):
            g_step.replay()
        t1.record()
        torch.cuda.synchronize()
    step_ms_total = max_over_ranks(t0.elapsed_time(t1), device)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ms_per_step = step_ms_total / K_steps
    tokens_per_step = int(seq.sum())
    value = whole_job_rate(tokens_per_step, ms_per_step, world)

    # ---- per-kernel durations (decode-only and append-only graphs, same stream)
    def time_graph(g, reps_):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps_):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (reps_ * S)

    reps_t = max(1, min(K_steps // S, 200))
    dec_ms = time_graph(g_dec, reps_t)
    app_ms = time_graph(g_app, reps_t)
    if B.tq_get_device_error() != B.TQ_OK:
        raise RuntimeError("device error during timed steps")
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9

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
        g_multi = capture(lambda i: decode_multi(i % R))
        g_multi.replay()
        torch.cuda.synchronize()
        mq_ms = time_graph(g_multi, reps_t)
        mq_bytes = dec_bytes + len(seq) * w.n_q_heads * (nQ - 1) * w.head_dim * (2 + 4)
        multi = {"n_queries": nQ, "ms": mq_ms, "gbs": mq_bytes / (mq_ms * 1e-3) / 1e9,
                 "query_token_attends_per_s": nQ * tokens_per_step / (mq_ms * 1e-3),
                 "vs_single_query_ms": dec_ms}

    # ---- end to end through the public API with host buffers: every step
    # copies its inputs (query, new K and V token) from one pinned host buffer
    # to the device, runs append + decode, and reads the output back to
    # pinned host memory; the steps are replayed from a CUDA graph like the
    # device-only steps, so the copies are in every step
    parts = [q, knew, vnew]
    nbytes = [t.numel() * t.element_size() for t in parts]
    offs = [0]
    for n in nbytes[:-1]:
        offs.append(offs[-1] + (n + 255) // 256 * 256)
    total_in = offs[-1] + nbytes[-1]
    hbuf = torch.empty(total_in, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(total_in, dtype=torch.uint8, device=device)
    for t, o, n in zip(parts, offs, nbytes):
        hbuf[o:o + n].copy_(t.contiguous().view(torch.uint8).view(-1).cpu())
    qd, kd, vd = (dbuf[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(parts, offs, nbytes))
    outh = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e_step(i):
        dbuf.copy_(hbuf, non_blocking=True)
        kr, vr, kwr, vwr = reps[i % R]
        B.tq_decode_step(cfg, tables, 0, qd, w.softmax_scale, kd, vd, seq_before, Tmax, kr, vr,
                         out, ws, k_win=kwr, v_win=vwr)
        outh.copy_(out, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    g_e2e = capture(e2e_step)
    g_e2e.replay()
    torch.cuda.synchronize()
    n_rep = max(1, K_steps // S)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(n_rep):
        g_e2e.replay()
    b.record()
    torch.cuda.synchronize()
    n_e2e = n_rep * S
    e2e_serial_ms = max_over_ranks(a.elapsed_time(b) / n_e2e, device)

    # the same steps pipelined as a server runs independent steps: step i's
    # host-to-device copy (copy-in stream) overlaps step i-1's kernels
    # (compute stream), and its device-to-host copy (copy-out stream) overlaps
    # step i+1's; inputs and outputs are double-buffered on the device and the
    # host, and graph edges order every reuse of a buffer
    dbufs = [dbuf, torch.empty_like(dbuf)]
    dviews = [tuple(d[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(parts, offs, nbytes))
              for d in dbufs]
    outs = [out, torch.empty_like(out)]
    ouths = [outh, torch.empty(out.shape, dtype=out.dtype).pin_memory()]

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

    g_pipe = capture_pipelined()
    g_pipe.replay()
    torch.cuda.synchronize()
    a.record()
    for _ in range(n_rep):
        g_pipe.replay()
    b.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b) / n_e2e, device)
    if B.tq_get_device_error() != B.TQ_OK:
        raise RuntimeError("device error during the end-to-end steps")
    # the host copies hold what the last steps computed
    for j in range(2):
        if not torch.equal(ouths[j], outs[j].cpu()):
            raise RuntimeError("pipelined end-to-end steps: host output differs from the device's")
    h2d = total_in
    d2h = outh.numel() * outh.element_size()

    # ---- sampled parity at full size, in the launch configuration timed above
    parity = None
    if not args.no_parity and rank == 0:
        # the timed steps rewrote one row and one window slot of every replica:
        # restore replica 0 from the inputs, as it stands before the step's
        # append, and check the output of one step
        quantize_all()
        reset_window(st, w)
        window_before_step(st, w, seq)
        parity = sampled_parity(B, w, st, q, out, reps[0], seq, step)

    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": K_steps, "warmup": warm, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp32", "data": "synthetic",
        "config": {
            "workload": w.name, "batch": w.batch, "q_heads": w.n_q_heads,
            "kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "context": int(seq.max()),
            "k_bits": w.k_bits, "v_bits": w.v_bits, "k_qjl": w.k_qjl, "k_sign": w.k_sign,
            "window": Wn,
            "new_tokens_per_step": 1, "parallelism": f"replicas x{world}",
            "sparse_v": args.sparse_v,
            "l2": f"{R} cache replicas cycled ({R * cache_bytes / 1e6:.0f} MB > 4 x L2 {l2 / 1e6:.0f} MB)",
            "graph_steps": S,
        },
        "roofline": {
            "kernel": "tq::decode_kernel", "bound": "hbm", "achieved": dec_gbs,
            "peak": hbm_peak, "unit": "GB/s", "frac": dec_gbs / hbm_peak,
            "peak_source": f"{peak_kind} hbm_gbs",
            "traffic": (args.decode_traffic if args.decode_traffic is not None
                        else captured_traffic("decode_kernel", w.name)),
            "bytes_per_launch": dec_bytes, "launch_ms": dec_ms,
        },
        "decode": {"ms": dec_ms, "gbs": dec_gbs, "frac_of_peak": dec_gbs / hbm_peak,
                   "tokens_per_s": tokens_per_step / (dec_ms * 1e-3), "bytes": dec_bytes},
        "append": {"ms": app_ms, "launches": launches_per_step - 1},
        "quantize": {"ms": q_ms, "gbs": q_gbs, "frac_of_peak": q_gbs / hbm_peak,
                     "vectors": 2 * n_vec, "bytes": q_bytes, "what": "bulk quantize of the "
                     "context's K and V (bf16 in, packed planes out)"},
        "e2e": {"value": whole_job_rate(tokens_per_step, e2e_ms, world), "unit": "tokens/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": n_e2e, "pipelined": True,
                "serial": {"value": whole_job_rate(tokens_per_step, e2e_serial_ms, world),
                           "ms_per_step": e2e_serial_ms,
                           "what": "each step's copy-in, kernels and copy-out one after another"}},
        "gpu_launches": K_steps * launches_per_step,
        "clocks": clocks.summary(),
        "parity": parity,
    }
    if multi is not None:
        res["multi_query"] = multi
    if qjl_proj is not None:
        res["qjl_projection"] = qjl_proj
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, st, q, seq, budget_s=args.cpu_seconds)
    return res


def _oracle_inputs(w, st, q, heads):
    """fp64 copies of the inputs of kv-heads `heads` (sequence 0)."""
    import numpy as np
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)
    K = f64(st["K"][:1, heads])
    V = f64(st["V"][:1, heads])
    g = w.group
    qh = [h * g + j for h in heads for j in range(g)]
    return K, V, f64(q[:1, qh])


def _oracle_cache(w, K, V, T):
    """The oracle's own compressed cache of K, V (sequence 0), plus window ring."""
    import numpy as np
    import oracle as O
    Wn = w.window
    nq = T - Wn
    ck, bk = O.codebook_fp32(w.k_bits, w.head_dim)
    cv, bv = O.codebook_fp32(w.v_bits, w.head_dim)
    sk = O.rotation_signs(w.codec_seed, 0, 0, w.head_dim)
    sv = O.rotation_signs(w.codec_seed, 0, 1, w.head_dim)
    qk = O.quantize_vectors(K[:, :, :nq], ck, bk, sk)
    qv = O.quantize_vectors(V[:, :, :nq], cv, bv, sv)
    qjl = None
    if w.k_qjl:
        S = O.qjl_matrix(w.codec_seed, 0, w.qjl_m, w.head_dim)
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
        kw = np.zeros((1, K.shape[1], Wn, w.head_dim))
        vw = np.zeros_like(kw)
        for t in range(nq, T):
            kw[:, :, t % Wn] = K[:, :, t]
            vw[:, :, t % Wn] = V[:, :, t]
    return dict(ck=ck, bk=bk, cv=cv, bv=bv, sk=sk, sv=sv, qk=qk, qv=qv, qjl=qjl, dsign=dsign,
                kw=kw, vw=vw)


def _oracle_decode(w, c, qs, T):
    import oracle as O
    return O.decode_attention(qs, c["qk"]["codes"], c["qk"]["norms"], c["qv"]["codes"],
                              c["qv"]["norms"], c["ck"], c["cv"], c["sk"], c["sv"], [T],
                              w.softmax_scale, window=w.window, k_win=c["kw"], v_win=c["vw"],
                              qjl=c["qjl"], dsign=c["dsign"])


def sampled_parity(B, w, st, q, out, rep0, seq, decode):
    """Oracle decode of a sample of kv-heads of sequence 0 at full context,
    against the CUDA output of the timed launch configuration."""
    import numpy as np
    import torch
    import oracle as O
    decode(0)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    heads = [0, w.n_kv_heads - 1] if w.n_kv_heads > 1 else [0]
    K, V, qs = _oracle_inputs(w, st, q, heads)
    T = int(seq[0])
    c = _oracle_cache(w, K, V, T)
    gk = O.unpack_codes(rep0[0].codes_view()[:1, heads].cpu().numpy(), w.k_bits, w.head_dim)
    band = O.near_boundary(c["qk"]["y"], c["bk"], w.head_dim)
    code_diff = int((gk != c["qk"]["codes"]).sum())
    outside = int(((gk != c["qk"]["codes"]) & ~band).sum())
    ref = _oracle_decode(w, c, qs, T)
    g = w.group
    qh = [h * g + j for h in heads for j in range(g)]
    mine = got[:1, qh]
    rel = np.linalg.norm(mine - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
    return {"max_rel_l2": float(rel.max()), "tolerance": 2e-3, "pass": bool(rel.max() < 2e-3),
            "kv_heads_checked": heads, "query_heads_checked": len(qh),
            "key_code_mismatches_in_boundary_band": code_diff - outside,
            "key_code_mismatches_outside_band": outside}


def cpu_baseline(w, st, q, seq, budget_s=15.0):
    """The oracle, as it stands, timed on this host's cores on a bounded sample:
    decode attention of one kv-head group of sequence 0 (the step's append of
    one token is negligible next to it), scaled to the workload."""
    import numpy as np
    cores = len(os.sched_getaffinity(0))
    T = int(seq[0])
    K, V, qs = _oracle_inputs(w, st, q, [0])
    c = _oracle_cache(w, K, V, T)
    n = 0
    t0 = time.perf_counter()
    while True:
        _oracle_decode(w, c, qs, T)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 1000:
            break
    per_group = el / n
    groups = w.batch * w.n_kv_heads
    step_s = per_group * groups * (float(np.mean(seq)) / T)
    tokens = float(np.sum(seq))
    return {"value": tokens / step_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} oracle decode(s) of one kv-head group ({w.group} query heads) "
                      f"over {T} tokens of sequence 0, {el:.1f} s, scaled x{groups} groups"}


# ------------------------------------------------------------ reference arm
def run_reference(args, w, rank, world):
    """The CPU oracle timed as the reference implementation, on the same
    workload, metric and unit; each step is a bounded sample (one kv-head group)."""
    import numpy as np
    import oracle as O
    from kv_cache_quantization_random_gb300 import workloads as WL
    if rank != 0:
        return None
    cores = len(os.sched_getaffinity(0))
    seq = WL.seq_lens(w)
    T, Wn = int(seq[0]), w.window
    nq = T - Wn
    f64 = lambda t: t.float().numpy().astype(np.float64)
    K, V = WL.make_kv(w, batch=1)
    K, V = f64(K[:, :1]), f64(V[:, :1])
    qs = f64(WL.make_q(w)[:1, :w.group])
    c = _oracle_cache(w, K, V, T)

    def step():
        # append: quantize the token leaving the window (one vector per kind)
        O.quantize_vectors(K[:, :, nq - 1:nq], c["ck"], c["bk"], c["sk"])
        O.quantize_vectors(V[:, :, nq - 1:nq], c["cv"], c["bv"], c["sv"])
        _oracle_decode(w, c, qs, T)

    for _ in range(max(args.warmup, 3)):
        step()
    steps = min(args.steps, args.reference_max_steps)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    el = time.perf_counter() - t0
    groups = w.batch * w.n_kv_heads
    ms_per_step = el / steps * groups * 1e3 * (float(np.mean(seq)) / T)
    value = float(np.sum(seq)) / (ms_per_step * 1e-3)
    sample = (f"each step: oracle append of 1 token + decode of one kv-head group "
              f"({w.group} query heads) over {T} tokens, scaled x{groups} groups")
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "batch": w.batch, "q_heads": w.n_q_heads,
                       "kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "context": T,
                       "k_bits": w.k_bits, "v_bits": w.v_bits, "window": Wn,
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b_32k")
    ap.add_argument("--no-parity", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reference-max-steps", type=int, default=200)
    ap.add_argument("--n-queries", type=int, default=1,
                    help="also time decode of N query tokens per sequence (causal, in the window)")
    ap.add_argument("--sparse-v", type=int, default=0,
                    help="skip a 32-token chunk's V sum when all its softmax weights are below "
                         "2^-N of the running maximum (0: exact, the default)")
    ap.add_argument("--decode-traffic", type=float, default=None,
                    help="dram bytes per decode launch from an ncu capture of the current kernel")
    args = ap.parse_args()

    from kv_cache_quantization_random_gb300 import workloads as WL
    w = WL.get(args.workload)
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
    res = run_ours(args, w, rank, world, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
