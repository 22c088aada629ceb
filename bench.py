#!/usr/bin/env python
"""Benchmark of the MLA hot path on GB300.

A step is one whole MLA decode layer step on the DeepSeek-V2-shaped decode
workload (d_model 5120, 128 heads, d_nope 128, d_rope 64, r_kv 512, r_q 1536,
batch 64, per-sequence cache lengths ~ U[1024, 4096], seed 0):
latent + query projection with the cache append, weight absorption, split-KV
latent attention, combine, W_UV, and the output projection.  ``value`` is
latent-cache bytes read per step (sum over sequences of L_b * (r_kv + d_rope)
* 2) divided by the step time, summed over ranks.  The prefill workload
(B=4, S=4096, same dims) is timed as a secondary figure in TFLOP/s.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs an independent replica (the path has no
cross-GPU exchange); rank 0 prints one JSON line.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import mla_synth as syn  # noqa: E402

METRIC = "MLA decode latent-cache HBM GB/s (% of peak); prefill TFLOP/s (% bf16 peak)"
DECODE = syn.WORKLOADS["dsv2_decode"]
PREFILL = syn.WORKLOADS["dsv2_prefill"]
MLRA = syn.WORKLOADS["mlra_decode"]
L2_FLUSH_BYTES = 512 << 20
NOMINAL_HBM_GBS = 7900.0  # the HBM3e bandwidth NVIDIA quotes for GB300 (context beside the measured peak)
# DRAM bytes (read + write) of one decode attention launch on this workload,
# from an ncu capture of the current kernel (dram__bytes_read.sum +
# dram__bytes_write.sum); None whenever the kernel changes until it is
# captured again.
DECODE_TRAFFIC_BYTES = 217263616  # 213,548,288 read + 3,715,328 written


def max_over_ranks(vals, world: int, device):
    """Element-wise maximum of per-rank timings, returned on every rank (the
    job is as slow as its slowest rank)."""
    vals = [float(v) for v in vals]
    if world <= 1:
        return vals
    import torch
    import torch.distributed as dist
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_rate(world: int, units_per_rank: float, ms: float) -> float:
    """Whole-job throughput: every rank processes units_per_rank in ms (weak
    scaling), so the job processes world times that."""
    return world * units_per_rank / (ms * 1e-3)


def spread(ms_list):
    """Median and 10th / 90th percentiles of per-step times (ms)."""
    a = np.asarray(ms_list, np.float64)
    return {"median": round(float(np.median(a)), 5), "p10": round(float(np.percentile(a, 10)), 5),
            "p90": round(float(np.percentile(a, 90)), 5)}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def decode_bytes(lens) -> int:
    return int(np.sum(lens)) * (DECODE.r_kv + DECODE.d_rope) * 2


def decode_call_extra_bytes(B: int) -> int:
    """Bytes an mla_decode call moves besides the cache rows: the absorption
    and value weights W_UK and W_UV, the queries read and the output written
    (bf16)."""
    w = DECODE
    weights = 2 * w.n_heads * w.d_nope * w.r_kv * 2
    q = B * w.n_heads * (w.d_nope + w.d_rope) * 2
    out = B * w.n_heads * w.d_v * 2
    return weights + q + out


def decode_flops(lens) -> float:
    w = DECODE
    return float(np.sum(lens)) * w.n_heads * 2 * ((w.r_kv + w.d_rope) + w.r_kv)


def prefill_flops(w=PREFILL) -> float:
    T = w.batch * w.seq
    H = w.n_heads
    # The query: compressed (W_DQ, then W_UQ and W_QR) or, in the small-model
    # form (r_q = 0), one W_Q.
    q_proj = (w.d_model * w.r_q + w.r_q * H * (w.d_nope + w.d_rope)) if w.r_q else w.d_model * H * w.d_nope
    proj = 2 * T * (w.d_model * (w.r_kv + w.d_rope) + q_proj + w.r_kv * H * (w.d_nope + w.d_v)
                    + H * w.d_v * w.d_model)
    attn = w.batch * H * (w.seq * (w.seq + 1) / 2) * 2 * ((w.d_nope + w.d_rope) + w.d_v)
    return proj + attn, attn


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str):
        self.index = index
        self.proc = None
        self.lines = []
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=5)

    def summary(self):
        rows = []
        for ts, line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            rows.append((ts, f))
        inside = [r for r in rows if any(a - 0.05 <= r[0] <= b + 0.05 for a, b in self.windows)]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        sm = [float(f[2]) for _, f in use if f[2].replace(".", "").isdigit()]
        smax = [float(f[3]) for _, f in use if f[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, f in use:
            for i, n in enumerate(names):
                if f[6 + i].lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(use), "samples_in_timed_region": len(inside)}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def timing_events(n):
    """n (begin, end) pairs of timing events, created eagerly (torch creates
    the underlying cudaEvent_t lazily, on first record) so that their handles
    can be handed to the library's profiling hook."""
    import torch
    out = []
    for _ in range(n):
        pair = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        for e in pair:
            e.record()
        out.append(pair)
    torch.cuda.synchronize()
    return out


def to_dev(stored, device):
    import torch
    if stored.dtype == np.uint16:
        return torch.from_numpy(stored.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(stored).to(device)


def build_layer(w, device, max_batch, max_seq, max_tokens, ws_max_len):
    import head_latent_attention_gb300 as mla
    cfg = mla.make_config(w.variant, w.dtype, w.d_model, w.n_heads, w.d_nope, w.d_rope, w.d_v,
                          w.r_kv, w.r_q, w.n_latent_heads, w.rope_base, max_batch, max_seq)
    dev_w = {k: to_dev(s, device) for k, (s, _) in syn.weights(w).items()}
    return mla.MlaLayer(cfg, dev_w, max_tokens, device=device, ws_max_len=ws_max_len)


def run_ours(args, rank, world, device):
    import torch
    import torch.distributed as dist
    from head_latent_attention_gb300 import _build
    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        dist.barrier()
    import head_latent_attention_gb300 as mla

    hbm_peak, tf_peak, tf_sust, peak_src = peaks()
    w = DECODE
    B = w.batch
    lens = syn.lengths(w)
    lay = build_layer(w, device, B, w.seq, B, 0)
    for b in range(B):
        ls, _ = syn.cache_rows(w, b, int(lens[b]))
        lay.cache_lat[b, :lens[b]] = to_dev(ls, device)
        rs, _ = syn.cache_rows(w, b, int(lens[b]), "cache_rope")
        lay.cache_rope[b, :lens[b]] = to_dev(rs, device)
    xs, _ = syn.activations(w, B)
    x = to_dev(xs, device)
    seq = torch.arange(B, dtype=torch.int32, device=device)
    pos = torch.from_numpy(lens - 1).to(device)
    sl = torch.from_numpy(lens).to(device)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    dt = torch.bfloat16
    qn = torch.empty(B, w.n_heads, w.d_nope, dtype=dt, device=device)
    qr = torch.empty(B, w.n_heads, w.d_rope, dtype=dt, device=device)
    o = torch.empty(B, w.n_heads, w.d_v, dtype=dt, device=device)
    y = torch.empty(B, w.d_model, dtype=dt, device=device)

    def check(st, what):
        if st != mla.MLA_OK:
            raise mla.MlaError(st, what)

    def step(x_in, pos_in, sl_in):
        check(mla.mla_project_latent(lay.h, lay.w, x_in, seq, pos_in, lay.cache, qn, qr, lay.ws),
              "mla_project_latent")
        check(mla.mla_decode(lay.h, lay.w, qn, qr, lay.cache, sl_in, B, o, lay.ws), "mla_decode")
        check(mla.mla_out_proj(lay.h, lay.w, o.view(B, -1), y, lay.ws), "mla_out_proj")

    # The step is captured once as a CUDA graph (its ~14 launches replay
    # without host overhead).  A second capture carries the profiling hook's
    # events around the decode attention kernel; event nodes cut the
    # programmatic overlap at that kernel's two edges, so the step is timed
    # from the graph without them and the kernel from the one with them,
    # both replayed in the timed loop.
    for _ in range(2):
        step(x, pos, sl)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    n_launch0 = mla.mla_launch_count()
    with torch.cuda.graph(graph):
        step(x, pos, sl)
    launches_per_step = mla.mla_launch_count() - n_launch0
    kb, ke = timing_events(1)[0]
    mla.mla_set_profile_events(mla.MLA_PROFILE_DECODE_ATTENTION, kb, ke)
    graph_k = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_k):
        step(x, pos, sl)
    mla.mla_set_profile_events(mla.MLA_PROFILE_DECODE_ATTENTION, None, None)
    # A third capture brackets the whole mla_decode call (absorption,
    # schedule, attention, merge, W_UV).
    cb, ce = timing_events(1)[0]
    mla.mla_set_profile_events(mla.MLA_PROFILE_DECODE_CALL, cb, ce)
    graph_c = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_c):
        step(x, pos, sl)
    mla.mla_set_profile_events(mla.MLA_PROFILE_DECODE_CALL, None, None)
    graphs = (graph, graph_k, graph_c)
    for _ in range(max(args.warmup, 3)):
        for g in graphs:
            flush.zero_()
            g.replay()
    torch.cuda.synchronize()

    uuid = str(getattr(torch.cuda.get_device_properties(device), "uuid", ""))
    sampler = ClockSampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else
                           (uuid or str(torch.cuda.current_device())))
    sampler.start()
    time.sleep(0.2)
    K = args.steps
    ev = timing_events(K)
    kern_ms, call_ms = [], []
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
        flush.zero_()
        graph_k.replay()
        flush.zero_()
        graph_c.replay()
        ce.synchronize()
        kern_ms.append(kb.elapsed_time(ke))
        call_ms.append(cb.elapsed_time(ce))
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        dist.barrier()
    launches = launches_per_step * len(graphs) * K  # the step graph and the two with timing events
    sampler.mark(t0, t1)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = sum(step_ms) / K
    kms = sum(kern_ms) / K
    cms = sum(call_ms) / K

    # End to end through the C ABI from pinned host buffers: H2D of the step's
    # inputs (token activations, positions, lengths: one pinned staging
    # buffer, one copy) and D2H of its output, captured with the step in one
    # graph.  Both copies go through mla_copy: the SMs move the bytes over the
    # host link and the copies chain with the step's kernels like any other
    # launch of the library.
    nx, ni = x.numel() * 2, B * 4
    inp_h = torch.empty(nx + 2 * ni, dtype=torch.uint8).pin_memory()
    inp_h[:nx].copy_(torch.from_numpy(np.ascontiguousarray(xs).view(np.uint8).reshape(-1)))
    inp_h[nx:nx + ni].copy_(torch.from_numpy((lens - 1).astype(np.int32).view(np.uint8)))
    inp_h[nx + ni:].copy_(torch.from_numpy(lens.astype(np.int32).view(np.uint8)))
    y_h = torch.empty(B, w.d_model, dtype=torch.bfloat16).pin_memory()
    inp_d = torch.empty(inp_h.numel(), dtype=torch.uint8, device=device)
    x_d = inp_d[:nx].view(torch.bfloat16).view(B, w.d_model)
    pos_d = inp_d[nx:nx + ni].view(torch.int32)
    sl_d = inp_d[nx + ni:].view(torch.int32)
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        check(mla.mla_copy(inp_d, inp_h), "mla_copy (inputs)")
        step(x_d, pos_d, sl_d)
        check(mla.mla_copy(y_h, y), "mla_copy (output)")
    for _ in range(2):
        g2.replay()
    eev = timing_events(K)
    torch.cuda.synchronize()
    t2 = time.time()
    for i in range(K):
        flush.zero_()
        eev[i][0].record(stream)
        g2.replay()
        eev[i][1].record(stream)
    torch.cuda.synchronize()
    t3 = time.time()
    sampler.mark(t2, t3)
    e2e_ms = sum(a.elapsed_time(b) for a, b in eev) / K
    launches += (launches_per_step + 2) * K  # the end-to-end graph: the step and its two copies
    h2d = inp_h.numel()
    d2h = y_h.numel() * 2

    # Secondary: prefill layer (project + causal attention + output projection).
    pre = run_prefill(args, lay_device=device) if args.prefill else None
    sampler.stop()
    clocks = sampler.summary()

    nbytes = decode_bytes(lens)
    ms, e2e_ms, kms, cms = max_over_ranks([ms, e2e_ms, kms, cms], world, device)
    value = job_rate(world, nbytes, ms) / 1e9
    call_bytes = nbytes + decode_call_extra_bytes(B)
    e2e_val = job_rate(world, nbytes, e2e_ms) / 1e9
    achieved = nbytes / (kms * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) caches/activations, N(0,1/fan_in) weights)",
        "config": {"workload": "dsv2_decode", "batch": B, "cache_len": "U[1024,4096] seed 0",
                   "sum_len": int(np.sum(lens)), "d_model": w.d_model, "heads": w.n_heads,
                   "d_nope": w.d_nope, "d_rope": w.d_rope, "r_kv": w.r_kv, "r_q": w.r_q,
                   "cache_bytes_per_step": nbytes,
                   "l2": "flushed between steps (512 MiB write, outside the step events)",
                   "timing": "step events around a graph of the step; the attention kernel's events "
                             "and the decode call's events in two more captures of the step replayed "
                             "after it in the same loop",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": "decode split-KV latent attention",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "peak_source": peak_src,
                     "kernel_ms": round(kms, 5), "traffic": DECODE_TRAFFIC_BYTES,
                     "traffic_unit": "bytes per launch",
                     "nominal": {"peak": NOMINAL_HBM_GBS, "frac": round(achieved / NOMINAL_HBM_GBS, 4)}},
        "decode_call": {"what": "one mla_decode call: absorption, split-KV attention, merge, W_UV",
                        "ms": round(cms, 5), "bytes": call_bytes,
                        "bytes_are": "cache rows read + W_UK + W_UV + q_nope + q_rope read + o written",
                        "GB/s": round(call_bytes / (cms * 1e-3) / 1e9, 1),
                        "frac": round(call_bytes / (cms * 1e-3) / 1e9 / hbm_peak, 4)},
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "step_ms": spread(step_ms),
        "kernel_ms_spread": spread(kern_ms),
        "clocks": clocks,
    }
    if pre:
        out["prefill"] = pre
    if args.small:
        out["small_lm_decode"] = run_small_decode(args, device)
        out["small_lm_prefill"] = run_prefill(args, device, syn.WORKLOADS["small_lm_prefill"])
    if args.cca:
        out["cca_prefill"] = run_cca(args, device, "cca_prefill")
        out["ccgqa_prefill"] = run_cca(args, device, "ccgqa_prefill")
    if args.mlra:
        out["mlra_decode"] = run_mlra(args, device)
        if world > 1:
            out["mlra_tp"] = run_mlra_tp(args, rank, world, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args)
    return out


def run_prefill(args, lay_device, w=None):
    """One prefill layer step (projection with the cache append, causal
    attention, output projection) of the DeepSeek-V2 prefill workload, or of
    another prefill workload `w` (the small-model form: no decoupled RoPE
    key, half-split RoPE on the decompressed query and keys)."""
    import torch
    import head_latent_attention_gb300 as mla
    hbm_peak, tf_peak, tf_sust, peak_src = peaks()
    if w is None:
        w = PREFILL if not args.prefill_batch else PREFILL.replace(batch=args.prefill_batch)
    B, S = w.batch, w.seq
    lay = build_layer(w, lay_device, B, S, B * S, S)
    xs, _ = syn.activations(w, B * S)
    x = to_dev(xs, lay_device)
    pos = torch.arange(S, dtype=torch.int32, device=lay_device).repeat(B)
    seq = torch.arange(B, dtype=torch.int32, device=lay_device).repeat_interleave(S)
    stream = torch.cuda.current_stream()

    dt = torch.bfloat16
    qn = torch.empty(B * S, w.n_heads, w.d_nope, dtype=dt, device=lay_device)
    qr = torch.empty(B * S, w.n_heads, w.d_rope, dtype=dt, device=lay_device) if w.d_rope else None
    o = torch.empty(B, S, w.n_heads, w.d_v, dtype=dt, device=lay_device)
    y = torch.empty(B * S, w.d_model, dtype=dt, device=lay_device)

    def check(st, what):
        if st != mla.MLA_OK:
            raise mla.MlaError(st, what)

    def step():
        check(mla.mla_project_latent(lay.h, lay.w, x, seq, pos, lay.cache, qn, qr, lay.ws), "mla_project_latent")
        check(mla.mla_prefill(lay.h, lay.w, qn, qr, lay.cache, B, S, None, o, lay.ws), "mla_prefill")
        check(mla.mla_out_proj(lay.h, lay.w, o.view(B * S, -1), y, lay.ws), "mla_out_proj")

    # Like the decode step: one graph of the layer step without timing hooks
    # (the step's figure) and one with events around the attention kernel
    # (its figure), replayed alternately.  The DeepSeek-V2 step moves several
    # GB, far more than L2 holds; a smaller workload's step fits in L2, so L2
    # is flushed before each replay (outside the events).
    footprint = B * S * (w.d_model * 4 + (w.r_kv + w.d_rope) * 2 + w.n_heads * (2 * w.d_nope + 2 * w.d_v)) * 2
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=lay_device) if footprint < (1 << 30) else None
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    kb, ke = timing_events(1)[0]
    mla.mla_set_profile_events(mla.MLA_PROFILE_PREFILL_ATTENTION, kb, ke)
    g_k = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_k):
        step()
    mla.mla_set_profile_events(mla.MLA_PROFILE_PREFILL_ATTENTION, None, None)
    for _ in range(3):
        g.replay()
        g_k.replay()
    torch.cuda.synchronize()
    K = max(args.prefill_steps, 1)
    ev = timing_events(K)
    step_ms, kern_ms = [], []
    for i in range(K):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        g.replay()
        ev[i][1].record(stream)
        if flush is not None:
            flush.zero_()
        g_k.replay()
        ke.synchronize()
        kern_ms.append(kb.elapsed_time(ke))
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = sum(step_ms) / K
    kms = sum(kern_ms) / K
    total, attn = prefill_flops(w)
    tf = total / (ms * 1e-3) / 1e12
    katt = attn / (kms * 1e-3) / 1e12
    del lay, g, g_k
    torch.cuda.empty_cache()
    return {"workload": w.name, "batch": B, "seq": S, "steps": K,
            "timing": "graph of the layer step; attention kernel events in a second graph of it",
            "l2": "flushed before each replay" if flush is not None else "step traffic far above L2: no flush",
            "ms_per_step": round(ms, 4), "step_ms": spread(step_ms), "tflops": round(tf, 2), "unit": "TFLOP/s",
            "frac_of_bf16_peak": round(tf / tf_peak, 4), "flops_per_step": total,
            "roofline": {"bound": "tensor", "kernel": "causal flash attention",
                         "achieved": round(katt, 2), "peak": tf_peak, "unit": "TFLOP/s",
                         "frac": round(katt / tf_peak, 4), "peak_source": peak_src,
                         "kernel_ms": round(kms, 4)}}


def run_mlra(args, device):
    """One MLRA decode layer step (latent projection with the cache append,
    split-KV attention over the L latent sub-heads, output projection) on
    the MLRA workload: 128 sequences, cache length 8192, L = 4 sub-heads of
    rank 256.  The 2.1 GB cache is larger than L2, so steps need no flush."""
    import torch
    import head_latent_attention_gb300 as mla
    hbm_peak, tf_peak, tf_sust, peak_src = peaks()
    w = MLRA
    B = w.batch
    lens = syn.lengths(w)
    lay = build_layer(w, device, B, w.seq, B, 0)
    for b in range(B):
        ls, _ = syn.cache_rows(w, b, int(lens[b]))
        lay.cache_lat[b, :lens[b]] = to_dev(ls, device)
    xs, _ = syn.activations(w, B)
    x = to_dev(xs, device)
    seq = torch.arange(B, dtype=torch.int32, device=device)
    pos = torch.from_numpy(lens - 1).to(device)
    sl = torch.from_numpy(lens).to(device)
    stream = torch.cuda.current_stream()

    def step():
        qn, _ = lay.project_latent(x, seq, pos)
        o = lay.decode(qn, None, sl)
        return lay.out_proj(o)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    K = args.mlra_steps
    ev = timing_events(K)
    kev = timing_events(K)
    for i in range(K):
        mla.mla_set_profile_events(mla.MLA_PROFILE_DECODE_ATTENTION, kev[i][0], kev[i][1])
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    mla.mla_set_profile_events(mla.MLA_PROFILE_DECODE_ATTENTION, None, None)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = sum(step_ms) / K
    kms = sum(a.elapsed_time(b) for a, b in kev) / K
    nbytes = int(np.sum(lens)) * w.r_kv * 2
    del lay
    torch.cuda.empty_cache()
    return {"workload": "mlra_decode", "batch": B, "cache_len": int(lens[0]), "latent_heads": w.n_latent_heads,
            "steps": K, "ms_per_step": round(ms, 4), "step_ms": spread(step_ms),
            "value": round(nbytes / (ms * 1e-3) / 1e9, 2),
            "unit": "GB/s", "cache_bytes_per_step": nbytes, "l2": "cache 2.1 GB > L2, no flush",
            "roofline": {"bound": "hbm", "kernel": "MLRA split-KV latent attention",
                         "achieved": round(nbytes / (kms * 1e-3) / 1e9, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(nbytes / (kms * 1e-3) / 1e9 / hbm_peak, 4), "peak_source": peak_src,
                         "kernel_ms": round(kms, 4)}}


def run_small_decode(args, device):
    """One small-LM decode layer step (latent projection with the cache
    append, the per-step decompression of each sequence's cached rows into
    keys (rotated) and values, causal attention of the one new query, output
    projection): 8 sequences, lengths ~ U[512, 1024].  RoPE sits between W_UK
    and the query in this form, so nothing can be absorbed; the decompression
    covers each sequence's rows up to its length.  Graph-captured, L2 flushed
    between steps."""
    import torch
    import head_latent_attention_gb300 as mla
    hbm_peak, tf_peak, tf_sust, peak_src = peaks()
    w = syn.WORKLOADS["small_lm_decode"]
    B = w.batch
    lens = syn.lengths(w)
    lay = build_layer(w, device, B, w.seq, B, w.seq)
    for b in range(B):
        ls, _ = syn.cache_rows(w, b, int(lens[b]))
        lay.cache_lat[b, :lens[b]] = to_dev(ls, device)
    xs, _ = syn.activations(w, B)
    x = to_dev(xs, device)
    seq = torch.arange(B, dtype=torch.int32, device=device)
    pos = torch.from_numpy(lens - 1).to(device)
    sl = torch.from_numpy(lens).to(device)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    dt = torch.bfloat16
    qn = torch.empty(B, w.n_heads, w.d_nope, dtype=dt, device=device)
    o = torch.empty(B, w.n_heads, w.d_v, dtype=dt, device=device)
    y = torch.empty(B, w.d_model, dtype=dt, device=device)

    def check(st, what):
        if st != mla.MLA_OK:
            raise mla.MlaError(st, what)

    def step():
        check(mla.mla_project_latent(lay.h, lay.w, x, seq, pos, lay.cache, qn, None, lay.ws), "mla_project_latent")
        check(mla.mla_decode(lay.h, lay.w, qn, None, lay.cache, sl, B, o, lay.ws), "mla_decode")
        check(mla.mla_out_proj(lay.h, lay.w, o.view(B, -1), y, lay.ws), "mla_out_proj")

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        g.replay()
    torch.cuda.synchronize()
    K = max(args.steps, 1)
    ev = timing_events(K)
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        g.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = sum(step_ms) / K
    rows = int(np.sum(lens))
    cache_bytes = rows * w.r_kv * 2
    # Bytes the step must move in this form: the cached rows read, their keys
    # and values (fp16) written and read back once, and the weights.
    kv_bytes = rows * 2 * w.n_heads * w.d_nope * 2
    weights = sum(int(np.prod(s)) for s in syn.weight_shapes(w).values()) * 2
    all_bytes = cache_bytes + 2 * kv_bytes + weights
    del lay, g
    torch.cuda.empty_cache()
    return {"workload": "small_lm_decode", "batch": B, "cache_len": "U[512,1024] seed 0", "sum_len": rows,
            "steps": K, "ms_per_step": round(ms, 5), "step_ms": spread(step_ms),
            "value": round(cache_bytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "cache_bytes_per_step": cache_bytes,
            "l2": "flushed between steps (512 MiB write, outside the step events)",
            "roofline": {"bound": "hbm", "kernel": "whole decode step (latency-bound at this size)",
                         "bytes": all_bytes,
                         "bytes_are": "cache rows + fp16 keys/values written and read back + weights",
                         "achieved": round(all_bytes / (ms * 1e-3) / 1e9, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(all_bytes / (ms * 1e-3) / 1e9 / hbm_peak, 4), "peak_source": peak_src}}


def cca_flops(w):
    """FLOPs of one CCA / CCGQA forward as the page computes it: the
    down-projections, both convolutions, causal attention in the latent
    (exact causal pairs) and the output projection."""
    T = w.batch * w.seq
    P = w.q_latent + w.kv_latent
    proj = 2.0 * T * w.d_model * (P + w.kv_latent) + 2.0 * T * w.q_latent * w.d_model
    conv = (2.0 * T * P * w.conv_kernel_seq if w.conv_layers >= 1 else 0.0) + \
           (2.0 * T * P * w.d_h * w.conv_kernel_ch if w.conv_layers >= 2 else 0.0)
    attn = w.batch * w.n_heads * (w.seq * (w.seq + 1) / 2) * 2 * (2 * w.d_h)
    return proj + conv + attn, attn


def run_cca(args, device, name):
    """One CCA / CCGQA layer forward (compressed convolutional attention,
    the layer on the same pages): 4 sequences of 2048 tokens, d_model 2048.
    Graph-captured; the attention kernel's events in a second graph."""
    import torch
    import head_latent_attention_gb300 as mla
    hbm_peak, tf_peak, tf_sust, peak_src = peaks()
    w = syn.CCA_WORKLOADS[name]
    cfg = mla.make_cca_config(w.d_model, w.n_heads, w.n_kv_heads, w.q_latent, w.kv_latent, w.conv_layers,
                              w.conv_kernel_seq, w.conv_kernel_ch, w.qk_mean, w.value_shift, w.rope_base,
                              w.key_temp, w.seq)
    lay = mla.CcaLayer(cfg, {k: to_dev(s, device) for k, (s, _) in syn.cca_weights(w).items()}, w.batch,
                       device=device)
    xs, _ = syn.cca_activations(w, w.batch * w.seq)
    x = to_dev(xs, device).view(w.batch, w.seq, w.d_model)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream()

    def step():
        st = mla.mla_cca_forward(lay.h, lay.w, x, w.batch, w.seq, y, lay.ws)
        if st != mla.MLA_OK:
            raise mla.MlaError(st, "mla_cca_forward")

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    kb, ke = timing_events(1)[0]
    mla.mla_set_profile_events(mla.MLA_PROFILE_PREFILL_ATTENTION, kb, ke)
    g_k = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_k):
        step()
    mla.mla_set_profile_events(mla.MLA_PROFILE_PREFILL_ATTENTION, None, None)
    for _ in range(3):
        g.replay()
        g_k.replay()
    torch.cuda.synchronize()
    K = max(args.prefill_steps, 1)
    ev = timing_events(K)
    kern_ms = []
    for i in range(K):
        ev[i][0].record(stream)
        g.replay()
        ev[i][1].record(stream)
        g_k.replay()
        ke.synchronize()
        kern_ms.append(kb.elapsed_time(ke))
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms, kms = sum(step_ms) / K, sum(kern_ms) / K
    total, attn = cca_flops(w)
    del lay, g, g_k
    torch.cuda.empty_cache()
    return {"workload": name, "batch": w.batch, "seq": w.seq, "heads": w.n_heads, "kv_heads": w.n_kv_heads,
            "d_h": w.d_h, "steps": K, "ms_per_step": round(ms, 4), "step_ms": spread(step_ms),
            "tflops": round(total / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "flops_per_step": total,
            "frac_of_bf16_peak": round(total / (ms * 1e-3) / 1e12 / tf_peak, 4),
            "roofline": {"bound": "tensor", "kernel": "causal flash attention in the latent",
                         "achieved": round(attn / (kms * 1e-3) / 1e12, 2), "peak": tf_peak, "unit": "TFLOP/s",
                         "frac": round(attn / (kms * 1e-3) / 1e12 / tf_peak, 4), "peak_source": peak_src,
                         "kernel_ms": round(kms, 4)}}


def run_mlra_tp(args, rank, world, device):
    """MLRA decode layer step with latent sub-head tensor parallelism across
    the ranks (mlra_attn module docstring: each device loads 1/L of the KV
    cache): rank s holds latent blocks [s L/n, (s+1) L/n), the heads that read
    them and the matching columns of W_O; its step appends its latent columns,
    attends with its heads and projects them, and one all-reduce (sum) of the
    partial outputs [B, d_model] over NCCL gives the layer's output.  Runs
    when the number of ranks divides L (= 4); the whole job reads the cache
    once per step."""
    import torch
    import torch.distributed as dist
    import head_latent_attention_gb300 as mla
    from head_latent_attention_gb300 import mlra_tp
    w = MLRA
    if w.n_latent_heads % world or w.n_heads % world:
        return {"workload": "mlra_decode", "n_shards": world,
                "skipped": f"{world} ranks do not divide L = {w.n_latent_heads} latent blocks"}
    B = w.batch
    lens = syn.lengths(w)
    cfg = mla.make_config(w.variant, w.dtype, w.d_model, w.n_heads, w.d_nope, w.d_rope, w.d_v, w.r_kv,
                          w.r_q, w.n_latent_heads, w.rope_base, B, w.seq)
    full = {k: to_dev(s, device) for k, (s, _) in syn.weights(w).items()}
    lay = mla.MlaLayer(cfg, mlra_tp.shard_weights(full, cfg, rank, world), B, device=device, ws_max_len=0,
                       shard=(rank, world))
    del full
    cols = mlra_tp.shard_cache_columns(cfg, rank, world)
    for b in range(B):
        ls, _ = syn.cache_rows(w, b, int(lens[b]))
        lay.cache_lat[b, :lens[b]] = to_dev(np.ascontiguousarray(ls[:, cols]), device)
    xs, _ = syn.activations(w, B)
    x = to_dev(xs, device)
    seq = torch.arange(B, dtype=torch.int32, device=device)
    pos = torch.from_numpy(lens - 1).to(device)
    sl = torch.from_numpy(lens).to(device)
    stream = torch.cuda.current_stream()

    def step():
        qn, _ = lay.project_latent(x, seq, pos)
        o = lay.decode(qn, None, sl)
        return mlra_tp.all_reduce_partial(lay.out_proj(o))

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    dist.barrier()
    K = args.mlra_steps
    ev = timing_events(K)
    for i in range(K):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks([sum(step_ms) / K], world, device)[0]
    nbytes = int(np.sum(lens)) * w.r_kv * 2  # the whole job's cache bytes per step
    del lay
    torch.cuda.empty_cache()
    return {"workload": "mlra_decode", "n_shards": world, "batch": B, "cache_len": int(lens[0]),
            "steps": K, "ms_per_step": round(ms, 4), "step_ms": spread(step_ms),
            "value": round(nbytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "cache_bytes_per_step": nbytes, "cache_bytes_per_gpu": nbytes // world,
            "collective": "NCCL all-reduce (sum) of the bf16 partial outputs [B, d_model] per step"}


# ---------------------------------------------------------------------------
# CPU baseline: the fp64 oracle on a bounded sample of the decode workload
# ---------------------------------------------------------------------------

def oracle_decode_sample(bs, lens, Wx, n_threads):
    import oracle
    w = DECODE
    xs, xe = syn.activations(w, w.batch)
    lat = np.zeros((len(bs), int(max(lens[b] for b in bs)), w.r_kv))
    rope = np.zeros((len(bs), lat.shape[1], w.d_rope))
    for i, b in enumerate(bs):
        lat[i, :lens[b]] = syn.cache_rows(w, b, int(lens[b]))[1]
        rope[i, :lens[b]] = syn.cache_rows(w, b, int(lens[b]), "cache_rope")[1]
    sub = w.replace(seq=lat.shape[1])
    t0 = time.perf_counter()
    oracle.decode(sub, xe[bs], np.asarray([lens[b] for b in bs], np.int32), lat, rope, Wx,
                  absorbed=True, n_threads=n_threads)
    return time.perf_counter() - t0


def cpu_baseline(args):
    import oracle
    oracle.build()
    n_threads = os.cpu_count() or 1
    w = DECODE
    lens = syn.lengths(w)
    Wx = {k: e for k, (_, e) in syn.weights(w).items()}
    done, secs, bs = 0, 0.0, []
    for b in range(w.batch):
        secs += oracle_decode_sample([b], lens, Wx, n_threads)
        bs.append(b)
        if secs >= args.cpu_seconds:
            break
    nbytes = decode_bytes(lens[bs])
    # The same oracle on one thread, over the shortest sequences until about
    # a third of the budget is spent.
    order = [int(b) for b in np.argsort(lens, kind="stable")]
    secs1, bs1 = 0.0, []
    for b in order:
        secs1 += oracle_decode_sample([b], lens, Wx, 1)
        bs1.append(b)
        if secs1 >= args.cpu_seconds / 3:
            break
    nbytes1 = decode_bytes(lens[bs1])
    return {"value": round(nbytes / secs / 1e9, 5), "unit": "GB/s", "cores": n_threads,
            "kind": "oracle",
            "sample": f"oracle decode step (projection, absorbed attention, W_UV, W_O; fp64) "
                      f"for sequences 0..{len(bs) - 1} of the dsv2_decode workload "
                      f"({int(np.sum(lens[bs]))} cached tokens, {secs:.1f} s)",
            "single_thread": {"value": round(nbytes1 / secs1 / 1e9, 6), "unit": "GB/s", "cores": 1,
                              "sample": f"the same oracle step on one thread for the {len(bs1)} shortest "
                                        f"sequences ({int(np.sum(lens[bs1]))} cached tokens, {secs1:.1f} s)"}}


def run_reference(args):
    """The oracle as the reference arm: each step is one sequence of the decode
    workload run through the fp64 oracle on the host cores."""
    import oracle
    oracle.build()
    n_threads = os.cpu_count() or 1
    w = DECODE
    lens = syn.lengths(w)
    Wx = {k: e for k, (_, e) in syn.weights(w).items()}
    for i in range(args.warmup):
        oracle_decode_sample([i % w.batch], lens, Wx, n_threads)
    secs, nbytes = 0.0, 0
    for i in range(args.steps):
        b = (args.warmup + i) % w.batch
        secs += oracle_decode_sample([b], lens, Wx, n_threads)
        nbytes += decode_bytes(lens[[b]])
    v = nbytes / secs / 1e9
    sample = (f"each step: one sequence of dsv2_decode through the fp64 oracle decode step "
              f"(sequences {args.warmup % w.batch}.., {nbytes // 1152} cached tokens over "
              f"{args.steps} steps)")
    return {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "dsv2_decode", "batch": w.batch,
                       "cache_len": "U[1024,4096] seed 0"},
            "cpu_baseline": {"value": round(v, 6), "unit": "GB/s", "cores": n_threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--prefill-steps", type=int, default=20)
    ap.add_argument("--no-prefill", dest="prefill", action="store_false")
    ap.add_argument("--no-mlra", dest="mlra", action="store_false")
    ap.add_argument("--no-small", dest="small", action="store_false")
    ap.add_argument("--no-cca", dest="cca", action="store_false")
    ap.add_argument("--mlra-steps", type=int, default=5)
    ap.add_argument("--mlra-only", action="store_true", help="time only the MLRA decode layer (profiling aid)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the prefill layer (profiling aid)")
    ap.add_argument("--prefill-batch", type=int, default=0,
                    help="sequences in the prefill workload (default 4)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch
    import torch.distributed as dist
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(device))
    if args.prefill_only or args.mlra_only:
        from head_latent_attention_gb300 import _build
        _build.build()
        out = run_prefill(args, device) if args.prefill_only else run_mlra(args, device)
        if rank == 0:
            print(json.dumps(out), flush=True)
        return
    out = run_ours(args, rank, world, device)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
