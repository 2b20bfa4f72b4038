#!/usr/bin/env python3
"""Benchmark of the MLA latent-cache decode hot path on GB300.

One *step* is one pass of the whole hot path for one attention layer: RoPE of
the new query's rope part, absorption of q_nope through W_UK, latent attention
over the cache (split-K flash decode + combine) and the W_UV projection.
Consecutive steps use the buffers (cache, weights, queries) of R distinct
layers whose total size exceeds the 129 MB L2, so no step finds its inputs in
L2 from the step before.

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle on the same workload instead (the reference arm).  ``--workload`` picks
another of the five workloads (default: dense bf16, B=1, T=4096).
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
sys.path.insert(0, ROOT)

METRIC = "MLA decode tokens/s and latent-cache HBM GB/s (% of GB300 roofline)"
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one decode +
# combine launch pair of the current kernels, from an ncu capture of this
# bench (cold caches between launches, so the split partials' round trip,
# 4.2 MB at B=1, is counted as a DRAM re-read that a warm L2 serves).
MEASURED_TRAFFIC = {"dense_bf16_b1_t4096_h128": 4952320 + 4226304}
L2_BYTES = 129 * 2 ** 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dense_bf16",
                    choices=["tiny_f32", "dense_bf16", "ragged_bf16", "sparse_bf16", "verify_bf16",
                             "verify_sparse_bf16"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args()


def workload(name):
    from mla_latent_kv_12_gb300 import workloads as W
    return {"tiny_f32": W.TINY_F32, "dense_bf16": W.DENSE_BF16, "ragged_bf16": W.RAGGED_BF16,
            "sparse_bf16": W.SPARSE_BF16, "verify_bf16": W.VERIFY_BF16,
            "verify_sparse_bf16": W.VERIFY_SPARSE_BF16}[name]


def layout_of(w):
    return "flat" if w.ragged else "padded"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), \
            d.get("bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def algorithmic(inp, with_sel=True):
    """(cache bytes, flops) of one decode launch: every visited (key, query row)
    reads one latent||rope row once per batch row and costs 2*H*(rank+rope+rank) flops."""
    w = inp.w
    esize = 4 if w.dtype == "f32" else 2
    row_bytes = (w.rank + w.rope) * esize
    if inp.sel is not None and with_sel:
        cnt = inp.sel_count.clamp(min=0)
        keys_rows = int(cnt.sum())                      # each (row, token) gathers its own rows
        byts = keys_rows * row_bytes + int(cnt.numel()) * 0 + keys_rows * 4
        visits = keys_rows
    else:
        byts = int(inp.kv_len.sum()) * row_bytes       # one pass over each batch row's window
        visits = 0
        for b in range(w.batch):
            for i in range(w.s_q):
                visits += max(int(inp.kv_len[b]) - w.s_q + i + 1, 0)
    flops = visits * 2 * w.heads * (w.rank + w.rope + w.rank)
    return byts, flops


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for s in self.samples for k in range(4)
                          if len(s) > 4 + k and s[4 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.samples)}


def max_over_ranks(x: float, device) -> float:
    """The largest value of ``x`` over all ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def time_oracle(inp, seconds, heads_per_row=None):
    """Times the float64 oracle (rotations + reconstructed attention) on whole
    query rows, or on ``heads_per_row`` heads of each row, until ~``seconds``
    of CPU work.  Returns (tokens/s scaled to whole rows, units done, elapsed,
    threads)."""
    from tests import helpers as H
    w = inp.w
    hs = None if heads_per_row is None else list(range(min(heads_per_row, w.heads)))
    frac = 1.0 if hs is None else len(hs) / w.heads
    t0 = time.perf_counter()
    done = 0
    while True:
        H.oracle_reference_out_only(inp, rows=[done % w.n_q], heads=hs)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds or done >= 64:
            break
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return done * frac / el, done, el, threads


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from mla_latent_kv_12_gb300 import workloads as W
    w = workload(args.workload)
    inp = W.make_inputs(w, layout=layout_of(w))
    # Each step: one query row of the workload on a fixed subset of heads (the
    # oracle's cost is linear in heads), so that K + W steps take minutes.
    heads = 8 if w.heads >= 64 else None
    rates = []
    threads = 1
    for k in range(args.warmup + args.steps):
        v, done, el, threads = time_oracle(inp, 0.0, heads_per_row=heads)
        if k >= args.warmup:
            rates.append(el / done)
    sec_per_unit = statistics.mean(rates)
    frac = 1.0 if heads is None else heads / w.heads
    value = frac / sec_per_unit
    sec_per_row = sec_per_unit / frac
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec_per_row * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "layers": 1, "l2": "cpu"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step one query row of {w.name} on {heads or w.heads} of "
                                   f"{w.heads} heads (scaled to whole rows), float64 "
                                   "reconstructed-path oracle (numpy BLAS)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from mla_latent_kv_12_gb300 import mla
    from mla_latent_kv_12_gb300 import workloads as W
    from mla_latent_kv_12_gb300.pipeline import DecodeStep

    w = workload(args.workload)
    inp = W.make_inputs(w, layout=layout_of(w))
    one = DecodeStep(inp, dev)
    layer_bytes = (one.latent.numel() + one.rope.numel() + one.kv_b_proj.numel()) * one.latent.element_size()
    R = max(1, min(16, -(-2 * L2_BYTES // layer_bytes)))
    steps = [one] + [DecodeStep(inp, dev) for _ in range(R - 1)]
    stream = torch.cuda.current_stream()

    # One CUDA graph per layer for the whole step, and one for its decode launches
    # (planner + decode + combine) to time the dominant kernel without host gaps.
    for s in steps:
        s.run()
        if s.fused:      # the decode-only graphs read the absorbed query of the separate entry points
            s.rope_q()
            s.absorb()
    torch.cuda.synchronize()
    g_step, g_att = [], []
    cap = torch.cuda.Stream()
    with torch.cuda.stream(cap):
        for s in steps:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                s.run()
            g_step.append(g)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                s.attend()
            g_att.append(g)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    for k in range(args.warmup):
        g_step[k % R].replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_dec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        start.record(stream)
        for k in range(args.steps):
            g_step[k % R].replay()
        stop.record(stream)
        torch.cuda.synchronize()
        # the decode launches alone, same layer rotation, bracketed one by one
        for k in range(args.steps):
            ev_dec[k][0].record(stream)
            g_att[k % R].replay()
            ev_dec[k][1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms_total = max_over_ranks(start.elapsed_time(stop), dev)
    ms_step = ms_total / args.steps
    dec_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_dec)
    tokens = w.n_q * args.steps * world
    value = tokens / (ms_total / 1e3)

    # end to end: pinned host query in, host result out, every step
    e2e_steps = max(10, args.steps // 4)
    hq = [inp.q_nope.reshape(w.n_q, w.heads, w.nope).pin_memory(), inp.q_rope_raw.pin_memory()]
    hout = torch.empty(one.out.shape, dtype=one.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in hq)
    d2h = hout.numel() * hout.element_size()
    def e2e_step(s):
        s.q_nope.copy_(hq[0], non_blocking=True)
        s.q_rope_raw.copy_(hq[1], non_blocking=True)
        s.run()
        hout.copy_(s.out, non_blocking=True)
    for k in range(3):
        e2e_step(steps[k % R])
    torch.cuda.synchronize()
    # one CUDA graph per layer holding the host->device copies, the step's
    # launches and the device->host copy, as a serving loop would replay it
    g_e2e = []
    with torch.cuda.stream(cap):
        for s in steps:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                e2e_step(s)
            g_e2e.append(g)
    for k in range(3):
        g_e2e[k % R].replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(e2e_steps):
        g_e2e[k % R].replay()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_value = w.n_q * world / (e2e_ms / 1e3)

    # the cache append of the page's forward (RMSNorm + RoPE of one new token per
    # batch row), timed alone over a scratch cache: one launch per call
    ap_lat = torch.zeros(w.batch, 4, w.rank, dtype=one.dtype, device=dev)
    ap_rope = torch.zeros(w.batch, 4, w.rope, dtype=one.dtype, device=dev)
    ap_len = torch.zeros(w.batch, dtype=torch.int32, device=dev)
    ap_in = inp.latent[:, :1].reshape(w.batch if inp.latent.shape[0] == w.batch else 1, 1, w.rank)
    ap_in = ap_in.expand(w.batch, 1, w.rank).contiguous().to(dev)
    ap_rin = torch.randn(w.batch, 1, w.rope, device=dev).to(one.dtype)
    ap_w = torch.ones(w.rank, dtype=one.dtype, device=dev)
    ap_per_graph, ap_reps = 20, 10
    for _ in range(3):
        mla.append_compressed(ap_in, ap_rin, ap_w, 1e-6, w.theta, ap_lat, ap_rope, None, ap_len)
    torch.cuda.synchronize()
    g_ap = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g_ap, stream=cap):
            for _ in range(ap_per_graph):
                mla.append_compressed(ap_in, ap_rin, ap_w, 1e-6, w.theta, ap_lat, ap_rope, None, ap_len)
    g_ap.replay()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(ap_reps):
        g_ap.replay()
    a1.record(stream)
    torch.cuda.synchronize()
    append_us = a0.elapsed_time(a1) / (ap_per_graph * ap_reps) * 1e3
    ap_bytes = w.batch * (w.rank + w.rope) * one.latent.element_size() * 2

    # the DSA top-k selection (2048 positions per query row from f32 scores over
    # the row's window), timed alone: 10 calls per CUDA graph, replayed
    sel_k = 2048
    sel_len = inp.kv_len.repeat_interleave(w.s_q).to(torch.int32).to(dev)
    sel_scores = torch.randn(w.n_q, int(inp.kv_len.max()), device=dev)
    sel_out = torch.empty(w.n_q, sel_k, dtype=torch.int32, device=dev)
    sel_cnt = torch.empty(w.n_q, dtype=torch.int32, device=dev)
    for _ in range(3):
        mla.select_topk(sel_scores, sel_len, sel_k, sel_out, sel_cnt)
    torch.cuda.synchronize()
    g_sel = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g_sel, stream=cap):
            for _ in range(10):
                mla.select_topk(sel_scores, sel_len, sel_k, sel_out, sel_cnt)
    g_sel.replay()
    torch.cuda.synchronize()
    a0.record(stream)
    for _ in range(5):
        g_sel.replay()
    a1.record(stream)
    torch.cuda.synchronize()
    select_us = a0.elapsed_time(a1) / 50 * 1e3
    sel_bytes = int(inp.kv_len.repeat_interleave(w.s_q).sum()) * 4

    # the speculative-round rollback of a right-aligned cache (8 rows x 65536
    # tokens of latent || rope, the verify batch's cache): one row-gather launch
    # per state array, 2 x 0.6 GB moved per call, larger than L2
    rb_B, rb_W = 8, 65536
    rb_lat = torch.randn(rb_B, rb_W, w.rank, device=dev).to(one.dtype)
    rb_rope = torch.randn(rb_B, rb_W, w.rope, device=dev).to(one.dtype)
    rb_off = np.full(rb_B, rb_W - 7)
    rb_off[::2] = rb_W                                     # half the rows fill the width
    rb_keep = np.arange(rb_B) % 5                          # 0..4 of 4 appended tokens kept (4 = all)
    rb_keep = np.minimum(rb_keep, 4)
    rb_shift, _, _, rb_w = mla.plan_rollback(rb_W - rb_off, rb_off, rb_off - 4, rb_keep, rb_W)
    rb_shift = rb_shift.to(dev)
    rb_dst = [torch.empty(rb_B, rb_w, a.shape[2], dtype=a.dtype, device=dev) for a in (rb_lat, rb_rope)]

    def rollback_call():
        for a, d in zip((rb_lat, rb_rope), rb_dst):
            mla.cache_shift_rows(a, d, shift=rb_shift)
    for _ in range(3):
        rollback_call()
    torch.cuda.synchronize()
    g_rb = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g_rb, stream=cap):
            for _ in range(5):
                rollback_call()
    g_rb.replay()
    torch.cuda.synchronize()
    a0.record(stream)
    for _ in range(4):
        g_rb.replay()
    a1.record(stream)
    torch.cuda.synchronize()
    rollback_us = a0.elapsed_time(a1) / 20 * 1e3
    rb_bytes = 2 * rb_B * rb_w * (w.rank + w.rope) * rb_lat.element_size()
    del rb_lat, rb_rope, rb_dst

    # the reconstructed prefill of a 4096-token prompt (RoPE of the query rope
    # part, per-head K/V materialisation, causal attention), three launches per
    # step, each part also timed alone; CUDA graphs of 3 steps, replayed
    from mla_latent_kv_12_gb300.pipeline import PrefillStep
    pf = PrefillStep(W.make_inputs(W.PREFILL_BF16), dev)

    def graph_us(fn, per_graph=3, reps=3):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for _ in range(per_graph):
                    fn()
        g.replay()
        torch.cuda.synchronize()
        a0.record(stream)
        for _ in range(reps):
            g.replay()
        a1.record(stream)
        torch.cuda.synchronize()
        return a0.elapsed_time(a1) / (per_graph * reps) * 1e3

    pf_step_us = graph_us(pf.run)
    pf_att_us = graph_us(pf.attend)
    pf_rec_us = graph_us(pf.reconstruct)
    pf_rope_us = graph_us(pf.rope_q)
    pfw = pf.w
    pf_pairs = sum(max(int(pf.inp.kv_len[b]) - pfw.s_q + i + 1, 0) for b in range(pfw.batch) for i in range(pfw.s_q))
    pf_att_flops = pf_pairs * 2 * pfw.heads * (pfw.nope + pfw.rope + pfw.v)
    pf_rec_flops = 2 * pf.latent.shape[0] * pf.latent.shape[1] * pfw.rank * pfw.heads * (pfw.nope + pfw.v)
    pf_status = int(pf.status.item())
    del pf

    hbm, tf_burst, tf_sus, src = load_peaks()
    byts, flops = algorithmic(inp)
    ach_gbs = byts / (dec_ms / 1e3) / 1e9
    ach_tf = flops / (dec_ms / 1e3) / 1e12
    mem_bound = (byts / hbm) >= (flops / 1e3 / tf_burst)
    roof = ({"bound": "hbm", "achieved": ach_gbs, "peak": hbm, "unit": "GB/s", "frac": ach_gbs / hbm}
            if mem_bound else
            {"bound": "tensor", "achieved": ach_tf, "peak": tf_burst, "unit": "TFLOP/s",
             "frac": ach_tf / tf_burst})
    roof.update({"traffic": MEASURED_TRAFFIC.get(w.name), "kernel": "mla_decode_attend (decode + combine)",
                 "peak_source": src, "algorithmic_bytes": byts, "algorithmic_flops": flops,
                 "kernel_ms": dec_ms, "tensor_tflops": ach_tf, "cache_gbs": ach_gbs})

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, done, el, threads = time_oracle(inp, args.cpu_seconds)
        cpu = {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{done} query rows (all heads) of {w.name}, float64 reconstructed-path "
                         f"oracle, {el:.1f} s"}
    kind = mla.decode_kernel_kind(w.heads, w.rank, w.rope, one.dtype, one.dtype)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "s_q": w.s_q, "heads": w.heads,
                   "rank": w.rank, "rope": w.rope, "layers": 1,
                   "l2": f"rotating {R} layers' buffers ({R * layer_bytes / 2**20:.0f} MiB > L2)",
                   "decode_kernel": "tcgen05" if kind == 1 else "cuda-core",
                   "parallelism": f"replicas{world}"},
        "clocks": clk.summary(),
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "timing": "CUDA graph per layer: host->device copies of the query, the step's launches, "
                          "device->host copy of the output; replayed"},
        "gpu_launches": one.launches_per_step() * args.steps,
        "timing": "CUDA graph per layer step, replayed; decode kernel timed on its own graph replays",
        "roofline": roof,
        "cpu_baseline": cpu,
        "cache_gbs": ach_gbs,
        "append": {"us_per_call": append_us, "tokens_per_call": w.batch, "bytes_per_call": ap_bytes,
                   "note": "mla_append_compressed (RMSNorm + RoPE of one new token per batch row), "
                           "20 calls per CUDA graph, replayed"},
        "select_topk": {"us_per_call": select_us, "rows": w.n_q, "top_k": sel_k, "score_bytes": sel_bytes,
                        "note": "mla_select_topk over f32 scores of each query row's window, "
                                "10 calls per CUDA graph, replayed"},
        "prefill": {"workload": W.PREFILL_BF16.name, "us_per_step": pf_step_us,
                    "tokens_per_s": pfw.n_q / (pf_step_us * 1e-6),
                    "attention_us": pf_att_us, "attention_tflops": pf_att_flops / (pf_att_us * 1e-6) / 1e12,
                    "attention_frac_of_measured_bf16_burst": pf_att_flops / (pf_att_us * 1e-6) / 1e12 / tf_burst,
                    "reconstruct_us": pf_rec_us,
                    "reconstruct_tflops": pf_rec_flops / (pf_rec_us * 1e-6) / 1e12,
                    "rope_us": pf_rope_us, "device_status": pf_status,
                    "note": "mla_rope_partial_interleaved + mla_reconstruct_kv + mla_prefill_attend; attention "
                            "flops = causal (query, key) pairs x 2 x H x (nope + rope + v); 3 steps per CUDA "
                            "graph, replayed"},
        "rollback": {"us_per_call": rollback_us, "bytes_per_call": rb_bytes,
                     "gbs": rb_bytes / (rollback_us * 1e-6) / 1e9,
                     "frac_of_measured_hbm": rb_bytes / (rollback_us * 1e-6) / 1e9 / hbm,
                     "note": "right-aligned rollback (mla_plan_rollback + two mla_cache_shift_rows) of "
                             "8 x 65536 tokens of latent || rope, read + write bytes, 5 calls per CUDA "
                             "graph, replayed"},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
