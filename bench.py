#!/usr/bin/env python3
"""Benchmark of the MLA latent-cache decode hot path on GB300.

One *step* is one pass of the whole hot path for one attention layer: RoPE of
the new query's rope part, absorption of q_nope through W_UK, latent attention
over the cache (split-K flash decode + combine) and the W_UV projection.
Consecutive steps use the buffers (cache, weights, queries) of R distinct
layers, R chosen so that the bytes one step touches, times R, exceed twice the
129 MB L2: no step finds its inputs in L2 from the step before.

The headline line is the batched ragged decode (B = 32 rows of U[1024, 32768]
cached keys, 128 heads), the largest one-token decode workload; ``per_config``
adds the other decode workloads (dense B = 1, sparse top-2048, multi-row
verify dense and sparse), each timed the same way.  ``--impl reference`` times
the float64 CPU oracle on the headline workload instead (the reference arm).
"""
from __future__ import annotations

import argparse
import dataclasses
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
# bench's workload; absent when the kernels changed after the capture.
MEASURED_TRAFFIC: dict = {"ragged_bf16_b32_len1k_32k_h128": 601_256_192}
L2_BYTES = 129 * 2 ** 20
WORKLOADS = ("tiny_f32", "dense_bf16", "ragged_bf16", "sparse_bf16", "verify_bf16", "verify_sparse_bf16")
HEADLINE = "ragged_bf16"
PER_CONFIG = ("dense_bf16", "ragged_bf16", "sparse_bf16", "verify_bf16", "verify_sparse_bf16")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=WORKLOADS)
    ap.add_argument("--no-per-config", action="store_true", help="time the headline workload only")
    ap.add_argument("--no-side", action="store_true", help="skip the append / top-k / rollback / prefill objects")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--layers", type=int, default=0,
                    help="rotate exactly this many layers' buffers (0: as many as flush the L2 between uses); "
                         "a smaller count keeps a profiler capture's device memory small")
    return ap.parse_args(argv)


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
        byts = keys_rows * row_bytes + keys_rows * 4    # rows + their indices
        visits = keys_rows
    else:
        byts = int(inp.kv_len.sum()) * row_bytes       # one pass over each batch row's window
        visits = 0
        for b in range(w.batch):
            for i in range(w.s_q):
                visits += max(int(inp.kv_len[b]) - w.s_q + i + 1, 0)
    flops = visits * 2 * w.heads * (w.rank + w.rope + w.rank)
    return byts, flops


def step_algorithmic(inp):
    """(bytes, flops) of the whole step: the decode's cache bytes and flops, plus
    W_UK and W_UV (read once each), the query in and the output out, and the
    absorb and projection flops."""
    w = inp.w
    esize = 4 if w.dtype == "f32" else 2
    byts, flops = algorithmic(inp)
    weights = w.heads * (w.nope + w.v) * w.rank * esize   # all of kv_b_proj: W_UK and W_UV once each
    q_in = w.n_q * w.heads * (w.nope + w.rope) * esize
    out = w.n_q * w.heads * w.v * esize
    flops += 2 * w.n_q * w.heads * w.rank * (w.nope + w.v)
    return byts + weights + q_in + out, flops


def roofline(byts, flops, seconds, hbm, tf_peak, src):
    """The benchmark spec's roofline: the slower of bytes at the HBM rate and flops at the bf16 rate."""
    ach_gbs = byts / seconds / 1e9
    ach_tf = flops / seconds / 1e12
    mem_bound = (byts / (hbm * 1e9)) >= (flops / (tf_peak * 1e12))
    if mem_bound:
        r = {"bound": "hbm", "achieved": ach_gbs, "peak": hbm, "unit": "GB/s", "frac": ach_gbs / hbm}
    else:
        r = {"bound": "tensor", "achieved": ach_tf, "peak": tf_peak, "unit": "TFLOP/s", "frac": ach_tf / tf_peak}
    r.update({"peak_source": src, "algorithmic_bytes": byts, "algorithmic_flops": flops,
              "seconds": seconds, "gbs": ach_gbs, "tflops": ach_tf})
    return r


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms while running."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.error = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError as e:
            self.proc = None
            self.error = str(e)
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 4 and parts[0].replace(".", "").isdigit():
                self.samples.append((time.perf_counter(), parts))

    def wait_samples(self, n, timeout=3.0, keep_busy=None):
        """Blocks until ``n`` samples have arrived (running ``keep_busy`` meanwhile)."""
        t0 = time.perf_counter()
        while self.proc is not None and len(self.samples) < n and time.perf_counter() - t0 < timeout:
            if keep_busy is not None:
                keep_busy()
            else:
                time.sleep(0.01)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, since=None):
        rows = [p for t, p in self.samples if since is None or t >= since]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0,
                    "error": self.error}
        sm = [float(s[0]) for s in rows]
        mx = [float(s[1]) for s in rows if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for s in rows for k in range(4)
                          if len(s) > 4 + k and s[4 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


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


# ---------------------------------------------------------------- the oracle on the host cores

def one_row_inputs(inp, b):
    """The inputs of batch row ``b`` alone (its window copied out, kv_start 0)."""
    import torch
    from mla_latent_kv_12_gb300.workloads import DecodeInputs
    w = inp.w
    bb = 0 if inp.packed_flat else b
    s, n = int(inp.kv_start[b]), int(inp.kv_len[b])
    w1 = dataclasses.replace(w, batch=1)
    rows = slice(b * w.s_q, (b + 1) * w.s_q)
    sel = inp.sel[rows].clone() if inp.sel is not None else None
    cnt = inp.sel_count[rows].clone() if inp.sel is not None else None
    return DecodeInputs(w1, inp.q_nope[b:b + 1].clone(), inp.q_rope_raw[b:b + 1].clone(),
                        inp.latent[bb:bb + 1, s:s + n].clone(), inp.rope_raw[bb:bb + 1, s:s + n].clone(),
                        inp.kv_b_proj, torch.zeros(1, dtype=torch.int32), torch.tensor([n], dtype=torch.int32),
                        inp.q_offset[b:b + 1].clone(), False, sel, cnt)


def _oracle_task(args):
    """One task of the host-core oracle pool: the reconstructed-path oracle for
    all query tokens of one batch row, on a subset of heads.  Returns seconds."""
    inp1, heads = args
    from tests import helpers as H
    t0 = time.perf_counter()
    H.oracle_reference_out_only(inp1, rows=list(range(inp1.w.s_q)), heads=heads)
    return time.perf_counter() - t0


class OraclePool:
    """The float64 oracle as it stands, run on the host cores by a pool of
    single-threaded processes (spawned, BLAS limited to one thread each), one
    task per (batch row, group of heads)."""

    def __init__(self, workers=None):
        import multiprocessing as mp
        self.workers = workers or (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                                   else os.cpu_count())
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(self.workers)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.pool.map(_oracle_task, [])            # workers up before any timing

    def run(self, inp, rows, heads_per_task):
        """Tokens/s equivalent of the oracle over ``rows`` batch rows, each cut
        into tasks of ``heads_per_task`` heads.  Returns (tokens, seconds)."""
        w = inp.w
        groups = [list(range(h, min(h + heads_per_task, w.heads))) for h in range(0, w.heads, heads_per_task)]
        tasks = [(one_row_inputs(inp, b), g) for b in rows for g in groups]
        t0 = time.perf_counter()
        self.pool.map(_oracle_task, tasks, chunksize=1)
        el = time.perf_counter() - t0
        return len(rows) * w.s_q, el

    def run_heads(self, inp, b, heads):
        """One batch row on the listed heads, one head per task."""
        inp1 = one_row_inputs(inp, b)
        t0 = time.perf_counter()
        self.pool.map(_oracle_task, [(inp1, [h]) for h in heads], chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.pool.terminate()
        self.pool.join()


def cpu_baseline(inp, seconds, pool):
    """The oracle on whole batch rows (all heads) until about ``seconds`` have passed."""
    w = inp.w
    heads_per_task = max(1, w.heads // pool.workers)
    done_tokens, el = 0, 0.0
    b = 0
    while el < seconds and b < w.batch:
        t, e = pool.run(inp, [b], heads_per_task)
        done_tokens += t
        el += e
        b += 1
    return {"value": done_tokens / el, "unit": "tokens/s", "cores": pool.workers, "kind": "oracle",
            "sample": f"{b} batch row(s) of {w.name} ({done_tokens} query tokens, all {w.heads} heads), "
                      f"float64 reconstructed-path oracle, {pool.workers} single-threaded processes "
                      f"(one per core, tasks of {heads_per_task} heads), {el:.1f} s"}


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from mla_latent_kv_12_gb300 import workloads as W
    w = workload(args.workload)
    inp = W.make_inputs(w, layout=layout_of(w))
    pool = OraclePool()
    # Each step: all query tokens of one batch row on one head per worker
    # (the oracle's cost is linear in heads), rows in turn.
    heads = list(range(min(pool.workers, w.heads)))
    times = []
    for k in range(args.warmup + args.steps):
        el = pool.run_heads(inp, k % w.batch, heads)
        if k >= args.warmup:
            times.append(el)
    pool.close()
    sec = statistics.mean(times)
    tokens = w.s_q * len(heads) / w.heads          # query tokens' worth of work per step
    value = tokens / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "layers": 1, "l2": "cpu"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": pool.workers, "kind": "oracle",
                         "sample": f"per step all {w.s_q} query token(s) of one batch row of {w.name} on "
                                   f"{len(heads)} of {w.heads} heads (one head per process, rows in turn); "
                                   f"value counts the work done ({tokens:.4g} tokens per step), float64 "
                                   "reconstructed-path oracle"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- the GPU arm

def layers_for(inp, step_bytes):
    """Distinct layers to rotate so that consecutive uses of one layer are
    separated by more than twice the L2 of other layers' bytes (one layer when
    a step alone touches that much)."""
    if step_bytes >= 2 * L2_BYTES:
        return 1
    return min(16, -(-2 * L2_BYTES // max(step_bytes, 1)) + 1)


def measure(w, steps, warmup, dev, world, peaks, e2e=False, clocks=None, layers=0):
    """Times the whole step and the decode launches of workload ``w`` on R
    rotating layers with CUDA-graph replays.  Returns a dict."""
    import torch
    from mla_latent_kv_12_gb300 import mla
    from mla_latent_kv_12_gb300 import workloads as W
    from mla_latent_kv_12_gb300.pipeline import DecodeStep

    hbm, tf_burst, _, src = peaks
    inp = W.make_inputs(w, layout=layout_of(w))
    byts, flops = algorithmic(inp)
    sbytes, sflops = step_algorithmic(inp)
    R = layers if layers > 0 else layers_for(inp, sbytes)
    steps_l = [DecodeStep(inp, dev) for _ in range(R)]
    one = steps_l[0]
    for s in steps_l:
        s.run()
        if s.fused:      # the decode-only graphs read the absorbed query of the separate entry points
            s.rope_q()
            s.absorb()
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    g_step, g_att = [], []
    with torch.cuda.stream(cap):
        for s in steps_l:
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
    for k in range(warmup):
        g_step[k % R].replay()
    kk = [warmup]

    def busy():
        g_step[kk[0] % R].replay()
        kk[0] += 1
        torch.cuda.synchronize()
    if clocks is not None:          # clocks sampled under this load, right before and during the timed region
        clocks.wait_samples(len(clocks.samples) + 3, keep_busy=busy)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    t_clk = time.perf_counter()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(steps):
        g_step[k % R].replay()
    stop.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms_total = max_over_ranks(start.elapsed_time(stop), dev)
    clk = clocks.summary(since=t_clk - 0.2) if clocks is not None else None
    # the decode launches alone (decode + combine, + planner), same layer rotation, one by one
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for k in range(steps):
        ev[k][0].record(stream)
        g_att[k % R].replay()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    dec_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    ms_step = ms_total / steps
    status = max(int(s.status.item()) for s in steps_l)
    res = {
        "workload": w.name, "batch": w.batch, "s_q": w.s_q, "heads": w.heads, "layers": R,
        "tokens_per_s": w.n_q * world / (ms_step / 1e3), "ms_per_step": ms_step, "kernel_ms": dec_ms,
        "cache_gbs": byts / (dec_ms / 1e3) / 1e9, "device_status": status,
        "step_launches": one.launches_per_step(), "decode_launches": one.attend_launches(),
        "roofline": roofline(byts, flops, dec_ms / 1e3, hbm, tf_burst, src),
        "step_roofline": roofline(sbytes, sflops, ms_step / 1e3, hbm, tf_burst, src),
        "kind": "tcgen05" if mla.decode_kernel_kind(w.heads, w.rank, w.rope, one.dtype, one.dtype) == 1
        else "cuda-core",
    }
    res["roofline"]["traffic"] = MEASURED_TRAFFIC.get(w.name)
    res["roofline"]["kernel"] = "mla_decode_attend (decode + combine)"
    res["step_roofline"]["note"] = ("whole step: cache bytes + W_UK + W_UV + query in + output out, "
                                    "absorb + attention + projection flops")
    if clk is not None:
        res["clocks"] = clk
    if e2e:
        res["e2e"] = measure_e2e(steps_l, inp, steps, cap, stream, world, dev)
    res["_inp"] = inp
    res["_steps"] = steps_l
    res["_cap"] = cap
    return res


E2E_GRAPH_STEPS = 8   # steps per captured graph of the end-to-end leg


def measure_e2e(steps_l, inp, steps, cap, stream, world, dev):
    """The same step through the public API with the query copied in from pinned
    host memory and the output copied back, every step, as a serving loop runs
    it: two sets of device buffers (layers) in turn, the query copy of step k+1
    and the output copy of step k-1 on their own streams, overlapping step k's
    launches.  One CUDA graph holds E2E_GRAPH_STEPS such steps; successive
    replays of it do not overlap, so one step in E2E_GRAPH_STEPS pays its
    copies in full."""
    import torch
    from mla_latent_kv_12_gb300.pipeline import DecodeStep
    w = inp.w
    objs = list(steps_l)
    if len(objs) < 2:                     # a second buffer set for the copies to land in
        extra = DecodeStep(inp, dev)
        extra.run()
        objs.append(extra)
    nb = len(objs)
    hq = [inp.q_nope.reshape(w.n_q, w.heads, w.nope).pin_memory(), inp.q_rope_raw.pin_memory()]
    hout = [torch.empty(objs[0].out.shape, dtype=objs[0].out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in hq)
    d2h = hout[0].numel() * hout[0].element_size()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()

    def body():
        """E2E_GRAPH_STEPS steps; object j % nb serves step j."""
        done = [None] * E2E_GRAPH_STEPS      # step j's launches completed
        out_done = [None] * E2E_GRAPH_STEPS  # step j's output copied out
        s_in.wait_stream(torch.cuda.current_stream())
        s_out.wait_stream(torch.cuda.current_stream())
        main = torch.cuda.current_stream()
        for j in range(E2E_GRAPH_STEPS):
            o = objs[j % nb]
            if j >= nb:                      # its buffers' previous step has read the query
                s_in.wait_event(done[j - nb])
            with torch.cuda.stream(s_in):
                o.q_nope.copy_(hq[0], non_blocking=True)
                o.q_rope_raw.copy_(hq[1], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            main.wait_event(ev_in)
            if j >= nb:                      # and its previous output has left
                main.wait_event(out_done[j - nb])
            o.run()
            done[j] = torch.cuda.Event()
            done[j].record(main)
            s_out.wait_event(done[j])
            with torch.cuda.stream(s_out):
                hout[j % 2].copy_(o.out, non_blocking=True)
                out_done[j] = torch.cuda.Event()
                out_done[j].record(s_out)
        main.wait_stream(s_in)
        main.wait_stream(s_out)

    with torch.cuda.stream(cap):
        body()                               # warm-up, outside any capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            body()
    for k in range(2):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(2, -(-max(10, steps) // E2E_GRAPH_STEPS))
    e0.record(stream)
    for k in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * E2E_GRAPH_STEPS)
    return {"value": w.n_q * world / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "timing": f"CUDA graph of {E2E_GRAPH_STEPS} steps on {nb} buffer sets in turn: each step copies its "
                      "query in from pinned host memory and its output back to pinned host memory on side "
                      "streams, overlapping the neighbouring steps' launches; replayed"}


def side_objects(w, one, inp, dev, cap, peaks):
    """The other kernels of the library, each timed alone with CUDA-graph replays."""
    import numpy as np
    import torch
    from mla_latent_kv_12_gb300 import mla
    from mla_latent_kv_12_gb300 import workloads as W
    from mla_latent_kv_12_gb300.pipeline import PrefillStep
    hbm, tf_burst, _, _ = peaks
    stream = torch.cuda.current_stream()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

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

    # the cache append of the page's forward (RMSNorm + RoPE of one new token per batch row)
    ap_lat = torch.zeros(w.batch, 4, w.rank, dtype=one.dtype, device=dev)
    ap_rope = torch.zeros(w.batch, 4, w.rope, dtype=one.dtype, device=dev)
    ap_len = torch.zeros(w.batch, dtype=torch.int32, device=dev)
    ap_in = torch.randn(w.batch, 1, w.rank, device=dev).to(one.dtype)
    ap_rin = torch.randn(w.batch, 1, w.rope, device=dev).to(one.dtype)
    ap_w = torch.ones(w.rank, dtype=one.dtype, device=dev)
    append_us = graph_us(lambda: mla.append_compressed(ap_in, ap_rin, ap_w, 1e-6, w.theta, ap_lat, ap_rope,
                                                       None, ap_len), per_graph=20, reps=10)
    ap_bytes = w.batch * (w.rank + w.rope) * one.latent.element_size() * 2

    # the DSA top-k selection (2048 positions per query row from f32 scores over the row's window)
    sel_k = 2048
    sel_len = inp.kv_len.repeat_interleave(w.s_q).to(torch.int32).to(dev)
    sel_scores = torch.randn(w.n_q, int(inp.kv_len.max()), device=dev)
    sel_out = torch.empty(w.n_q, sel_k, dtype=torch.int32, device=dev)
    sel_cnt = torch.empty(w.n_q, dtype=torch.int32, device=dev)
    select_us = graph_us(lambda: mla.select_topk(sel_scores, sel_len, sel_k, sel_out, sel_cnt), per_graph=10,
                         reps=5)
    sel_bytes = int(inp.kv_len.repeat_interleave(w.s_q).sum()) * 4
    del sel_scores

    # the speculative-round rollback of a right-aligned cache (8 rows x 65536 tokens of latent || rope)
    rb_B, rb_W = 8, 65536
    rb_lat = torch.randn(rb_B, rb_W, w.rank, device=dev).to(one.dtype)
    rb_rope = torch.randn(rb_B, rb_W, w.rope, device=dev).to(one.dtype)
    rb_off = np.full(rb_B, rb_W - 7)
    rb_off[::2] = rb_W                                     # half the rows fill the width
    rb_keep = np.minimum(np.arange(rb_B) % 5, 4)           # 0..4 of 4 appended tokens kept
    rb_shift, _, _, rb_w = mla.plan_rollback(rb_W - rb_off, rb_off, rb_off - 4, rb_keep, rb_W)
    rb_shift = rb_shift.to(dev)
    rb_dst = [torch.empty(rb_B, rb_w, a.shape[2], dtype=a.dtype, device=dev) for a in (rb_lat, rb_rope)]

    def rollback_call():
        for a, d in zip((rb_lat, rb_rope), rb_dst):
            mla.cache_shift_rows(a, d, shift=rb_shift)
    rollback_us = graph_us(rollback_call, per_graph=5, reps=4)
    rb_bytes = 2 * rb_B * rb_w * (w.rank + w.rope) * rb_lat.element_size()
    del rb_lat, rb_rope, rb_dst

    # the reconstructed prefill of a 4096-token prompt (query RoPE, K/V materialisation, causal attention)
    pf = PrefillStep(W.make_inputs(W.PREFILL_BF16), dev)
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
    return {
        "append": {"us_per_call": append_us, "tokens_per_call": w.batch, "bytes_per_call": ap_bytes,
                   "note": "mla_append_compressed (RMSNorm + RoPE of one new token per batch row), "
                           "20 calls per CUDA graph, replayed"},
        "select_topk": {"us_per_call": select_us, "rows": w.n_q, "top_k": sel_k, "score_bytes": sel_bytes,
                        "gbs": sel_bytes / (select_us * 1e-6) / 1e9,
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


def public(res):
    return {k: v for k, v in res.items() if not k.startswith("_")}


def ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    # the host-core oracle pool is spawned before the first CUDA call
    pool = OraclePool() if (rank == 0 and not args.no_cpu_baseline) else None
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()

    w = workload(args.workload)
    with ClockSampler(local) as clk:
        head = measure(w, args.steps, args.warmup, dev, world, peaks, e2e=True, clocks=clk, layers=args.layers)
    inp, one, cap = head["_inp"], head["_steps"][0], head["_cap"]
    side = {} if args.no_side else side_objects(w, one, inp, dev, cap, peaks)
    del head["_steps"]
    per_config = {}
    if not args.no_per_config:
        for name in PER_CONFIG:
            if name == args.workload:
                per_config[workload(name).name] = {k: v for k, v in public(head).items() if k not in ("e2e", "clocks")}
                continue
            r = measure(workload(name), max(args.steps, 20), max(args.warmup, 3), dev, world, peaks, layers=args.layers)
            per_config[r["workload"]] = public(r)
            del r
            torch.cuda.empty_cache()
    cpu = None
    if pool is not None:
        cpu = cpu_baseline(inp, args.cpu_seconds, pool)
        pool.close()
    roof = dict(head["roofline"])
    line = {
        "metric": METRIC, "value": head["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "s_q": w.s_q, "heads": w.heads,
                   "rank": w.rank, "rope": w.rope, "cached_keys": int(inp.kv_len.sum()), "layers": 1,
                   "l2": (f"rotating {head['layers']} layers' buffers (inputs of one step x layers > 2 x L2)"
                          if args.layers <= 0 else f"{head['layers']} layers fixed by --layers (L2 not flushed)"),
                   "decode_kernel": head["kind"], "parallelism": f"replicas{world}"},
        "clocks": head.get("clocks"),
        "e2e": head["e2e"],
        "gpu_launches": head["step_launches"] * args.steps,
        "timing": "CUDA graph per layer step, replayed; decode kernel timed on its own graph replays",
        "roofline": roof,
        "step_roofline": head["step_roofline"],
        "cpu_baseline": cpu,
        "cache_gbs": head["cache_gbs"],
        "per_config": per_config,
    }
    line.update(side)
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
