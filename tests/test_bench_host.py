"""Host-side logic of bench.py: max-over-ranks timing with two gloo ranks on CPU,
the reference arm's rank rule, and the algorithmic byte / flop counts."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    v = bench.max_over_ranks(10.0 + 5.0 * rank, torch.device("cpu"))
    q.put((rank, v))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5


def _run_ref(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "tiny_f32", "--steps", "2", "--warmup", "1",
                           "--cpu-seconds", "0.2"], env=env, capture_output=True, text=True,
                          timeout=300)


def test_reference_arm_rank_rule():
    r1 = _run_ref(1, 2)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _run_ref(0, 2)
    assert r0.returncode == 0, r0.stderr
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_algorithmic_counts():
    from mla_latent_kv_12_gb300 import workloads as W
    inp = W.make_inputs(W.DENSE_BF16)
    byts, flops = bench.algorithmic(inp)
    assert byts == 4096 * 1152
    assert flops == 4096 * 2 * 128 * (576 + 512)
    import dataclasses
    w = dataclasses.replace(W.VERIFY_BF16, t=100)
    inp = W.make_inputs(w, rows=2)
    byts, flops = bench.algorithmic(inp)
    assert byts == 2 * 100 * 1152                 # each row's window read once
    assert flops == 2 * (97 + 98 + 99 + 100) * 2 * 128 * 1088
