"""Host-side logic of bench.py: max-over-ranks timing with two gloo ranks on CPU,
the reference arm's rank rule, the algorithmic byte / flop counts, the
roofline's bound and fraction, and the clock record's summary."""
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
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # the reported step time is the time measured per step (not scaled up)
    assert line["ms_per_step"] < 60_000


def test_one_row_inputs_give_the_same_oracle_rows():
    # the host-core oracle pool works on one batch row at a time: the row cut
    # out of a ragged packed batch gives the oracle's rows of the whole batch
    import dataclasses
    import numpy as np
    from mla_latent_kv_12_gb300 import workloads as W
    from tests import helpers as H
    w = dataclasses.replace(W.RAGGED_BF16, heads=4)
    inp = W.make_inputs(w, layout="flat", rows=3, t_override=200)
    for b in range(3):
        one = bench.one_row_inputs(inp, b)
        a = H.oracle_reference_out_only(one, rows=[0], heads=[0, 3])
        full = H.oracle_reference_out_only(inp, rows=[b], heads=[0, 3])
        assert np.allclose(a[0], full[b], rtol=1e-12, atol=1e-12)
    w = dataclasses.replace(W.VERIFY_SPARSE_BF16, heads=2, top_k=20)
    inp = W.make_inputs(w, rows=2, t_override=60)
    one = bench.one_row_inputs(inp, 1)
    a = H.oracle_reference_out_only(one, rows=[0, 1, 2, 3], heads=[1])
    full = H.oracle_reference_out_only(inp, rows=[4, 5, 6, 7], heads=[1])
    assert np.allclose(a[:4], full[4:8], rtol=1e-12, atol=1e-12)


def test_step_bytes_and_layer_rotation():
    from mla_latent_kv_12_gb300 import workloads as W
    inp = W.make_inputs(W.DENSE_BF16)
    byts, flops = bench.step_algorithmic(inp)
    weights = 128 * 256 * 512 * 2
    assert byts == 4096 * 1152 + weights + 128 * 192 * 2 + 128 * 128 * 2
    assert flops == 4096 * 2 * 128 * 1088 + 2 * 128 * 512 * 256
    R = bench.layers_for(inp, byts)
    assert (R - 1) * byts >= 2 * bench.L2_BYTES            # other layers' bytes between two uses
    assert bench.layers_for(inp, 10 ** 12) == 1


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


def test_roofline_takes_the_slower_bound():
    # The ragged pair: 573.8 MB of cache and 138.7 GFLOP in 130.4 us -> HBM-bound.
    r = bench.roofline(573_754_752, 138_721_148_928, 130.4e-6, 6687.1, 1935.2, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6687.1
    assert r["achieved"] == pytest.approx(573_754_752 / 130.4e-6 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6687.1)
    assert 0.65 < r["frac"] < 0.67
    # The verify pair: 604 MB and 584 GFLOP (967 flop/B, above the ridge) -> tensor-bound.
    v = bench.roofline(603_979_776, 584_102_182_912, 433.4e-6, 6687.1, 1935.2, "measured")
    assert v["bound"] == "tensor" and v["unit"] == "TFLOP/s"
    assert v["frac"] == pytest.approx(584_102_182_912 / 433.4e-6 / 1e12 / 1935.2)
    # exactly at the ridge the bytes decide
    ridge = bench.roofline(6687.1e9, 1935.2e12, 1.0, 6687.1, 1935.2, "measured")
    assert ridge["bound"] == "hbm" and ridge["frac"] == pytest.approx(1.0)


def test_clock_summary_reasons():
    cs = bench.ClockSampler(0)
    assert cs.summary()["reasons"] == ["unavailable"] and cs.summary()["samples"] == 0
    row = lambda sm, cap: [sm, "2070", "1100.5", "0x0", "Not Active", "Not Active", "Not Active", cap]
    cs.samples = [(1.0, row("2070", "Not Active")), (2.0, row("2040", "Active")), (3.0, row("2070", "Not Active"))]
    s = cs.summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    # samples before the timed region are left out
    assert cs.summary(since=2.5)["reasons"] == [] and cs.summary(since=2.5)["samples"] == 1
