"""Reconstructed prefill on the device (per-head K/V materialisation on
tcgen05, then causal attention on tcgen05) against the oracle's
reconstructed definition, through the C ABI: small blocks whole (several
query and key tiles, ragged tails, left-padded and packed rows), the
4096-token prompt on sampled rows and heads, and the degenerate cases."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import mla_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from mla_latent_kv_12_gb300 import mla
    from mla_latent_kv_12_gb300 import workloads as W
    from mla_latent_kv_12_gb300.pipeline import PrefillStep
else:
    from mla_latent_kv_12_gb300 import workloads as W

DEV = "cuda"


def _check(step, inp, rows, heads, dtype="bf16"):
    want, want_lse = H.oracle_prefill(inp, rows, heads)
    w = inp.w
    ri, hi = torch.tensor(rows), torch.tensor(heads)
    got = step.out.view(w.n_q, w.heads, w.v).cpu()[ri][:, hi]
    lse = step.lse.cpu()[ri][:, hi].to(torch.float64).numpy()
    H.assert_close(got, want[rows], dtype, "prefill out")
    wl = want_lse[rows]
    fin = np.isfinite(wl)
    assert np.array_equal(np.isfinite(lse), fin), "lse finiteness"
    assert np.max(np.abs(lse[fin] - wl[fin]), initial=0.0) <= 2e-2, "lse"


def test_reconstruct_matches_the_oracle():
    g = torch.Generator().manual_seed(100)
    rows, Hh, rank = 300, 128, 512
    lat = torch.randn(rows, rank, generator=g)
    lat = (lat * torch.rsqrt(lat.square().mean(-1, keepdim=True))).to(torch.bfloat16)
    wkv = (torch.randn(Hh * 256, rank, generator=g) * rank ** -0.5).to(torch.bfloat16)
    kv = torch.full((rows, Hh, 256), float("nan"), dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.reconstruct_kv(lat.to(DEV), wkv.to(DEV), kv[..., :128], kv[..., 128:], Hh, 128, 128, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    k_want, v_want = O.reconstruct_kv(lat.to(torch.float64).numpy(), wkv.to(torch.float64).numpy(), Hh, 128, 128)
    H.assert_close(kv[..., :128].cpu(), k_want, "bf16", "k_nope")
    H.assert_close(kv[..., 128:].cpu(), v_want, "bf16", "v")


@pytest.mark.parametrize("layout", ["padded", "flat"])
def test_prefill_small_blocks_match_the_oracle(layout):
    # two rows with different earlier caches, a 300-token block (three query
    # tiles, the last ragged) and windows of 400..700 keys (left-padded rows)
    w = dataclasses.replace(W.PREFILL_BF16, name="prefill_small", batch=2, s_q=300, t=0, seed=6,
                            ragged=(100, 400))
    inp = W.make_inputs(w, layout=layout)
    step = PrefillStep(inp, DEV)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    _check(step, inp, list(range(w.n_q)), [0, 5, 64, 127])


def test_prefill_f32_output_and_short_windows():
    # kv_len < s_q: the block's first tokens see no key (zeros, lse -inf)
    w = dataclasses.replace(W.PREFILL_BF16, name="prefill_short", batch=2, s_q=160, t=150, seed=7)
    inp = W.make_inputs(w)
    inp.q_offset = torch.zeros_like(inp.q_offset)          # keep RoPE positions non-negative
    step = PrefillStep(inp, DEV, out_dtype=torch.float32)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    out = step.out.view(w.n_q, w.heads, w.v).cpu()
    assert torch.all(out[:10] == 0) and torch.all(step.lse.cpu()[:10] == -float("inf"))
    _check(step, inp, list(range(w.n_q)), [1, 77])


def test_prefill_4096_token_block_sampled():
    inp = W.make_inputs(W.PREFILL_BF16)
    step = PrefillStep(inp, DEV)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    rows = [0, 1, 127, 128, 129, 1000, 2047, 2048, 3968, 4094, 4095]
    _check(step, inp, rows, [0, 31, 64, 127])


def test_prefill_flags_a_window_outside_the_buffer():
    w = dataclasses.replace(W.PREFILL_BF16, name="prefill_bad", batch=2, s_q=64, t=200, seed=8)
    inp = W.make_inputs(w)
    step = PrefillStep(inp, DEV)
    step.kv_len[1] = step.t_max + 1                       # row 1 runs past its buffer rows
    step.out.fill_(3.0)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == mla.DEVICE_INDEX_OUT_OF_RANGE
    out = step.out.view(w.n_q, w.heads, w.v).cpu()
    assert torch.all(out[w.s_q:] == 3.0)                   # the bad row is skipped
    step.kv_len[1] = int(inp.kv_len[1])
    step.status.zero_()
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    _check(step, inp, list(range(0, w.n_q, 7)), [3])


def test_chunked_prefill_after_a_long_cache_sampled():
    # a 512-token chunk appended after ~3000 cached tokens per row (packed rows):
    # the chunk's queries see the whole earlier cache plus their causal prefix
    w = dataclasses.replace(W.PREFILL_BF16, name="prefill_chunk", batch=3, s_q=512, t=0, seed=9,
                            ragged=(2900, 3100))
    inp = W.make_inputs(w, layout="flat")
    step = PrefillStep(inp, DEV)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    rows = [0, 127, 128, 511, 512, 700, 1023, 1024, 1300, 1535]
    _check(step, inp, rows, [2, 100])


def test_single_token_prefill_equals_the_decode_path():
    # S_q = 1 through the prefill path matches the absorbed decode step on the same inputs
    w = dataclasses.replace(W.DENSE_BF16, name="prefill_one", t=1000, seed=10)
    inp = W.make_inputs(w)
    step = PrefillStep(inp, DEV)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    _check(step, inp, [0], list(range(0, 128, 9)))
    from mla_latent_kv_12_gb300.pipeline import DecodeStep
    dstep = DecodeStep(inp, DEV)
    dstep.run()
    torch.cuda.synchronize()
    H.assert_close(step.out.cpu(), dstep.out.cpu().to(torch.float64).numpy(), "bf16", "prefill vs decode")
