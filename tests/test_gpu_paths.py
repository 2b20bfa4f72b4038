"""CUDA paths that the headline workloads do not reach, against the float64 oracle.

* 64 heads: the tensor-core kernels pad the MMA's 128 rows with zero queries.
* More than 128 query rows: the decode plans its split with a separate
  planner launch instead of in its prologue, and the projections run in
  several row blocks.
* Long rows: the split plan charges each row start, in the prologue and in
  the planner launch.
* Many split pieces per row: the combine loads a batch of pieces at once and
  merges the batches online (a rescale when a later batch holds a larger
  maximum); the fused tail's thread groups share a row's pieces.
* A cache whose batch stride is not a whole number of rows: selected rows
  are gathered with 16-byte cp.async loads instead of TMA gather4.
* The fp16 exchange of the two half scores of an SM pair: the range over
  which it stays within the bf16 tolerance, and the status bit beyond it.
"""
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
    from mla_latent_kv_12_gb300.pipeline import DecodeStep
else:  # collected on CPU-only machines, skipped by the marker filter
    from mla_latent_kv_12_gb300 import workloads as W

DEV = "cuda"


def _granular_and_fused(inp, rows=None, heads=None, expect_fused=True):
    ref = H.oracle_reference(inp, rows, heads)
    step = DecodeStep(inp, DEV, fused=False)
    step.run()
    torch.cuda.synchronize()
    H.compare_step(step, ref, inp.w.dtype)
    assert int(step.status.item()) == 0
    fstep = DecodeStep(inp, DEV, fused=True)
    assert fstep.fused == expect_fused
    if fstep.fused:
        fstep.run()
        torch.cuda.synchronize()
        H.compare_step(fstep, ref, inp.w.dtype)
        assert int(fstep.status.item()) == 0
    return step


# ---------------------------------------------------------------- 64 heads

H64 = dataclasses.replace(W.DENSE_BF16, name="dense_bf16_h64", heads=64)


@pytest.mark.parametrize("case", ["dense", "ragged", "sparse", "verify", "verify_sparse"])
def test_64_heads_whole_step(case):
    if case == "dense":
        inp = W.make_inputs(dataclasses.replace(H64, batch=3, t=1500))
    elif case == "ragged":
        w = dataclasses.replace(W.RAGGED_BF16, heads=64)
        inp = W.make_inputs(w, layout="flat", rows=5, t_override=1500)
    elif case == "sparse":
        w = dataclasses.replace(W.SPARSE_BF16, heads=64, top_k=300)
        inp = W.make_inputs(w, rows=3, t_override=5000)
    else:
        w = dataclasses.replace(W.VERIFY_BF16, heads=64, top_k=200 if case == "verify_sparse" else 0)
        inp = W.make_inputs(w, rows=3, t_override=1100)
    step = _granular_and_fused(inp)
    assert mla.decode_kernel_kind(64, 512, 64) == 1
    assert step.attend_launches() == 2


def test_64_heads_projection_row_blocks():
    # 150 query rows: the absorb in one block of 256, the projection in three of 64.
    g = torch.Generator().manual_seed(64)
    n_q = 150
    q = torch.randn(n_q, 64, 128, generator=g).to(torch.bfloat16)
    kv = (torch.randn(64 * 256, 512, generator=g) / 512 ** 0.5).to(torch.bfloat16)
    out = torch.zeros(n_q, 64, 576, dtype=torch.bfloat16, device=DEV)
    mla.absorb_q(q.to(DEV), kv.to(DEV), out, 64, 128, 128, 512)
    H.assert_close(out[..., :512], O.absorb_q(H.f64(q), H.f64(kv), 64, 128, 128), "bf16", "absorb")
    ctx = (torch.randn(n_q, 64, 512, generator=g) * 0.05).to(torch.bfloat16)
    pv = torch.empty(n_q, 64 * 128, dtype=torch.float32, device=DEV)
    mla.project_v(ctx.to(DEV), kv.to(DEV), pv, 64, 128, 128)
    H.assert_close(pv, O.project_v(H.f64(ctx), H.f64(kv), 64, 128, 128), "bf16", "project_v")


@pytest.mark.parametrize("n_q", [257, 600])
def test_absorb_and_project_many_row_blocks(n_q):
    # more than one 256-row absorb block (a ragged last block) and many 64-row
    # projection blocks, 128 heads
    g = torch.Generator().manual_seed(n_q)
    q = torch.randn(n_q, 128, 128, generator=g).to(torch.bfloat16)
    kv = (torch.randn(128 * 256, 512, generator=g) / 512 ** 0.5).to(torch.bfloat16)
    out = torch.zeros(n_q, 128, 576, dtype=torch.bfloat16, device=DEV)
    mla.absorb_q(q.to(DEV), kv.to(DEV), out, 128, 128, 128, 512)
    rows = [0, 1, 255, 256, n_q - 1]
    want = O.absorb_q(H.f64(q[rows]), H.f64(kv), 128, 128, 128)
    H.assert_close(out[rows][..., :512], want, "bf16", "absorb")
    assert torch.count_nonzero(out[..., 512:]) == 0
    ctx = (torch.randn(n_q, 128, 512, generator=g) * 0.05).to(torch.bfloat16)
    pv = torch.empty(n_q, 128 * 128, dtype=torch.bfloat16, device=DEV)
    mla.project_v(ctx.to(DEV), kv.to(DEV), pv, 128, 128, 128)
    H.assert_close(pv[rows], O.project_v(H.f64(ctx[rows]), H.f64(kv), 128, 128, 128), "bf16", "project_v")


# ---------------------------------------------------------------- the planner launch (> 128 query rows)

PLANNER_ROWS = [0, 1, 63, 64, 127, 128, 129, 158, 159]


def _plan_charge(step, n_units):
    # the decode workspace starts with the split plan: the prefix over work
    # units, then the start charge per unit
    return int(step.workspace[: 4 * (n_units + 2)].view(torch.int32)[n_units + 1].item())


def test_planner_path_ragged_160_rows():
    w = dataclasses.replace(W.RAGGED_BF16, batch=160)
    inp = W.make_inputs(w, layout="flat", t_override=900)
    step = _granular_and_fused(inp, rows=PLANNER_ROWS, heads=[0, 7, 64, 127], expect_fused=False)
    assert step.attend_launches() == 3          # planner + decode + combine
    assert torch.all(torch.isfinite(step.ctx.float()))
    assert _plan_charge(step, 160) == 0         # ~15 tiles per SM pair: no start charge


@pytest.mark.parametrize("rows,t", [(32, 12000), (160, 6000)])
def test_charged_split_plan_every_row(rows, t):
    # Rows long enough that every SM pair streams 32 tiles or more: the plan
    # charges each row start (in the decode prologue for 32 rows, in the
    # planner launch for 160), so ranges move, and a range that ends inside a
    # row's charge holds none of that row.  Every row, three heads.
    w = dataclasses.replace(W.RAGGED_BF16, batch=rows)
    inp = W.make_inputs(w, layout="flat", t_override=t)
    step = _granular_and_fused(inp, heads=[0, 77, 127], expect_fused=rows <= 64)
    assert _plan_charge(step, rows) > 0


@pytest.mark.parametrize("batch,t", [(1, 40000), (3, 20000)])
def test_combine_merges_many_pieces_per_row(batch, t):
    # One row of 40,000 keys is 625 tiles; the 76 SM pairs of a GB300 take
    # ranges of 9 (no row-start charge at this length), so the row has 70
    # pieces: five batches of the combine's 16, and nine pieces for each of the
    # fused tail's eight thread groups.  Three rows of 20,000 keys: ~24 pieces
    # each.
    w = dataclasses.replace(W.DENSE_BF16, batch=batch, t=t)
    inp = W.make_inputs(w)
    _granular_and_fused(inp, heads=[0, 127] if batch == 1 else [9, 64])


@pytest.mark.parametrize("top_k", [0, 120])
def test_planner_path_verify_80_rows_of_2_tokens(top_k):
    # dense: groups of 2 clusters in lockstep per batch row; sparse: one query row per unit
    w = dataclasses.replace(W.VERIFY_BF16, batch=80, s_q=2, top_k=top_k)
    inp = W.make_inputs(w, rows=80, t_override=700)
    step = _granular_and_fused(inp, rows=PLANNER_ROWS, heads=[0, 31, 100], expect_fused=False)
    assert step.attend_launches() == 3


# ---------------------------------------------------------------- cp.async row gather

def _odd_batch_stride_copy(t: torch.Tensor, extra: int) -> torch.Tensor:
    """A device copy of ``t`` [B, T, F] whose batch stride is T*F + extra elements
    (not a whole number of rows)."""
    B, T, F = t.shape
    bs = T * F + extra
    buf = torch.zeros(B * bs + 64, dtype=t.dtype, device=DEV)
    view = torch.as_strided(buf, (B, T, F), (bs, F, 1))
    view.copy_(t.to(DEV))
    return view


@pytest.mark.parametrize("selected", [True, False])
def test_odd_batch_stride_takes_the_cp_async_gather(selected):
    w = dataclasses.replace(W.SPARSE_BF16, top_k=300)
    inp = W.make_inputs(w, rows=3, t_override=5000, layout="padded")
    inp.sel_count[1] = -1                       # one dense row among the selected ones
    step = DecodeStep(inp, DEV, fused=False)
    step.run()                                  # the query (absorbed + rotated) and the rotated cache
    torch.cuda.synchronize()
    lat = _odd_batch_stride_copy(step.latent, 8)    # 16 bytes past each batch row
    rope = _odd_batch_stride_copy(step.rope, 8)
    assert lat.stride(0) % lat.stride(1) != 0 and rope.stride(0) % rope.stride(1) != 0
    sel = step.sel if selected else None
    cnt = step.sel_count if selected else None
    ctx = torch.full_like(step.ctx, float("nan"))
    lse = torch.full_like(step.lse, float("nan"))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.decode_attend(step.q, lat, rope, step.kv_start, step.kv_len, 3, 1, step.scale, ctx, lse,
                      sel=sel, sel_count=cnt, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = H.oracle_reference(inp, with_selection=selected)
    H.assert_close(ctx.cpu(), ref["ctx"], "bf16", "ctx")
    assert np.max(np.abs(H.f64(lse) - ref["lse"])) <= 2e-2
    # the same ctx as the TMA gather4 / tiled layout, within the tolerance
    ctx2 = torch.empty_like(ctx)
    mla.decode_attend(step.q, step.latent, step.rope, step.kv_start, step.kv_len, 3, 1, step.scale, ctx2,
                      sel=sel, sel_count=cnt)
    torch.cuda.synchronize()
    H.assert_close(ctx.cpu(), ctx2.cpu(), "bf16", "cp.async vs gather4")
    if selected:
        out = torch.full((3, 300, 576), 7, dtype=torch.bfloat16, device=DEV)
        mla.gather_selected(lat, rope, step.kv_start, step.kv_len, 3, 1, step.sel, step.sel_count, 300, out, st)
        torch.cuda.synchronize()
        want = O.gather_selected(step.latent.cpu().view(torch.int16).numpy(),
                                 step.rope.cpu().view(torch.int16).numpy(), inp.kv_start.numpy(),
                                 inp.kv_len.numpy(), 1, inp.sel.numpy(), inp.sel_count.numpy(), 300)
        assert np.array_equal(out.cpu().view(torch.int16).numpy(), want)


# ---------------------------------------------------------------- fp16 score exchange range

def _half_scores_max(q, lat, rope, kv_start, kv_len):
    """Largest |half score| the SM pair exchanges, in float64: CTA r holds
    q_lat[256r:256r+256] . latent[256r:...] + q_rope[32r:32r+32] . rope[32r:...]."""
    best = 0.0
    for b in range(q.shape[0]):
        s, n = int(kv_start[b]), int(kv_len[b])
        L, R = lat[b, s:s + n], rope[b, s:s + n]
        for r in range(2):
            h = q[b, :, 256 * r:256 * r + 256] @ L[:, 256 * r:256 * r + 256].T + \
                q[b, :, 512 + 32 * r:512 + 32 * r + 32] @ R[:, 32 * r:32 * r + 32].T
            best = max(best, float(np.max(np.abs(h))))
    return best


@pytest.mark.parametrize("gain", [1, 4, 8, 16, 64])
def test_score_exchange_range(gain):
    # Queries scaled by `gain` (exact in bf16): half scores grow with it.  Within
    # the documented range the result meets the bf16 tolerance and no bit is
    # set; past it MLA_DEVICE_SCORE_RANGE is set.
    w = dataclasses.replace(W.DENSE_BF16, batch=2, t=2000)
    inp = W.make_inputs(w)
    step = DecodeStep(inp, DEV, fused=False)
    step.rope_q()
    step.absorb()
    q = (step.q.float() * gain).to(torch.bfloat16)
    assert torch.equal(q.float(), step.q.float() * gain)
    ctx = torch.empty_like(step.ctx)
    lse = torch.empty_like(step.lse)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.decode_attend(q, step.latent, step.rope, step.kv_start, step.kv_len, 2, 1, step.scale, ctx, lse,
                      device_status=st)
    torch.cuda.synchronize()
    qf, lat, rp = H.f64(q), H.f64(step.latent), H.f64(step.rope)
    kv_start, kv_len = inp.kv_start.numpy(), inp.kv_len.numpy()
    want_ctx, want_lse = O.attend_latent(qf[..., :512], qf[..., 512:], lat, rp, kv_start, kv_len, 1,
                                         scale=step.scale)
    half = _half_scores_max(qf, lat, rp, kv_start, kv_len)
    got = H.f64(ctx)
    rl = H.rel_l2(got, want_ctx)
    err = float(np.max(np.abs(got - want_ctx)))
    flagged = bool(int(st.item()) & mla.DEVICE_SCORE_RANGE)
    print(f"gain {gain}: max |half score| {half:.1f}, ctx rel-L2 {rl:.2e} max-abs {err:.2e}, flagged {flagged}")
    assert flagged == (half > mla.FP16_SCORE_LIMIT)
    if not flagged:
        H.assert_close(got, want_ctx, "bf16", f"ctx at gain {gain}")
        assert np.max(np.abs(H.f64(lse) - want_lse)) <= 2e-2
