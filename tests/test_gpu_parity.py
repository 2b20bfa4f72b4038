"""CUDA path vs the float64 oracle, element by element, through the C ABI.

Small cases run whole; the full-size workloads compare sampled query rows and
heads (the oracle computes those one by one) in the launch configuration the
benchmark uses.
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


def run_and_compare(inp, rows=None, heads=None, with_selection=True):
    """The four entry points one by one (every intermediate checked), then the
    fused step where it serves the shapes (out and lse checked)."""
    ref = H.oracle_reference(inp, rows, heads, with_selection)
    step = DecodeStep(inp, DEV, with_selection=with_selection, fused=False)
    step.run()
    torch.cuda.synchronize()
    res = H.compare_step(step, ref, inp.w.dtype)
    assert int(step.status.item()) == 0
    fstep = DecodeStep(inp, DEV, with_selection=with_selection, fused=True)
    if fstep.fused:
        fstep.run()
        torch.cuda.synchronize()
        res["fused"] = H.compare_step(fstep, ref, inp.w.dtype)
        assert int(fstep.status.item()) == 0
    return step, res


# ---------------------------------------------------------------- RoPE

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_rope_matches_oracle(dtype):
    g = torch.Generator().manual_seed(7)
    x = torch.randn(3, 5, 4, 80, generator=g).to(dtype)      # width 80: 64 rotated + 16 tail
    offs = torch.tensor([0, 17, 131000], dtype=torch.int32)
    out = torch.empty_like(x, device=DEV)
    mla.rope_partial_interleaved(x.to(DEV), out, 64, 10000.0, row_offsets=offs.to(DEV))
    want = O.rope_partial_interleaved(H.f64(x), offs.numpy(), 64, 10000.0)
    got = H.f64(out)
    if dtype == torch.float32:
        assert H.rel_l2(got, want) <= 1e-6
    else:
        H.assert_close(got, want, "bf16", "rope")
    # the kept tail and the position-0 permutation are bit-exact
    assert torch.equal(out[..., 64:].cpu(), x[..., 64:])
    perm = torch.cat([x[0, 0, :, 0:64:2], x[0, 0, :, 1:64:2]], -1)
    assert torch.equal(out[0, 0, :, :64].cpu(), perm)


def test_rope_in_place_and_scalar_offset():
    g = torch.Generator().manual_seed(8)
    x = torch.randn(2, 7, 3, 64, generator=g)
    xd = x.to(DEV)
    mla.rope_partial_interleaved(xd, xd, 64, 10000.0, position_offset=4093)
    want = O.rope_partial_interleaved(H.f64(x), 4093, 64, 10000.0)
    assert H.rel_l2(H.f64(xd), want) <= 1e-6


def test_rope_strided_views_into_packed_query():
    # q_rope raw [B,S,H,64] -> columns 512.. of a packed [B,S,H,576] buffer.
    g = torch.Generator().manual_seed(9)
    x = torch.randn(2, 4, 8, 64, generator=g).to(torch.bfloat16)
    packed = torch.zeros(2, 4, 8, 576, dtype=torch.bfloat16, device=DEV)
    mla.rope_partial_interleaved(x.to(DEV), packed[..., 512:], 64, 10000.0,
                                 row_offsets=torch.tensor([10, 20], dtype=torch.int32, device=DEV))
    want = O.rope_partial_interleaved(H.f64(x), [10, 20], 64, 10000.0)
    H.assert_close(packed[..., 512:], want, "bf16", "rope strided")
    assert torch.count_nonzero(packed[..., :512]) == 0


# ---------------------------------------------------------------- absorb / project

@pytest.mark.parametrize("n_q", [1, 7, 32, 33])
def test_absorb_matches_oracle(n_q):
    w = W.DENSE_BF16
    g = torch.Generator().manual_seed(n_q)
    q = torch.randn(n_q, w.heads, w.nope, generator=g).to(torch.bfloat16)
    kv = (torch.randn(w.heads * 256, 512, generator=g) / 512 ** 0.5).to(torch.bfloat16)
    out = torch.zeros(n_q, w.heads, 576, dtype=torch.bfloat16, device=DEV)
    mla.absorb_q(q.to(DEV), kv.to(DEV), out, w.heads, 128, 128, 512)
    want = O.absorb_q(H.f64(q), H.f64(kv), w.heads, 128, 128)
    H.assert_close(out[..., :512], want, "bf16", "absorb")
    assert torch.count_nonzero(out[..., 512:]) == 0


@pytest.mark.parametrize("n_q,out_dtype", [(1, torch.bfloat16), (32, torch.bfloat16), (5, torch.float32)])
def test_project_v_matches_oracle(n_q, out_dtype):
    g = torch.Generator().manual_seed(100 + n_q)
    ctx = (torch.randn(n_q, 128, 512, generator=g) * 0.05).to(torch.bfloat16)
    kv = (torch.randn(128 * 256, 512, generator=g) / 512 ** 0.5).to(torch.bfloat16)
    out = torch.empty(n_q, 128 * 128, dtype=out_dtype, device=DEV)
    mla.project_v(ctx.to(DEV), kv.to(DEV), out, 128, 128, 128)
    want = O.project_v(H.f64(ctx), H.f64(kv), 128, 128, 128)
    H.assert_close(out, want, "bf16", "project_v")


# ---------------------------------------------------------------- whole step, small cases

def test_tiny_f32_whole_step():
    inp = W.make_inputs(W.TINY_F32)
    run_and_compare(inp)


def test_dense_bf16_whole_step():
    inp = W.make_inputs(W.DENSE_BF16)
    run_and_compare(inp)


@pytest.mark.parametrize("layout", ["padded", "flat", "aligned"])
def test_ragged_reduced(layout):
    inp = W.make_inputs(W.RAGGED_BF16, layout=layout, rows=5, t_override=1500)
    run_and_compare(inp)


def test_sparse_reduced():
    w = dataclasses.replace(W.SPARSE_BF16, top_k=300)
    inp = W.make_inputs(w, rows=3, t_override=5000)
    run_and_compare(inp)


@pytest.mark.parametrize("top_k", [0, 200])
def test_verify_reduced(top_k):
    w = dataclasses.replace(W.VERIFY_BF16, top_k=top_k)
    inp = W.make_inputs(w, rows=3, t_override=1100)
    run_and_compare(inp)


def test_verify_f32_tiny_causal():
    w = dataclasses.replace(W.TINY_F32, batch=2, s_q=4, t=70)
    inp = W.make_inputs(w)
    run_and_compare(inp)


@pytest.mark.parametrize("batch", [2, 3, 4])
def test_matrix_vector_absorb_row_counts(batch):
    # 2..4 query rows take the CUDA-core absorb (with the query RoPE folded in
    # the fused step); the granular run checks q_lat and the rotated q_rope.
    w = dataclasses.replace(W.DENSE_BF16, batch=batch, t=700)
    run_and_compare(W.make_inputs(w), heads=[0, 9, 64, 127])


@pytest.mark.parametrize("batch", [1, 17, 64])
def test_fused_step_row_counts(batch):
    # 1, 17 and 64 query rows: N = 16, 32 and 64 in the fused projection MMA,
    # rows finished in place and split rows mixed.
    w = dataclasses.replace(W.DENSE_BF16, batch=batch, t=900 if batch > 1 else 4096)
    inp = W.make_inputs(w)
    rows = list(range(batch)) if batch <= 17 else [0, 1, 31, 62, 63]
    ref = H.oracle_reference(inp, rows, [0, 5, 64, 127])
    step = DecodeStep(inp, DEV, fused=True)
    assert step.fused
    step.run()
    torch.cuda.synchronize()
    H.compare_step(step, ref, "bf16")
    assert int(step.status.item()) == 0


def test_fused_step_refuses_unserved_shapes():
    inp = W.make_inputs(W.TINY_F32)
    step = DecodeStep(inp, DEV)
    assert not step.fused                       # f32: composed from the four entry points
    w = W.DENSE_BF16
    assert mla.decode_step_workspace_size(65, 1, w.heads, w.nope, w.v, w.rank, w.rope, 4096) == 0
    assert mla.decode_step_workspace_size(64, 1, w.heads, w.nope, w.v, w.rank, w.rope, 4096) > 0


def test_decode_rescale_in_some_heads_only():
    # Softmax scale 1 and a planted key aligned with head 5's query late in the
    # window: head 5's running maximum jumps by far more than the lazy-rescale
    # threshold in a later tile while its warp neighbours' does not, so the O
    # rescale runs for some heads of a warp only.
    w = dataclasses.replace(W.DENSE_BF16, batch=2, t=2000)
    inp = W.make_inputs(w)
    g = torch.Generator().manual_seed(11)
    q = (torch.randn(2, 128, 576, generator=g) * 0.1).to(torch.bfloat16)
    lat = inp.latent.clone()
    for b in range(2):
        d = q[b, 5, :512].float()
        lat[b, 1300] = (d / d.square().mean().sqrt()).to(torch.bfloat16)
    kv_len = inp.kv_len.clone()
    ctx = torch.empty(2, 128, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(2, 128, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.decode_attend(q.to(DEV), lat.to(DEV), inp.rope_raw.to(DEV), None, kv_len.to(DEV), 2, 1, 1.0, ctx, lse,
                      device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want_ctx, want_lse = O.attend_latent(H.f64(q[..., :512]), H.f64(q[..., 512:]), H.Rows(lat),
                                         H.Rows(inp.rope_raw), [0, 0], kv_len.numpy(), 1, scale=1.0)
    H.assert_close(ctx, want_ctx, "bf16", "ctx")
    assert np.max(np.abs(H.f64(lse) - want_lse)) <= 2e-2


# ---------------------------------------------------------------- cache append (NEXT-3)

def _append_case(dtype, cache_dtype, B=4, S=3, T=64, packed=False, offsets=None, seed=50):
    g = torch.Generator().manual_seed(seed)
    rank, rope_dim = 512, 64
    bb = 1 if packed else B
    lat = torch.randn(bb, T, rank, generator=g).to(cache_dtype)
    rp = torch.randn(bb, T, rope_dim, generator=g).to(cache_dtype)
    lat_raw = (torch.randn(B, S, rank, generator=g) * 2.0).to(dtype)
    rope_raw = torch.randn(B, S, rope_dim, generator=g).to(dtype)
    w = (1.0 + 0.1 * torch.randn(rank, generator=g)).to(dtype)
    if packed:
        kv_start = torch.tensor([0, 16, 32, 48][:B], dtype=torch.int32)
        kv_len = torch.tensor([3, 13, 0, 16][:B], dtype=torch.int32)        # row 3: 48 + 16 + S > 64
    else:
        kv_start = torch.tensor([0, 2, 0, 1][:B], dtype=torch.int32)
        kv_len = torch.tensor([5, 20, 0, 63][:B], dtype=torch.int32)        # row 3: 1 + 63 + S > 64
    return lat, rp, lat_raw, rope_raw, w, kv_start, kv_len


@pytest.mark.parametrize("dtype,cache_dtype,packed,S", [
    (torch.bfloat16, torch.bfloat16, False, 3), (torch.bfloat16, torch.bfloat16, False, 1),
    (torch.float32, torch.float32, False, 3), (torch.float32, torch.bfloat16, True, 3),
    (torch.bfloat16, torch.float32, True, 2)])
def test_append_matches_oracle(dtype, cache_dtype, packed, S):
    lat, rp, lat_raw, rope_raw, w, kv_start, kv_len = _append_case(dtype, cache_dtype, S=S, packed=packed)
    offsets = torch.tensor([7, 0, 100000, 3], dtype=torch.int32) if packed else None
    d = {k: v.to(DEV) for k, v in dict(lat=lat, rp=rp, lat_raw=lat_raw, rope_raw=rope_raw, w=w,
                                        kv_start=kv_start, kv_len=kv_len).items()}
    out_len = torch.full_like(d["kv_len"], -7)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.append_compressed(d["lat_raw"], d["rope_raw"], d["w"], 1e-6, 10000.0, d["lat"], d["rp"], d["kv_start"],
                          d["kv_len"], kv_len_out=out_len,
                          row_offsets=offsets.to(DEV) if offsets is not None else None, device_status=st)
    torch.cuda.synchronize()
    want_lat, want_rp, want_len, overflow = O.append_compressed(
        H.f64(lat), H.f64(rp), H.f64(lat_raw), H.f64(rope_raw), H.f64(w), 1e-6, 10000.0, kv_start.numpy(),
        kv_len.numpy(), row_offsets=offsets.numpy() if offsets is not None else None)
    assert overflow == [3]
    assert int(st.item()) & mla.DEVICE_INDEX_OUT_OF_RANGE
    assert out_len.cpu().tolist() == list(want_len)
    tol = "f32" if cache_dtype == torch.float32 and dtype == torch.float32 else "bf16"
    for b in range(4):
        if b in overflow:
            continue
        bb = 0 if packed else b
        first = int(kv_start[b] + kv_len[b])
        H.assert_close(d["lat"][bb, first:first + S], want_lat[bb, first:first + S], tol, f"latent row {b}")
        H.assert_close(d["rp"][bb, first:first + S], want_rp[bb, first:first + S], tol, f"rope row {b}")
    # everything else in the cache is untouched, bit for bit
    touched = torch.zeros(lat.shape[:2], dtype=torch.bool)
    for b in range(4):
        if b not in overflow:
            bb = 0 if packed else b
            first = int(kv_start[b] + kv_len[b])
            touched[bb, first:first + S] = True
    assert torch.equal(d["lat"].cpu()[~touched], lat[~touched])
    assert torch.equal(d["rp"].cpu()[~touched], rp[~touched])


def test_append_then_decode_matches_oracle():
    # The page's forward: append the new token, then attend.  The cache is set
    # up without its last key; the append writes it (normalised, rotated at its
    # position) and updates kv_len in place; the decode step then matches the
    # oracle over the full window.
    w = dataclasses.replace(W.DENSE_BF16, t=700)
    inp = W.make_inputs(w)
    step = DecodeStep(inp, DEV)
    last = int(inp.kv_len[0]) - 1
    step.latent[0, last] = 3.0
    step.rope[0, last] = -2.0
    step.kv_len -= 1
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ones = torch.ones(w.rank, dtype=torch.bfloat16, device=DEV)
    mla.append_compressed(inp.latent[:, last:last + 1].to(DEV), inp.rope_raw[:, last:last + 1].to(DEV), ones,
                          1e-6, w.theta, step.latent, step.rope, step.kv_start, step.kv_len,
                          kv_len_out=step.kv_len, device_status=st)
    step.run()
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(step.kv_len[0].item()) == last + 1
    ref = H.oracle_reference(inp)
    H.compare_step(step, ref, "bf16")


# ---------------------------------------------------------------- DSA top-k selection (NEXT-2)

def _select_and_compare(scores, lengths, top_k):
    n = scores.shape[0]
    sel = torch.full((n, top_k), -5, dtype=torch.int32, device=DEV)
    cnt = torch.full((n,), -9, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.select_topk(scores.to(DEV), lengths.to(DEV), top_k, sel, cnt, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sel, cnt = sel.cpu(), cnt.cpu()
    for r in range(n):
        want = O.select_topk(scores[r, :int(lengths[r])].numpy(), top_k)
        if want is None:
            assert int(cnt[r]) == -1 and torch.all(sel[r] == -5)
        else:
            assert int(cnt[r]) == top_k
            assert np.array_equal(sel[r].numpy().astype(np.int64), want), f"row {r}"
    return sel, cnt


@pytest.mark.parametrize("top_k", [1, 7, 2048])
def test_select_topk_bit_exact(top_k):
    g = torch.Generator().manual_seed(70 + top_k)
    T = 131072
    lengths = torch.tensor([100, 5000, T, 2048, 2049, 1], dtype=torch.int32)
    normal = torch.randn(6, T, generator=g)
    _select_and_compare(normal, lengths, top_k)
    ties = torch.randint(0, 10, (6, T), generator=g).to(torch.float32)     # heavy ties at the threshold
    _select_and_compare(ties, lengths, top_k)


def test_select_topk_special_values():
    g = torch.Generator().manual_seed(80)
    x = torch.randn(4, 3000, generator=g)
    x[0, ::7] = float("inf")
    x[0, 3::11] = float("-inf")
    x[1, :] = 0.0
    x[1, ::2] = -0.0                   # +0 ranks above -0
    x[2, 100:110] = float("nan")       # positive NaN ranks first and makes the threshold NaN
    x[3, 50:60] = -float("nan")        # negative NaN ranks last
    lengths = torch.tensor([3000, 3000, 3000, 3000], dtype=torch.int32)
    for k in (5, 64, 2999):
        _select_and_compare(x, lengths, k)


def test_select_then_sparse_decode():
    # indexer-style scores -> device top-k -> selected-position decode, against
    # the oracle over the oracle's selection (identical, bit for bit)
    w = dataclasses.replace(W.SPARSE_BF16, top_k=256)
    inp = W.make_inputs(w, rows=3, t_override=4000)
    g = torch.Generator().manual_seed(90)
    scores = torch.randn(3, 4000, generator=g)
    lengths = inp.kv_len.clone()
    lengths[1] = 200                                   # a short row: dense
    sel, cnt = _select_and_compare(scores, lengths, 256)
    inp2 = dataclasses.replace(inp, sel=sel.clone(), sel_count=cnt.clone())
    inp2.kv_len[1] = 200
    run_and_compare(inp2)


# ---------------------------------------------------------------- edge cases

def test_selection_edge_cases_flags_and_skips():
    w = dataclasses.replace(W.SPARSE_BF16, top_k=64)
    inp = W.make_inputs(w, rows=4, t_override=700)
    # row 0: dense (-1); row 1: duplicates + unsorted; row 2: one out-of-range entry; row 3: count 0
    inp.sel_count[0] = -1
    inp.sel[1, :5] = torch.tensor([9, 3, 3, 600, 9], dtype=torch.int32)
    inp.sel_count[1] = 5
    inp.sel[2, 10] = 700          # == kv_len: outside the window
    inp.sel_count[3] = 0
    step = DecodeStep(inp, DEV, fused=False)
    step.run()
    fstep = DecodeStep(inp, DEV, fused=True)
    assert fstep.fused
    fstep.run()
    torch.cuda.synchronize()
    for s in (step, fstep):
        st = int(s.status.item())
        assert st & mla.DEVICE_INDEX_OUT_OF_RANGE and st & mla.DEVICE_BAD_SELECTION_COUNT
    # the oracle: row 2 without the bad entry, row 3 attends to nothing
    sel, cnt = inp.sel.clone(), inp.sel_count.clone()
    sel[2, 10:cnt[2] - 1] = inp.sel[2, 11:cnt[2]].clone()
    cnt[2] -= 1
    cnt[3] = 1                     # placeholder; row 3 checked separately
    inp2 = dataclasses.replace(inp, sel=sel, sel_count=cnt)
    ref = H.oracle_reference(inp2, rows=[0, 1, 2])
    H.compare_step(step, ref, "bf16")
    H.compare_step(fstep, ref, "bf16")
    assert torch.count_nonzero(step.ctx[3]) == 0
    for s in (step, fstep):
        assert torch.count_nonzero(s.out[3]) == 0
        assert torch.all(torch.isneginf(s.lse[3]))


def test_empty_and_short_rows():
    w = dataclasses.replace(W.VERIFY_BF16, top_k=0)
    inp = W.make_inputs(w, rows=3, t_override=400)
    inp.kv_len[1] = 0              # empty row: ctx 0, lse -inf
    inp.kv_len[2] = 2              # 4 query tokens over 2 keys: tokens 0, 1 see nothing
    ref = H.oracle_reference(inp)
    for fused in (False, True):
        step = DecodeStep(inp, DEV, fused=fused)
        assert step.fused == fused
        step.run()
        torch.cuda.synchronize()
        H.compare_step(step, ref, "bf16")


def test_gather_is_bit_exact():
    w = dataclasses.replace(W.SPARSE_BF16, top_k=128)
    inp = W.make_inputs(w, rows=3, t_override=3000, layout="padded")
    inp.sel_count[2] = -1
    dev = {k: getattr(inp, k).to(DEV) for k in ("latent", "rope_raw", "kv_start", "kv_len", "sel", "sel_count")}
    out = torch.full((3, 128, 576), 7, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.gather_selected(dev["latent"], dev["rope_raw"], dev["kv_start"], dev["kv_len"], 3, 1,
                        dev["sel"], dev["sel_count"], 128, out, st)
    want = O.gather_selected(inp.latent.view(torch.int16).numpy(), inp.rope_raw.view(torch.int16).numpy(),
                             inp.kv_start.numpy(), inp.kv_len.numpy(), 1, inp.sel.numpy(),
                             inp.sel_count.numpy(), 128)
    assert np.array_equal(out.cpu().view(torch.int16).numpy(), want)
    assert int(st.item()) == 0


# ---------------------------------------------------------------- full-size workloads (sampled)

SAMPLE_HEADS = [0, 1, 63, 64, 127]


@pytest.mark.slow
def test_ragged_full_size_sampled():
    inp = W.make_inputs(W.RAGGED_BF16, layout="flat")
    lens = inp.kv_len.numpy()
    rows = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 0, 31})
    run_and_compare(inp, rows=rows, heads=SAMPLE_HEADS)


@pytest.mark.slow
def test_sparse_full_size_sampled():
    inp = W.make_inputs(W.SPARSE_BF16)
    run_and_compare(inp, rows=[0, 7], heads=SAMPLE_HEADS)


@pytest.mark.slow
def test_verify_full_size_sampled():
    inp = W.make_inputs(W.VERIFY_SPARSE_BF16)
    rows = [0, 1, 2, 3, 30, 31]
    run_and_compare(inp, rows=rows, heads=SAMPLE_HEADS, with_selection=False)
    run_and_compare(inp, rows=rows, heads=SAMPLE_HEADS, with_selection=True)
