"""Cache row operations on the device (rollback, filter, merge of the
right-aligned layout; rollback of the per-row window layout) against the
oracle: bit-exact for the moved rows, and a decode over a rolled-back cache
against the oracle's attention over each row's accepted prefix."""
import numpy as np
import pytest
import torch

from oracle import mla_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from mla_latent_kv_12_gb300 import cache_rows as CR
    from mla_latent_kv_12_gb300 import mla

DEV = "cuda"


def _states(g, B, width):
    """latent bf16 [.,512], rope bf16 [.,64], indexer keys f32 [.,128], and two odd
    widths (f32 x3, bf16 x5) that take the narrower vector paths; pads hold junk."""
    shapes = [(512, torch.bfloat16), (64, torch.bfloat16), (128, torch.float32), (3, torch.float32),
              (5, torch.bfloat16)]
    return [torch.randn(B, width, f, generator=g).to(dt) for f, dt in shapes]


def _f64(t):
    return t.to(torch.float64).numpy()


def _same_bits(got, want64, what):
    want = torch.from_numpy(want64).to(got.dtype)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bits = torch.int16 if got.dtype == torch.bfloat16 else torch.int32
    assert torch.equal(got.cpu().view(bits), want.view(bits)), what


def test_rollback_is_the_oracles_rotation_bit_exact():
    g = torch.Generator().manual_seed(90)
    B, width, appended = 7, 777, 5
    offs = np.array([777, 700, 5, 431, 777, 6, 100])
    pad = width - offs
    before = offs - appended
    keep = np.array([5, 0, 0, 3, 2, 5, 1])
    states = _states(g, B, width)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, new_width, new_off, new_pad = CR.rollback([s.to(DEV) for s in states], pad, offs, before, keep,
                                                   device_status=st)
    torch.cuda.synchronize()
    want, w, off_o, pad_o = O.rollback_right_aligned([_f64(s) for s in states], pad, offs, before, keep)
    assert int(st.item()) == 0 and new_width == w
    assert list(new_off.numpy()) == list(off_o) and list(new_pad.numpy()) == list(pad_o)
    for k, (a, b) in enumerate(zip(out, want)):
        _same_bits(a, b, f"state {k}")


def test_filter_and_merge_are_the_oracles_bit_exact():
    g = torch.Generator().manual_seed(91)
    width = 300
    offs = np.array([120, 0, 299, 37])
    pad = width - offs
    states = _states(g, 4, width)
    dev_states = [s.to(DEV) for s in states]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    keep = [3, 0, 0, 1]                                       # duplicates and an empty row
    out, w, off, new_pad = CR.filter_rows(dev_states, pad, offs, keep, device_status=st)
    want, w_o, off_o, pad_o = O.filter_right_aligned([_f64(s) for s in states], pad, offs, keep)
    torch.cuda.synchronize()
    assert w == w_o == 120                                   # the longest kept row (120) fills the width
    for k, (a, b) in enumerate(zip(out, want)):
        _same_bits(a, b, f"filter state {k}")
    # merge: the filtered cache, an empty cache (width 0) and a wider one
    g2 = torch.Generator().manual_seed(92)
    width3, offs3 = 450, np.array([3, 450])
    states3 = _states(g2, 2, width3)
    empty = [torch.empty((2, 0, s.shape[2]), dtype=s.dtype) for s in states]
    caches_dev = [(out, new_pad.numpy(), off.numpy()), ([e.to(DEV) for e in empty], [0, 0], [0, 0]),
                  ([s.to(DEV) for s in states3], width3 - offs3, offs3)]
    merged, w_m, off_m, pad_m = CR.merge(caches_dev, device_status=st)
    torch.cuda.synchronize()
    caches_o = [([b for b in want], pad_o, off_o), ([_f64(e) for e in empty], [0, 0], [0, 0]),
                ([_f64(s) for s in states3], width3 - offs3, offs3)]
    want_m, w_mo, off_mo, pad_mo = O.merge_right_aligned(caches_o)
    assert int(st.item()) == 0 and w_m == w_mo == 450
    assert list(off_m.numpy()) == list(off_mo) and list(pad_m.numpy()) == list(pad_mo)
    for k, (a, b) in enumerate(zip(merged, want_m)):
        _same_bits(a, b, f"merge state {k}")


def test_decode_over_a_rolled_back_cache_attends_to_the_accepted_prefix():
    g = torch.Generator().manual_seed(93)
    B, width, H_, rank, rope_dim = 4, 1100, 128, 512, 64
    offs = np.array([1100, 640, 1033, 70])
    pad = width - offs
    before = offs - 4
    keep = np.array([1, 4, 0, 2])
    lat = torch.randn(B, width, rank, generator=g).to(torch.bfloat16)
    rp = torch.randn(B, width, rope_dim, generator=g).to(torch.bfloat16)
    (lat2, rp2), w2, off2, pad2 = CR.rollback([lat.to(DEV), rp.to(DEV)], pad, offs, before, keep)
    q = (torch.randn(B, H_, rank + rope_dim, generator=g) * 0.05).to(torch.bfloat16)
    ctx = torch.empty(B, H_, rank, dtype=torch.float32, device=DEV)
    lse = torch.empty(B, H_, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    scale = 1.0 / np.sqrt(192.0)
    mla.decode_attend(q.to(DEV), lat2, rp2, pad2.to(DEV), off2.to(DEV), B, 1, scale, ctx, lse_out=lse,
                      device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    qf = _f64(q)
    want, want_lse = O.attend_latent(qf[..., :rank], qf[..., rank:], H.Rows(lat), H.Rows(rp), pad,
                                     before + keep, 1, None, None, scale)
    H.assert_close(ctx.cpu(), want, "bf16", "ctx")          # bf16 cache, Q and P: the bf16 bound
    assert np.max(np.abs(lse.cpu().numpy() - want_lse)) < 1e-3


def test_rollback_lengths_in_place_and_flags_bad_rows():
    kv_len = torch.tensor([10, 7, 3, 9], dtype=torch.int32, device=DEV)
    before = torch.tensor([6, 7, 1, 2], dtype=torch.int32, device=DEV)
    keep = torch.tensor([2, 0, 5, 3], dtype=torch.int32, device=DEV)    # row 2 would keep 6 of 3
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.rollback_lengths(before, keep, kv_len, device_status=st)
    torch.cuda.synchronize()
    assert kv_len.cpu().tolist() == [8, 7, 3, 5]
    assert int(st.item()) == mla.DEVICE_INDEX_OUT_OF_RANGE


def test_shift_rows_flags_a_bad_source_row_and_leaves_it_unwritten():
    src = torch.randn(2, 40, 64, device=DEV).to(torch.bfloat16)
    dst = torch.full((3, 40, 64), 7.0, device=DEV, dtype=torch.bfloat16)
    rows = torch.tensor([1, 2, 0], dtype=torch.int32, device=DEV)          # 2 is outside [0, 2)
    shift = torch.tensor([0, 0, -3], dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.cache_shift_rows(src, dst, shift=shift, src_row=rows, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == mla.DEVICE_INDEX_OUT_OF_RANGE
    assert torch.equal(dst[0], src[1]) and torch.all(dst[1] == 7.0)
    assert torch.equal(dst[2], torch.roll(src[0], 3, dims=0))                # column c takes (c - 3) mod 40
