"""Host logic of the cache row operations (cache_rows.py): the library's host
plans plus the composition that slices them per state array and per merged
source, checked on CPU against the oracle.  The row gather itself is the GPU
kernel; here a CPU stand-in of its documented contract takes its place (only
in this test), so that everything around it runs as on the device."""
import numpy as np
import pytest
import torch

from oracle import mla_oracle as O


def _gather_contract(src, dst, shift=None, src_row=None, zero_below=None, device_status=None, stream=None):
    """dst[i, c] = c < zero_below[i] ? 0 : src[src_row[i], (c + shift[i]) mod src_width]."""
    n, width = dst.shape[0], dst.shape[1]
    for i in range(n):
        r = i if src_row is None else int(src_row[i])
        z = 0 if zero_below is None else int(zero_below[i])
        sh = 0 if shift is None else int(shift[i])
        for c in range(width):
            dst[i, c] = 0 if c < z else src[r, (c + sh) % src.shape[1]]
    return dst


@pytest.fixture()
def cr(monkeypatch):
    from mla_latent_kv_12_gb300 import cache_rows, mla
    monkeypatch.setattr(mla, "cache_shift_rows", _gather_contract)
    return cache_rows


def _tagged(offsets, width, feats=2):
    a = torch.full((len(offsets), width, feats), -1.0, dtype=torch.float64)
    for b, o in enumerate(offsets):
        for j in range(o):
            a[b, width - o + j] = torch.tensor([b, j], dtype=torch.float64)[:feats]
    return a, np.array([width - o for o in offsets]), np.array(offsets)


def test_rollback_composition_matches_the_oracle(cr):
    before, keep = [4, 1, 6], [2, 0, 3]
    offsets = [b + 3 for b in before]
    a, pad, offs = _tagged(offsets, 9)
    b2 = a * 10.0
    (o1, o2), w, off, new_pad = cr.rollback([a, b2], pad, offs, before, keep)
    (w1, w2), ww, woff, wpad = O.rollback_right_aligned([a.numpy(), b2.numpy()], pad, offs, before, keep)
    assert w == ww and list(off.numpy()) == list(woff) and list(new_pad.numpy()) == list(wpad)
    assert np.array_equal(o1.numpy(), w1) and np.array_equal(o2.numpy(), w2)


def test_filter_and_merge_composition_matches_the_oracle(cr):
    a, pad, offs = _tagged([3, 7, 0, 5], 8)
    out, w, off, new_pad = cr.filter_rows([a], pad, offs, [3, 0, 0])
    want, ww, woff, wpad = O.filter_right_aligned([a.numpy()], pad, offs, [3, 0, 0])
    assert w == ww and np.array_equal(out[0].numpy(), want[0])
    # three sources of different widths, one of them empty (width 0)
    b, pad_b, offs_b = _tagged([6, 2], 6)
    e = torch.empty((2, 0, 2), dtype=torch.float64)
    a0 = a.clone()
    for r in range(4):
        a0[r, :pad[r]] = 0.0
    merged, wm, offm, padm = cr.merge([([a0], pad, offs), ([e], [0, 0], [0, 0]), ([b], pad_b, offs_b)])
    want, wmo, offmo, padmo = O.merge_right_aligned([([a0.numpy()], pad, offs), ([e.numpy()], [0, 0], [0, 0]),
                                                     ([b.numpy()], pad_b, offs_b)])
    assert wm == wmo == 7 and list(offm.numpy()) == list(offmo) and list(padm.numpy()) == list(padmo)
    assert np.array_equal(merged[0].numpy(), want[0])
