"""The C-ABI library: it loads without a GPU, exports every function that
include/mla.h declares, and rejects bad arguments on the host before any
launch (these calls never reach a kernel)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "mla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from mla_latent_kv_12_gb300 import mla
    return mla


def test_library_exports_every_header_function(lib):
    names = header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib.lib, n), n
    assert set(lib.EXPORTS) == set(names)


def test_status_strings(lib):
    assert lib.status_string(0) == "ok"
    assert lib.status_string(1) == "invalid argument"
    assert lib.status_string(99) == "unknown status"
    assert lib.lib.mla_version() >> 16 == 1


def _strides(*v):
    return (ctypes.c_int64 * 3)(*v)


@pytest.mark.parametrize("kw,needle", [
    (dict(rotary_dims=7), "rotary_dims"),
    (dict(rotary_dims=0), "rotary_dims"),
    (dict(rotary_dims=80), "rotary_dims"),
    (dict(theta=0.0), "theta"),
    (dict(theta=float("nan")), "theta"),
    (dict(offset=-1), "offset"),
    (dict(dtype=5), "dtype"),
    (dict(rows=0), "positive"),
])
def test_rope_validation(lib, kw, needle):
    a = dict(rotary_dims=64, theta=1e4, offset=0, dtype=1, rows=1)
    a.update(kw)
    s = _strides(64, 64, 64)
    st = lib.lib.mla_rope_partial_interleaved(16, 16, a["dtype"], a["rows"], 1, 1, 64, s, s,
                                              a["rotary_dims"], a["theta"], None, a["offset"], None)
    assert st == 1
    assert needle in lib.lib.mla_last_error_detail().decode()


def test_decode_validation(lib):
    L = lib.lib
    args = [16, 576, 576, 16, 576, 0, 16, 576, 0, 1, None, 16, 1, 1, 128, 512, 64, 4096,
            None, None, 0, 0.07, 16, 65536, 512, 1, None, None, 0, None, None]
    bad = list(args); bad[21] = -1.0                     # softmax scale
    assert L.mla_decode_attend(*bad) == 1
    bad = list(args); bad[11] = None                     # kv_len
    assert L.mla_decode_attend(*bad) == 1
    bad = list(args); bad[18] = 16                       # selection without counts
    assert L.mla_decode_attend(*bad) == 1
    bad = list(args); bad[2] = 100                       # head stride < rank + rope
    assert L.mla_decode_attend(*bad) == 1
    assert L.mla_decode_workspace_size(0, 1, 128, 512, 64, 4096, 0, 0, 1) == 0
    assert L.mla_decode_kernel_kind(128, 512, 64, 7, 1) == -1


def test_bf16_shapes_outside_the_fast_path_are_refused(lib):
    # bf16 is served for heads 64 / 128, rank 512, rope 64 (nope 128, v 128 for
    # the projections); anything else returns MLA_ERR_UNSUPPORTED before any
    # launch (the pointers here are not device memory: a launch would fault).
    L = lib.lib
    args = [16, 576, 576, 16, 576, 0, 16, 576, 0, 1, None, 16, 1, 1, 128, 512, 64, 4096,
            None, None, 0, 0.07, 16, 65536, 512, 1, None, None, 0, None, None]
    for i, v in [(14, 16), (14, 96), (15, 256), (16, 32)]:   # heads 16 / 96, rank 256, rope 32
        bad = list(args); bad[i] = v
        assert L.mla_decode_attend(*bad) == 2, (i, v)
        assert "bf16 is served" in L.mla_last_error_detail().decode()
    assert L.mla_decode_kernel_kind(128, 512, 64, 1, 1) == 1
    assert L.mla_decode_kernel_kind(64, 512, 64, 1, 1) == 1
    assert L.mla_decode_kernel_kind(16, 512, 64, 1, 1) == -1
    assert L.mla_decode_kernel_kind(16, 32, 8, 0, 0) == 0          # f32: CUDA cores, any shape
    assert L.mla_decode_workspace_size(1, 1, 16, 512, 64, 4096, 0, 0, 1) == 0
    assert L.mla_decode_workspace_size(1, 1, 64, 512, 64, 4096, 0, 0, 1) > 0
    # absorb: q_nope, strides, kv_b_proj, q_out, strides, dtype, n_q, heads, nope, v, rank
    assert L.mla_absorb_q(16, 0, 128, 16, 16, 0, 576, 1, 1, 16, 128, 128, 512, None) == 2
    assert L.mla_absorb_q(16, 0, 64, 16, 16, 0, 576, 1, 1, 128, 64, 128, 512, None) == 2
    assert "bf16 is served" in L.mla_last_error_detail().decode()
    # project: ctx, strides, kv_b_proj, dtype, out, stride, out dtype, n_q, heads, nope, v, rank
    assert L.mla_project_v(16, 0, 512, 16, 1, 16, 16 * 128, 1, 1, 16, 128, 128, 512, None) == 2
    assert L.mla_project_v(16, 0, 512, 16, 1, 16, 128 * 64, 1, 1, 128, 128, 64, 512, None) == 2


def test_default_scale_and_workspace_limits(lib):
    L = lib.lib
    import numpy as np
    assert L.mla_default_softmax_scale(128, 64) == np.float32(1.0 / np.sqrt(192.0))
    assert L.mla_default_softmax_scale(16, 8) == np.float32(1.0 / np.sqrt(24.0))
    assert L.mla_default_softmax_scale(0, 0) == 0.0
    assert lib.default_scale(128, 64) == float(np.float32(1.0 / np.sqrt(192.0)))
    # batch * s_q past the limits (and past int32) gives 0, not a wrapped size
    assert L.mla_decode_workspace_size(1 << 16, 1 << 16, 128, 512, 64, 4096, 0, 0, 1) == 0
    assert L.mla_decode_workspace_size(1 << 20, 2, 128, 512, 64, 4096, 0, 0, 1) == 0
    assert L.mla_decode_workspace_size(1 << 20, 1, 128, 512, 64, 4096, 0, 0, 1) > 0
    assert L.mla_decode_workspace_size(1 << 16, 1 << 16, 4, 32, 8, 64, 0, 0, 0) == 0


def test_absorb_and_project_validation(lib):
    L = lib.lib
    assert L.mla_absorb_q(None, 0, 128, 16, 16, 0, 576, 1, 1, 128, 128, 128, 512, None) == 1
    assert L.mla_absorb_q(16, 0, 128, 16, 16, 0, 576, 1, 0, 128, 128, 128, 512, None) == 1
    assert L.mla_project_v(16, 0, 512, 16, 1, 16, 100, 1, 1, 128, 128, 128, 512, None) == 1
    assert L.mla_gather_selected(16, 576, 0, 16, 576, 0, 1, None, 16, 1, 1, 512, 64, 100,
                                 16, None, 8, 16, None, None) == 1


def test_decode_step_validation(lib):
    L = lib.lib
    # q_nope, strides, q_rope, strides, offsets, offset, theta, kv_b_proj, latent, strides, rope, strides,
    # dtype, kv_start, kv_len, B, S, H, nope, v, rank, rope, T, sel, counts, k_max, scale, out, stride,
    # out dtype, lse, workspace, bytes, status, stream
    args = [16, 16384, 128, 16, 8192, 64, None, 0, 1e4, 16, 16, 512, 0, 16, 64, 0,
            1, None, 16, 1, 1, 128, 128, 128, 512, 64, 4096, None, None, 0, 0.07, 16, 16384,
            1, None, 256, 1 << 30, None, None]
    bad = list(args); bad[0] = None                      # q_nope
    assert L.mla_decode_step(*bad) == 1
    bad = list(args); bad[8] = 0.0                       # theta
    assert L.mla_decode_step(*bad) == 1
    bad = list(args); bad[16] = 0                        # f32: not served by the fused step
    assert L.mla_decode_step(*bad) == 2
    assert "compose" in L.mla_last_error_detail().decode()
    bad = list(args); bad[19] = 65                       # 65 query rows
    assert L.mla_decode_step(*bad) == 2
    bad = list(args); bad[36] = 1024                     # workspace too small
    assert L.mla_decode_step(*bad) == 1
    assert L.mla_decode_step_workspace_size(1, 1, 128, 128, 128, 512, 64, 4096, 0, 0, 1) > 0
    assert L.mla_decode_step_workspace_size(1, 1, 64, 128, 128, 512, 64, 4096, 0, 0, 1) > 0
    assert L.mla_decode_step_workspace_size(1, 1, 32, 128, 128, 512, 64, 4096, 0, 0, 1) == 0
    assert L.mla_decode_step_workspace_size(1, 1, 128, 128, 128, 512, 64, 4096, 0, 0, 0) == 0


def test_append_validation(lib):
    L = lib.lib
    # latent_raw, strides, rope_raw, strides, dtype, weight, eps, theta, offsets, latent, strides, rope, strides,
    # cache dtype, kv_start, kv_len, kv_len_out, B, S, rank, rope, T, status, stream
    args = [16, 512, 512, 16, 64, 64, 1, 16, 1e-6, 1e4, None, 16, 512, 0, 16, 64, 0, 1, None, 16, None,
            1, 1, 512, 64, 128, None, None]
    for i, v in [(0, None), (8, -1.0), (9, 0.0), (23, 2048), (24, 63), (21, 0), (19, None), (6, 5)]:
        bad = list(args); bad[i] = v
        assert L.mla_append_compressed(*bad) == 1, i
    assert "epsilon" in (bad := list(args), bad.__setitem__(8, float("nan")), L.mla_append_compressed(*bad),
                         L.mla_last_error_detail().decode())[3]


def test_select_validation(lib):
    L = lib.lib
    args = [16, 4096, 16, 2, 64, 16, 64, 16, None, None]
    for i, v in [(0, None), (3, 0), (4, 0), (6, 32), (2, None)]:
        bad = list(args); bad[i] = v
        assert L.mla_select_topk(*bad) == 1, i


def test_selftest_validation(lib):
    L = lib.lib
    assert L.mla_selftest_bounded_wait(1000, None, None, None) == 1
    assert L.mla_selftest_bounded_wait(0, 16, None, None) == 1
    assert L.mla_selftest_bounded_wait((1 << 32) + 1, 16, None, None) == 1


def test_shift_rows_and_rollback_lengths_validation(lib):
    L = lib.lib
    # src, token stride, batch stride, src batch, src width, dst, token stride, batch stride, dst width,
    # features, dtype, src_row, shift, zero_below, n_rows, status, stream
    MB = 1 << 20
    args = [16 * MB, 512, 512 * 64, 2, 64, 64 * MB, 512, 512 * 64, 60, 512, 1, None, None, None, 2, None, None]
    for i, v in [(0, None), (5, None), (10, 5), (9, 0), (14, 0), (14, 70000), (1, 256), (6, 256), (7, 512),
                 (4, -1), (8, -1), (5, 16 * MB + 4096)]:          # the last one: destination overlaps source
        bad = list(args); bad[i] = v
        assert L.mla_cache_shift_rows(*bad) == 1, i
    assert "overlap" in L.mla_last_error_detail().decode()
    zero_width = list(args); zero_width[8] = 0                    # nothing to write: no launch, ok
    assert L.mla_cache_shift_rows(*zero_width) == 0
    assert L.mla_rollback_lengths(None, 16, 16, 16, 4, None, None) == 1
    assert L.mla_rollback_lengths(16, 16, 16, 16, 0, None, None) == 1


# ------------------------------------------------ host plans of the cache row operations

def _right_aligned(rng_, B, width, lo=0):
    offs = rng_.integers(lo, width + 1, B)
    return width - offs, offs


def _apply_plan(a, width_out, shift, src_row=None, zero_below=None):
    """The gather the row kernel performs, per its contract, on a host array."""
    B_out = len(shift)
    out = np.zeros((B_out, width_out, a.shape[2]), a.dtype)
    for i in range(B_out):
        r = i if src_row is None else src_row[i]
        for c in range(width_out):
            if zero_below is not None and c < zero_below[i]:
                continue
            out[i, c] = a[r, (c + int(shift[i])) % a.shape[1]]
    return out


def test_rollback_plan_matches_the_oracle(lib):
    from oracle import mla_oracle as O
    r = np.random.default_rng(80)
    for trial in range(20):
        B, appended = int(r.integers(1, 6)), int(r.integers(0, 5))
        width = int(r.integers(appended, 20))
        pad, offs = _right_aligned(r, B, width, lo=appended)
        before = offs - appended
        keep = r.integers(0, appended + 1, B)
        a = r.standard_normal((B, width, 3))
        shift, new_pad, new_off, new_width = lib.plan_rollback(pad, offs, before, keep, width)
        (want,), w, off_o, pad_o = O.rollback_right_aligned([a], pad, offs, before, keep)
        assert new_width == w and list(new_off) == list(off_o) and list(new_pad) == list(pad_o)
        assert np.array_equal(_apply_plan(a, new_width, shift.numpy()), want)


def test_filter_and_merge_plans_match_the_oracle(lib):
    from oracle import mla_oracle as O
    r = np.random.default_rng(81)
    for trial in range(20):
        B, width = int(r.integers(1, 6)), int(r.integers(1, 16))
        pad, offs = _right_aligned(r, B, width)
        a = r.standard_normal((B, width, 2))
        for b in range(B):
            a[b, :pad[b]] = 0.0
        keep = r.integers(0, B, int(r.integers(1, B + 2)))
        shift, new_pad, new_off, new_width = lib.plan_filter(pad, offs, keep, width)
        (want,), w, off_o, pad_o = O.filter_right_aligned([a], pad, offs, keep)
        assert new_width == w and list(new_off) == list(off_o) and list(new_pad) == list(pad_o)
        assert np.array_equal(_apply_plan(a, new_width, shift.numpy(), src_row=keep), want)
        # merge this cache with a second one of another width
        B2, width2 = int(r.integers(1, 4)), int(r.integers(1, 24))
        pad2, offs2 = _right_aligned(r, B2, width2)
        a2 = r.standard_normal((B2, width2, 2))
        shift, zero, new_pad, w_m = lib.plan_merge([width] * B + [width2] * B2, list(pad) + list(pad2),
                                                   list(offs) + list(offs2))
        (want,), w, off_o, pad_o = O.merge_right_aligned([([a], pad, offs), ([a2], pad2, offs2)])
        assert w_m == w and list(new_pad) == list(pad_o)
        if w:
            got = np.concatenate([_apply_plan(a, w, shift[:B].numpy(), zero_below=zero[:B].numpy()),
                                  _apply_plan(a2, w, shift[B:].numpy(), zero_below=zero[B:].numpy())])
            assert np.array_equal(got, want)


def test_row_plans_reject_bad_bookkeeping(lib):
    with pytest.raises(lib.MLAError, match="right-aligned"):
        lib.plan_rollback([1, 0], [3, 3], [1, 1], [0, 0], 4)             # 0 + 3 != 4
    with pytest.raises(lib.MLAError, match="keeps"):
        lib.plan_rollback([0, 1], [4, 3], [2, 2], [3, 0], 4)             # keeps 5 of 4
    with pytest.raises(lib.MLAError, match="outside"):
        lib.plan_filter([0, 1], [4, 3], [2], 4)
    with pytest.raises(lib.MLAError, match="right-aligned"):
        lib.plan_merge([4, 5], [0, 1], [4, 3])


def test_reconstruct_and_prefill_validation(lib):
    L = lib.lib
    MB = 1 << 20
    # latent, row stride, rows, kv_b_proj, H, nope, v, rank, k, k strides, v, v strides, dtype, status, stream
    rec = [16 * MB, 512, 300, 64 * MB, 128, 128, 128, 512, 128 * MB, 128 * 256, 256, 128 * MB + 256, 128 * 256,
           256, 1, None, None]
    for i, v, want in [(0, None, 1), (2, 0, 1), (14, 5, 1), (1, 256, 1), (9, 64, 1), (5, 64, 2), (14, 0, 2),
                       (0, 16 * MB + 2, 1)]:
        bad = list(rec); bad[i] = v
        assert L.mla_reconstruct_kv(*bad) == want, (i, v)
    # q_nope + strides, q_rope + strides, k + strides, v + strides, rope + stride, packed, dtype, kv_start,
    # kv_len, B, S, H, nope, rope, v, t_max, scale, out, out stride, out dtype, lse, status, stream
    pf = [16 * MB, 128 * 128, 128, 20 * MB, 128 * 64, 64, 32 * MB, 128 * 256, 256, 32 * MB + 256, 128 * 256, 256,
          48 * MB, 64, 0, 1, 16, 32, 2, 300, 128, 128, 64, 128, 700, 0.07, 64 * MB, 128 * 128, 1, None, None, None]
    for i, v, want in [(0, None, 1), (16, None, 1), (19, 0, 1), (25, 0.0, 1), (25, float("inf"), 1),
                       (27, 1000, 1), (21, 96, 2), (22, 96, 1), (15, 0, 2), (26, 64 * MB + 8, 1), (1, 100, 1)]:
        bad = list(pf); bad[i] = v
        assert L.mla_prefill_attend(*bad) == want, (i, v)


def test_row_plans_random_cases_match_the_oracle(lib):
    # many random right-aligned caches: bookkeeping and the planned gather
    # reproduce the oracle's rollback, filter and merge exactly
    from oracle import mla_oracle as O
    r = np.random.default_rng(82)
    for trial in range(200):
        B, width = int(r.integers(1, 5)), int(r.integers(0, 12))
        appended = int(r.integers(0, width + 1))
        offs = r.integers(appended, width + 1, B)
        pad = width - offs
        a = r.integers(-50, 50, (B, max(width, 1), 1)).astype(np.float64)[:, :width]
        before = offs - appended
        keep = r.integers(0, appended + 1, B)
        shift, new_pad, new_off, new_width = lib.plan_rollback(pad, offs, before, keep, width)
        (want,), w, off_o, pad_o = O.rollback_right_aligned([a], pad, offs, before, keep)
        assert (new_width, list(new_off), list(new_pad)) == (w, list(off_o), list(pad_o))
        if width:
            assert np.array_equal(_apply_plan(a, new_width, shift.numpy()), want)
            keep_rows = r.integers(0, B, int(r.integers(1, 4)))
            shift, new_pad, new_off, new_width = lib.plan_filter(pad, offs, keep_rows, width)
            (want,), w, off_o, pad_o = O.filter_right_aligned([a], pad, offs, keep_rows)
            assert (new_width, list(new_off), list(new_pad)) == (w, list(off_o), list(pad_o))
            assert np.array_equal(_apply_plan(a, new_width, shift.numpy(), src_row=keep_rows), want)
