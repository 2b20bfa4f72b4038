"""The C-ABI library: it loads without a GPU, exports every function that
include/mla.h declares, and rejects bad arguments on the host before any
launch (these calls never reach a kernel)."""
import ctypes
import os
import re

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
    assert L.mla_decode_step_workspace_size(1, 1, 64, 128, 128, 512, 64, 4096, 0, 0, 1) == 0
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
