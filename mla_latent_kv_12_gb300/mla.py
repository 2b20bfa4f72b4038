"""Thin ctypes binding of libmla (the C ABI declared in ``include/mla.h``).

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream.  Importing this module
fails loudly if the built library is missing; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla.so")

F32, BF16 = 0, 1
DEVICE_BAD_SELECTION_COUNT = 1 << 1
DEVICE_INDEX_OUT_OF_RANGE = 1 << 4
DEVICE_TIMEOUT = 1 << 5
DEVICE_LAYOUT = 1 << 6
DEVICE_SCORE_RANGE = 1 << 7
DEVICE_VALUE_RANGE = 1 << 8
FP16_SCORE_LIMIT = 256.0

_DT = {torch.float32: F32, torch.bfloat16: BF16}

EXPORTS = (
    "mla_status_string", "mla_last_error_detail", "mla_version", "mla_default_softmax_scale",
    "mla_rope_partial_interleaved", "mla_absorb_q", "mla_decode_attend",
    "mla_decode_workspace_size", "mla_decode_kernel_kind", "mla_project_v",
    "mla_gather_selected", "mla_decode_attend_no_alloc", "mla_decode_step",
    "mla_decode_step_workspace_size", "mla_append_compressed", "mla_select_topk",
    "mla_selftest_bounded_wait", "mla_plan_rollback", "mla_plan_filter", "mla_plan_merge",
    "mla_cache_shift_rows", "mla_rollback_lengths", "mla_reconstruct_kv", "mla_prefill_attend",
)


class MLAError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"mla status {status}: {detail}")
        self.status = status
        self.detail = detail


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmla.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    i64, i32, vp, f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_float
    sz = ctypes.c_size_t
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_status_string.argtypes = [ctypes.c_int]
    lib.mla_last_error_detail.restype = ctypes.c_char_p
    lib.mla_last_error_detail.argtypes = []
    lib.mla_version.restype = ctypes.c_int
    lib.mla_default_softmax_scale.restype = f32
    lib.mla_default_softmax_scale.argtypes = [i32, i32]
    lib.mla_rope_partial_interleaved.restype = ctypes.c_int
    lib.mla_rope_partial_interleaved.argtypes = [vp, vp, ctypes.c_int, i64, i64, i64, i64, i64p, i64p,
                                                 i32, f32, vp, i64, vp]
    lib.mla_absorb_q.restype = ctypes.c_int
    lib.mla_absorb_q.argtypes = [vp, i64, i64, vp, vp, i64, i64, ctypes.c_int, i32, i32, i32, i32, i32, vp]
    lib.mla_decode_attend.restype = ctypes.c_int
    lib.mla_decode_attend.argtypes = [vp, i64, i64, vp, i64, i64, vp, i64, i64, ctypes.c_int, vp, vp,
                                      i32, i32, i32, i32, i32, i64, vp, vp, i32, f32, vp, i64, i64,
                                      ctypes.c_int, vp, vp, sz, vp, vp]
    lib.mla_decode_workspace_size.restype = sz
    lib.mla_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i64, i32, ctypes.c_int, ctypes.c_int]
    lib.mla_decode_kernel_kind.restype = ctypes.c_int
    lib.mla_decode_kernel_kind.argtypes = [i32, i32, i32, ctypes.c_int, ctypes.c_int]
    lib.mla_project_v.restype = ctypes.c_int
    lib.mla_project_v.argtypes = [vp, i64, i64, vp, ctypes.c_int, vp, i64, ctypes.c_int, i32, i32, i32,
                                  i32, i32, vp]
    lib.mla_decode_attend_no_alloc.restype = ctypes.c_int
    lib.mla_decode_attend_no_alloc.argtypes = [vp, i64, i64, vp, i64, i64, vp, i64, i64, ctypes.c_int, vp,
                                               vp, i32, i32, i32, i32, i32, i64, vp, vp, i32, f32, vp, i64,
                                               i64, ctypes.c_int, vp, vp, vp]
    lib.mla_decode_step.restype = ctypes.c_int
    lib.mla_decode_step.argtypes = [vp, i64, i64, vp, i64, i64, vp, i64, f32, vp, vp, i64, i64, vp, i64, i64,
                                    ctypes.c_int, vp, vp, i32, i32, i32, i32, i32, i32, i32, i64, vp, vp, i32,
                                    f32, vp, i64, ctypes.c_int, vp, vp, sz, vp, vp]
    lib.mla_decode_step_workspace_size.restype = sz
    lib.mla_decode_step_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i64, i32, ctypes.c_int,
                                                   ctypes.c_int]
    lib.mla_append_compressed.restype = ctypes.c_int
    lib.mla_append_compressed.argtypes = [vp, i64, i64, vp, i64, i64, ctypes.c_int, vp, f32, f32, vp, vp, i64,
                                          i64, vp, i64, i64, ctypes.c_int, vp, vp, vp, i32, i32, i32, i32, i64,
                                          vp, vp]
    lib.mla_select_topk.restype = ctypes.c_int
    lib.mla_select_topk.argtypes = [vp, i64, vp, i32, i32, vp, i64, vp, vp, vp]
    lib.mla_selftest_bounded_wait.restype = ctypes.c_int
    lib.mla_selftest_bounded_wait.argtypes = [i64, vp, vp, vp]
    for name, args in (("mla_plan_rollback", [i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]),
                       ("mla_plan_filter", [i32, i32, vp, vp, vp, i32, vp, vp, vp, vp]),
                       ("mla_plan_merge", [i32, vp, vp, vp, vp, vp, vp, vp]),
                       ("mla_cache_shift_rows", [vp, i64, i64, i32, i32, vp, i64, i64, i32, i32,
                                                 ctypes.c_int, vp, vp, vp, i32, vp, vp]),
                       ("mla_rollback_lengths", [vp, vp, vp, vp, i32, vp, vp]),
                       ("mla_reconstruct_kv", [vp, i64, i64, vp, i32, i32, i32, i32, vp, i64, i64, vp, i64, i64,
                                               ctypes.c_int, vp, vp]),
                       ("mla_prefill_attend", [vp, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64,
                                               ctypes.c_int, ctypes.c_int, vp, vp, i32, i32, i32, i32, i32, i32,
                                               i64, f32, vp, i64, ctypes.c_int, vp, vp, vp])):
        getattr(lib, name).restype = ctypes.c_int
        getattr(lib, name).argtypes = args
    lib.mla_gather_selected.restype = ctypes.c_int
    lib.mla_gather_selected.argtypes = [vp, i64, i64, vp, i64, i64, ctypes.c_int, vp, vp, i32, i32, i32,
                                        i32, i64, vp, vp, i32, vp, vp, vp]
    return lib


lib = _load()


def _check(status: int) -> None:
    if status != 0:
        raise MLAError(status, lib.mla_last_error_detail().decode())


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dt(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return _DT[t.dtype]


def status_string(status: int) -> str:
    return lib.mla_status_string(status).decode()


# ---------------------------------------------------------------- entry points

def rope_partial_interleaved(x: torch.Tensor, out: torch.Tensor, rotary_dims: int, theta: float,
                             position_offset: int = 0, row_offsets: Optional[torch.Tensor] = None,
                             stream=None) -> torch.Tensor:
    """``x`` / ``out``: 4-D ``[rows, tokens, inner, width]`` views (last dim contiguous)."""
    assert x.dim() == 4 and out.shape == x.shape and x.dtype == out.dtype
    assert x.stride(3) == 1 and out.stride(3) == 1
    ins = (ctypes.c_int64 * 3)(*x.stride()[:3])
    outs = (ctypes.c_int64 * 3)(*out.stride()[:3])
    _check(lib.mla_rope_partial_interleaved(
        _ptr(x), _ptr(out), _dt(x), x.shape[0], x.shape[1], x.shape[2], x.shape[3], ins, outs,
        rotary_dims, float(theta), _ptr(row_offsets), int(position_offset), _stream(stream)))
    return out


def absorb_q(q_nope: torch.Tensor, kv_b_proj: torch.Tensor, q_out: torch.Tensor, heads: int,
             nope: int, v_dim: int, rank: int, stream=None) -> torch.Tensor:
    """``q_nope`` ``[n_q, H, >=nope]`` view; writes ``q_out[:, :, :rank]``."""
    assert q_nope.dim() == 3 and q_out.dim() == 3 and q_nope.stride(2) == 1 and q_out.stride(2) == 1
    assert kv_b_proj.is_contiguous()
    _check(lib.mla_absorb_q(_ptr(q_nope), q_nope.stride(0), q_nope.stride(1), _ptr(kv_b_proj),
                            _ptr(q_out), q_out.stride(0), q_out.stride(1), _dt(q_nope),
                            q_nope.shape[0], heads, nope, v_dim, rank, _stream(stream)))
    return q_out


def decode_workspace_size(batch, s_q, heads, rank, rope_dim, t_max, k_max=0, selected=False,
                          dtype=torch.bfloat16) -> int:
    return lib.mla_decode_workspace_size(batch, s_q, heads, rank, rope_dim, t_max, k_max,
                                         1 if selected else 0, _DT[dtype])


def decode_kernel_kind(heads, rank, rope_dim, dtype=torch.bfloat16, out_dtype=torch.bfloat16) -> int:
    return lib.mla_decode_kernel_kind(heads, rank, rope_dim, _DT[dtype], _DT[out_dtype])


def decode_attend(q: torch.Tensor, latent: torch.Tensor, rope: torch.Tensor, kv_start, kv_len,
                  batch: int, s_q: int, softmax_scale: float, ctx_out: torch.Tensor,
                  lse_out: Optional[torch.Tensor] = None, sel: Optional[torch.Tensor] = None,
                  sel_count: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                  device_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """``q`` ``[n_q, H, rank+rope]``; ``latent`` ``[B_buf, T_max, rank]`` and ``rope``
    ``[B_buf, T_max, rope]`` views (a batch stride of 0 for the packed-flat layout is
    expressed by passing ``B_buf == 1``); ``ctx_out`` ``[n_q, H, rank]``."""
    n_q, heads, _ = q.shape
    rank, rope_dim = latent.shape[-1], rope.shape[-1]
    t_max = latent.shape[1]
    lat_bs = latent.stride(0) if latent.shape[0] > 1 else 0
    rope_bs = rope.stride(0) if rope.shape[0] > 1 else 0
    k_max = sel.shape[1] if sel is not None else 0
    if workspace is None:
        nbytes = decode_workspace_size(batch, s_q, heads, rank, rope_dim, t_max, k_max,
                                       sel is not None, latent.dtype)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    _check(lib.mla_decode_attend(
        _ptr(q), q.stride(0), q.stride(1), _ptr(latent), latent.stride(1), lat_bs,
        _ptr(rope), rope.stride(1), rope_bs, _dt(latent), _ptr(kv_start), _ptr(kv_len),
        batch, s_q, heads, rank, rope_dim, t_max, _ptr(sel), _ptr(sel_count), k_max,
        float(softmax_scale), _ptr(ctx_out), ctx_out.stride(0), ctx_out.stride(1), _dt(ctx_out),
        _ptr(lse_out), _ptr(workspace), workspace.numel(), _ptr(device_status), _stream(stream)))
    return ctx_out


def project_v(ctx: torch.Tensor, kv_b_proj: torch.Tensor, out: torch.Tensor, heads: int, nope: int,
              v_dim: int, stream=None) -> torch.Tensor:
    """``ctx`` ``[n_q, H, rank]`` view; ``out`` ``[n_q, H*v]`` (row stride free)."""
    n_q, _, rank = ctx.shape
    assert ctx.stride(2) == 1 and out.stride(1) == 1 and kv_b_proj.is_contiguous()
    _check(lib.mla_project_v(_ptr(ctx), ctx.stride(0), ctx.stride(1), _ptr(kv_b_proj), _dt(ctx),
                             _ptr(out), out.stride(0), _dt(out), n_q, heads, nope, v_dim, rank,
                             _stream(stream)))
    return out


def decode_step_workspace_size(batch, s_q, heads, nope, v_dim, rank, rope_dim, t_max, k_max=0,
                               selected=False, dtype=torch.bfloat16) -> int:
    return lib.mla_decode_step_workspace_size(batch, s_q, heads, nope, v_dim, rank, rope_dim, t_max, k_max,
                                              1 if selected else 0, _DT[dtype])


def decode_step(q_nope: torch.Tensor, q_rope: torch.Tensor, theta: float, kv_b_proj: torch.Tensor,
                latent: torch.Tensor, rope: torch.Tensor, kv_start, kv_len, batch: int, s_q: int, nope: int,
                v_dim: int, softmax_scale: float, out: torch.Tensor, lse_out: Optional[torch.Tensor] = None,
                row_offsets: Optional[torch.Tensor] = None, position_offset: int = 0,
                sel: Optional[torch.Tensor] = None, sel_count: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None, device_status: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    """Fused decode step.  ``q_nope`` ``[n_q, H, >=nope]`` and ``q_rope`` ``[n_q, H, >=rope]`` views
    (raw, pair-interleaved); cache views as for ``decode_attend``; ``out`` ``[n_q, H*v]``."""
    n_q, heads, _ = q_nope.shape
    rank, rope_dim = latent.shape[-1], rope.shape[-1]
    t_max = latent.shape[1]
    lat_bs = latent.stride(0) if latent.shape[0] > 1 else 0
    rope_bs = rope.stride(0) if rope.shape[0] > 1 else 0
    k_max = sel.shape[1] if sel is not None else 0
    if workspace is None:
        nbytes = decode_step_workspace_size(batch, s_q, heads, nope, v_dim, rank, rope_dim, t_max, k_max,
                                            sel is not None, latent.dtype)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=latent.device)
    _check(lib.mla_decode_step(
        _ptr(q_nope), q_nope.stride(0), q_nope.stride(1), _ptr(q_rope), q_rope.stride(0), q_rope.stride(1),
        _ptr(row_offsets), int(position_offset), float(theta), _ptr(kv_b_proj),
        _ptr(latent), latent.stride(1), lat_bs, _ptr(rope), rope.stride(1), rope_bs, _dt(latent),
        _ptr(kv_start), _ptr(kv_len), batch, s_q, heads, nope, v_dim, rank, rope_dim, t_max,
        _ptr(sel), _ptr(sel_count), k_max, float(softmax_scale), _ptr(out), out.stride(0), _dt(out),
        _ptr(lse_out), _ptr(workspace), workspace.numel(), _ptr(device_status), _stream(stream)))
    return out


def append_compressed(latent_raw: torch.Tensor, rope_raw: torch.Tensor, norm_weight: torch.Tensor, eps: float,
                      theta: float, latent: torch.Tensor, rope: torch.Tensor, kv_start, kv_len,
                      kv_len_out: Optional[torch.Tensor] = None, row_offsets: Optional[torch.Tensor] = None,
                      device_status: Optional[torch.Tensor] = None, stream=None):
    """``latent_raw`` ``[B, S, rank]`` / ``rope_raw`` ``[B, S, rope]`` views (last dim contiguous); cache
    views ``[B_buf, T_max, .]`` as for ``decode_attend`` (``B_buf == 1``: packed rows)."""
    B, S, rank = latent_raw.shape
    rope_dim = rope.shape[-1]
    lat_bs = latent.stride(0) if latent.shape[0] > 1 else 0
    rope_bs = rope.stride(0) if rope.shape[0] > 1 else 0
    _check(lib.mla_append_compressed(
        _ptr(latent_raw), latent_raw.stride(0), latent_raw.stride(1), _ptr(rope_raw), rope_raw.stride(0),
        rope_raw.stride(1), _dt(latent_raw), _ptr(norm_weight), float(eps), float(theta), _ptr(row_offsets),
        _ptr(latent), latent.stride(1), lat_bs, _ptr(rope), rope.stride(1), rope_bs, _dt(latent),
        _ptr(kv_start), _ptr(kv_len), _ptr(kv_len_out), B, S, rank, rope_dim, latent.shape[1],
        _ptr(device_status), _stream(stream)))


def select_topk(scores: torch.Tensor, lengths: torch.Tensor, top_k: int, selected: torch.Tensor,
                counts: torch.Tensor, device_status=None, stream=None):
    """``scores`` ``[n_rows, >=max length]`` f32 (last dim contiguous); ``selected`` ``[n_rows, >=top_k]``
    int32; ``counts`` ``[n_rows]`` int32."""
    assert scores.dtype == torch.float32 and scores.stride(1) == 1 and selected.stride(1) == 1
    _check(lib.mla_select_topk(_ptr(scores), scores.stride(0), _ptr(lengths), scores.shape[0], top_k,
                               _ptr(selected), selected.stride(0), _ptr(counts), _ptr(device_status),
                               _stream(stream)))


def selftest_bounded_wait(limit_cycles: int, device_status: torch.Tensor,
                          waited: Optional[torch.Tensor] = None, stream=None) -> None:
    _check(lib.mla_selftest_bounded_wait(int(limit_cycles), _ptr(device_status), _ptr(waited), _stream(stream)))


def gather_selected(latent: torch.Tensor, rope: torch.Tensor, kv_start, kv_len, batch: int, s_q: int,
                    sel: Optional[torch.Tensor], sel_count: torch.Tensor, k_max: int,
                    out: torch.Tensor, device_status=None, stream=None) -> torch.Tensor:
    lat_bs = latent.stride(0) if latent.shape[0] > 1 else 0
    rope_bs = rope.stride(0) if rope.shape[0] > 1 else 0
    _check(lib.mla_gather_selected(
        _ptr(latent), latent.stride(1), lat_bs, _ptr(rope), rope.stride(1), rope_bs, _dt(latent),
        _ptr(kv_start), _ptr(kv_len), batch, s_q, latent.shape[-1], rope.shape[-1], latent.shape[1],
        _ptr(sel), _ptr(sel_count), k_max, _ptr(out), _ptr(device_status), _stream(stream)))
    return out


# ---------------------------------------------------------------- cache row operations

def _host_i32(values) -> torch.Tensor:
    t = torch.as_tensor(values, dtype=torch.int32, device="cpu").contiguous()
    return t


def plan_rollback(left_pad, row_offsets, before_offsets, keep, width: int):
    """Host plan of a speculative-round rollback of a right-aligned cache.
    Returns ``(shift, new_left_pad, new_row_offsets, new_width)`` (CPU int32 tensors, int)."""
    lp, ro, bo, kp = (_host_i32(x) for x in (left_pad, row_offsets, before_offsets, keep))
    B = lp.numel()
    shift, pad, off = (torch.empty(B, dtype=torch.int32) for _ in range(3))
    w = ctypes.c_int32(0)
    _check(lib.mla_plan_rollback(B, int(width), _ptr(lp), _ptr(ro), _ptr(bo), _ptr(kp), _ptr(shift), _ptr(pad),
                                 _ptr(off), ctypes.addressof(w)))
    return shift, pad, off, w.value


def plan_filter(left_pad, row_offsets, keep_rows, width: int):
    """Host plan of a row filter. Returns ``(shift, new_left_pad, new_row_offsets, new_width)``."""
    lp, ro, kr = (_host_i32(x) for x in (left_pad, row_offsets, keep_rows))
    n = kr.numel()
    shift, pad, off = (torch.empty(n, dtype=torch.int32) for _ in range(3))
    w = ctypes.c_int32(0)
    _check(lib.mla_plan_filter(lp.numel(), int(width), _ptr(lp), _ptr(ro), _ptr(kr), n, _ptr(shift), _ptr(pad),
                               _ptr(off), ctypes.addressof(w)))
    return shift, pad, off, w.value


def plan_merge(source_width, left_pad, row_offsets):
    """Host plan of a merge of rows listed in merge order (each with its source's width).
    Returns ``(shift, zero_below, new_left_pad, new_width)``."""
    sw, lp, ro = (_host_i32(x) for x in (source_width, left_pad, row_offsets))
    n = lp.numel()
    shift, zero, pad = (torch.empty(n, dtype=torch.int32) for _ in range(3))
    w = ctypes.c_int32(0)
    _check(lib.mla_plan_merge(n, _ptr(sw), _ptr(lp), _ptr(ro), _ptr(shift), _ptr(zero), _ptr(pad),
                              ctypes.addressof(w)))
    return shift, zero, pad, w.value


def cache_shift_rows(src: torch.Tensor, dst: torch.Tensor, shift: Optional[torch.Tensor] = None,
                     src_row: Optional[torch.Tensor] = None, zero_below: Optional[torch.Tensor] = None,
                     device_status=None, stream=None) -> torch.Tensor:
    """``dst[i, c] = c < zero_below[i] ? 0 : src[src_row[i], (c + shift[i]) mod width]`` on views
    ``[B, width, F]`` (last dim contiguous); the index arrays are device int32 ``[dst rows]``."""
    assert src.dtype == dst.dtype and src.stride(-1) == 1 and dst.stride(-1) == 1
    _check(lib.mla_cache_shift_rows(_ptr(src), src.stride(1), src.stride(0), src.shape[0], src.shape[1],
                                    _ptr(dst), dst.stride(1), dst.stride(0), dst.shape[1], src.shape[2],
                                    _dt(src), _ptr(src_row), _ptr(shift), _ptr(zero_below), dst.shape[0],
                                    _ptr(device_status), _stream(stream)))
    return dst


def rollback_lengths(kv_len_before: torch.Tensor, keep: torch.Tensor, kv_len: torch.Tensor,
                     kv_len_out: Optional[torch.Tensor] = None, device_status=None, stream=None) -> torch.Tensor:
    """Per-row window layout: ``kv_len_out = kv_len_before + keep`` (in place when ``kv_len_out`` is None)."""
    out = kv_len if kv_len_out is None else kv_len_out
    _check(lib.mla_rollback_lengths(_ptr(kv_len_before), _ptr(keep), _ptr(kv_len), _ptr(out), kv_len.numel(),
                                    _ptr(device_status), _stream(stream)))
    return out


# ---------------------------------------------------------------- reconstructed prefill

def reconstruct_kv(latent: torch.Tensor, kv_b_proj: torch.Tensor, k_nope: torch.Tensor, v: torch.Tensor,
                   heads: int, nope: int, v_dim: int, device_status=None, stream=None):
    """``latent`` ``[rows, rank]`` view; ``k_nope`` ``[rows, H, nope]`` and ``v`` ``[rows, H, v]`` views."""
    assert latent.stride(-1) == 1 and k_nope.stride(-1) == 1 and v.stride(-1) == 1
    assert kv_b_proj.is_contiguous()
    _check(lib.mla_reconstruct_kv(_ptr(latent), latent.stride(0), latent.shape[0], _ptr(kv_b_proj), heads, nope,
                                  v_dim, latent.shape[1], _ptr(k_nope), k_nope.stride(0), k_nope.stride(1), _ptr(v),
                                  v.stride(0), v.stride(1), _dt(latent), _ptr(device_status), _stream(stream)))


def prefill_attend(q_nope: torch.Tensor, q_rope: torch.Tensor, k_nope: torch.Tensor, v: torch.Tensor,
                   rope: torch.Tensor, kv_start, kv_len, batch: int, s_q: int, t_max: int, packed: bool,
                   softmax_scale: float, out: torch.Tensor, lse_out: Optional[torch.Tensor] = None,
                   device_status=None, stream=None) -> torch.Tensor:
    """``q_nope`` ``[n_q, H, nope]`` / ``q_rope`` ``[n_q, H, rope]`` (rotated) views; ``k_nope`` / ``v``
    ``[buffer rows, H, .]``; ``rope`` ``[buffer rows, rope]``; ``out`` ``[n_q, H*v]``."""
    _, heads, nope = q_nope.shape
    _check(lib.mla_prefill_attend(
        _ptr(q_nope), q_nope.stride(0), q_nope.stride(1), _ptr(q_rope), q_rope.stride(0), q_rope.stride(1),
        _ptr(k_nope), k_nope.stride(0), k_nope.stride(1), _ptr(v), v.stride(0), v.stride(1), _ptr(rope),
        rope.stride(0), 1 if packed else 0, _dt(q_nope), _ptr(kv_start), _ptr(kv_len), batch, s_q, heads, nope,
        q_rope.shape[-1], v.shape[-1], int(t_max), float(softmax_scale), _ptr(out), out.stride(0), _dt(out),
        _ptr(lse_out), _ptr(device_status), _stream(stream)))
    return out


def default_scale(nope: int, rope_dim: int) -> float:
    """The page's softmax scale ``1/sqrt(qk_nope + qk_rope)``, as the library computes it."""
    return float(lib.mla_default_softmax_scale(nope, rope_dim))
