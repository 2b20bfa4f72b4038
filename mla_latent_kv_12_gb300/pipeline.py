"""One MLA decode step on the device, composed from the C-ABI entry points.

``DecodeStep`` owns the device buffers of one attention layer's decode step and
runs the hot path in order: RoPE of the new query's rope part (written into
the packed query), absorption of ``q_nope`` through ``W_UK`` (into the same
packed query), latent attention over the cache (split-K + combine), and the
``W_UV`` projection.  ``run`` takes the fused entry point (three launches)
where it serves the shapes and the four entry points otherwise; the four
methods stay callable one by one.  Cache keys are rotated once at set-up with
the same RoPE entry point (as an append would), at their positions
``0 .. kv_len-1``.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import mla
from .workloads import DTYPES, DecodeInputs


def rotate_cache_keys(inp: DecodeInputs, rope_raw_dev: torch.Tensor, rope_dev: torch.Tensor,
                      kv_start: torch.Tensor, kv_len: torch.Tensor, theta: float) -> None:
    """Rotate every row's cached keys at positions 0..kv_len-1 (one call per batch row)."""
    rope_dim = rope_dev.shape[-1]
    for b in range(inp.w.batch):
        bb = 0 if inp.packed_flat else b
        s, n = int(kv_start[b]), int(kv_len[b])
        if n == 0:
            continue
        src = rope_raw_dev[bb, s:s + n].reshape(1, n, 1, rope_dim)
        dst = rope_dev[bb, s:s + n].reshape(1, n, 1, rope_dim)
        mla.rope_partial_interleaved(src, dst, rope_dim, theta, position_offset=0)


class DecodeStep:
    def __init__(self, inp: DecodeInputs, device="cuda", out_dtype: Optional[torch.dtype] = None,
                 with_selection: bool = True, fused: bool = True):
        w = inp.w
        self.w, self.inp = w, inp
        dt = DTYPES[w.dtype]
        self.dtype = dt
        self.out_dtype = out_dtype or dt
        B, S, H = w.batch, w.s_q, w.heads
        self.n_q = n_q = B * S
        dev = torch.device(device)
        self.kv_start = inp.kv_start.to(dev)
        self.kv_len = inp.kv_len.to(dev)
        self.q_offset = inp.q_offset.to(dev)
        self.latent = inp.latent.to(dev)
        rope_raw = inp.rope_raw.to(dev)
        self.rope = torch.empty_like(rope_raw)
        rotate_cache_keys(inp, rope_raw, self.rope, inp.kv_start, inp.kv_len, w.theta)
        del rope_raw
        self.kv_b_proj = inp.kv_b_proj.to(dev).contiguous()
        self.sel = inp.sel.to(dev) if (with_selection and inp.sel is not None) else None
        self.sel_count = inp.sel_count.to(dev) if self.sel is not None else None
        # per-step inputs
        self.q_nope = inp.q_nope.to(dev).reshape(n_q, H, w.nope)
        self.q_rope_raw = inp.q_rope_raw.to(dev)                         # [B, S, H, rope]
        # work buffers
        D = w.rank + w.rope
        self.q = torch.empty(n_q, H, D, dtype=dt, device=dev)
        self.ctx = torch.empty(n_q, H, w.rank, dtype=dt, device=dev)
        self.lse = torch.empty(n_q, H, dtype=torch.float32, device=dev)
        self.out = torch.empty(n_q, H * w.v, dtype=self.out_dtype, device=dev)
        k_max = self.sel.shape[1] if self.sel is not None else 0
        nbytes = mla.decode_workspace_size(B, S, H, w.rank, w.rope, self.latent.shape[1], k_max,
                                           self.sel is not None, dt)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.scale = mla.default_scale(w.nope, w.rope)
        step_bytes = mla.decode_step_workspace_size(B, S, H, w.nope, w.v, w.rank, w.rope, self.latent.shape[1],
                                                    k_max, self.sel is not None, dt)
        self.fused = step_bytes > 0 and fused
        self.step_workspace = (torch.empty(step_bytes, dtype=torch.uint8, device=dev) if self.fused else None)

    # The four steps; each is one (or two) kernel launches on the current stream.
    def rope_q(self, stream=None):
        w = self.w
        qv = self.q.view(w.batch, w.s_q, w.heads, -1)[..., w.rank:]
        mla.rope_partial_interleaved(self.q_rope_raw, qv, w.rope, w.theta,
                                     row_offsets=self.q_offset, stream=stream)

    def absorb(self, stream=None):
        w = self.w
        mla.absorb_q(self.q_nope, self.kv_b_proj, self.q, w.heads, w.nope, w.v, w.rank, stream=stream)

    def attend(self, stream=None):
        mla.decode_attend(self.q, self.latent, self.rope, self.kv_start, self.kv_len, self.w.batch,
                          self.w.s_q, self.scale, self.ctx, self.lse, self.sel, self.sel_count,
                          self.workspace, self.status, stream=stream)

    def project(self, stream=None):
        w = self.w
        mla.project_v(self.ctx, self.kv_b_proj, self.out, w.heads, w.nope, w.v, stream=stream)

    def run_fused(self, stream=None) -> torch.Tensor:
        w = self.w
        mla.decode_step(self.q_nope, self.q_rope_raw.view(self.n_q, w.heads, w.rope), w.theta, self.kv_b_proj,
                        self.latent, self.rope, self.kv_start, self.kv_len, w.batch, w.s_q, w.nope, w.v,
                        self.scale, self.out, self.lse, row_offsets=self.q_offset, sel=self.sel,
                        sel_count=self.sel_count, workspace=self.step_workspace, device_status=self.status,
                        stream=stream)
        return self.out

    def run(self, stream=None) -> torch.Tensor:
        if self.fused:
            return self.run_fused(stream)
        self.rope_q(stream)
        self.absorb(stream)
        self.attend(stream)
        self.project(stream)
        return self.out

    def launches_per_step(self) -> int:
        """Kernels one ``run`` launches: three for the fused step (absorb + RoPE,
        decode, combine + projection); else RoPE, absorb, the decode launches,
        project."""
        if self.fused:
            return 3
        return 3 + self.attend_launches()

    def attend_launches(self) -> int:
        """Tensor-core decode: decode + combine (+ a planner launch above 128
        query rows).  CUDA-core decode: the decode kernel, plus a combine when
        it splits the keys."""
        w = self.w
        if mla.decode_kernel_kind(w.heads, w.rank, w.rope, self.dtype, self.dtype) == 1:
            return 2 if self.n_q <= 128 else 3
        k_max = self.sel.shape[1] if self.sel is not None else 0
        nbytes = mla.decode_workspace_size(w.batch, w.s_q, w.heads, w.rank, w.rope,
                                           self.latent.shape[1], k_max, self.sel is not None,
                                           self.dtype)
        return 2 if nbytes > 0 else 1


class PrefillStep:
    """Reconstructed prefill of one attention layer ("glm52-mla.ts",
    Glm52Mla.attendReconstructed): the block's ``S_q`` new tokens are the last
    keys of each row's window (appended before attending), RoPE rotates the
    query rope part at each row's offset, ``kv_b_proj`` materialises the
    per-head no-PE keys and values of every buffer row, and causal attention
    reads them with the cache's shared rope key.  Three launches per ``run``.
    """

    def __init__(self, inp: DecodeInputs, device="cuda", out_dtype: Optional[torch.dtype] = None):
        w = inp.w
        self.w, self.inp = w, inp
        dt = DTYPES[w.dtype]
        self.dtype = dt
        self.out_dtype = out_dtype or dt
        dev = torch.device(device)
        n_q, H = w.n_q, w.heads
        self.kv_start = inp.kv_start.to(dev)
        self.kv_len = inp.kv_len.to(dev)
        self.q_offset = inp.q_offset.to(dev)
        self.latent = inp.latent.to(dev)
        rope_raw = inp.rope_raw.to(dev)
        self.rope = torch.empty_like(rope_raw)
        rotate_cache_keys(inp, rope_raw, self.rope, inp.kv_start, inp.kv_len, w.theta)
        del rope_raw
        self.kv_b_proj = inp.kv_b_proj.to(dev).contiguous()
        self.q_nope = inp.q_nope.to(dev).reshape(n_q, H, w.nope)
        self.q_rope_raw = inp.q_rope_raw.to(dev)                          # [B, S, H, rope]
        self.q_rope = torch.empty(w.batch, w.s_q, H, w.rope, dtype=dt, device=dev)
        self.t_max = self.latent.shape[1]
        rows = self.latent.shape[0] * self.t_max
        self.kv = torch.empty(rows, H, w.nope + w.v, dtype=dt, device=dev)
        self.k_nope = self.kv[..., :w.nope]
        self.v = self.kv[..., w.nope:]
        self.out = torch.empty(n_q, H * w.v, dtype=self.out_dtype, device=dev)
        self.lse = torch.empty(n_q, H, dtype=torch.float32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.scale = mla.default_scale(w.nope, w.rope)

    def rope_q(self, stream=None):
        mla.rope_partial_interleaved(self.q_rope_raw, self.q_rope, self.w.rope, self.w.theta,
                                     row_offsets=self.q_offset, stream=stream)

    def reconstruct(self, stream=None):
        w = self.w
        mla.reconstruct_kv(self.latent.view(-1, w.rank), self.kv_b_proj, self.k_nope, self.v, w.heads, w.nope,
                           w.v, device_status=self.status, stream=stream)

    def attend(self, stream=None):
        w = self.w
        mla.prefill_attend(self.q_nope, self.q_rope.view(w.n_q, w.heads, w.rope), self.k_nope, self.v,
                           self.rope.view(-1, w.rope), self.kv_start, self.kv_len, w.batch, w.s_q, self.t_max,
                           self.inp.packed_flat, self.scale, self.out, self.lse, device_status=self.status,
                           stream=stream)

    def run(self, stream=None) -> torch.Tensor:
        self.rope_q(stream)
        self.reconstruct(stream)
        self.attend(stream)
        return self.out

    def launches_per_step(self) -> int:
        return 3
