"""Seeded synthetic inputs for MLA latent-cache decode.

This module only draws numbers: it holds shapes, seeds and value distributions,
and none of the attention arithmetic.  Both the CUDA path (tests, bench) and the
float64 oracle read the tensors it returns, so they see identical values.

Value distributions (GLM/DeepSeek-shaped MLA, "glm52-mla.ts" on the mlx-bun
0.0.13 page, `Glm52MlaProjection` and the `kv_b_proj` layout):

* ``q_nope`` ``[B, S_q, H, nope]`` and the raw, still pair-interleaved
  ``q_rope`` ``[B, S_q, H, rope]``: i.i.d. N(0, 1).
* ``latent`` ``[B, T, rank]``: i.i.d. N(0, 1) rows scaled to unit root mean
  square (the cached latent is the output of an RMS normalisation with unit
  weight, eps 1e-6, computed in f32 as on the page).
* ``rope_raw`` ``[B, T, rope]``: i.i.d. N(0, 1), pair-interleaved and not yet
  rotated; each side rotates cached keys at their own positions.
* ``kv_b_proj`` ``[H*(nope+v), rank]``: i.i.d. N(0, 1/rank) (fan-in scaling).

Every tensor is produced on the CPU in float32 from a ``torch.Generator`` and then
rounded once (round-to-nearest-even) to the storage dtype.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode workload: shapes, storage dtype and the cache geometry."""

    name: str
    batch: int
    s_q: int              # query tokens per row (1 = decode, >1 = causal verify)
    t: int                # cached keys per row (dense layouts) incl. the new tokens
    heads: int
    rank: int             # kv_lora_rank
    nope: int             # qk_nope_head_dim
    rope: int             # qk_rope_head_dim
    v: int                # v_head_dim
    theta: float
    dtype: str            # "f32" | "bf16"
    seed: int
    ragged: Optional[tuple] = None   # (lo, hi) inclusive cached-length range
    top_k: int = 0                   # selected positions per query row (0 = dense)

    @property
    def n_q(self) -> int:
        return self.batch * self.s_q

    @property
    def qk_head_dim(self) -> int:
        return self.nope + self.rope


# The five workloads of the hot path (names describe what they are).
TINY_F32 = Workload("tiny_f32_t64_h4", 1, 1, 64, 4, 32, 16, 8, 16, 10000.0, "f32", 0)
DENSE_BF16 = Workload("dense_bf16_b1_t4096_h128", 1, 1, 4096, 128, 512, 128, 64, 128,
                      10000.0, "bf16", 1)
RAGGED_BF16 = Workload("ragged_bf16_b32_len1k_32k_h128", 32, 1, 0, 128, 512, 128, 64, 128,
                       10000.0, "bf16", 2, ragged=(1024, 32768))
SPARSE_BF16 = Workload("sparse_bf16_b8_t131072_top2048_h128", 8, 1, 131072, 128, 512, 128,
                       64, 128, 10000.0, "bf16", 3, top_k=2048)
VERIFY_BF16 = Workload("verify_bf16_b8_sq4_t65536_h128", 8, 4, 65536, 128, 512, 128, 64,
                       128, 10000.0, "bf16", 4)
VERIFY_SPARSE_BF16 = dataclasses.replace(VERIFY_BF16, name="verify_sparse_bf16_b8_sq4_t65536_top2048_h128",
                                         top_k=2048)

# Reconstructed prefill (the pages' second workload: a dense long prompt block,
# causal, appended before attending): one row, 4096 new tokens, no earlier cache.
PREFILL_BF16 = Workload("prefill_bf16_b1_s4096_h128", 1, 4096, 4096, 128, 512, 128, 64, 128,
                        10000.0, "bf16", 5)

ALL = (TINY_F32, DENSE_BF16, RAGGED_BF16, SPARSE_BF16, VERIFY_BF16, VERIFY_SPARSE_BF16)


def _gen(seed: int, salt: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed) * 1_000_003 + int(salt))


def normal(shape, seed: int, salt: int, std: float = 1.0) -> torch.Tensor:
    """i.i.d. N(0, std^2) float32 tensor, seeded by (seed, salt)."""
    x = torch.randn(*shape, generator=_gen(seed, salt), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def unit_rms_rows(shape, seed: int, salt: int, eps: float = 1e-6) -> torch.Tensor:
    """Gaussian rows scaled to unit root mean square along the last axis (f32)."""
    x = normal(shape, seed, salt)
    x.mul_(torch.rsqrt(x.square().mean(-1, keepdim=True) + eps))
    return x


@dataclasses.dataclass
class DecodeInputs:
    """CPU tensors of one workload (storage dtype), plus int32 geometry.

    Cache rows of batch row ``b`` live at ``latent[b, kv_start[b] + t]`` for
    ``t < kv_len[b]`` (``latent`` is ``[B, T_max, rank]``; for the packed-flat
    layout ``B_buf == 1`` and ``kv_start`` holds prefix sums).  ``rope_pos[b, t]``
    is the RoPE position of cache row ``kv_start[b] + t``, which is ``t``.
    """

    w: Workload
    q_nope: torch.Tensor          # [B, S_q, H, nope]
    q_rope_raw: torch.Tensor      # [B, S_q, H, rope] pair-interleaved, unrotated
    latent: torch.Tensor          # [B_buf, T_max, rank]
    rope_raw: torch.Tensor        # [B_buf, T_max, rope] pair-interleaved, unrotated
    kv_b_proj: torch.Tensor       # [H*(nope+v), rank]
    kv_start: torch.Tensor        # int32 [B]
    kv_len: torch.Tensor          # int32 [B]
    q_offset: torch.Tensor        # int32 [B]: RoPE position of query token 0
    packed_flat: bool
    sel: Optional[torch.Tensor] = None      # int32 [B*S_q, k_max]
    sel_count: Optional[torch.Tensor] = None  # int32 [B*S_q]


def ragged_lengths(w: Workload) -> torch.Tensor:
    lo, hi = w.ragged
    g = _gen(w.seed, 101)
    return torch.randint(lo, hi + 1, (w.batch,), generator=g, dtype=torch.int64).to(torch.int32)


def make_inputs(w: Workload, layout: str = "padded", rows: Optional[int] = None,
                t_override: Optional[int] = None) -> DecodeInputs:
    """Draw the inputs of workload ``w``.

    ``layout``: ``"padded"`` puts every row in a ``[B, T_max]`` buffer, right
    aligned with ``kv_start[b] = T_max - kv_len[b]`` (the page's left-padded
    batch rows); ``"flat"`` packs all rows back to back in one ``[1, sum, .]``
    buffer with ``kv_start`` = prefix sums; ``"aligned"`` puts row ``b`` at
    ``kv_start[b] = 0`` of its own ``[T_max]`` slot.
    ``rows`` / ``t_override`` shrink the workload (same distributions) for fast
    tests.
    """
    if rows is not None or t_override is not None:
        w = dataclasses.replace(w, batch=rows or w.batch, t=t_override or w.t)
    dt = DTYPES[w.dtype]
    B, S = w.batch, w.s_q
    if w.ragged:
        cached = ragged_lengths(w)
        if t_override is not None:
            cached = torch.clamp(cached * t_override // w.ragged[1], min=1).to(torch.int32)
        kv_len = cached + S            # the S new tokens are appended before attending
        q_offset = cached.clone()
    else:
        kv_len = torch.full((B,), w.t, dtype=torch.int32)
        q_offset = kv_len - S
    q_nope = normal((B, S, w.heads, w.nope), w.seed, 1).to(dt)
    q_rope_raw = normal((B, S, w.heads, w.rope), w.seed, 2).to(dt)
    kv_b_proj = normal((w.heads * (w.nope + w.v), w.rank), w.seed, 3,
                       std=(1.0 / w.rank) ** 0.5).to(dt)
    if layout == "flat":
        total = int(kv_len.sum())
        kv_start = torch.zeros(B, dtype=torch.int32)
        kv_start[1:] = torch.cumsum(kv_len, 0)[:-1].to(torch.int32)
        latent = unit_rms_rows((1, total, w.rank), w.seed, 4).to(dt)
        rope_raw = normal((1, total, w.rope), w.seed, 5).to(dt)
    else:
        t_max = int(kv_len.max())
        kv_start = (t_max - kv_len).to(torch.int32) if layout == "padded" else \
            torch.zeros(B, dtype=torch.int32)
        latent = unit_rms_rows((B, t_max, w.rank), w.seed, 4).to(dt)
        rope_raw = normal((B, t_max, w.rope), w.seed, 5).to(dt)
    inp = DecodeInputs(w, q_nope, q_rope_raw, latent, rope_raw, kv_b_proj,
                       kv_start.to(torch.int32), kv_len.to(torch.int32),
                       q_offset.to(torch.int32), layout == "flat")
    if w.top_k:
        inp.sel, inp.sel_count = sorted_unique_selection(
            kv_len, S, w.top_k, w.seed)
    return inp


def sorted_unique_selection(kv_len: torch.Tensor, s_q: int, top_k: int, seed: int):
    """Per query row (b, i): ``top_k`` sorted unique uniform positions below the
    number of keys token i can see (``kv_len[b] - s_q + i + 1``)."""
    B = kv_len.numel()
    sel = torch.empty((B * s_q, top_k), dtype=torch.int32)
    cnt = torch.empty((B * s_q,), dtype=torch.int32)
    for b in range(B):
        for i in range(s_q):
            n = b * s_q + i
            limit = int(kv_len[b]) - s_q + i + 1
            k = min(top_k, limit)
            g = _gen(seed, 1000 + n)
            pos = torch.randperm(limit, generator=g)[:k].sort().values
            sel[n, :k] = pos.to(torch.int32)
            sel[n, k:] = 0
            cnt[n] = k
    return sel, cnt


def cache_positions(inp: DecodeInputs) -> torch.Tensor:
    """RoPE position of every buffer row (int64 ``[B_buf, T_max]``): row
    ``kv_start[b] + t`` of batch row ``b`` sits at position ``t``; padding rows
    get position 0."""
    B_buf, T_max = inp.latent.shape[0], inp.latent.shape[1]
    pos = torch.zeros((B_buf, T_max), dtype=torch.int64)
    for b in range(inp.w.batch):
        bb = 0 if inp.packed_flat else b
        s, n = int(inp.kv_start[b]), int(inp.kv_len[b])
        pos[bb, s:s + n] = torch.arange(n, dtype=torch.int64)
    return pos
