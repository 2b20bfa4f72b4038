"""Float64 CPU oracle for MLA decode over a compressed latent KV cache.

TEST INFRASTRUCTURE.  Only the tests, the package's ``smoke()`` self-check and
the CPU-baseline leg of the benchmark may import this module.  It shares no code
with the CUDA path: it is a plain, slow restatement of what the pages compute,
in float64 with numpy (``matmul`` is the only library primitive used as a step).

Source pages (cited by page title, function and section):

* "mlx-bun 0.0.11 -> 0.0.13 / package/src/model/glm52-mla.ts" (called *MLA page*
  below): ``partialInterleavedRopeMlx`` (partial interleaved RoPE),
  ``Glm52Mla.attendReconstructed`` (the definition this oracle computes),
  ``Glm52Mla.attendAbsorbed`` (the weight-absorbed form, implemented separately
  so that the two can be checked against each other) and the batched per-row
  loop of ``Glm52Mla.forward`` (row windows, per-row nullable selections).
* "mlx-bun 0.2.0 -> 0.4.0 / package/src/model/glm52-mla.ts" hunk (called *pad
  hunk*): the left-pad mask added to ``attendReconstructed``.
* "mlx-bun 0.2.0 -> 0.4.0 / package/src/model/glm52-cache.ts":
  ``Glm52Cache.specRoundRollback``, ``filter`` and ``mergeRows``, the row
  operations of the right-aligned compressed cache.
* "mlx-bun 0.4.0 -> 1.0.0 / package/src/model/glm52.ts" (deleted file),
  ``Glm52DecoderLayer.attend``: the sparse verify window evaluates query token
  ``i`` after appending tokens ``0..i``, each with its own selection.

Readings taken where the pages are silent (each is listed in the design notes):

* Cache row geometry: batch row ``b`` owns buffer rows ``kv_start[b] ..
  kv_start[b] + kv_len[b] - 1``; ``kv_start`` is the page's ``leftPad`` and the
  window is the page's right-aligned row.  Key ``t`` of the window is visible to
  query token ``i`` of ``S_q`` iff ``t <= kv_len - S_q + i`` (causal mask of
  ``attendReconstructed``), which for ``S_q == 1`` is every key.
* Selected positions index the row window (``takeAxis`` on the sliced row); they
  form a multiset (duplicates count twice).  A count of ``-1`` means dense
  (the page's ``null`` row), ``0`` is an error (the page throws on an empty
  selection), a position outside the visible window is an error (the page
  throws for host lists).
* ``lse`` (a side output the pages do not have) is ``log(sum(exp(s)))`` over the
  visible scaled scores; an empty visible set gives ``out = 0``, ``lse = -inf``.

Parity pins: see ``tests/test_oracle_pins.py``.  Every function here is pinned.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

F64 = np.float64


# --------------------------------------------------------------------------
# Partial interleaved RoPE  (MLA page, partialInterleavedRopeMlx)
# --------------------------------------------------------------------------

def rope_inverse_frequencies(rotary_dims: int, theta: float) -> np.ndarray:
    """Inverse frequency of each rotated pair, as float32 values.

    The page builds its angle table on the host with f32 rounding at three
    places: the exponent ``f32(f32(-2 j) / d)``, the inverse frequency
    ``f32(pow(f32(theta), exponent))`` and the angle ``f32(position * invf)``.
    """
    if rotary_dims <= 0 or rotary_dims % 2:
        raise ValueError("RoPE dimensions must be positive and even")
    if not np.isfinite(theta) or theta <= 0:
        raise ValueError("RoPE theta must be positive")
    half = rotary_dims // 2
    out = np.empty(half, dtype=np.float32)
    theta32 = F64(np.float32(theta))
    for j in range(half):
        exponent = np.float32(F64(np.float32(-2.0 * j)) / F64(rotary_dims))
        out[j] = np.float32(theta32 ** F64(exponent))
    return out


def rope_angles(positions: np.ndarray, rotary_dims: int, theta: float) -> np.ndarray:
    """f32 angle of every (position, pair): ``f32(p * invf_j)`` (exact product)."""
    invf = rope_inverse_frequencies(rotary_dims, theta).astype(F64)
    p = np.asarray(positions, dtype=F64)
    return (p[..., None] * invf).astype(np.float32)


def rope_partial_interleaved(x: np.ndarray, position_offset, rotary_dims: int,
                             theta: float) -> np.ndarray:
    """Rotate the first ``rotary_dims`` features of ``x``; keep the tail.

    ``x`` has shape ``[rows, tokens, *inner, width]``; tokens advance along
    axis 1 (the page's default ``tokenAxis``).  ``position_offset`` is an int
    (all rows) or a sequence of per-row ints (axis 0).  The rotary prefix enters
    pair-interleaved ``[a0, b0, a1, b1, ...]`` and leaves as split halves
    ``[r0.., i0..]`` with ``r = a cos - b sin`` and ``i = b cos + a sin``.
    The result is float64.
    """
    x = np.asarray(x, dtype=F64)
    if x.ndim < 3:
        raise ValueError("expect [rows, tokens, ..., width]")
    rows, tokens, width = x.shape[0], x.shape[1], x.shape[-1]
    if rotary_dims > width:
        raise ValueError("RoPE dimensions must fit the feature axis")
    if np.ndim(position_offset) == 0:
        offsets = np.full(rows, int(position_offset), dtype=np.int64)
    else:
        offsets = np.asarray(position_offset, dtype=np.int64)
        if offsets.shape != (rows,):
            raise ValueError("per-row offsets must match the row count")
    if np.any(offsets < 0):
        raise ValueError("RoPE position offset must be non-negative")
    half = rotary_dims // 2
    positions = offsets[:, None] + np.arange(tokens, dtype=np.int64)[None, :]
    ang = rope_angles(positions, rotary_dims, theta).astype(F64)   # [rows, tokens, half]
    cos, sin = np.cos(ang), np.sin(ang)
    bshape = (rows, tokens) + (1,) * (x.ndim - 3) + (half,)
    cos, sin = cos.reshape(bshape), sin.reshape(bshape)
    pairs = x[..., :rotary_dims].reshape(x.shape[:-1] + (half, 2))
    even, odd = pairs[..., 0], pairs[..., 1]
    real = even * cos - odd * sin
    imag = odd * cos + even * sin
    return np.concatenate([real, imag, x[..., rotary_dims:]], axis=-1)


# --------------------------------------------------------------------------
# RMSNorm and the compressed-state append  (MLA page, rmsNormF32Mlx;
# Glm52Mla.project and Glm52Mla.forward: the new tokens' latent is
# RMS-normalised, their rope key rotated at the row's offset, and both are
# appended to the row before attention)
# --------------------------------------------------------------------------

def rms_norm(x: np.ndarray, weight: np.ndarray, eps: float) -> np.ndarray:
    """``x * (mean(x^2) + eps)^(-1/2) * weight`` over the last axis, float64.

    The page computes it in f32 (square, mean, add eps, rsqrt, multiply by the
    input, multiply by the weight); this is the same definition in float64.
    """
    x = np.asarray(x, dtype=F64)
    w = np.asarray(weight, dtype=F64)
    if w.shape != (x.shape[-1],):
        raise ValueError("RMSNorm weight must match the feature axis")
    if not np.isfinite(eps) or eps < 0:
        raise ValueError("RMSNorm epsilon must be non-negative")
    mean_sq = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(mean_sq + eps) * w


def append_compressed(cache_latent: np.ndarray, cache_rope: np.ndarray, latent_raw: np.ndarray,
                      rope_raw: np.ndarray, weight: np.ndarray, eps: float, theta: float,
                      kv_start: Sequence[int], kv_len: Sequence[int],
                      row_offsets: Optional[Sequence[int]] = None):
    """Append ``S`` new tokens to every batch row of a compressed cache.

    ``latent_raw [B, S, rank]`` and ``rope_raw [B, S, rope]`` (pair-interleaved)
    are the new tokens' compressed projections.  Token ``t`` of row ``b`` is
    RMS-normalised / rotated at position ``row_offsets[b] + t`` (default: the
    row's current length ``kv_len[b]``, the page's right-aligned row offset)
    and written to buffer row ``kv_start[b] + kv_len[b] + t``.  Returns new
    float64 copies of the two cache buffers ``[B_buf, T_max, .]`` (a single
    buffer row ``B_buf = 1`` is shared by all rows, the packed layout) and the
    new lengths ``kv_len + S``.  A row whose new tokens would pass ``T_max`` is
    left unchanged and reported in the returned ``overflow`` list.
    """
    lat = np.array(cache_latent, dtype=F64, copy=True)
    rp = np.array(cache_rope, dtype=F64, copy=True)
    latent_raw = np.asarray(latent_raw, dtype=F64)
    rope_raw = np.asarray(rope_raw, dtype=F64)
    B, S = latent_raw.shape[0], latent_raw.shape[1]
    rope_dim = rope_raw.shape[-1]
    offsets = np.asarray(kv_len if row_offsets is None else row_offsets, dtype=np.int64)
    normed = rms_norm(latent_raw, weight, eps)
    rotated = rope_partial_interleaved(rope_raw, offsets, rope_dim, theta)
    t_max = lat.shape[1]
    new_len = np.asarray(kv_len, dtype=np.int64).copy()
    overflow = []
    for b in range(B):
        bb = b if lat.shape[0] > 1 else 0
        first = int(kv_start[b]) + int(kv_len[b])
        if first + S > t_max:
            overflow.append(b)
            continue
        lat[bb, first:first + S] = normed[b]
        rp[bb, first:first + S] = rotated[b]
        new_len[b] += S
    return lat, rp, new_len, overflow


# --------------------------------------------------------------------------
# Deterministic DSA top-k selection  ("mlx-bun ... glm52-dsa.ts",
# selectGlm52DsaDevice and its two key kernels; the scores come from the
# indexer, whose score function is not on the pages)
# --------------------------------------------------------------------------

def dsa_rank_keys(scores: np.ndarray) -> np.ndarray:
    """The rank key of each f32 score: the order-preserving map of the f32 bits
    to uint32 (negative values: all bits flipped; others: sign bit flipped),
    complemented so that ascending keys are descending scores."""
    bits = np.ascontiguousarray(scores, dtype=np.float32).view(np.uint32)
    ascending = np.where(bits & np.uint32(0x80000000), ~bits, bits ^ np.uint32(0x80000000))
    return (~ascending).astype(np.uint32)


def select_topk(scores: np.ndarray, top_k: int) -> Optional[np.ndarray]:
    """Positions selected from one row's scores, in the contract's order.

    Stable ascending sort of the rank keys (equal scores keep ascending
    positions), the first ``top_k`` positions, threshold = the minimum selected
    score; the output lists the selected positions whose score is above the
    threshold in ascending order, then the threshold ties in ascending order.
    A row with at most ``top_k`` scores is dense: ``None``.
    """
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    if top_k <= 0:
        raise ValueError("top_k must be positive")
    if scores.shape[0] <= top_k:
        return None
    ranked = np.argsort(dsa_rank_keys(scores), kind="stable")
    chosen = ranked[:top_k]
    chosen_scores = scores[chosen]
    threshold = np.min(chosen_scores)
    order_class = np.where(chosen_scores > threshold, 0, 1)
    order = np.lexsort((chosen, order_class))        # class first, then position
    return chosen[order].astype(np.int64)


# --------------------------------------------------------------------------
# kv_b_proj slicing (MLA page, attendReconstructed / attendAbsorbed)
# --------------------------------------------------------------------------

def head_weights(kv_b_proj: np.ndarray, head: int, nope: int, v: int):
    """``(W_UK_h [nope, rank], W_UV_h [v, rank])``: head ``h`` owns rows
    ``h*(nope+v) ..`` of ``kv_b_proj``, the first ``nope`` for keys, the next
    ``v`` for values."""
    row = head * (nope + v)
    return kv_b_proj[row:row + nope], kv_b_proj[row + nope:row + nope + v]


def reconstruct_kv(latent_rows: np.ndarray, kv_b_proj: np.ndarray, heads: int,
                   nope: int, v: int):
    """Per-head no-PE keys and values of cached latent rows ``[N, rank]``:
    ``kv_b_proj`` applied as a linear layer (``y = x W^T``), reshaped to
    ``[N, H, nope+v]`` and split (MLA page, attendReconstructed)."""
    lat = np.asarray(latent_rows, dtype=F64)
    w = np.asarray(kv_b_proj, dtype=F64)
    flat = lat @ w.T
    per_head = flat.reshape(lat.shape[0], heads, nope + v)
    return per_head[..., :nope], per_head[..., nope:]


# --------------------------------------------------------------------------
# Which cached rows a query row attends to
# --------------------------------------------------------------------------

def visible_rows(b: int, i: int, s_q: int, kv_start: Sequence[int], kv_len: Sequence[int],
                 sel: Optional[np.ndarray] = None, sel_count: Optional[Sequence[int]] = None
                 ) -> np.ndarray:
    """Buffer rows attended by query token ``i`` of batch row ``b``.

    Dense: window keys ``t`` with ``t <= kv_len - s_q + i`` (causal mask of
    attendReconstructed; ``kv_start`` plays the page's left pad).  Selected:
    ``kv_start + p`` for each listed ``p`` (gather semantics of attendAbsorbed),
    with ``p`` required to lie in the visible window.
    """
    start, length = int(kv_start[b]), int(kv_len[b])
    limit = length - s_q + i + 1          # keys visible to this token
    n = b * s_q + i
    if sel is None or sel_count is None or int(sel_count[n]) == -1:
        return start + np.arange(max(limit, 0), dtype=np.int64)
    count = int(sel_count[n])
    if count <= 0:
        raise ValueError("DSA selection cannot be empty")
    pos = np.asarray(sel[n, :count], dtype=np.int64)
    if np.any(pos < 0) or np.any(pos >= limit):
        raise ValueError("DSA position is outside the cached prefix")
    return start + pos


def _softmax_rows(scores: np.ndarray):
    """Max-subtracted softmax along the last axis, with log-sum-exp."""
    m = scores.max(axis=-1, keepdims=True)
    e = np.exp(scores - m)
    s = e.sum(axis=-1, keepdims=True)
    return e / s, (m + np.log(s))[..., 0]


# --------------------------------------------------------------------------
# The definition: reconstructed attention (MLA page attendReconstructed + pad hunk)
# --------------------------------------------------------------------------

def attend_reconstructed(q_nope, q_rope, latent, rope, kv_b_proj, kv_start, kv_len,
                         heads: int, nope: int, v: int, s_q: int,
                         sel=None, sel_count=None, scale: Optional[float] = None,
                         rows: Optional[Sequence[int]] = None,
                         head_subset: Optional[Sequence[int]] = None,
                         batch_buffer_rows: Optional[Sequence[int]] = None):
    """Attention output ``[n_q, len(heads), v]`` and ``lse`` ``[n_q, len(heads)]``.

    ``q_nope`` ``[n_q, H, nope]`` and ``q_rope`` ``[n_q, H, rope]`` (already
    rotated) for query rows ``n = b*s_q + i``; ``latent`` ``[B_buf, T, rank]``
    and ``rope`` ``[B_buf, T, rope]`` (already rotated) hold the cache; batch
    row ``b`` reads buffer ``batch_buffer_rows[b]`` (default ``b``).

    Per query row and head: K = [latent W_UK_h^T || rope] (rope shared by all
    heads), Q = [q_nope_h || q_rope_h], s = Q.K / sqrt(nope + rope) over the
    visible keys, softmax, out = sum p V with V = latent W_UV_h^T.  ``rows``
    and ``head_subset`` restrict the computation to a sample (outputs keep the
    full query-row count; unsampled entries are NaN).
    """
    q_nope = np.asarray(q_nope, dtype=F64)
    q_rope = np.asarray(q_rope, dtype=F64)
    n_q, H = q_nope.shape[0], q_nope.shape[1]
    rope_dim = q_rope.shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(nope + rope_dim)
    hs = list(range(H)) if head_subset is None else list(head_subset)
    out = np.full((n_q, len(hs), v), np.nan)
    lse = np.full((n_q, len(hs)), np.nan)
    rows = list(range(n_q)) if rows is None else list(rows)
    w_all = np.asarray(kv_b_proj, dtype=F64)
    # Query rows of one batch row share its cache; K/V of a row's window are
    # reconstructed once per head and each token takes the keys it sees.
    for b in sorted({n // s_q for n in rows}):
        bb = b if batch_buffer_rows is None else int(batch_buffer_rows[b])
        toks = [n for n in rows if n // s_q == b]
        keys_of = {n: visible_rows(b, n % s_q, s_q, kv_start, kv_len, sel, sel_count) for n in toks}
        union = np.unique(np.concatenate([keys_of[n] for n in toks] + [np.zeros(0, np.int64)]))
        where = {int(k): j for j, k in enumerate(union)}
        lat = np.asarray(latent[bb][union], dtype=F64)            # [U, rank]
        rp = np.asarray(rope[bb][union], dtype=F64)               # [U, rope]
        for j, h in enumerate(hs):
            w_uk, w_uv = head_weights(w_all, h, nope, v)
            k_nope, values = reconstruct_kv(lat, np.concatenate([w_uk, w_uv]), 1, nope, v)
            key = np.concatenate([k_nope[:, 0, :], rp], axis=-1)            # [U, nope+rope]
            for n in toks:
                idx = np.array([where[int(k)] for k in keys_of[n]], dtype=np.int64)
                if idx.size == 0:
                    out[n, j] = 0.0
                    lse[n, j] = -np.inf
                    continue
                query = np.concatenate([q_nope[n, h], q_rope[n, h]])        # [nope+rope]
                scores = (key[idx] @ query) * scale
                p, l = _softmax_rows(scores[None, :])
                out[n, j] = p[0] @ values[idx, 0, :]
                lse[n, j] = l[0]
    return out, lse


# --------------------------------------------------------------------------
# The weight-absorbed form (MLA page attendAbsorbed), and its pieces
# --------------------------------------------------------------------------

def absorb_q(q_nope, kv_b_proj, heads: int, nope: int, v: int) -> np.ndarray:
    """Latent-space query ``q_nope_h @ W_UK_h`` for every row and head:
    ``[n_q, H, nope] -> [n_q, H, rank]``."""
    q = np.asarray(q_nope, dtype=F64)
    w = np.asarray(kv_b_proj, dtype=F64)
    out = np.empty(q.shape[:2] + (w.shape[1],))
    for h in range(heads):
        w_uk, _ = head_weights(w, h, nope, v)
        out[:, h, :] = q[:, h, :] @ w_uk
    return out


def project_v(ctx, kv_b_proj, heads: int, nope: int, v: int) -> np.ndarray:
    """Per-head value projection of the latent context, heads concatenated:
    ``out[n, h*v:(h+1)*v] = ctx[n, h] @ W_UV_h^T`` (``[n_q, H, rank] -> [n_q, H*v]``)."""
    c = np.asarray(ctx, dtype=F64)
    w = np.asarray(kv_b_proj, dtype=F64)
    out = np.empty((c.shape[0], heads * v))
    for h in range(heads):
        _, w_uv = head_weights(w, h, nope, v)
        out[:, h * v:(h + 1) * v] = c[:, h, :] @ w_uv.T
    return out


def attend_latent(q_latent, q_rope, latent, rope, kv_start, kv_len, s_q: int,
                  sel=None, sel_count=None, scale: float = 1.0,
                  rows: Optional[Sequence[int]] = None,
                  head_subset: Optional[Sequence[int]] = None,
                  batch_buffer_rows: Optional[Sequence[int]] = None):
    """Attention in latent space: ``s = q_lat . latent + q_rope . rope``, scaled,
    softmax over the visible keys, ``ctx = sum p latent``.

    ``q_latent`` ``[n_q, H, rank]``; returns ``ctx`` ``[n_q, len(heads), rank]``
    and ``lse`` ``[n_q, len(heads)]`` (NaN for unsampled rows).
    """
    q_latent = np.asarray(q_latent, dtype=F64)
    q_rope = np.asarray(q_rope, dtype=F64)
    n_q, H, rank = q_latent.shape
    hs = list(range(H)) if head_subset is None else list(head_subset)
    ctx = np.full((n_q, len(hs), rank), np.nan)
    lse = np.full((n_q, len(hs)), np.nan)
    rows = range(n_q) if rows is None else rows
    for n in rows:
        b, i = divmod(n, s_q)
        bb = b if batch_buffer_rows is None else int(batch_buffer_rows[b])
        keys = visible_rows(b, i, s_q, kv_start, kv_len, sel, sel_count)
        if keys.size == 0:
            ctx[n] = 0.0
            lse[n] = -np.inf
            continue
        lat = np.asarray(latent[bb][keys], dtype=F64)
        rp = np.asarray(rope[bb][keys], dtype=F64)
        scores = (q_latent[n, hs] @ lat.T + q_rope[n, hs] @ rp.T) * scale   # [h, N]
        p, l = _softmax_rows(scores)
        ctx[n] = p @ lat
        lse[n] = l
    return ctx, lse


def attend_absorbed(q_nope, q_rope, latent, rope, kv_b_proj, kv_start, kv_len,
                    heads: int, nope: int, v: int, s_q: int, sel=None, sel_count=None,
                    scale: Optional[float] = None, rows=None, batch_buffer_rows=None):
    """Weight-absorbed attention: absorb, latent attention, value projection.
    Returns ``(out [n_q, H, v], ctx [n_q, H, rank], lse [n_q, H], q_latent)``."""
    rope_dim = np.asarray(q_rope).shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(nope + rope_dim)
    q_lat = absorb_q(q_nope, kv_b_proj, heads, nope, v)
    ctx, lse = attend_latent(q_lat, q_rope, latent, rope, kv_start, kv_len, s_q,
                             sel, sel_count, scale, rows=rows,
                             batch_buffer_rows=batch_buffer_rows)
    out = project_v(np.nan_to_num(ctx), kv_b_proj, heads, nope, v)
    return out.reshape(ctx.shape[0], heads, v), ctx, lse, q_lat


def gather_selected(latent, rope, kv_start, kv_len, s_q: int, sel, sel_count, k_max: int,
                    batch_buffer_rows=None):
    """Selected cache rows ``latent || rope`` copied to ``[n_q, k_max, rank+rope]``
    (``takeAxis`` of attendAbsorbed), in the storage dtype; unused slots are 0.
    A dense row (count -1) lists its visible window keys in order, at most ``k_max``."""
    latent = np.asarray(latent)
    rope = np.asarray(rope)
    n_q = len(sel_count)
    out = np.zeros((n_q, k_max, latent.shape[-1] + rope.shape[-1]), dtype=latent.dtype)
    for n in range(n_q):
        b, i = divmod(n, s_q)
        bb = b if batch_buffer_rows is None else int(batch_buffer_rows[b])
        keys = visible_rows(b, i, s_q, kv_start, kv_len, sel, sel_count)[:k_max]
        out[n, :keys.size, :latent.shape[-1]] = latent[bb][keys]
        out[n, :keys.size, latent.shape[-1]:] = rope[bb][keys]
    return out


# --------------------------------------------------------------------------
# Row operations of the right-aligned compressed cache  ("mlx-bun 0.2.0 ->
# 0.4.0 / package/src/model/glm52-cache.ts", Glm52Cache.specRoundRollback,
# Glm52Cache.filter and Glm52Cache.mergeRows).  Every state array has shape
# [B, width, features]; row b holds row_offsets[b] valid tokens in columns
# left_pad[b] .. width - 1, so left_pad[b] + row_offsets[b] == width.
# --------------------------------------------------------------------------

def rollback_right_aligned(arrays, left_pad, row_offsets, before_offsets, keep):
    """Undo the rejected part of a speculative round, keeping rows right-aligned.

    Row ``b`` had ``before_offsets[b]`` tokens when the round began and keeps
    ``keep[b]`` of the tokens appended since; the rest (``rejected[b]``) are
    dropped.  Each row is rotated right by its rejected count (column ``c``
    takes column ``(c - rejected + width) mod width``), which carries the
    rejected tail round to the front, and the leading columns that are pad in
    every row afterwards are cut.  Returns ``(new arrays, new width, new
    row_offsets, new left_pad)``.  The uniform case (the page hands it to
    ``trim``, whose body is not on the pages) goes through the same rotation.
    """
    left_pad = np.asarray(left_pad, dtype=np.int64)
    offsets = np.asarray(row_offsets, dtype=np.int64)
    next_offsets = np.asarray(before_offsets, dtype=np.int64) + np.asarray(keep, dtype=np.int64)
    rejected = offsets - next_offsets
    if np.any(rejected < 0) or np.any(next_offsets < 0):
        raise ValueError("rollback keeps more tokens than the round appended")
    B, width = np.asarray(arrays[0]).shape[:2]
    pads = left_pad + rejected
    removable = int(pads.min())
    columns = np.arange(width)
    index = (columns[None, :] - rejected[:, None] + width) % width     # [B, width]
    out = []
    for a in arrays:
        a = np.asarray(a)
        shifted = np.take_along_axis(a, index[:, :, None], axis=1)
        out.append(shifted[:, removable:].copy())
    return out, width - removable, next_offsets, pads - removable


def filter_right_aligned(arrays, left_pad, row_offsets, keep_rows):
    """Keep the rows ``keep_rows`` (in that order) and cut the leading columns
    that are pad in every kept row.  Returns ``(arrays, width, row_offsets,
    left_pad)``."""
    keep_rows = np.asarray(keep_rows, dtype=np.int64)
    if keep_rows.size == 0:
        raise ValueError("filter keeps no row")
    pads = np.asarray(left_pad, dtype=np.int64)[keep_rows]
    removable = int(pads.min())
    width = np.asarray(arrays[0]).shape[1]
    out = [np.asarray(a)[keep_rows, removable:].copy() for a in arrays]
    return out, width - removable, np.asarray(row_offsets, dtype=np.int64)[keep_rows], pads - removable


def merge_right_aligned(caches):
    """Concatenate the rows of several right-aligned caches into one.

    ``caches`` is a list of ``(arrays, left_pad, row_offsets)``.  Each row's
    valid tokens (its ``fetchRow``) are placed right-aligned in a common width
    equal to the largest row offset; pad columns are zero (the pages build
    empty rows from zeros; the pad content of longer merges is not shown).
    Returns ``(arrays, width, row_offsets, left_pad)``.
    """
    rows = []
    for arrays, left_pad, row_offsets in caches:
        for b in range(len(row_offsets)):
            pad, off = int(left_pad[b]), int(row_offsets[b])
            rows.append(([np.asarray(a)[b, pad:pad + off] for a in arrays], off))
    width = max(off for _, off in rows)
    n_arrays = len(caches[0][0])
    out = []
    for k in range(n_arrays):
        proto = np.asarray(caches[0][0][k])
        merged = np.zeros((len(rows), width, proto.shape[2]), dtype=proto.dtype)
        for i, (tokens, off) in enumerate(rows):
            if off:
                merged[i, width - off:] = tokens[k]
        out.append(merged)
    offsets = np.array([off for _, off in rows], dtype=np.int64)
    return out, width, offsets, width - offsets
