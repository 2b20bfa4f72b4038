"""Shared helpers of the parity tests: tolerances, oracle adapters, comparisons.

Tolerances of the path's contract: bf16 caches -- max-abs <= 2e-2 and relative L2
<= 5e-3; f32 caches -- relative L2 <= 1e-4; gathers and indices -- bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import mla_oracle as O

BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
F32_REL_L2 = 1e-4


def f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def rel_l2(got: np.ndarray, want: np.ndarray) -> float:
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def assert_close(got, want, dtype: str, what: str = "") -> dict:
    got, want = f64(got), f64(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = float(np.max(np.abs(got - want))) if got.size else 0.0
    rl = rel_l2(got, want)
    if dtype == "bf16":
        assert err <= BF16_MAX_ABS and rl <= BF16_REL_L2, f"{what}: max-abs {err:.3e} rel-L2 {rl:.3e}"
    else:
        assert rl <= F32_REL_L2, f"{what}: rel-L2 {rl:.3e} (max-abs {err:.3e})"
    return {"max_abs": err, "rel_l2": rl}


class Rows:
    """Indexable view ``view[bb][rows]`` of a CPU tensor that returns float64 numpy."""

    def __init__(self, t: torch.Tensor):
        self.t = t

    def __getitem__(self, bb):
        t = self.t[bb]

        class _R:
            def __getitem__(_, idx):
                idx = torch.as_tensor(np.asarray(idx, dtype=np.int64))
                return t.index_select(0, idx).to(torch.float64).numpy()
        return _R()


def oracle_rotated_cache_rope(inp, batch_rows, storage: torch.dtype):
    """The oracle's own rotation of the cached keys of the listed batch rows
    (positions 0..kv_len-1), rounded once to the cache storage dtype.  Returns a
    dict ``buffer row -> float64 [T_max, rope]`` (rows outside windows are 0)."""
    out = {}
    rope_dim = inp.rope_raw.shape[-1]
    for b in batch_rows:
        bb = 0 if inp.packed_flat else b
        s, n = int(inp.kv_start[b]), int(inp.kv_len[b])
        arr = out.setdefault(bb, np.zeros((inp.rope_raw.shape[1], rope_dim)))
        if n == 0:
            continue
        raw = inp.rope_raw[bb, s:s + n].to(torch.float64).numpy().reshape(1, n, 1, rope_dim)
        rot = O.rope_partial_interleaved(raw, 0, rope_dim, inp.w.theta).reshape(n, rope_dim)
        arr[s:s + n] = torch.from_numpy(rot).to(storage).to(torch.float64).numpy()
    return out


def oracle_rotated_q_rope(inp) -> np.ndarray:
    """Rotated query rope ``[n_q, H, rope]`` (float64, not rounded)."""
    w = inp.w
    raw = inp.q_rope_raw.to(torch.float64).numpy()                     # [B, S, H, rope]
    rot = O.rope_partial_interleaved(raw, inp.q_offset.numpy().astype(np.int64), w.rope, w.theta)
    return rot.reshape(w.n_q, w.heads, w.rope)


def batch_buffer_rows(inp):
    return [0] * inp.w.batch if inp.packed_flat else None


def oracle_reference(inp, rows=None, heads=None, with_selection=True):
    """Oracle outputs for sampled query rows / heads of a workload:
    ``out`` (reconstructed definition), ``ctx`` and ``lse`` (latent form),
    ``q_lat``, ``q_rope`` -- all float64."""
    w = inp.w
    rows = list(range(w.n_q)) if rows is None else list(rows)
    hs = list(range(w.heads)) if heads is None else list(heads)
    brows = sorted({n // w.s_q for n in rows})
    storage = inp.latent.dtype
    rope = oracle_rotated_cache_rope(inp, brows, storage)
    q_rope = oracle_rotated_q_rope(inp)
    q_nope = inp.q_nope.to(torch.float64).numpy().reshape(w.n_q, w.heads, w.nope)
    wkv = inp.kv_b_proj.to(torch.float64).numpy()
    sel = inp.sel.numpy() if (with_selection and inp.sel is not None) else None
    cnt = inp.sel_count.numpy() if sel is not None else None
    kv_start, kv_len = inp.kv_start.numpy(), inp.kv_len.numpy()
    bbr = batch_buffer_rows(inp)
    out, lse_r = O.attend_reconstructed(q_nope, q_rope, Rows(inp.latent), rope, wkv, kv_start, kv_len,
                                        w.heads, w.nope, w.v, w.s_q, sel, cnt, rows=rows,
                                        head_subset=hs, batch_buffer_rows=bbr)
    q_lat = O.absorb_q(q_nope, wkv, w.heads, w.nope, w.v)
    scale = 1.0 / np.sqrt(w.nope + w.rope)
    ctx, lse = O.attend_latent(q_lat[:, hs], q_rope[:, hs], Rows(inp.latent), rope, kv_start, kv_len,
                               w.s_q, sel, cnt, scale, rows=rows, batch_buffer_rows=bbr)
    return dict(rows=rows, heads=hs, out=out, lse_rec=lse_r, ctx=ctx, lse=lse, q_lat=q_lat,
                q_rope=q_rope)


def compare_step(step, ref, dtype: str) -> dict:
    """Compare a finished ``DecodeStep`` against ``oracle_reference`` output.
    A fused step keeps its query and context in its workspace: only ``out``
    and ``lse`` are compared for it."""
    w = step.w
    rows, hs = ref["rows"], ref["heads"]
    ri = torch.tensor(rows)
    hi = torch.tensor(hs)
    out = step.out.view(w.n_q, w.heads, w.v).cpu()[ri][:, hi]
    lse = step.lse.cpu()[ri][:, hi]
    res = {}
    res["out"] = assert_close(out, ref["out"][rows], dtype, "out")
    if not getattr(step, "fused", False):
        ctx = step.ctx.cpu()[ri][:, hi]
        q = step.q.cpu()
        res["ctx"] = assert_close(ctx, ref["ctx"][rows], dtype, "ctx")
        res["q_lat"] = assert_close(q[..., :w.rank], ref["q_lat"], dtype, "q_lat")
        res["q_rope"] = assert_close(q[..., w.rank:], ref["q_rope"], dtype, "q_rope")
    l_got, l_want = f64(lse), ref["lse"][rows]
    fin = np.isfinite(l_want)
    assert np.array_equal(np.isfinite(l_got), fin), "lse: -inf pattern differs"
    tol = 2e-2 if dtype == "bf16" else 1e-4
    assert np.max(np.abs(l_got[fin] - l_want[fin]), initial=0.0) <= tol, "lse"
    assert np.allclose(ref["lse"][rows][fin], ref["lse_rec"][rows][fin], rtol=1e-9)
    return res


def oracle_reference_out_only(inp, rows, heads=None):
    """The oracle's whole step for the listed query rows (all heads, or the
    listed ones): rotate the query rope and the rows' cached keys, then the
    reconstructed attention.  Returns ``out`` ``[n_q, len(heads), v]`` (NaN
    outside ``rows``)."""
    w = inp.w
    brows = sorted({n // w.s_q for n in rows})
    rope = oracle_rotated_cache_rope(inp, brows, inp.latent.dtype)
    q_rope = oracle_rotated_q_rope(inp)
    q_nope = inp.q_nope.to(torch.float64).numpy().reshape(w.n_q, w.heads, w.nope)
    wkv = inp.kv_b_proj.to(torch.float64).numpy()
    out, _ = O.attend_reconstructed(q_nope, q_rope, Rows(inp.latent), rope, wkv,
                                    inp.kv_start.numpy(), inp.kv_len.numpy(), w.heads, w.nope, w.v,
                                    w.s_q, inp.sel.numpy() if inp.sel is not None else None,
                                    inp.sel_count.numpy() if inp.sel is not None else None,
                                    rows=rows, head_subset=heads,
                                    batch_buffer_rows=batch_buffer_rows(inp))
    return out


def oracle_prefill(inp, rows, heads):
    """The reconstructed definition (``attendReconstructed``) for sampled query rows and heads
    of a prefill block: ``out [n_q, len(heads), v]`` and ``lse`` (float64; unsampled rows NaN)."""
    w = inp.w
    brows = sorted({n // w.s_q for n in rows})
    rope = oracle_rotated_cache_rope(inp, brows, inp.latent.dtype)
    q_rope = oracle_rotated_q_rope(inp)
    q_nope = inp.q_nope.to(torch.float64).numpy().reshape(w.n_q, w.heads, w.nope)
    wkv = inp.kv_b_proj.to(torch.float64).numpy()
    return O.attend_reconstructed(q_nope, q_rope, Rows(inp.latent), rope, wkv, inp.kv_start.numpy(),
                                  inp.kv_len.numpy(), w.heads, w.nope, w.v, w.s_q, rows=list(rows),
                                  head_subset=list(heads), batch_buffer_rows=batch_buffer_rows(inp))
