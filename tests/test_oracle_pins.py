"""Pins of the float64 oracle to facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: closed forms,
a worked example, invariants, brute force on tiny inputs, or a textbook library
routine (torch's CPU float64 scaled-dot-product attention).  The choice is such
that a plausible slip (a dropped term, a sign, an index, a transposed operand,
the wrong half of ``kv_b_proj``) fails at least one test.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import mla_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- RoPE pins

def test_rope_position_zero_is_the_deinterleave_permutation():
    # At position 0 every angle is 0: the prefix leaves as [a0.., b0..], tail kept.
    x = rng(0).standard_normal((2, 1, 3, 12)).astype(np.float32)
    y = O.rope_partial_interleaved(x, 0, 8, 10000.0)
    want = np.concatenate([x[..., 0:8:2], x[..., 1:8:2], x[..., 8:]], axis=-1)
    assert np.array_equal(y, want.astype(np.float64))


def test_rope_pair_zero_closed_form():
    # invf_0 = theta^0 = 1, so pair 0 turns by exactly `position` radians.
    assert O.rope_inverse_frequencies(64, 10000.0)[0] == np.float32(1.0)
    x = rng(1).standard_normal((1, 5, 1, 64))
    y = O.rope_partial_interleaved(x, 37, 64, 10000.0)
    for t in range(5):
        p = 37 + t
        a, b = x[0, t, 0, 0], x[0, t, 0, 1]
        assert y[0, t, 0, 0] == pytest.approx(a * math.cos(p) - b * math.sin(p), abs=1e-12)
        assert y[0, t, 0, 32] == pytest.approx(b * math.cos(p) + a * math.sin(p), abs=1e-12)


def test_rope_inverse_frequencies_closed_form():
    d, theta = 64, 10000.0
    invf = O.rope_inverse_frequencies(d, theta)
    # theta^(-2j/d) at j = d/8 and j = d/4 is 10^-1 and 10^-2.
    assert invf[8] == np.float32(0.1)
    assert invf[16] == np.float32(0.01)
    exact = np.array([theta ** (-2.0 * j / d) for j in range(d // 2)])
    assert np.all(np.abs(invf - exact) <= 2.0 ** -22 * exact)   # f32 rounding only
    assert np.all(np.diff(invf) < 0)


def test_rope_worked_example():
    # d = 4, theta = 1e4, position 1: pair angles (1, 0.01); width 6 keeps a tail of 2.
    ex = json.load(open(os.path.join(GOLDEN, "rope_worked_example.json")))
    x = np.array(ex["input"], dtype=np.float64).reshape(1, 1, 1, 6)
    y = O.rope_partial_interleaved(x, ex["position"], ex["rotary_dims"], ex["theta"])[0, 0, 0]
    a0, b0, a1, b1, t0, t1 = ex["input"]
    c1, s1 = math.cos(1.0), math.sin(1.0)
    th = float(np.float32(0.01))
    c2, s2 = math.cos(th), math.sin(th)
    want = [a0 * c1 - b0 * s1, a1 * c2 - b1 * s2, b0 * c1 + a0 * s1, b1 * c2 + a1 * s2, t0, t1]
    assert np.allclose(y, want, rtol=0, atol=1e-12)
    assert np.allclose(y, ex["expected"], rtol=0, atol=1e-12)


def test_rope_preserves_pair_norms_and_relative_positions():
    r = rng(2)
    q = r.standard_normal((1, 1, 1, 64))
    k = r.standard_normal((1, 1, 1, 64))
    for p in (0, 5, 4095, 131071):
        y = O.rope_partial_interleaved(q, p, 64, 10000.0)[0, 0, 0]
        pairs = q[0, 0, 0].reshape(32, 2)
        assert np.allclose(y[:32] ** 2 + y[32:] ** 2, (pairs ** 2).sum(-1), rtol=1e-12)
    def dot(m, n):
        return float(O.rope_partial_interleaved(q, m, 64, 10000.0)[0, 0, 0]
                     @ O.rope_partial_interleaved(k, n, 64, 10000.0)[0, 0, 0])
    # <R(q,m), R(k,n)> depends on m - n only (up to the f32 angle rounding).
    for m, n, delta in ((7, 3, 100), (50, 49, 900), (1000, 0, 24)):
        assert dot(m, n) == pytest.approx(dot(m + delta, n + delta), abs=1e-3)


def test_rope_per_row_offsets_match_scalar_calls():
    x = rng(3).standard_normal((3, 4, 2, 16))
    offs = [0, 9, 1000]
    y = O.rope_partial_interleaved(x, offs, 16, 10000.0)
    for r, o in enumerate(offs):
        assert np.array_equal(y[r:r + 1], O.rope_partial_interleaved(x[r:r + 1], o, 16, 10000.0))


def test_rope_rejects_what_the_page_rejects():
    x = np.zeros((1, 1, 1, 8))
    for bad in (dict(rotary_dims=3), dict(rotary_dims=0), dict(rotary_dims=10)):
        with pytest.raises(ValueError):
            O.rope_partial_interleaved(x, 0, bad["rotary_dims"], 10000.0)
    with pytest.raises(ValueError):
        O.rope_partial_interleaved(x, -1, 8, 10000.0)
    with pytest.raises(ValueError):
        O.rope_partial_interleaved(x, 0, 8, 0.0)


# ---------------------------------------------------------------- attention helpers

def tiny(seed=0, B=2, S=1, T=9, H=3, rank=6, nope=4, rope=4, v=5):
    r = rng(seed)
    return dict(
        q_nope=r.standard_normal((B * S, H, nope)),
        q_rope=r.standard_normal((B * S, H, rope)),
        latent=r.standard_normal((B, T, rank)),
        rope=r.standard_normal((B, T, rope)),
        kv_b_proj=r.standard_normal((H * (nope + v), rank)) / math.sqrt(rank),
        dims=dict(heads=H, nope=nope, v=v, s_q=S),
    )


def run_rec(d, kv_start, kv_len, **kw):
    out, lse = O.attend_reconstructed(d["q_nope"], d["q_rope"], d["latent"], d["rope"],
                                      d["kv_b_proj"], kv_start, kv_len, **d["dims"], **kw)
    return out, lse


def run_abs(d, kv_start, kv_len, **kw):
    return O.attend_absorbed(d["q_nope"], d["q_rope"], d["latent"], d["rope"],
                             d["kv_b_proj"], kv_start, kv_len, **d["dims"], **kw)


# ---------------------------------------------------------------- attention pins

def test_brute_force_loops_tiny():
    """Pure-Python loops (no numpy algebra) on a tiny causal, left-padded case."""
    d = tiny(seed=4, B=2, S=2, T=6, H=2, rank=3, nope=2, rope=2, v=2)
    kv_start, kv_len = [1, 0], [5, 6]
    out, lse = run_rec(d, kv_start, kv_len)
    H, nope, v = 2, 2, 2
    W = d["kv_b_proj"]
    for n in range(4):
        b, i = divmod(n, 2)
        last = kv_len[b] - 2 + i                       # last visible window key
        for h in range(H):
            scores, vals = [], []
            for t in range(last + 1):
                row = kv_start[b] + t
                lat = d["latent"][b][row]
                kn = [sum(W[h * (nope + v) + c][r] * lat[r] for r in range(3)) for c in range(nope)]
                vv = [sum(W[h * (nope + v) + nope + c][r] * lat[r] for r in range(3)) for c in range(v)]
                s = sum(d["q_nope"][n][h][c] * kn[c] for c in range(nope))
                s += sum(d["q_rope"][n][h][c] * d["rope"][b][row][c] for c in range(2))
                scores.append(s / math.sqrt(nope + 2))
                vals.append(vv)
            mx = max(scores)
            e = [math.exp(s - mx) for s in scores]
            z = sum(e)
            want = [sum(e[t] * vals[t][c] for t in range(len(e))) / z for c in range(v)]
            assert np.allclose(out[n, h], want, rtol=1e-12, atol=1e-14)
            assert lse[n, h] == pytest.approx(mx + math.log(z), rel=1e-12)


def test_reconstructed_matches_torch_sdpa_float64():
    """Textbook scaled-dot-product attention (torch CPU, float64) with an explicit mask."""
    d = tiny(seed=5, B=2, S=3, T=11, H=4, rank=8, nope=6, rope=4, v=5)
    kv_start, kv_len = [2, 0], [9, 11]
    out, _ = run_rec(d, kv_start, kv_len)
    H, nope, v, S = 4, 6, 5, 3
    W = torch.tensor(d["kv_b_proj"])
    for b in range(2):
        lat = torch.tensor(d["latent"][b])
        kv = torch.einsum("tr,or->to", lat, W).reshape(-1, H, nope + v)
        k = torch.cat([kv[..., :nope], torch.tensor(d["rope"][b])[:, None, :].expand(-1, H, -1)], -1)
        val = kv[..., nope:]
        q = torch.cat([torch.tensor(d["q_nope"][b * S:(b + 1) * S]),
                       torch.tensor(d["q_rope"][b * S:(b + 1) * S])], -1)        # [S, H, 10]
        T = lat.shape[0]
        mask = torch.zeros(S, T, dtype=torch.bool)
        for i in range(S):
            lo, hi = kv_start[b], kv_start[b] + kv_len[b] - S + i
            mask[i, lo:hi + 1] = True
        ref = torch.nn.functional.scaled_dot_product_attention(
            q.transpose(0, 1), k.transpose(0, 1), val.transpose(0, 1), attn_mask=mask)
        assert np.allclose(out[b * S:(b + 1) * S], ref.transpose(0, 1).numpy(), rtol=1e-10, atol=1e-12)


def test_absorbed_equals_reconstructed():
    """The page's two forms compute one function (absorption is exact algebra)."""
    d = tiny(seed=6, B=3, S=2, T=13, H=3, rank=16, nope=8, rope=4, v=8)
    kv_start, kv_len = [0, 3, 1], [13, 10, 7]
    rec, lse_r = run_rec(d, kv_start, kv_len)
    out, ctx, lse_a, _ = run_abs(d, kv_start, kv_len)
    assert np.allclose(out, rec, rtol=1e-12, atol=1e-13)
    assert np.allclose(lse_a, lse_r, rtol=1e-12)
    # and with a selection
    sel = np.array([[0, 2, 5], [1, 1, 4], [0, 8, 3], [8, 2, 0], [3, 5, 1], [0, 6, 2]], np.int64)
    cnt = [3, 2, 3, 2, 1, 3]
    rec, _ = run_rec(d, kv_start, kv_len, sel=sel, sel_count=cnt)
    out, _, _, _ = run_abs(d, kv_start, kv_len, sel=sel, sel_count=cnt)
    assert np.allclose(out, rec, rtol=1e-12, atol=1e-13)


def test_one_visible_key_returns_its_value():
    d = tiny(seed=7)
    sel = np.array([[4], [2]])
    out, lse = run_rec(d, [0, 0], [9, 9], sel=sel, sel_count=[1, 1])
    H, nope, v = 3, 4, 5
    for b, t in ((0, 4), (1, 2)):
        for h in range(H):
            _, w_uv = O.head_weights(d["kv_b_proj"], h, nope, v)
            assert np.allclose(out[b, h], w_uv @ d["latent"][b][t], rtol=1e-12)
            w_uk, _ = O.head_weights(d["kv_b_proj"], h, nope, v)
            s = (d["q_nope"][b, h] @ (w_uk @ d["latent"][b][t]) + d["q_rope"][b, h] @ d["rope"][b][t]) / math.sqrt(8)
            assert lse[b, h] == pytest.approx(s, rel=1e-12)


def test_zero_query_averages_values():
    d = tiny(seed=8)
    d["q_nope"][:] = 0.0
    d["q_rope"][:] = 0.0
    out, lse = run_rec(d, [0, 2], [9, 7])
    for b, (s, n) in enumerate(((0, 9), (2, 7))):
        for h in range(3):
            _, w_uv = O.head_weights(d["kv_b_proj"], h, 4, 5)
            assert np.allclose(out[b, h], (w_uv @ d["latent"][b][s:s + n].T).mean(-1), rtol=1e-12)
            assert lse[b, h] == pytest.approx(math.log(n), rel=1e-12)


def test_value_and_key_halves_of_kv_b_proj():
    d = tiny(seed=9)
    H, nope, v = 3, 4, 5
    w = d["kv_b_proj"].copy()
    for h in range(H):                       # zero every W_UV_h: output must vanish
        w[h * (nope + v) + nope:(h + 1) * (nope + v)] = 0.0
    out, _ = O.attend_reconstructed(d["q_nope"], d["q_rope"], d["latent"], d["rope"], w,
                                    [0, 0], [9, 9], **d["dims"])
    assert np.all(out == 0.0)
    w = d["kv_b_proj"].copy()
    for h in range(H):                       # zero every W_UK_h: scores are the rope term only
        w[h * (nope + v):h * (nope + v) + nope] = 0.0
    out, _ = O.attend_reconstructed(d["q_nope"], d["q_rope"], d["latent"], d["rope"], w,
                                    [0, 0], [9, 9], **d["dims"])
    for b in range(2):
        for h in range(H):
            s = d["rope"][b] @ d["q_rope"][b, h] / math.sqrt(8)
            p = np.exp(s - s.max()); p /= p.sum()
            _, w_uv = O.head_weights(w, h, nope, v)
            assert np.allclose(out[b, h], p @ (d["latent"][b] @ w_uv.T), rtol=1e-12)


def test_selection_semantics():
    d = tiny(seed=10, T=12)
    kv_start, kv_len = [0, 2], [12, 10]
    dense, _ = run_rec(d, kv_start, kv_len)
    all_sel = np.array([np.arange(12), np.r_[np.arange(10), 0, 0]])
    out, _ = run_rec(d, kv_start, kv_len, sel=all_sel, sel_count=[12, 10])
    assert np.allclose(out, dense, rtol=1e-12)             # all positions == dense
    perm = np.array([rng(11).permutation(12), np.r_[rng(12).permutation(10), 0, 0]])
    out_p, _ = run_rec(d, kv_start, kv_len, sel=perm, sel_count=[12, 10])
    assert np.allclose(out_p, dense, rtol=1e-12)           # order does not matter
    # a unique subset == dense attention over a cache that holds only those rows
    sub = np.array([[1, 4, 7, 11], [0, 3, 9, 0]])
    out_s, _ = run_rec(d, kv_start, kv_len, sel=sub, sel_count=[4, 3])
    for b, rows in ((0, [1, 4, 7, 11]), (1, [2 + 0, 2 + 3, 2 + 9])):
        d2 = dict(d, latent=d["latent"][b:b + 1, rows], rope=d["rope"][b:b + 1, rows],
                  q_nope=d["q_nope"][b:b + 1], q_rope=d["q_rope"][b:b + 1])
        ref, _ = run_rec(d2, [0], [len(rows)])
        assert np.allclose(out_s[b], ref[0], rtol=1e-12)
    # a duplicated position counts twice (multiset / gather semantics)
    dup = np.array([[5, 5, 6], [0, 0, 0]])
    out_d, _ = run_rec(d, kv_start, kv_len, sel=dup, sel_count=[3, -1])
    d3 = dict(d, latent=d["latent"][0:1, [5, 5, 6]], rope=d["rope"][0:1, [5, 5, 6]],
              q_nope=d["q_nope"][0:1], q_rope=d["q_rope"][0:1])
    ref, _ = run_rec(d3, [0], [3])
    assert np.allclose(out_d[0], ref[0], rtol=1e-12)
    assert np.allclose(out_d[1], dense[1], rtol=1e-12)     # count -1 == dense row


def test_selection_errors_and_empty_rows():
    d = tiny(seed=13)
    with pytest.raises(ValueError):
        run_rec(d, [0, 0], [9, 9], sel=np.array([[0], [0]]), sel_count=[0, 1])
    with pytest.raises(ValueError):
        run_rec(d, [0, 0], [9, 9], sel=np.array([[9], [0]]), sel_count=[1, 1])
    out, lse = run_rec(d, [0, 0], [0, 9])
    assert np.all(out[0] == 0.0) and np.all(lse[0] == -np.inf)


def test_verify_token_equals_single_token_decode():
    """Token i of a causal S_q-token block sees the prefix a serial decode sees."""
    S = 4
    d = tiny(seed=14, B=2, S=S, T=16)
    kv_start, kv_len = [0, 3], [16, 13]
    out, _ = run_rec(d, kv_start, kv_len)
    for b in range(2):
        for i in range(S):
            n = b * S + i
            d1 = dict(d, q_nope=d["q_nope"][n:n + 1], q_rope=d["q_rope"][n:n + 1],
                      latent=d["latent"][b:b + 1], rope=d["rope"][b:b + 1],
                      dims=dict(d["dims"], s_q=1))
            ref, _ = run_rec(d1, [kv_start[b]], [kv_len[b] - S + i + 1])
            assert np.allclose(out[n], ref[0], rtol=1e-12)


def test_left_padding_content_is_ignored():
    d = tiny(seed=15)
    out, _ = run_rec(d, [3, 0], [6, 9])
    d["latent"][0, :3] = 1e6
    d["rope"][0, :3] = -1e6
    out2, _ = run_rec(d, [3, 0], [6, 9])
    assert np.array_equal(out, out2)


def test_absorb_and_project_match_einsum():
    d = tiny(seed=16, H=3, rank=6, nope=4, v=5)
    q_lat = O.absorb_q(d["q_nope"], d["kv_b_proj"], 3, 4, 5)
    W = torch.tensor(d["kv_b_proj"]).reshape(3, 9, 6)
    ref = torch.einsum("nhk,hkr->nhr", torch.tensor(d["q_nope"]), W[:, :4])
    assert np.allclose(q_lat, ref.numpy(), rtol=1e-12)
    ctx = rng(17).standard_normal((2, 3, 6))
    out = O.project_v(ctx, d["kv_b_proj"], 3, 4, 5)
    ref = torch.einsum("nhr,hvr->nhv", torch.tensor(ctx), W[:, 4:]).reshape(2, 15)
    assert np.allclose(out, ref.numpy(), rtol=1e-12)


def test_gather_selected_is_indexing():
    r = rng(18)
    lat = r.integers(-30000, 30000, size=(2, 10, 6)).astype(np.int16)
    rp = r.integers(-30000, 30000, size=(2, 10, 2)).astype(np.int16)
    sel = np.array([[3, 1, 0], [8, 4, 4]])
    g = O.gather_selected(lat, rp, [0, 1], [10, 9], 1, sel, [2, 3], 3)
    assert np.array_equal(g[0, 0], np.r_[lat[0, 3], rp[0, 3]])
    assert np.array_equal(g[0, 1], np.r_[lat[0, 1], rp[0, 1]])
    assert np.all(g[0, 2] == 0)
    assert np.array_equal(g[1, 0], np.r_[lat[1, 1 + 8], rp[1, 9]])
    assert np.array_equal(g[1, 2], np.r_[lat[1, 5], rp[1, 5]])


def test_gather_selected_dense_rows_list_the_window_in_order():
    # Count -1 (the page's null selection): the row's visible window, first key
    # first, cut after k_max entries; slots past the window stay zero.  Written
    # out by hand from the buffer indices (kv_start + t), not through the oracle.
    r = rng(19)
    lat = r.integers(-30000, 30000, size=(3, 12, 4)).astype(np.int16)
    rp = r.integers(-30000, 30000, size=(3, 12, 2)).astype(np.int16)
    row = lambda bb, t: np.r_[lat[bb, t], rp[bb, t]]
    sel = np.zeros((3, 5), dtype=np.int64)
    # row 0: window of 9 keys at buffer rows 2..10, k_max 5 -> rows 2, 3, 4, 5, 6
    # row 1: window of 3 keys at buffer rows 7..9 -> rows 7, 8, 9, then zeros
    # row 2: mixed with a listed row -- count 2 takes the listed positions
    sel[2, :2] = [4, 0]
    g = O.gather_selected(lat, rp, [2, 7, 1], [9, 3, 6], 1, sel, [-1, -1, 2], 5)
    assert [np.array_equal(g[0, j], row(0, 2 + j)) for j in range(5)] == [True] * 5
    assert [np.array_equal(g[1, j], row(1, 7 + j)) for j in range(3)] == [True] * 3
    assert np.all(g[1, 3:] == 0)
    assert np.array_equal(g[2, 0], row(2, 5)) and np.array_equal(g[2, 1], row(2, 1))
    assert np.all(g[2, 2:] == 0)
    # verify rows (s_q = 2): token 0 sees one key fewer than token 1, in order
    g = O.gather_selected(lat, rp, [0], [4], 2, np.zeros((2, 6), np.int64), [-1, -1], 6)
    assert [np.array_equal(g[0, j], row(0, j)) for j in range(3)] == [True] * 3
    assert np.all(g[0, 3:] == 0)
    assert [np.array_equal(g[1, j], row(0, j)) for j in range(4)] == [True] * 4
    assert np.all(g[1, 4:] == 0)


# ---------------------------------------------------------------- RMSNorm / append pins

def test_rms_norm_closed_forms():
    # eps = 0, unit weight: the output has unit root mean square whatever the input.
    x = rng(40).standard_normal((3, 7, 512)) * 3.7
    y = O.rms_norm(x, np.ones(512), 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-12)
    # a constant row c with eps: every element is c / sqrt(c^2 + eps) * w_i
    c, eps = -0.3, 1e-2
    w = rng(41).standard_normal(16)
    y = O.rms_norm(np.full((1, 16), c), w, eps)
    assert np.allclose(y[0], c / math.sqrt(c * c + eps) * w, rtol=1e-13)
    # scale invariance (eps = 0) and the weight acting elementwise
    x = rng(42).standard_normal((4, 32))
    w = rng(43).standard_normal(32)
    assert np.allclose(O.rms_norm(5.5 * x, w, 0.0), O.rms_norm(x, w, 0.0), rtol=1e-12)
    assert np.allclose(O.rms_norm(x, w, 0.0), O.rms_norm(x, np.ones(32), 0.0) * w, rtol=1e-13)
    # a one-hot row: mean of squares is 1/n, so the hot entry becomes sqrt(n)
    e = np.zeros((1, 64)); e[0, 9] = 1.0
    assert np.isclose(O.rms_norm(e, np.ones(64), 0.0)[0, 9], 8.0, rtol=1e-14)
    with pytest.raises(ValueError):
        O.rms_norm(x, w, -1.0)
    with pytest.raises(ValueError):
        O.rms_norm(x, np.ones(31), 0.0)


def test_append_places_normalised_and_rotated_rows():
    r = rng(44)
    B, S, T, rank, rope = 3, 2, 20, 16, 8
    lat = r.standard_normal((B, T, rank))
    rp = r.standard_normal((B, T, rope))
    lat_raw = r.standard_normal((B, S, rank))
    rope_raw = r.standard_normal((B, S, rope))
    w = r.standard_normal(rank)
    kv_start = [0, 3, 1]
    kv_len = [5, 10, 18]          # row 2 overflows: 1 + 18 + 2 > 20
    new_lat, new_rp, new_len, overflow = O.append_compressed(lat, rp, lat_raw, rope_raw, w, 1e-6, 10000.0,
                                                             kv_start, kv_len)
    assert overflow == [2] and list(new_len) == [7, 12, 18]
    for b in range(2):
        first = kv_start[b] + kv_len[b]
        for t in range(S):
            x = lat_raw[b, t]
            want = x / math.sqrt(float(np.mean(x * x)) + 1e-6) * w
            assert np.allclose(new_lat[b, first + t], want, rtol=1e-12)
            # position kv_len[b] + t, checked against the pinned RoPE on one vector
            want_r = O.rope_partial_interleaved(rope_raw[b, t].reshape(1, 1, rope), kv_len[b] + t, rope,
                                                10000.0)[0, 0]
            assert np.allclose(new_rp[b, first + t], want_r, rtol=1e-12)
        # every other buffer row is untouched
        keep = [i for i in range(T) if not first <= i < first + S]
        assert np.array_equal(new_lat[b, keep], lat[b, keep]) and np.array_equal(new_rp[b, keep], rp[b, keep])
    assert np.array_equal(new_lat[2], lat[2]) and np.array_equal(new_rp[2], rp[2])
    # explicit row offsets move only the rotation, not the placement
    _, rp2, _, _ = O.append_compressed(lat, rp, lat_raw, rope_raw, w, 1e-6, 10000.0, kv_start, kv_len,
                                       row_offsets=[0, 0, 0])
    assert np.allclose(rp2[0, 5], np.concatenate([rope_raw[0, 0, 0::2], rope_raw[0, 0, 1::2]]), rtol=0)


def test_append_exact_fit_and_packed_buffer():
    # a row whose new tokens end exactly at T_max is appended; one token more is not
    r = rng(45)
    lat = r.standard_normal((1, 12, 8)); rp = r.standard_normal((1, 12, 4))
    lat_raw = r.standard_normal((2, 2, 8)); rope_raw = r.standard_normal((2, 2, 4))
    # packed layout: both rows share buffer row 0; row 0 = [0, 5), row 1 = [5, 10) + 2 new = 12 = T_max
    new_lat, _, new_len, overflow = O.append_compressed(lat, rp, lat_raw, rope_raw, np.ones(8), 0.0, 10000.0,
                                                        [0, 5], [3, 5])
    assert overflow == [] and list(new_len) == [5, 7]
    assert np.allclose(new_lat[0, 10:12], O.rms_norm(lat_raw[1], np.ones(8), 0.0))
    assert np.allclose(new_lat[0, 3:5], O.rms_norm(lat_raw[0], np.ones(8), 0.0))
    _, _, _, overflow = O.append_compressed(lat, rp, lat_raw, rope_raw, np.ones(8), 0.0, 10000.0, [0, 6], [3, 5])
    assert overflow == [1]


# ---------------------------------------------------------------- DSA top-k pins

def test_rank_keys_order_floats():
    # the key order is the float order, descending, over signs, zeros and infinities
    v = np.array([-np.inf, -3.5, -1e-30, -0.0, 0.0, 1e-30, 2.0, np.inf], dtype=np.float32)
    k = O.dsa_rank_keys(v)
    assert np.all(np.diff(k.astype(np.int64)) < 0)          # larger score -> smaller key
    x = rng(60).standard_normal(1000).astype(np.float32)
    assert np.array_equal(np.argsort(O.dsa_rank_keys(x), kind="stable"), np.argsort(-x, kind="stable"))


def test_select_topk_distinct_scores_brute_force():
    x = rng(61).permutation(5000).astype(np.float32) * 0.25 - 300.0     # distinct values
    got = O.select_topk(x, 64)
    want = np.sort(np.argsort(x)[::-1][:64])                           # the 64 largest, then ascending
    # distinct: only the k-th is at the threshold, so it comes last
    assert np.array_equal(np.sort(got), want)
    thr_pos = int(np.argsort(x)[::-1][63])
    assert got[-1] == thr_pos and np.array_equal(got[:-1], np.sort(want[want != thr_pos]))


def test_select_topk_ties_and_order():
    # all equal: the first k positions, ascending (equal scores keep ascending positions)
    assert np.array_equal(O.select_topk(np.zeros(100, np.float32), 10), np.arange(10))
    # a tie group straddling the boundary: above-threshold positions first, then the
    # lowest-position members of the tie group, each ascending
    x = np.zeros(20, np.float32)
    x[[3, 17]] = 5.0                    # above
    x[[1, 4, 9, 12, 18]] = 2.0          # the tie group at the threshold
    got = O.select_topk(x, 5)
    assert list(got) == [3, 17, 1, 4, 9]
    # -inf and +inf take part like any value; -0.0 and +0.0 are equal scores
    y = np.array([1.0, -np.inf, np.inf, 0.0, -0.0, -1.0], np.float32)
    assert list(O.select_topk(y, 3)) == [0, 2, 3]
    assert list(O.select_topk(y, 4)) == [0, 2, 3, 4]
    # short rows are dense
    assert O.select_topk(np.ones(8, np.float32), 8) is None
    assert O.select_topk(np.ones(9, np.float32), 8) is not None
    with pytest.raises(ValueError):
        O.select_topk(np.ones(4, np.float32), 0)


def test_select_topk_set_is_permutation_equivariant():
    r = rng(62)
    x = r.integers(0, 40, 3000).astype(np.float32)     # many ties
    perm = r.permutation(3000)
    inv = np.argsort(perm)
    a = O.select_topk(x, 300)
    b = O.select_topk(x[perm], 300)
    # the above-threshold set is the same set of values' positions mapped through the permutation
    thr = x[a].min()
    assert set(a[x[a] > thr]) == set(perm[b][x[perm][b] > thr].tolist()) == set(np.nonzero(x > thr)[0].tolist())
    assert len(a) == 300 and np.all(np.diff(a[x[a] > thr]) > 0) and np.all(np.diff(a[x[a] == thr]) > 0)
    del inv


# ---------------------------------------------------------------- right-aligned cache row operations

def _tagged_cache(offsets, width, features=3, fill=-1.0):
    """A right-aligned cache whose valid token j of row b holds (b, j, b*1000+j)
    and whose pad holds ``fill``: every token says where it came from."""
    B = len(offsets)
    a = np.full((B, width, features), fill)
    pad = np.array([width - o for o in offsets])
    for b, o in enumerate(offsets):
        for j in range(o):
            a[b, pad[b] + j] = [b, j, b * 1000 + j][:features]
    return a, pad, np.array(offsets)


def _valid_tokens(a, pad, b):
    return a[b, pad[b]:]


def test_rollback_keeps_each_rows_accepted_prefix_in_order():
    before = [5, 2, 7, 0]
    appended = 4
    offsets = [o + appended for o in before]
    a, pad, offs = _tagged_cache(offsets, width=12)
    keep = [4, 0, 2, 1]
    (out,), width, new_off, new_pad = O.rollback_right_aligned([a], pad, offs, before, keep)
    assert list(new_off) == [9, 2, 9, 1]
    # the width loses the columns that are pad in every row afterwards
    assert width == 12 - min(pad[b] + (offsets[b] - new_off[b]) for b in range(4)) == 9
    assert np.all(new_pad + new_off == width)
    for b in range(4):
        tokens = _valid_tokens(out, new_pad, b)
        assert tokens.shape[0] == new_off[b]
        assert np.array_equal(tokens[:, 0], np.full(new_off[b], b))           # the row's own tokens
        assert np.array_equal(tokens[:, 1], np.arange(new_off[b]))            # its first tokens, in order


def test_rollback_uniform_rejection_drops_the_last_columns():
    # every row rejects r tokens and one row fills the width: the result is the
    # cache without its last r columns (what trimming the tail gives)
    before = [6, 3]
    offsets = [9, 6]
    a = rng(70).standard_normal((2, 9, 4))
    _, pad, offs = _tagged_cache(offsets, 9)
    (out,), width, new_off, new_pad = O.rollback_right_aligned([a], pad, offs, before, [1, 1])
    assert width == 7 and list(new_off) == [7, 4] and list(new_pad) == [0, 3]
    assert np.array_equal(out, a[:, :7])
    # nothing rejected and a full row: identity
    (same,), w2, off2, pad2 = O.rollback_right_aligned([a], pad, offs, before, [3, 3])
    assert w2 == 9 and np.array_equal(same, a) and list(off2) == offsets and list(pad2) == list(pad)


def test_rollback_rejects_more_than_was_appended():
    a, pad, offs = _tagged_cache([4, 4], 4)
    with pytest.raises(ValueError):
        O.rollback_right_aligned([a], pad, offs, [2, 2], [3, 0])
    # a row may go back to empty
    (out,), width, new_off, new_pad = O.rollback_right_aligned([a], pad, offs, [0, 2], [0, 0])
    assert list(new_off) == [0, 2] and width == 2 and list(new_pad) == [2, 0]
    assert np.array_equal(out[1, :, 1], [0, 1])


def test_rollback_then_attention_equals_attention_over_the_accepted_prefix():
    # decode over the rolled-back cache attends exactly to each row's accepted prefix
    r = rng(71)
    before, offsets, keep = [3, 5], [6, 8], [2, 1]
    width, rank, rope_dim, H = 10, 8, 4, 2
    lat = r.standard_normal((2, width, rank)); rp = r.standard_normal((2, width, rope_dim))
    pad = np.array([width - o for o in offsets])
    q_lat = r.standard_normal((2, H, rank)); q_rope = r.standard_normal((2, H, rope_dim))
    (lat2, rp2), w2, off2, pad2 = O.rollback_right_aligned([lat, rp], pad, offsets, before, keep)
    got, _ = O.attend_latent(q_lat, q_rope, lat2, rp2, pad2, off2, 1, None, None, 0.5)
    want, _ = O.attend_latent(q_lat, q_rope, lat, rp, pad, np.add(before, keep), 1, None, None, 0.5)
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13)


def test_filter_keeps_rows_and_cuts_the_common_pad():
    a, pad, offs = _tagged_cache([3, 7, 5, 1], 9)
    (out,), width, new_off, new_pad = O.filter_right_aligned([a], pad, offs, [2, 0, 3])
    assert width == 5 == max(5, 3, 1)                     # the longest kept row now fills the width
    assert list(new_off) == [5, 3, 1] and list(new_pad) == [0, 2, 4]
    for i, src in enumerate([2, 0, 3]):
        assert np.array_equal(_valid_tokens(out, new_pad, i), _valid_tokens(a, pad, src))
    with pytest.raises(ValueError):
        O.filter_right_aligned([a], pad, offs, [])


def test_merge_right_aligns_rows_in_the_longest_width():
    a, pad_a, off_a = _tagged_cache([2, 4], 6, fill=7.0)        # width above its longest row
    b, pad_b, off_b = _tagged_cache([5, 0], 5, fill=7.0)
    (out,), width, offs, pads = O.merge_right_aligned([([a], pad_a, off_a), ([b], pad_b, off_b)])
    assert width == 5 and list(offs) == [2, 4, 5, 0] and list(pads) == [3, 1, 0, 5]
    assert np.array_equal(_valid_tokens(out, pads, 0), _valid_tokens(a, pad_a, 0))
    assert np.array_equal(_valid_tokens(out, pads, 1), _valid_tokens(a, pad_a, 1))
    assert np.array_equal(_valid_tokens(out, pads, 2), _valid_tokens(b, pad_b, 0))
    for i in range(4):
        assert np.all(out[i, :pads[i]] == 0.0)                      # pad columns are zero


def test_filter_then_merge_round_trip():
    r = rng(72)
    offsets = [4, 9, 6, 2, 9]
    width = 9
    a = r.standard_normal((5, width, 3))
    pad = np.array([width - o for o in offsets])
    for b in range(5):
        a[b, :pad[b]] = 0.0
    parts = [O.filter_right_aligned([a], pad, offsets, rows) for rows in ([0, 1], [2], [3, 4])]
    (out,), w, offs, pads = O.merge_right_aligned([(arrs, p, o) for arrs, _, o, p in parts])
    assert w == width and list(offs) == offsets and list(pads) == list(pad)
    assert np.array_equal(out, a)
