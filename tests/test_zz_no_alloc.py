"""The decode entry point that allocates nothing (mla_decode_attend_no_alloc).

Some callers cannot allocate device memory at decode time -- a server whose
pool already owns the free memory, a plugin host without an allocator, a
latency-bound loop.  For them the library keeps the split-K scratch in a
built-in device array.  This file checks, through the C ABI, that this entry
point gives what mla_decode_attend gives with a caller-allocated workspace and
what the float64 oracle gives, on two calls in a row and on calls of
different shapes in turn (the shared array keeps the previous call's
contents), and that a request too large for the array is refused without a
launch.  It is collected last so that a failure here never hides another
test's result.
"""
import dataclasses

import numpy as np
import pytest
import torch

from tests import helpers as H

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from mla_latent_kv_12_gb300 import mla
    from mla_latent_kv_12_gb300 import workloads as W
    from mla_latent_kv_12_gb300.pipeline import DecodeStep


def _no_alloc(step, ctx, lse, status):
    q, lat, rope = step.q, step.latent, step.rope
    k_max = step.sel.shape[1] if step.sel is not None else 0
    return mla.lib.mla_decode_attend_no_alloc(
        q.data_ptr(), q.stride(0), q.stride(1), lat.data_ptr(), lat.stride(1),
        lat.stride(0) if lat.shape[0] > 1 else 0, rope.data_ptr(), rope.stride(1),
        rope.stride(0) if rope.shape[0] > 1 else 0, mla._dt(lat), step.kv_start.data_ptr(),
        step.kv_len.data_ptr(), step.w.batch, step.w.s_q, step.w.heads, step.w.rank, step.w.rope,
        lat.shape[1], None if step.sel is None else step.sel.data_ptr(),
        None if step.sel is None else step.sel_count.data_ptr(), k_max, step.scale, ctx.data_ptr(),
        ctx.stride(0), ctx.stride(1), mla._dt(ctx), lse.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


CASES = {
    "dense_t4096": lambda: W.make_inputs(W.DENSE_BF16),
    "ragged_150_rows": lambda: W.make_inputs(dataclasses.replace(W.RAGGED_BF16, batch=150), layout="flat",
                                             t_override=700),
    "ragged_flat": lambda: W.make_inputs(W.RAGGED_BF16, layout="flat", rows=5, t_override=1500),
    "sparse": lambda: W.make_inputs(dataclasses.replace(W.SPARSE_BF16, top_k=300), rows=3, t_override=5000),
    "verify": lambda: W.make_inputs(dataclasses.replace(W.VERIFY_BF16, top_k=0), rows=3, t_override=1100),
    "tiny_f32": lambda: W.make_inputs(W.TINY_F32),
}


# query rows checked against the oracle (all rows of the small cases)
ORACLE_ROWS = {"dense_t4096": None, "ragged_150_rows": [0, 1, 127, 128, 149], "ragged_flat": None,
               "sparse": None, "verify": None, "tiny_f32": None}
ORACLE_HEADS = {"dense_t4096": [0, 9, 64, 127], "ragged_150_rows": [0, 64, 127]}


def _check_call(case, step, ref, call):
    """One no-alloc call: against the workspace entry point's result and the oracle."""
    w = step.w
    ctx = torch.full_like(step.ctx, float("nan"))
    lse = torch.full_like(step.lse, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _no_alloc(step, ctx, lse, status)
    assert rc == 0, mla.lib.mla_last_error_detail().decode()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    H.assert_close(ctx, step.ctx, w.dtype, f"{case} ctx call {call} vs workspace entry point")
    fin = torch.isfinite(step.lse)
    assert torch.equal(torch.isfinite(lse), fin)
    assert torch.max(torch.abs(lse[fin] - step.lse[fin])).item() <= 2e-2
    rows, hs = ref["rows"], ref["heads"]
    ri, hi = torch.tensor(rows), torch.tensor(hs)
    H.assert_close(ctx.cpu()[ri][:, hi], ref["ctx"][rows], w.dtype, f"{case} ctx call {call} vs oracle")
    l_got, l_want = H.f64(lse.cpu()[ri][:, hi]), ref["lse"][rows]
    ok = np.isfinite(l_want)
    assert np.array_equal(np.isfinite(l_got), ok)
    assert np.max(np.abs(l_got[ok] - l_want[ok]), initial=0.0) <= (2e-2 if w.dtype == "bf16" else 1e-4)


def _prepare(case):
    inp = CASES[case]()
    step = DecodeStep(inp, "cuda", fused=False)
    step.run()                                  # reference: caller-allocated workspace
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    ref = H.oracle_reference(inp, ORACLE_ROWS[case], ORACLE_HEADS.get(case))
    return step, ref


@pytest.mark.parametrize("case", sorted(CASES))
def test_no_alloc_matches_workspace_entry_point_and_oracle(case):
    step, ref = _prepare(case)
    for call in range(2):                       # two calls in a row on the shared array
        _check_call(case, step, ref, call)


def test_no_alloc_calls_of_different_shapes_in_turn():
    # The shared array is not cleared between calls: each call must write all
    # it reads, whatever a larger call before it left there.
    order = ["ragged_150_rows", "sparse", "dense_t4096", "verify", "ragged_flat", "dense_t4096",
             "ragged_150_rows", "verify"]
    prepared = {c: _prepare(c) for c in sorted(set(order))}
    for k, case in enumerate(order):
        step, ref = prepared[case]
        _check_call(case, step, ref, k)


def test_no_alloc_refuses_requests_beyond_its_array():
    inp = W.make_inputs(W.DENSE_BF16)
    step = DecodeStep(inp, "cuda", fused=False)
    big_batch = 4096                            # far more split slots than the array holds
    need = mla.decode_workspace_size(big_batch, 1, 128, 512, 64, 4096, 0, False, torch.bfloat16)
    assert need > (64 << 20)
    ctx = torch.zeros_like(step.ctx)
    lse = torch.zeros_like(step.lse)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    w = dataclasses.replace(step.w, batch=big_batch)
    step.w = w
    rc = _no_alloc(step, ctx, lse, status)
    assert rc == 2                              # MLA_ERR_UNSUPPORTED
    assert "built-in" in mla.lib.mla_last_error_detail().decode()
    torch.cuda.synchronize()
    assert torch.count_nonzero(ctx) == 0        # nothing was launched
