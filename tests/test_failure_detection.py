"""Failure detection without a GPU fault: a bounded device wait on a barrier
that nothing completes gives up, records MLA_DEVICE_TIMEOUT and returns; the
context stays usable (a decode step afterwards matches the oracle)."""
import dataclasses

import pytest
import torch

from tests import helpers as H

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from mla_latent_kv_12_gb300 import mla
    from mla_latent_kv_12_gb300 import workloads as W
    from mla_latent_kv_12_gb300.pipeline import DecodeStep


def test_bounded_wait_times_out_and_context_survives():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    limit = 2_000_000                      # about a millisecond of SM clock
    mla.selftest_bounded_wait(limit, st, waited)
    torch.cuda.synchronize()
    assert int(st.item()) == mla.DEVICE_TIMEOUT
    assert limit <= int(waited.item()) < 50 * limit
    # the context is healthy: an ordinary decode step still matches the oracle
    inp = W.make_inputs(dataclasses.replace(W.DENSE_BF16, t=300))
    step = DecodeStep(inp, "cuda")
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    H.compare_step(step, H.oracle_reference(inp), "bf16")
