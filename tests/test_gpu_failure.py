"""Failure detection without a GPU fault: a bounded wait that runs out.

With CPATTN_TEST_STALL=1 the tensor-core prefill's MMA thread waits on a
barrier that nothing arrives at.  The wait gives up after its limit, the
kernel drains its copies and MMAs, frees its tensor memory and returns, and
the host reads CP_ERR_DEVICE_TIMEOUT from the device status word.  The
context stays usable: the next call runs normally and matches the oracle.
"""

import math
import os

import numpy as np
import pytest
import torch

import cp_workloads as W
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cp():
    import __graft_entry__
    __graft_entry__.ensure_built()
    import context_long_attention_gb300 as cp
    return cp


def test_bounded_wait_reports_timeout_and_context_survives(cp, monkeypatch):
    new_len, prefix_len, C = [300], [40], 2
    q, k, v = W.prefill_inputs(new_len, prefix_len, 4, 2, 64, "bf16", seed=5, device="cuda")
    plan = cp.cp_shard_plan(cp.CP_ZIGZAG, C, new_len, prefix_len, device="cuda")
    cp.cp_device_error_check()  # clean start
    monkeypatch.setenv("CPATTN_TEST_STALL", "1")
    cp.cp_prefill_attn(plan, q, k, v, 1 / 8)
    with pytest.raises(cp.CpError) as ei:
        cp.cp_device_error_check()
    assert ei.value.status == -4 and "bounded wait" in str(ei.value)
    monkeypatch.delenv("CPATTN_TEST_STALL")
    cp.cp_device_error_check()  # the status word was cleared
    o, lse = cp.cp_prefill_attn(plan, q, k, v, 1 / 8)
    cp.cp_device_error_check()
    ref = oracle.prefill_reference(oracle.zigzag_plan(new_len, prefix_len, C), new_len, prefix_len,
                                   q.double().cpu().numpy(), k.double().cpu().numpy(),
                                   v.double().cpu().numpy(), 1 / 8)
    ro = plan.rank_off
    for r in range(C):
        _, o_ref, l_ref = ref[r]
        assert np.abs(o[ro[r]:ro[r + 1]].double().cpu().numpy() - o_ref).max() <= 2e-2
        assert np.abs(lse[ro[r]:ro[r + 1]].double().cpu().numpy() - l_ref).max() <= 1e-3
