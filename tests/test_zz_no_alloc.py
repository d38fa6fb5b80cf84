"""The allocation-free decode entry point, checked against the workspace one.

cp_decode_attn_noalloc serves callers that cannot allocate device memory at
the point of the call — code inside a CUDA-graph capture that must not grow
the memory pool, serving loops with a fixed memory budget, plugins reached
through a C interface without an allocator.  Its split-KV scratch lives in a
static device array inside the library instead of a caller workspace.

The test calls it through the C ABI twice in a row, on a schedule that splits
KV ranges across workers (so the scratch array is really used), and compares
each result with cp_decode_attn given a torch-allocated workspace, within the
FP8-cache tolerance of the parity tests.  This file is collected last so that
a run stopping at its first failure has run every other test before it.
"""

import math

import numpy as np
import pytest
import torch

import cp_workloads as W

pytestmark = pytest.mark.gpu

TOL_FP8_MAX_ABS = 6e-2
TOL_LSE = 1e-3


@pytest.fixture(scope="module")
def cp():
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")
    import __graft_entry__
    __graft_entry__.ensure_built()
    import context_long_attention_gb300 as cp
    return cp


def test_noalloc_decode_matches_workspace_decode_twice(cp):
    ctx = [0, 1, 3, 129, 1000, 4097, 2500]
    C = 8
    data = W.mla_decode_inputs(ctx, H=64, seed=77, device="cuda")
    plan = cp.cp_decode_plan(C, ctx, n_workers=5, device="cuda")
    assert plan.n_parts > 0  # the schedule splits pairs: scratch is used
    need = cp.cp_decode_workspace_size(plan, 64, 512)
    assert 0 < need <= cp._binding.NOALLOC_SCRATCH_BYTES
    shards, scales = cp.cp_kv_shard_pack(plan, data["kv_fp8"], data["kv_scale"])
    scale = 1.0 / math.sqrt(576)
    ref_o, ref_l = cp.cp_decode_attn(plan, cp.CP_DECODE_MLA, data["q"], shards,
                                     shard_scale=scales, sm_scale=scale)
    cp.cp_device_error_check()
    ref_o, ref_l = ref_o.double().cpu().numpy(), ref_l.double().cpu().numpy()
    for _ in range(2):
        o, l = cp.cp_decode_attn_noalloc(plan, cp.CP_DECODE_MLA, data["q"], shards,
                                         shard_scale=scales, sm_scale=scale)
        cp.cp_device_error_check()
        o, l = o.double().cpu().numpy(), l.double().cpu().numpy()
        assert np.array_equal(np.isneginf(l), np.isneginf(ref_l))
        fin = np.isfinite(ref_l)
        assert np.abs(l[fin] - ref_l[fin]).max() <= TOL_LSE
        assert np.abs(o - ref_o).max() <= TOL_FP8_MAX_ABS


def test_noalloc_rejects_plans_beyond_its_scratch(cp):
    ctx = [131072] * 16
    plan = cp.cp_decode_plan(8, ctx, n_workers=2048, device=None)  # host-only plan
    need = cp.cp_decode_workspace_size(plan, 64, 512)
    assert need > cp._binding.NOALLOC_SCRATCH_BYTES
    q = torch.empty((16, 64, 576), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cp.CpError) as ei:
        cp.cp_decode_attn_noalloc(plan, cp.CP_DECODE_MLA, q, [q] * 8,
                                  shard_scale=[q.float()] * 8)
    assert ei.value.status == -5 and "fixed" in str(ei.value)
