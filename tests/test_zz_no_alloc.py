"""The allocation-free decode entry point, checked against the workspace one.

cp_decode_attn_noalloc serves callers that cannot allocate device memory at
the point of the call: serving loops held to a fixed memory budget, and
plugins reached through a C interface that gives them no allocator.  Its
split-KV scratch lives in a static device array inside the library instead
of a caller workspace.

Both entry points run the same kernels on the same plan and inputs; only the
place of the scratch differs, so their outputs must be bit-identical.  The
tests call it through the C ABI twice in a row on schedules that split KV
ranges across workers (so the array is really used): an FP8 MLA plan, then a
smaller bf16 GQA plan run after a larger one, whose leftovers in the array
must never be read.  The workspace calls get a NaN-filled workspace, so a
read of a slot the call did not write shows up as a difference.  This file
is collected last so that a run stopping at its first failure has run every
other test before it.
"""

import math

import pytest
import torch

import cp_workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cp():
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")
    import __graft_entry__
    __graft_entry__.ensure_built()
    import context_long_attention_gb300 as cp
    return cp


def nan_workspace(cp, plan, H, Dv):
    need = cp.cp_decode_workspace_size(plan, H, Dv)
    assert 0 < need <= cp._binding.NOALLOC_SCRATCH_BYTES
    return torch.full((need // 4 + 4,), float("nan"), dtype=torch.float32, device="cuda").view(torch.uint8)


def assert_bit_identical(a, b):
    for x, y in zip(a, b):
        assert x.shape == y.shape and torch.equal(x.view(torch.int32), y.view(torch.int32))


def test_noalloc_decode_matches_workspace_decode_twice(cp):
    ctx = [0, 1, 3, 129, 1000, 4097, 2500]
    C = 8
    data = W.mla_decode_inputs(ctx, H=64, seed=77, device="cuda")
    plan = cp.cp_decode_plan(C, ctx, n_workers=5, device="cuda")
    assert plan.n_parts > 0  # the schedule splits pairs: scratch is used
    shards, scales = cp.cp_kv_shard_pack(plan, data["kv_fp8"], data["kv_scale"])
    scale = 1.0 / math.sqrt(576)
    ref = cp.cp_decode_attn(plan, cp.CP_DECODE_MLA, data["q"], shards, shard_scale=scales,
                            sm_scale=scale, ws=nan_workspace(cp, plan, 64, 512))
    cp.cp_device_error_check()
    for _ in range(2):
        out = cp.cp_decode_attn_noalloc(plan, cp.CP_DECODE_MLA, data["q"], shards,
                                        shard_scale=scales, sm_scale=scale)
        cp.cp_device_error_check()
        assert_bit_identical(out, ref)


def test_noalloc_leftovers_of_a_larger_plan_are_never_read(cp):
    # a large MLA plan fills much of the array first
    big_ctx = [20000, 30000, 9000]
    big = W.mla_decode_inputs(big_ctx, H=64, seed=5, device="cuda", bf16=True, fp8=False)
    bplan = cp.cp_decode_plan(8, big_ctx, n_workers=40, device="cuda")
    assert bplan.n_parts > 0
    bsh, _ = cp.cp_kv_shard_pack(bplan, big["kv_bf16"])
    cp.cp_decode_attn_noalloc(bplan, cp.CP_DECODE_MLA, big["q"], bsh, sm_scale=1 / 24)
    # then a smaller bf16 GQA plan whose pairs are split across workers
    ctx = [700, 5, 2049, 300]
    Hq, Hkv, D = 16, 4, 128
    q, k, v = W.gqa_decode_inputs(len(ctx), ctx, Hq, Hkv, D, "bf16", seed=9, device="cuda")
    plan = cp.cp_decode_plan(4, ctx, n_workers=7, device="cuda")
    assert plan.n_parts > 0
    sk, _ = cp.cp_kv_shard_pack(plan, k)
    sv, _ = cp.cp_kv_shard_pack(plan, v)
    scale = 1.0 / math.sqrt(D)
    ref = cp.cp_decode_attn(plan, cp.CP_DECODE_GQA, q, sk, sv, sm_scale=scale,
                            ws=nan_workspace(cp, plan, Hq, D))
    cp.cp_device_error_check()
    for _ in range(2):
        out = cp.cp_decode_attn_noalloc(plan, cp.CP_DECODE_GQA, q, sk, sv, sm_scale=scale)
        cp.cp_device_error_check()
        assert_bit_identical(out, ref)


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
