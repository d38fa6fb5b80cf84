"""The hot path inside a CUDA graph.

Plans are built once outside the graph: their host-to-device copy comes from
pageable memory.  The attention calls and the merge are captured with the
caller's preallocated outputs and workspace and replayed.  Each replay must
give the eager call's results bit for bit, and so must a replay after new
query values are written into the captured query buffer.
"""

import math

import pytest
import torch

import cp_workloads as W
from test_gpu_parity import DEV, cp  # noqa: F401

pytestmark = pytest.mark.gpu


def capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()  # warm-up on a side stream, as torch asks before a capture
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_prefill_decode_merge_replay(cp):
    nl, pl, C, Hq, Hkv, D = [700, 64], [128, 0], 4, 8, 2, 128
    q, k, v = W.prefill_inputs(nl, pl, Hq, Hkv, D, "bf16", seed=31, device=DEV)
    plan = cp.cp_shard_plan(cp.CP_ZIGZAG, C, nl, pl, device=DEV)
    o = torch.empty_like(q)
    lse = torch.empty((q.shape[0], Hq), dtype=torch.float32, device=DEV)

    ctx, H = [3, 300, 4100], 64
    data = W.mla_decode_inputs(ctx, H=H, seed=32, device=DEV, bf16=False)
    dplan = cp.cp_decode_plan(C, ctx, n_workers=7, device=DEV)
    assert dplan.n_split > 0  # split pairs: the fixup kernel is in the graph too
    shards, scales = cp.cp_kv_shard_pack(dplan, data["kv_fp8"], data["kv_scale"])
    dq = data["q"].clone()
    B = len(ctx)
    o_part = torch.empty((C, B, H, 512), dtype=torch.float32, device=DEV)
    lse_part = torch.empty((C, B, H), dtype=torch.float32, device=DEV)
    ws = torch.empty(max(cp.cp_decode_workspace_size(dplan, H, 512), 16), dtype=torch.uint8, device=DEV)
    od = torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV)
    ld = torch.empty((B, H), dtype=torch.float32, device=DEV)

    def step():
        cp.cp_prefill_attn(plan, q, k, v, 1.0 / math.sqrt(D), out=o, lse=lse)
        cp.cp_decode_attn(dplan, cp.CP_DECODE_MLA, dq, shards, shard_scale=scales, sm_scale=1.0 / 24,
                          o_part=o_part, lse_part=lse_part, ws=ws)
        cp.cp_lse_merge(o_part, lse_part, out=od, lse=ld)

    step()
    cp.cp_device_error_check()
    ref = [t.clone() for t in (o, lse, od, ld)]
    g = capture(step)
    for t in (o, lse, od, ld):
        t.zero_()
    g.replay()
    cp.cp_device_error_check()
    for got, want in zip((o, lse, od, ld), ref):
        assert torch.equal(got, want)

    # new query values through the captured buffers
    q.copy_(W.prefill_inputs(nl, pl, Hq, Hkv, D, "bf16", seed=33, device=DEV)[0])
    dq.copy_(W.mla_decode_inputs(ctx, H=H, seed=34, device=DEV, bf16=False)["q"])
    g.replay()
    cp.cp_device_error_check()
    replayed = [t.clone() for t in (o, lse, od, ld)]
    step()
    cp.cp_device_error_check()
    for got, want in zip(replayed, (o, lse, od, ld)):
        assert torch.equal(got, want)
