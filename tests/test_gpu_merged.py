"""GPU parity of cp_decode_attn_merged (the decode and the LSE merge of its
shard partials in one call; "How GPUs Share a Long Context During LLM
Inference" §3.3, "DeepSeek-V4 Attention Inference Systems" §5): the merged
(O, LSE) of every request (every query row) against the oracle's attention
over the whole cache.  For the MLA caches (FP8 and bf16) a worker's
consecutive items of one request accumulate as one run, so the cases mix
short requests (whole runs), long ones (cut by worker boundaries into parts),
empty ones and tiny worker counts; GQA caches go through the per-shard
partials and must match cp_decode_attn + cp_lse_merge bit for bit."""

import math

import numpy as np
import pytest
import torch

import cp_workloads as W
import oracle
from test_gpu_parity import DEV, TOL_BF16, TOL_FP8, check_lse, check_o, cp, np64  # noqa: F401

pytestmark = pytest.mark.gpu


def kv_fp64(data, b, fp8):
    ctx = data["ctx"]
    base = np.concatenate([[0], np.cumsum(ctx)])
    sl = slice(int(base[b]), int(base[b + 1]))
    if fp8:
        lat = oracle.e4m3_decode(data["kv_fp8"][sl].cpu().numpy())
        return oracle.mla_cache_to_kv(lat, data["kv_scale"][sl].double().cpu().numpy())
    return oracle.mla_cache_to_kv(np64(data["kv_bf16"][sl]))


def merged_mla(cp, data, C, s_q, H, fp8, contiguous, n_workers, out_dtype):
    ctx = data["ctx"]
    B = len(ctx)
    plan = cp.cp_decode_plan_ex(C, ctx, layout=int(contiguous), s_q=s_q, n_workers=n_workers, device=DEV)
    q = data["q"].reshape(B, s_q, H, 576) if s_q > 1 else data["q"]
    if fp8:
        shards, scales = cp.cp_kv_shard_pack(plan, data["kv_fp8"], data["kv_scale"])
    else:
        shards, scales = cp.cp_kv_shard_pack(plan, data["kv_bf16"])
    o, lse = cp.cp_decode_attn_merged(plan, cp.CP_DECODE_MLA, q, shards, shard_scale=scales,
                                      sm_scale=1.0 / math.sqrt(576), out_dtype=out_dtype)
    cp.cp_device_error_check()
    return plan, o.reshape(B, s_q, H, 512), lse.reshape(B, s_q, H)


def check_merged(data, s_q, H, fp8, o, lse, reqs=None):
    ctx = data["ctx"]
    B = len(ctx)
    qn = np64(data["q"]).reshape(B, s_q, H, 576)
    scale = 1.0 / math.sqrt(576)
    tol = TOL_FP8 if fp8 else TOL_BF16
    for b in (range(B) if reqs is None else reqs):
        L = ctx[b]
        if L == 0:
            assert torch.all(o[b] == 0) and torch.all(lse[b] == -math.inf)
            continue
        K, V = kv_fp64(data, b, fp8)
        for i in range(s_q):
            fo, fl = oracle.decode_attention(qn[b, i], K[:L - s_q + i + 1], V[:L - s_q + i + 1], scale)
            check_o(o[b, i], fo, what=f"merged b{b} row{i}", **tol)
            check_lse(lse[b, i], fl)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("C,nw", [(8, 3), (8, 152), (4, 1), (1, 5), (8, 41)])
def test_merged_mla_fp8(cp, C, nw, out_dtype):
    ctx = [0, 1, 3, 129, 1000, 4097, 20000, 700, 5]
    data = W.mla_decode_inputs(ctx, H=64, seed=500 + C + nw, device=DEV)
    data["ctx"] = ctx
    plan, o, lse = merged_mla(cp, data, C, 1, 64, True, False, nw, out_dtype)
    assert o.dtype == out_dtype
    check_merged(data, 1, 64, True, o, lse)
    if C > 1 and nw <= 5:  # long runs across several pairs and shards
        assert any(len(set(int(p) % len(ctx) for p in plan.work[a:b2, 0])) < b2 - a
                   for a, b2 in zip(plan.worker_off[:-1], plan.worker_off[1:]))


@pytest.mark.parametrize("contiguous", [False, True])
@pytest.mark.parametrize("s_q,H", [(2, 32), (3, 20)])
def test_merged_mla_fp8_query_rows(cp, contiguous, s_q, H):
    """Several query rows (a row reads the tokens up to L - s_q + i): runs
    that start on a pair's last rows, masked for some rows, and go on to
    another shard's first tokens."""
    ctx = [s_q, 130, 1031, 4100, 257, 2 * 128 * 8 + 1, 6]
    data = W.mla_decode_inputs(ctx, H=s_q * H, seed=520 + s_q, device=DEV)
    data["ctx"] = ctx
    for nw in (2, 9, 64):
        _, o, lse = merged_mla(cp, data, 8, s_q, H, True, contiguous, nw, torch.float32)
        check_merged(data, s_q, H, True, o, lse)


def test_merged_mla_fp8_scale_spread(cp):
    """Per-token scales growing along each request by up to 2^6, so that the
    weights' scale exponent must fall as a run goes on across shards."""
    ctx = [3000, 700, 129, 9000]
    data = W.mla_decode_inputs(ctx, H=40, seed=541, device=DEV)
    g = torch.Generator().manual_seed(543)
    k = torch.cat([torch.clamp(torch.arange(L) * 7 // L + torch.randint(0, 2, (L,), generator=g), max=6)
                   for L in ctx]).to(torch.float32)
    scale = (data["kv_scale"].cpu() * torch.pow(2.0, k)).to(DEV)
    data["kv_fp8"] = (data["kv_bf16"].float() / scale[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    data["kv_scale"] = scale
    data["ctx"] = ctx
    for C, nw in [(8, 3), (2, 1), (8, 30)]:
        _, o, lse = merged_mla(cp, data, C, 1, 40, True, False, nw, torch.float32)
        check_merged(data, 1, 40, True, o, lse)


def test_merged_mla_fp8_full_size_sampled(cp):
    """64 x 131,072 tokens, C = 8 (the decode benchmark's batch): sampled
    requests against the oracle."""
    w = W.WORKLOADS["mla"]
    data = W.mla_decode_inputs([w["ctx"]] * w["B"], H=w["H"], seed=W.SEEDS["mla"], device=DEV, fp8=True,
                               bf16=False)
    data["ctx"] = [w["ctx"]] * w["B"]
    _, o, lse = merged_mla(cp, data, w["C"], 1, w["H"], True, False, 0, torch.bfloat16)
    check_merged(data, 1, w["H"], True, o, lse, reqs=[0, 29, 63])
    del data
    torch.cuda.empty_cache()


@pytest.mark.parametrize("C,nw,s_q,H", [(8, 3, 1, 64), (8, 152, 1, 64), (1, 5, 1, 64), (8, 9, 3, 20),
                                        (4, 64, 2, 32)])
def test_merged_mla_bf16(cp, C, nw, s_q, H):
    """The bf16 MLA kernel's runs, as the FP8 one's."""
    ctx = [0, 1, 3, 129, 1000, 4097, 20000, 5] if s_q == 1 else [s_q, 130, 1031, 4100, 2 * 128 * 8 + 1, 6]
    data = W.mla_decode_inputs(ctx, H=s_q * H, seed=570 + C + nw + s_q, device=DEV, fp8=False, bf16=True)
    data["ctx"] = ctx
    _, o, lse = merged_mla(cp, data, C, s_q, H, False, False, nw, torch.float32)
    check_merged(data, s_q, H, False, o, lse)


def test_merged_gqa_matches_decode_then_merge(cp):
    """A GQA cache takes the per-shard partials in the workspace: the same
    kernels as cp_decode_attn + cp_lse_merge, the same bits."""
    ctx = [0, 9, 300, 4100]
    plan = cp.cp_decode_plan(8, ctx, n_workers=7, device=DEV)
    Hq, Hkv, D = 16, 4, 128
    q, k, v = W.gqa_decode_inputs(len(ctx), ctx, Hq, Hkv, D, "bf16", seed=561, device=DEV, std=0.3)
    sk, _ = cp.cp_kv_shard_pack(plan, k)
    sv, _ = cp.cp_kv_shard_pack(plan, v)
    o, lse = cp.cp_decode_attn_merged(plan, cp.CP_DECODE_GQA, q, sk, sv, sm_scale=1 / math.sqrt(D))
    op, lp = cp.cp_decode_attn(plan, cp.CP_DECODE_GQA, q, sk, sv, sm_scale=1 / math.sqrt(D))
    o2, lse2 = cp.cp_lse_merge(op, lp, out_dtype=torch.bfloat16)
    cp.cp_device_error_check()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_pair_split_into_more_than_64_parts(cp):
    """One shard (C = 1) and a long request over 152 workers: its only pair is
    cut into more than 64 parts, which the split merge (cp_decode_attn) and
    the runs' merge (cp_decode_attn_merged) both take in lane-sized chunks."""
    ctx = [70000, 300]
    data = W.mla_decode_inputs(ctx, H=64, seed=580, device=DEV)
    data["ctx"] = ctx
    plan = cp.cp_decode_plan(1, ctx, n_workers=152, device=DEV)
    pairs = plan.pairs
    assert int(pairs[0, 3]) > 64  # n_parts of the long pair
    shards, scales = cp.cp_kv_shard_pack(plan, data["kv_fp8"], data["kv_scale"])
    op, lp = cp.cp_decode_attn(plan, cp.CP_DECODE_MLA, data["q"], shards, shard_scale=scales,
                               sm_scale=1.0 / math.sqrt(576))
    o1, l1 = cp.cp_lse_merge(op, lp, out_dtype=torch.float32)
    cp.cp_device_error_check()
    check_merged(data, 1, 64, True, o1.reshape(2, 1, 64, 512), l1.reshape(2, 1, 64))
    assert int(max(n for _, _, n in plan.merge_list)) > 64
    _, o2, l2 = merged_mla(cp, data, 1, 1, 64, True, False, 152, torch.float32)
    check_merged(data, 1, 64, True, o2, l2)
