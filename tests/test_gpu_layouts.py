"""GPU parity of the contiguous-chunk decode layout (vLLM DCP post §4) and
of decode steps with several query rows per request ("DeepSeek-V4 Attention
Inference Systems" §2.2, MTP / speculative decode), against the oracle:
the pack bit-exact, every shard's partial (O, LSE) and the merged result."""

import math

import numpy as np
import pytest
import torch

import cp_workloads as W
import oracle
from test_gpu_paged import make_pages
from test_gpu_parity import DEV, TOL_BF16, TOL_FP8, check_lse, check_o, cp, np64  # noqa: F401

pytestmark = pytest.mark.gpu


def token_map(L, C, contiguous):
    return (oracle.decode_shard_map_contiguous if contiguous else oracle.decode_shard_map)(L, C)


@pytest.mark.parametrize("contiguous", [False, True])
def test_pack_bit_exact(cp, contiguous):
    ctx = [0, 1, 7, 129, 1000, 4099]
    C = 8
    plan = cp.cp_decode_plan_ex(C, ctx, layout=int(contiguous), device=DEV)
    g = torch.Generator(device=DEV).manual_seed(3)
    T = sum(ctx)
    kv = torch.randint(0, 255, (T, 576), dtype=torch.uint8, device=DEV, generator=g)
    sc = torch.rand(T, device=DEV, generator=g)
    shards, scales = cp.cp_kv_shard_pack(plan, kv, sc)
    kvh, sch = kv.cpu().numpy(), sc.cpu().numpy()
    base = np.concatenate([[0], np.cumsum(ctx)])
    off = [0] * C
    for b, L in enumerate(ctx):
        shard, row = token_map(L, C, contiguous)
        for r in range(C):
            toks = [p for p in range(L) if shard[p] == r]
            assert [row[p] for p in toks] == list(range(len(toks)))
            got = shards[r][off[r]:off[r] + len(toks)].cpu().numpy()
            assert np.array_equal(got, kvh[base[b] + np.asarray(toks, dtype=np.int64)])
            assert np.array_equal(scales[r][off[r]:off[r] + len(toks)].cpu().numpy(),
                                  sch[base[b] + np.asarray(toks, dtype=np.int64)])
            off[r] += len(toks)
    assert [s.shape[0] for s in shards] == off


def run_mla(cp, data, ctx, C, s_q, H, fp8, contiguous, n_workers=0):
    plan = cp.cp_decode_plan_ex(C, ctx, layout=int(contiguous), s_q=s_q, n_workers=n_workers, device=DEV)
    B = len(ctx)
    q = data["q"].reshape(B, s_q, H, 576) if s_q > 1 else data["q"]
    if fp8:
        shards, scales = cp.cp_kv_shard_pack(plan, data["kv_fp8"], data["kv_scale"])
    else:
        shards, scales = cp.cp_kv_shard_pack(plan, data["kv_bf16"])
    scale = 1.0 / math.sqrt(576)
    o_part, lse_part = cp.cp_decode_attn(plan, cp.CP_DECODE_MLA, q, shards, shard_scale=scales,
                                         sm_scale=scale)
    N = B * s_q
    o, lse = cp.cp_lse_merge(o_part.reshape(C, N, H, 512), lse_part.reshape(C, N, H),
                             out_dtype=torch.float32)
    cp.cp_device_error_check()
    return plan, o_part.reshape(C, B, s_q, H, 512), lse_part.reshape(C, B, s_q, H), \
        o.reshape(B, s_q, H, 512), lse.reshape(B, s_q, H)


def check_mla(data, ctx, C, s_q, H, fp8, contiguous, o_part, lse_part, o, lse, reqs=None):
    tol = TOL_FP8 if fp8 else TOL_BF16
    base = np.concatenate([[0], np.cumsum(ctx)])
    B = len(ctx)
    qn = np64(data["q"]).reshape(B, s_q, H, 576)
    scale = 1.0 / math.sqrt(576)
    for b in (range(B) if reqs is None else reqs):
        L = ctx[b]
        if fp8:
            lat = oracle.e4m3_decode(data["kv_fp8"][base[b]:base[b] + L].cpu().numpy())
            K, V = oracle.mla_cache_to_kv(lat, data["kv_scale"][base[b]:base[b] + L].double().cpu().numpy())
        else:
            K, V = oracle.mla_cache_to_kv(np64(data["kv_bf16"][base[b]:base[b] + L]))
        po, pl = oracle.query_rows_partials(qn[b], K, V, C, scale, contiguous=contiguous)
        for r in range(C):
            for i in range(s_q):
                check_o(o_part[r, b, i], po[r, i], what=f"partial r{r} b{b} row{i}", **tol)
                check_lse(lse_part[r, b, i], pl[r, i])
        for i in range(s_q):
            fo, fl = oracle.decode_attention(qn[b, i], K[:L - s_q + i + 1], V[:L - s_q + i + 1], scale)
            check_o(o[b, i], fo, what=f"merged b{b} row{i}", **tol)
            check_lse(lse[b, i], fl)


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("contiguous", [False, True])
@pytest.mark.parametrize("s_q,H", [(1, 64), (2, 32), (4, 16), (3, 20)])
def test_mla_layout_and_query_rows(cp, fp8, contiguous, s_q, H):
    ctx = [max(s_q, 1), 5, 130, 1031, 4100]
    data = W.mla_decode_inputs(ctx, H=s_q * H, seed=41 + s_q, device=DEV)
    C = 8
    _, o_part, lse_part, o, lse = run_mla(cp, data, ctx, C, s_q, H, fp8, contiguous, n_workers=7)
    check_mla(data, ctx, C, s_q, H, fp8, contiguous, o_part, lse_part, o, lse)


def test_mla_query_rows_tiny_requests(cp):
    """Requests of exactly s_q tokens and shards that hold only tokens past a
    row's position (that row's partial there is empty)."""
    s_q, H, C = 4, 16, 8
    ctx = [4, 5, 6, 9, 12]
    for fp8 in (True, False):
        data = W.mla_decode_inputs(ctx, H=s_q * H, seed=77, device=DEV)
        for contiguous in (False, True):
            _, o_part, lse_part, o, lse = run_mla(cp, data, ctx, C, s_q, H, fp8, contiguous)
            check_mla(data, ctx, C, s_q, H, fp8, contiguous, o_part, lse_part, o, lse)


def gqa_rows_case(cp, ctx, Hq, Hkv, s_q, contiguous, seed, C=4, n_workers=5, D=128, dtype="bf16"):
    """GQA decode with s_q query rows per request: every shard's partials and
    the merged rows against the oracle."""
    B = len(ctx)
    q, k, v = W.gqa_decode_inputs(B, ctx, Hq * s_q, Hkv, D, dtype, seed=seed, device=DEV, std=0.3)
    plan = cp.cp_decode_plan_ex(C, ctx, layout=int(contiguous), s_q=s_q, n_workers=n_workers, device=DEV)
    qq = q.reshape(B, s_q, Hq, D) if s_q > 1 else q
    sk, _ = cp.cp_kv_shard_pack(plan, k)
    sv, _ = cp.cp_kv_shard_pack(plan, v)
    scale = 1.0 / math.sqrt(D)
    o_part, lse_part = cp.cp_decode_attn(plan, cp.CP_DECODE_GQA, qq, sk, sv, sm_scale=scale)
    o_part = o_part.reshape(C, B, s_q, Hq, D)
    lse_part = lse_part.reshape(C, B, s_q, Hq)
    o, lse = cp.cp_lse_merge(o_part.reshape(C, B * s_q, Hq, D), lse_part.reshape(C, B * s_q, Hq),
                             out_dtype=torch.float32)
    o, lse = o.reshape(B, s_q, Hq, D), lse.reshape(B, s_q, Hq)
    cp.cp_device_error_check()
    base = np.concatenate([[0], np.cumsum(ctx)])
    qn, kn, vn = np64(q).reshape(B, s_q, Hq, D), np64(k), np64(v)
    for b, L in enumerate(ctx):
        K, V = kn[base[b]:base[b] + L], vn[base[b]:base[b] + L]
        po, pl = oracle.query_rows_partials(qn[b], K, V, C, scale, contiguous=contiguous)
        for r in range(C):
            for i in range(s_q):
                check_o(o_part[r, b, i], po[r, i], what=f"GQA partial r{r} b{b} row{i}", **TOL_BF16)
                check_lse(lse_part[r, b, i], pl[r, i])
        for i in range(s_q):
            fo, fl = oracle.decode_attention(qn[b, i], K[:L - s_q + i + 1], V[:L - s_q + i + 1], scale)
            check_o(o[b, i], fo, what=f"GQA merged b{b} row{i}", **TOL_BF16)
            check_lse(lse[b, i], fl)


@pytest.mark.parametrize("contiguous", [False, True])
@pytest.mark.parametrize("s_q", [1, 3])
def test_gqa_layout_and_query_rows(cp, contiguous, s_q):
    gqa_rows_case(cp, [s_q, 40, 300, 4100], 8, 2, s_q, contiguous, seed=60 + s_q)


@pytest.mark.parametrize("Hq,Hkv,s_q,D", [(32, 4, 3, 128), (32, 4, 6, 128), (32, 16, 1, 128), (64, 8, 1, 128),
                                          (64, 8, 2, 128), (8, 8, 1, 128), (8, 2, 1, 64), (32, 4, 3, 64),
                                          (32, 4, 6, 64), (32, 8, 1, 64), (32, 32, 1, 128), (32, 32, 3, 128),
                                          (64, 32, 1, 64)])
def test_gqa_column_widths(cp, Hq, Hkv, s_q, D):
    """The tensor-core GQA decode pads a kv head's G s_q query columns to 16,
    32 or 64: each width at head dim 128 and 64, 16 kv heads, G = 1, ragged
    tiles and split pairs; 32 kv heads (multi-head attention among them),
    whose query operands load one kv head at a time."""
    ctx = [s_q, 129, 1000, 2600] + ([0] if s_q == 1 else [])
    gqa_rows_case(cp, ctx, Hq, Hkv, s_q, False, seed=Hq + 3 * Hkv + s_q + D, n_workers=7, D=D)


@pytest.mark.parametrize("Hq,Hkv,s_q,D,contiguous", [(8, 2, 2, 64, False), (8, 2, 3, 128, True),
                                                     (16, 1, 4, 64, False)])
def test_gqa_fp32_query_rows(cp, Hq, Hkv, s_q, D, contiguous):
    """fp32 caches on the tf32 GQA decode with several query rows (up to 64
    columns per kv head) and both shard layouts."""
    gqa_rows_case(cp, [s_q, 129, 1000, 2600], Hq, Hkv, s_q, contiguous, seed=400 + Hq + s_q + D,
                  n_workers=7, D=D, dtype="fp32")


def test_gqa_full_size_sampled(cp):
    """16 requests x 131,072 tokens, 32 q / 8 kv heads, head dim 128, C = 8:
    sampled requests against the oracle (whole context)."""
    B, L, Hq, Hkv, D, C = 16, 131072, 32, 8, 128, 8
    ctx = [L] * B
    q, k, v = W.gqa_decode_inputs(B, ctx, Hq, Hkv, D, "bf16", seed=71, device=DEV)
    plan = cp.cp_decode_plan(C, ctx, device=DEV)
    sk, _ = cp.cp_kv_shard_pack(plan, k)
    sv, _ = cp.cp_kv_shard_pack(plan, v)
    scale = 1.0 / math.sqrt(D)
    o_part, lse_part = cp.cp_decode_attn(plan, cp.CP_DECODE_GQA, q, sk, sv, sm_scale=scale)
    o, lse = cp.cp_lse_merge(o_part, lse_part, out_dtype=torch.float32)
    cp.cp_device_error_check()
    qn = np64(q)
    for b in (0, 11):
        K, V = np64(k[b * L:(b + 1) * L]), np64(v[b * L:(b + 1) * L])
        fo, fl = oracle.decode_attention(qn[b], K, V, scale)
        check_o(o[b], fo, what=f"full-size GQA b{b}", **TOL_BF16)
        check_lse(lse[b], fl)


def test_paged_contiguous_query_rows_match_unpaged(cp):
    """The paged pool with a contiguous-layout MTP plan gives bit-identical
    partials to the per-shard buffers."""
    s_q, H, C, page = 2, 32, 4, 64
    ctx = [2, 200, 1500]
    data = W.mla_decode_inputs(ctx, H=s_q * H, seed=91, device=DEV)
    plan, o_ref, l_ref, _, _ = run_mla(cp, data, ctx, C, s_q, H, True, True, n_workers=6)
    pages = make_pages(cp, plan, page, seed=5)
    pool, spool = cp.cp_kv_shard_pack_paged(plan, pages, data["kv_fp8"], data["kv_scale"])
    q = data["q"].reshape(len(ctx), s_q, H, 576)
    o_p, l_p = cp.cp_decode_attn_paged(plan, pages, cp.CP_DECODE_MLA, q, pool, scale_pool=spool,
                                       sm_scale=1.0 / math.sqrt(576))
    cp.cp_device_error_check()
    assert torch.equal(o_p.reshape(o_ref.shape), o_ref) and torch.equal(l_p.reshape(l_ref.shape), l_ref)


def test_mla_query_rows_full_size_sampled(cp):
    """64 requests x 131,072 tokens, 2 query rows of 32 heads, FP8, C = 8:
    sampled requests and rows against the oracle."""
    B, L, s_q, H, C = 64, 131072, 2, 32, 8
    ctx = [L] * B
    data = W.mla_decode_inputs(ctx, H=s_q * H, seed=55, device=DEV, bf16=False)
    _, o_part, lse_part, o, lse = run_mla(cp, data, ctx, C, s_q, H, True, False)
    scale = 1.0 / math.sqrt(576)
    qn = np64(data["q"]).reshape(B, s_q, H, 576)
    for b in (0, 41):
        lat = oracle.e4m3_decode(data["kv_fp8"][b * L:(b + 1) * L].cpu().numpy())
        K, V = oracle.mla_cache_to_kv(lat, data["kv_scale"][b * L:(b + 1) * L].double().cpu().numpy())
        for i in range(s_q):
            fo, fl = oracle.decode_attention(qn[b, i], K[:L - s_q + i + 1], V[:L - s_q + i + 1], scale)
            check_o(o[b, i], fo, what=f"full-size MTP b{b} row{i}", **TOL_FP8)
            check_lse(lse[b, i], fl)


def test_gqa_paged_query_rows_match_unpaged(cp):
    """GQA with 3 query rows over a paged pool: bit-identical to the per-shard buffers."""
    ctx = [3, 130, 900]
    B, Hq, Hkv, D, C, s_q = len(ctx), 8, 2, 64, 4, 3
    q, k, v = W.gqa_decode_inputs(B, ctx, Hq * s_q, Hkv, D, "bf16", seed=66, device=DEV, std=0.3)
    plan = cp.cp_decode_plan_ex(C, ctx, s_q=s_q, n_workers=5, device=DEV)
    qq = q.reshape(B, s_q, Hq, D)
    sk, _ = cp.cp_kv_shard_pack(plan, k)
    sv, _ = cp.cp_kv_shard_pack(plan, v)
    o_ref, l_ref = cp.cp_decode_attn(plan, cp.CP_DECODE_GQA, qq, sk, sv, sm_scale=0.125)
    pages = make_pages(cp, plan, 64, seed=6)
    kp, _ = cp.cp_kv_shard_pack_paged(plan, pages, k)
    vp, _ = cp.cp_kv_shard_pack_paged(plan, pages, v)
    o_p, l_p = cp.cp_decode_attn_paged(plan, pages, cp.CP_DECODE_GQA, qq, kp, vp, sm_scale=0.125)
    cp.cp_device_error_check()
    assert torch.equal(o_p, o_ref) and torch.equal(l_p, l_ref)


def gqa_fp8_rows_case(cp, ctx, Hq, Hkv, s_q, contiguous, seed, C=4, n_workers=5):
    """GQA over an E4M3 cache (one scale per token for its K and V rows) with
    s_q query rows per request: every shard's partials and the merged rows
    against the oracle (codes decoded bit by bit, times the scale)."""
    B, D = len(ctx), 128
    q, kc, vc, sc = W.gqa_decode_inputs_fp8(B, ctx, Hq * s_q, Hkv, D, seed=seed, device=DEV, std=0.3)
    plan = cp.cp_decode_plan_ex(C, ctx, layout=int(contiguous), s_q=s_q, n_workers=n_workers, device=DEV)
    qq = q.reshape(B, s_q, Hq, D) if s_q > 1 else q
    sk, ss = cp.cp_kv_shard_pack(plan, kc, sc)
    sv, _ = cp.cp_kv_shard_pack(plan, vc)
    scale = 1.0 / math.sqrt(D)
    o_part, lse_part = cp.cp_decode_attn(plan, cp.CP_DECODE_GQA, qq, sk, sv, shard_scale=ss, sm_scale=scale)
    o_part = o_part.reshape(C, B, s_q, Hq, D)
    lse_part = lse_part.reshape(C, B, s_q, Hq)
    o, lse = cp.cp_lse_merge(o_part.reshape(C, B * s_q, Hq, D), lse_part.reshape(C, B * s_q, Hq),
                             out_dtype=torch.float32)
    o, lse = o.reshape(B, s_q, Hq, D), lse.reshape(B, s_q, Hq)
    cp.cp_device_error_check()
    base = np.concatenate([[0], np.cumsum(ctx)])
    s64 = sc.double().cpu().numpy()[:, None, None]
    kn = oracle.e4m3_decode(kc.cpu().numpy()) * s64
    vn = oracle.e4m3_decode(vc.cpu().numpy()) * s64
    qn = np64(q).reshape(B, s_q, Hq, D)
    for b, L in enumerate(ctx):
        K, V = kn[base[b]:base[b] + L], vn[base[b]:base[b] + L]
        po, pl = oracle.query_rows_partials(qn[b], K, V, C, scale, contiguous=contiguous)
        for r in range(C):
            for i in range(s_q):
                check_o(o_part[r, b, i], po[r, i], what=f"FP8 GQA partial r{r} b{b} row{i}", **TOL_FP8)
                check_lse(lse_part[r, b, i], pl[r, i])
        for i in range(s_q):
            fo, fl = oracle.decode_attention(qn[b, i], K[:L - s_q + i + 1], V[:L - s_q + i + 1], scale)
            check_o(o[b, i], fo, what=f"FP8 GQA merged b{b} row{i}", **TOL_FP8)
            check_lse(lse[b, i], fl)


@pytest.mark.parametrize("Hq,Hkv,s_q,contiguous", [(8, 2, 2, False), (8, 2, 3, True), (16, 4, 2, True),
                                                   (32, 8, 1, False), (16, 16, 1, False), (32, 1, 1, True)])
def test_gqa_fp8_query_rows_and_widths(cp, Hq, Hkv, s_q, contiguous):
    """The FP8 tensor-core GQA decode pads a kv head's G s_q query columns to
    16 or 32: several query rows, both shard layouts, one query head per kv
    head, one kv head for 32 query heads, ragged tiles and split pairs."""
    ctx = [s_q, 129, 1000, 2600] + ([0] if s_q == 1 else [])
    gqa_fp8_rows_case(cp, ctx, Hq, Hkv, s_q, contiguous, seed=300 + Hq + Hkv + s_q, n_workers=7)


def test_gqa_fp8_full_size_sampled(cp):
    """16 requests x 131,072 tokens over an E4M3 cache, 32 q / 8 kv heads,
    head dim 128, C = 8 (the benchmark's GQA workload): one sampled request,
    whole context, against the oracle."""
    B, L, Hq, Hkv, D, C = 16, 131072, 32, 8, 128, 8
    ctx = [L] * B
    q, kc, vc, sc = W.gqa_decode_inputs_fp8(B, ctx, Hq, Hkv, D, seed=72, device=DEV)
    plan = cp.cp_decode_plan(C, ctx, device=DEV)
    sk, ss = cp.cp_kv_shard_pack(plan, kc, sc)
    sv, _ = cp.cp_kv_shard_pack(plan, vc)
    scale = 1.0 / math.sqrt(D)
    o_part, lse_part = cp.cp_decode_attn(plan, cp.CP_DECODE_GQA, q, sk, sv, shard_scale=ss, sm_scale=scale)
    o, lse = cp.cp_lse_merge(o_part, lse_part, out_dtype=torch.float32)
    cp.cp_device_error_check()
    b = 9
    s64 = sc[b * L:(b + 1) * L].double().cpu().numpy()[:, None, None]
    K = oracle.e4m3_decode(kc[b * L:(b + 1) * L].cpu().numpy()) * s64
    V = oracle.e4m3_decode(vc[b * L:(b + 1) * L].cpu().numpy()) * s64
    fo, fl = oracle.decode_attention(np64(q)[b], K, V, scale)
    check_o(o[b], fo, what=f"full-size FP8 GQA b{b}", **TOL_FP8)
    check_lse(lse[b], fl)
