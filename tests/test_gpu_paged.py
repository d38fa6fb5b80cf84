"""GPU parity of the paged token-sharded decode cache against the oracle.

The pool layout is the oracle's enumeration (token p -> shard p mod C, row
p // C -> page table); packing is bit-exact, the decode partials and the
merge meet the same tolerances as the contiguous cache, and the paged decode
reproduces the contiguous decode bit for bit (the same products in the same
order, rows read from elsewhere)."""

import math

import numpy as np
import pytest
import torch

import cp_workloads as W
import oracle
from test_gpu_parity import DEV, TOL_BF16, TOL_FP8, check_lse, check_o, cp, np64  # noqa: F401

pytestmark = pytest.mark.gpu


def make_pages(cp, plan, page_size, seed, spare=3):
    """Random distinct page ids for every pair's pages, `spare` unused pages
    in the pool, -1 in the unused table entries."""
    rows = plan.pairs[:, 0]
    need = [-(-int(n) // page_size) for n in rows]
    maxp = max(1, max(need))
    rng = np.random.default_rng(seed)
    num_pages = sum(need) + spare
    ids = rng.permutation(num_pages)
    table = np.full((len(rows), maxp), -1, np.int32)
    k = 0
    for pr, n in enumerate(need):
        table[pr, :n] = ids[k:k + n]
        k += n
    return cp.PageTable(table, page_size, num_pages, device=DEV)


def expected_pool_rows(ctx, C, pages):
    """(global token index, pool row) of every token, from the oracle's rule."""
    base = np.concatenate([[0], np.cumsum(ctx)])
    rows = oracle.paged_token_rows(ctx, C, pages.host, pages.page_size)
    return np.array([base[b] + p for b, p, _ in rows], np.int64), np.array([x for _, _, x in rows], np.int64)


@pytest.mark.parametrize("kind", ["fp8", "bf16", "gqa"])
@pytest.mark.parametrize("C,page_size", [(8, 64), (3, 128), (1, 192)])
def test_paged_pack_bit_exact(cp, kind, C, page_size):
    ctx = [0, 1, 77, 300, 4100]
    plan = cp.cp_decode_plan(C, ctx, device=DEV)
    pages = make_pages(cp, plan, page_size, seed=C + page_size)
    if kind == "gqa":
        _, k, _ = W.gqa_decode_inputs(len(ctx), ctx, 8, 2, 64, "bf16", seed=3, device=DEV)
        kv, sc = k, None
    else:
        d = W.mla_decode_inputs(ctx, H=4, seed=4, device=DEV, fp8=kind == "fp8", bf16=kind == "bf16")
        kv, sc = (d["kv_fp8"], d["kv_scale"]) if kind == "fp8" else (d["kv_bf16"], None)
    pool, spool = cp.cp_kv_shard_pack_paged(plan, pages, kv, sc)
    torch.cuda.synchronize()
    tok, prow = expected_pool_rows(ctx, C, pages)
    tok_t, prow_t = torch.as_tensor(tok, device=DEV), torch.as_tensor(prow, device=DEV)
    assert torch.equal(pool[prow_t].view(torch.uint8), kv[tok_t].view(torch.uint8))
    if sc is not None:
        assert torch.equal(spool[prow_t], sc[tok_t])
    # rows past each pair's last row on its last page are zero
    for pr, n in enumerate(plan.pairs[:, 0]):
        n = int(n)
        end = -(-n // page_size) * page_size
        for i in range(n, end):
            row = int(pages.host[pr, i // page_size]) * page_size + i % page_size
            assert not pool[row].view(torch.uint8).any(), f"pair {pr} tail row {i} not zero"
            if spool is not None:
                assert spool[row].item() == 0.0


def mla_paged_case(cp, data, C, fp8, nw, page_size, seed):
    ctx = data["ctx"]
    scale = 1.0 / math.sqrt(576)
    plan = cp.cp_decode_plan(C, ctx, n_workers=nw, device=DEV)
    pages = make_pages(cp, plan, page_size, seed)
    kv, sc = (data["kv_fp8"], data["kv_scale"]) if fp8 else (data["kv_bf16"], None)
    pool, spool = cp.cp_kv_shard_pack_paged(plan, pages, kv, sc)
    o_part, lse_part = cp.cp_decode_attn_paged(plan, pages, cp.CP_DECODE_MLA, data["q"], pool,
                                               scale_pool=spool, sm_scale=scale)
    o, lse = cp.cp_lse_merge(o_part, lse_part, out_dtype=torch.bfloat16)
    # the contiguous cache through the same kernels
    shards, sscales = cp.cp_kv_shard_pack(plan, kv, sc)
    o_c, lse_c = cp.cp_decode_attn(plan, cp.CP_DECODE_MLA, data["q"], shards, shard_scale=sscales,
                                   sm_scale=scale)
    cp.cp_device_error_check()
    assert torch.equal(o_part, o_c) and torch.equal(lse_part, lse_c), "paged differs from contiguous"
    tol = TOL_FP8 if fp8 else TOL_BF16
    base = np.concatenate([[0], np.cumsum(ctx)])
    qn = np64(data["q"])
    for b, L in enumerate(ctx):
        if fp8:
            lat = oracle.e4m3_decode(data["kv_fp8"][base[b]:base[b] + L].cpu().numpy())
            K, V = oracle.mla_cache_to_kv(lat, data["kv_scale"][base[b]:base[b] + L].double().cpu().numpy())
        else:
            K, V = oracle.mla_cache_to_kv(np64(data["kv_bf16"][base[b]:base[b] + L]))
        po, pl = oracle.decode_shard_partials(qn[b], K, V, C, scale)
        for r in range(C):
            check_o(o_part[r, b], po[r], what=f"paged partial r{r} b{b}", **tol)
            check_lse(lse_part[r, b], pl[r])
        fo, fl = oracle.decode_attention(qn[b], K, V, scale)
        check_o(o[b], fo, what=f"paged merged b{b}", **tol)
        check_lse(lse[b], fl)


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("C,nw,page_size", [(8, 5, 64), (4, 0, 128), (1, 3, 192)])
def test_paged_decode_mla(cp, fp8, C, nw, page_size):
    ctx = [0, 1, 3, 129, 1000, 4097]
    data = W.mla_decode_inputs(ctx, H=64, seed=51 + C, device=DEV)
    mla_paged_case(cp, data, C, fp8, nw, page_size, seed=7 * C + page_size)


def test_paged_decode_gqa(cp):
    ctx = [0, 2, 300, 4100]
    C, Hq, Hkv, D = 4, 16, 4, 128
    q, k, v = W.gqa_decode_inputs(len(ctx), ctx, Hq, Hkv, D, "bf16", seed=61, device=DEV, std=0.3)
    scale = 1.0 / math.sqrt(D)
    plan = cp.cp_decode_plan(C, ctx, n_workers=7, device=DEV)
    pages = make_pages(cp, plan, 64, seed=62)
    kpool, _ = cp.cp_kv_shard_pack_paged(plan, pages, k)
    vpool, _ = cp.cp_kv_shard_pack_paged(plan, pages, v)
    o_part, lse_part = cp.cp_decode_attn_paged(plan, pages, cp.CP_DECODE_GQA, q, kpool, vpool,
                                               sm_scale=scale)
    ks, _ = cp.cp_kv_shard_pack(plan, k)
    vs, _ = cp.cp_kv_shard_pack(plan, v)
    o_c, lse_c = cp.cp_decode_attn(plan, cp.CP_DECODE_GQA, q, ks, vs, sm_scale=scale)
    cp.cp_device_error_check()
    assert torch.equal(o_part, o_c) and torch.equal(lse_part, lse_c), "paged differs from contiguous"
    base = np.concatenate([[0], np.cumsum(ctx)])
    qn, kn, vn = np64(q), np64(k), np64(v)
    for b, L in enumerate(ctx):
        Kb, Vb = kn[base[b]:base[b] + L], vn[base[b]:base[b] + L]
        po, pl = oracle.decode_shard_partials(qn[b], Kb, Vb, C, scale)
        for r in range(C):
            check_o(o_part[r, b], po[r], what=f"paged GQA partial r{r} b{b}", **TOL_BF16)
            check_lse(lse_part[r, b], pl[r])


def test_paged_decode_gqa_fp8(cp):
    """GQA over an E4M3 pool: scales read through the page table; the paged
    partials against the oracle, and within the FP8 bound of the per-shard
    ones (which take the tensor-core kernel)."""
    ctx = [0, 5, 300, 2100]
    C, Hq, Hkv, D = 4, 8, 2, 128
    q, kc, vc, sc = W.gqa_decode_inputs_fp8(len(ctx), ctx, Hq, Hkv, D, seed=63, device=DEV, std=0.3)
    scale = 1.0 / math.sqrt(D)
    plan = cp.cp_decode_plan(C, ctx, n_workers=5, device=DEV)
    pages = make_pages(cp, plan, 64, seed=64)
    kpool, spool = cp.cp_kv_shard_pack_paged(plan, pages, kc, sc)
    vpool, _ = cp.cp_kv_shard_pack_paged(plan, pages, vc)
    o_p, l_p = cp.cp_decode_attn_paged(plan, pages, cp.CP_DECODE_GQA, q, kpool, vpool, scale_pool=spool,
                                       sm_scale=scale)
    ks, ss = cp.cp_kv_shard_pack(plan, kc, sc)
    vs, _ = cp.cp_kv_shard_pack(plan, vc)
    o_c, l_c = cp.cp_decode_attn(plan, cp.CP_DECODE_GQA, q, ks, vs, shard_scale=ss, sm_scale=scale)
    cp.cp_device_error_check()
    assert (o_p - o_c).abs().max().item() <= 6e-2
    s64 = sc.double().cpu().numpy()[:, None, None]
    kn = oracle.e4m3_decode(kc.cpu().numpy()) * s64
    vn = oracle.e4m3_decode(vc.cpu().numpy()) * s64
    qn = np64(q)
    base = np.concatenate([[0], np.cumsum(ctx)])
    for b, L in enumerate(ctx):
        po, pl = oracle.decode_shard_partials(qn[b], kn[base[b]:base[b] + L], vn[base[b]:base[b] + L], C, scale)
        for r in range(C):
            check_o(o_p[r, b], po[r], what=f"paged FP8 GQA partial r{r} b{b}", **TOL_FP8)
            check_lse(l_p[r, b], pl[r])
