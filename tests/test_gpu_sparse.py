"""GPU parity of sparse decode with an exact sharded top-k ("DeepSeek-V4
Attention Inference Systems" §5.2): the selected token indices bit-exact
against the oracle's local-lists-then-merge (and brute force), the owners'
selection buffers bit-exact, and the sparse attention's partials and merged
result against the oracle."""

import math

import numpy as np
import pytest
import torch

import cp_workloads as W
import oracle
from test_gpu_parity import DEV, TOL_BF16, TOL_FP8, check_lse, check_o, cp, np64  # noqa: F401

pytestmark = pytest.mark.gpu


def token_map(L, C, contiguous):
    return (oracle.decode_shard_map_contiguous if contiguous else oracle.decode_shard_map)(L, C)


def shard_scores(scores, ctx, C, plan, contiguous):
    """Each shard's scores in its row order, placed by the oracle's map."""
    s = scores.cpu().numpy()
    base = np.concatenate([[0], np.cumsum(ctx)])
    maps = [np.asarray(token_map(L, C, contiguous)[0], dtype=np.int64) for L in ctx]
    out = []
    for r in range(C):
        rows = np.concatenate([base[b] + np.nonzero(m == r)[0] for b, m in enumerate(maps)]).astype(np.int64)
        out.append(torch.from_numpy(s[rows].copy()).to(DEV))
        assert out[-1].shape[0] == sum(int(plan.pairs[r * len(ctx) + b, 0]) for b in range(len(ctx)))
    return out


def oracle_selection(scores, ctx, C, k, contiguous):
    s = scores.cpu().numpy()
    base = np.concatenate([[0], np.cumsum(ctx)])
    return [oracle.sharded_topk(s[base[b]:base[b] + L], C, k, contiguous=contiguous)[0]
            for b, L in enumerate(ctx)]


@pytest.mark.parametrize("contiguous", [False, True])
@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("C,k", [(1, 7), (4, 1), (8, 64), (8, 512), (3, 2048), (4, 4096)])
def test_topk_bit_exact(cp, contiguous, ties, C, k):
    ctx = [0, 1, 5, 300, 4100, 20000]
    scores = W.index_scores(ctx, seed=C * 100 + k, device=DEV, ties=ties)
    plan = cp.cp_decode_plan_ex(C, ctx, layout=int(contiguous), n_workers=11, device=DEV)
    sel, cnt, _ = cp.cp_sparse_topk(plan, shard_scores(scores, ctx, C, plan, contiguous), k)
    cp.cp_device_error_check()
    sel, cnt = sel.cpu().numpy(), cnt.cpu().numpy()
    want = oracle_selection(scores, ctx, C, k, contiguous)
    s = scores.cpu().numpy()
    base = np.concatenate([[0], np.cumsum(ctx)])
    for b, L in enumerate(ctx):
        assert cnt[b] == min(k, L)
        assert sel[b, :cnt[b]].tolist() == want[b], f"request {b}"
        assert np.all(sel[b, cnt[b]:] == -1)
        if L <= 4100:  # brute force over the whole request
            sb = s[base[b]:base[b] + L]
            assert want[b] == sorted(sorted(range(L), key=lambda p: (-float(sb[p]), p))[:k])


@pytest.mark.parametrize("contiguous", [False, True])
@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("C,k", [(1, 100), (2, 3000), (8, 4096)])
def test_topk_unstaged(cp, contiguous, ties, C, k):
    """Pairs longer than the 32,768 scores a block stages, requests whose C k
    candidates pass the 16,384 the merge stages, and a context past the
    131,072 token indices the merge orders at a time: the same exact selection."""
    ctx = [200003, 70001, 40000, 33]
    scores = W.index_scores(ctx, seed=C * 7 + k, device=DEV, ties=ties)
    plan = cp.cp_decode_plan_ex(C, ctx, layout=int(contiguous), device=DEV)
    sel, cnt, _ = cp.cp_sparse_topk(plan, shard_scores(scores, ctx, C, plan, contiguous), k)
    cp.cp_device_error_check()
    sel, cnt = sel.cpu().numpy(), cnt.cpu().numpy()
    s = scores.cpu().numpy()
    base = np.concatenate([[0], np.cumsum(ctx)])
    for b, L in enumerate(ctx):
        sb = s[base[b]:base[b] + L]
        order = np.lexsort((np.arange(L), -sb.astype(np.float64)))
        assert cnt[b] == min(k, L)
        assert sel[b, :cnt[b]].tolist() == sorted(order[:k].tolist()), f"request {b}"
        assert np.all(sel[b, cnt[b]:] == -1)


@pytest.mark.parametrize("contiguous", [False, True])
@pytest.mark.parametrize("k", [1, 100, 700])
def test_topk_sixty_four_shards(cp, contiguous, k):
    """C = 64, the largest: the merge reads two shards' counts per lane."""
    ctx = [20000, 64, 0, 5001]
    C = 64
    scores = W.index_scores(ctx, seed=640 + k, device=DEV)
    plan = cp.cp_decode_plan_ex(C, ctx, layout=int(contiguous), device=DEV)
    sel, cnt, _ = cp.cp_sparse_topk(plan, shard_scores(scores, ctx, C, plan, contiguous), k)
    cp.cp_device_error_check()
    sel, cnt = sel.cpu().numpy(), cnt.cpu().numpy()
    s = scores.cpu().numpy()
    base = np.concatenate([[0], np.cumsum(ctx)])
    for b, L in enumerate(ctx):
        sb = s[base[b]:base[b] + L]
        order = np.lexsort((np.arange(L), -sb.astype(np.float64)))
        assert cnt[b] == min(k, L)
        assert sel[b, :cnt[b]].tolist() == sorted(order[:k].tolist()), f"request {b}"
        assert np.all(sel[b, cnt[b]:] == -1)


@pytest.mark.parametrize("contiguous", [False, True])
def test_topk_infinite_scores(cp, contiguous):
    """Masked tokens scored -inf (most of some requests, so the k-th key is
    -inf) and a few +inf: the order still counts them as numbers."""
    ctx = [9000, 30000, 5000]
    C, k = 4, 2048
    scores = W.index_scores(ctx, seed=99, device=DEV)
    g = torch.Generator(device="cpu").manual_seed(5)
    u = torch.rand(sum(ctx), generator=g)
    s = scores.cpu()
    base = 0
    for L, masked in zip(ctx, (0.9, 0.5, 0.7)):
        s[base:base + L][u[base:base + L] < masked] = -math.inf
        s[base:base + L][u[base:base + L] > 0.999] = math.inf
        base += L
    scores = s.to(DEV)
    plan = cp.cp_decode_plan_ex(C, ctx, layout=int(contiguous), device=DEV)
    sel, cnt, _ = cp.cp_sparse_topk(plan, shard_scores(scores, ctx, C, plan, contiguous), k)
    cp.cp_device_error_check()
    sel, cnt = sel.cpu().numpy(), cnt.cpu().numpy()
    want = oracle_selection(scores, ctx, C, k, contiguous)
    sn = scores.cpu().numpy()
    off = np.concatenate([[0], np.cumsum(ctx)])
    for b, L in enumerate(ctx):
        sb = sn[off[b]:off[b] + L]
        order = np.lexsort((np.arange(L), -sb.astype(np.float64)))
        assert want[b] == sorted(order[:k].tolist())
        assert cnt[b] == min(k, L)
        assert sel[b, :cnt[b]].tolist() == want[b], f"request {b}"


def test_topk_full_size_sampled(cp):
    """64 requests x 131,072 tokens, C = 8, k = 2048: sampled requests exact."""
    ctx = [131072] * 64
    C, k = 8, 2048
    scores = W.index_scores(ctx, device=DEV)
    plan = cp.cp_decode_plan_ex(C, ctx, device=DEV)
    # round robin: shard r's rows of request b are tokens r, r + C, ...
    st = scores.view(64, 131072 // C, C)
    shards = [st[:, :, r].contiguous().view(-1) for r in range(C)]
    sel, cnt, _ = cp.cp_sparse_topk(plan, shards, k)
    cp.cp_device_error_check()
    sel = sel.cpu().numpy()
    s = scores.cpu().numpy()
    for b in (0, 17, 63):
        sb = s[b * 131072:(b + 1) * 131072]
        order = np.lexsort((np.arange(131072), -sb.astype(np.float64)))
        assert sel[b].tolist() == sorted(order[:k].tolist())
    assert np.all(cnt.cpu().numpy() == k)


def run_sparse(cp, kind, ctx, C, k, contiguous, seed):
    B = len(ctx)
    plan = cp.cp_decode_plan_ex(C, ctx, layout=int(contiguous), n_workers=9, device=DEV)
    scores = W.index_scores(ctx, seed=seed, device=DEV)
    sel, cnt, ws = cp.cp_sparse_topk(plan, shard_scores(scores, ctx, C, plan, contiguous), k)
    splan = cp.cp_sparse_plan(C, B, k, n_workers=7, device=DEV)
    if kind == "gqa":
        q, kc, vc = W.gqa_decode_inputs(B, ctx, 16, 4, 128, "bf16", seed=seed, device=DEV, std=0.3)
        sk, _ = cp.cp_kv_shard_pack(plan, kc)
        sv, _ = cp.cp_kv_shard_pack(plan, vc)
        selk, _, pc = cp.cp_sparse_gather(plan, k, ws, sk)
        selv, _, pc2 = cp.cp_sparse_gather(plan, k, ws, sv)
        assert torch.equal(pc, pc2)
        o_part, lse_part = cp.cp_sparse_decode_attn(splan, pc, cp.CP_DECODE_GQA, q, selk, selv,
                                                    sm_scale=1.0 / math.sqrt(128))
        merged = cp.cp_sparse_decode_attn_merged(splan, pc, cp.CP_DECODE_GQA, q, selk, selv,
                                                 sm_scale=1.0 / math.sqrt(128), out_dtype=torch.float32)
        data = {"q": q, "k": kc, "v": vc}
        shards, selb = sk, selk
    else:
        fp8 = kind == "fp8"
        data = W.mla_decode_inputs(ctx, H=64, seed=seed, device=DEV, fp8=fp8, bf16=not fp8)
        kv, ksc = (data["kv_fp8"], data["kv_scale"]) if fp8 else (data["kv_bf16"], None)
        shards, shsc = cp.cp_kv_shard_pack(plan, kv, ksc)
        selb, selsc, pc = cp.cp_sparse_gather(plan, k, ws, shards, shsc)
        o_part, lse_part = cp.cp_sparse_decode_attn(splan, pc, cp.CP_DECODE_MLA, data["q"], selb,
                                                    sel_scale=selsc, sm_scale=1.0 / math.sqrt(576))
        merged = cp.cp_sparse_decode_attn_merged(splan, pc, cp.CP_DECODE_MLA, data["q"], selb, sel_scale=selsc,
                                                 sm_scale=1.0 / math.sqrt(576), out_dtype=torch.float32)
    o, lse = cp.cp_lse_merge(o_part, lse_part, out_dtype=torch.float32)
    cp.cp_device_error_check()
    data["merged"] = merged  # cp_sparse_decode_attn_merged's (O, LSE)
    return plan, scores, sel, cnt, pc, shards, selb, data, o_part, lse_part, o, lse


@pytest.mark.parametrize("contiguous", [False, True])
def test_gather_bit_exact(cp, contiguous):
    ctx = [3, 70, 1000, 4100]
    C, k = 4, 300
    plan, scores, sel, cnt, pc, shards, selb, _, _, _, _, _ = run_sparse(cp, "fp8", ctx, C, k, contiguous, 5)
    want = oracle_selection(scores, ctx, C, k, contiguous)
    pcn = pc.cpu().numpy()
    for b, L in enumerate(ctx):
        shard, row = token_map(L, C, contiguous)
        off = [int(plan.pairs[r * len(ctx) + b, 1]) for r in range(C)]
        for r in range(C):
            mine = [p for p in want[b] if shard[p] == r]  # in token order
            assert pcn[r * len(ctx) + b] == len(mine)
            kp = cp.sparse_slot_rows(k)
            got = selb[r][b * kp:b * kp + len(mine)].cpu()
            pad = selb[r][b * kp + len(mine):b * kp + min(kp, -(-len(mine) // 128) * 128)].cpu()
            assert not pad.any()  # zeros up to the tile boundary
            src = shards[r][[off[r] + row[p] for p in mine]].cpu() if mine else got
            assert torch.equal(got, src)


@pytest.mark.parametrize("kind", ["fp8", "bf16", "gqa"])
@pytest.mark.parametrize("contiguous", [False, True])
def test_sparse_decode(cp, kind, contiguous):
    ctx = [1, 9, 500, 4100, 9000]
    C, k = 8, 512
    plan, scores, sel, cnt, pc, _, _, data, o_part, lse_part, o, lse = run_sparse(
        cp, kind, ctx, C, k, contiguous, 21)
    want = oracle_selection(scores, ctx, C, k, contiguous)
    assert [sel[b, :cnt[b]].tolist() for b in range(len(ctx))] == want
    base = np.concatenate([[0], np.cumsum(ctx)])
    for b, L in enumerate(ctx):
        if kind == "gqa":
            qn = np64(data["q"][b])
            K, V = np64(data["k"][base[b]:base[b] + L]), np64(data["v"][base[b]:base[b] + L])
            scale, tol = 1.0 / math.sqrt(128), TOL_BF16
        else:
            qn = np64(data["q"][b])
            if kind == "fp8":
                lat = oracle.e4m3_decode(data["kv_fp8"][base[b]:base[b] + L].cpu().numpy())
                K, V = oracle.mla_cache_to_kv(lat, data["kv_scale"][base[b]:base[b] + L].double().cpu().numpy())
                tol = TOL_FP8
            else:
                K, V = oracle.mla_cache_to_kv(np64(data["kv_bf16"][base[b]:base[b] + L]))
                tol = TOL_BF16
            scale = 1.0 / math.sqrt(576)
        po, pl = oracle.sparse_partials(qn, K, V, want[b], C, scale, contiguous=contiguous)
        for r in range(C):
            check_o(o_part[r, b], po[r], what=f"{kind} partial r{r} b{b}", **tol)
            check_lse(lse_part[r, b], pl[r])
        fo, fl = oracle.decode_attention(qn, K, V, scale, keys=np.asarray(want[b], dtype=np.int64))
        check_o(o[b], fo, what=f"{kind} merged b{b}", **tol)
        check_lse(lse[b], fl)
        om, lm = data["merged"]  # decode and merge in one call
        check_o(om[b], fo, what=f"{kind} one-call merged b{b}", **tol)
        check_lse(lm[b], fl)
    if kind == "gqa":  # the same kernels as decode + merge: the same bits
        assert torch.equal(data["merged"][0], o) and torch.equal(data["merged"][1], lse)


def test_sparse_decode_full_size_sampled(cp):
    """64 x 131,072 tokens, C = 8, k = 2048, FP8: sampled requests' merged
    sparse attention against the oracle over the oracle's selection."""
    B, L, C, k = 64, 131072, 8, 2048
    ctx = [L] * B
    plan = cp.cp_decode_plan_ex(C, ctx, device=DEV)
    scores = W.index_scores(ctx, seed=77, device=DEV)
    st = scores.view(B, L // C, C)
    shards_s = [st[:, :, r].contiguous().view(-1) for r in range(C)]
    sel, cnt, ws = cp.cp_sparse_topk(plan, shards_s, k)
    data = W.mla_decode_inputs(ctx, H=64, seed=78, device=DEV, bf16=False)
    sh, sc = cp.cp_kv_shard_pack(plan, data["kv_fp8"], data["kv_scale"])
    selk, selsc, pc = cp.cp_sparse_gather(plan, k, ws, sh, sc)
    splan = cp.cp_sparse_plan(C, B, k, device=DEV)
    scale = 1.0 / math.sqrt(576)
    o_part, lse_part = cp.cp_sparse_decode_attn(splan, pc, cp.CP_DECODE_MLA, data["q"], selk,
                                                sel_scale=selsc, sm_scale=scale)
    o, lse = cp.cp_lse_merge(o_part, lse_part, out_dtype=torch.float32)
    cp.cp_device_error_check()
    s = scores.cpu().numpy()
    for b in (3, 60):
        sb = s[b * L:(b + 1) * L]
        want = sorted(np.lexsort((np.arange(L), -sb.astype(np.float64)))[:k].tolist())
        assert sel[b].tolist() == want
        lat = oracle.e4m3_decode(data["kv_fp8"][b * L:(b + 1) * L].cpu().numpy())
        K, V = oracle.mla_cache_to_kv(lat, data["kv_scale"][b * L:(b + 1) * L].double().cpu().numpy())
        fo, fl = oracle.decode_attention(np64(data["q"][b]), K, V, scale, keys=np.asarray(want))
        check_o(o[b], fo, what=f"full-size sparse b{b}", **TOL_FP8)
        check_lse(lse[b], fl)
