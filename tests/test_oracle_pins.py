"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Nothing here touches a GPU.  Each test checks the oracle against something
other than itself: a value the pages print (fixtures in tests/golden/, each
with its citation), a closed form, an invariant, a library routine
(torch scaled_dot_product_attention / logsumexp / float8 casts in fp64), or
brute force on tiny inputs.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ maps


def test_zigzag_cp4_16_tokens_matches_page():
    g = golden("zigzag_cp4_16tokens.json")
    plan = oracle.zigzag_plan(g["new_len"], g["prefix_len"], g["C"])
    assert [sorted(o) for o in plan["order"]] == g["rank_tokens"]
    for b, e in oracle.zigzag_block_bounds(16, 4):
        assert e - b == g["tokens_per_block"]


def test_interleave_cp4_16_tokens_matches_page():
    g = golden("interleave_cp4_16tokens.json")
    plan = oracle.interleave_plan(g["new_len"], g["prefix_len"], g["C"])
    assert plan["order"] == g["rank_tokens"]


def test_interleave_batch_5_3_matches_page():
    g = golden("interleave_batch_5_3.json")
    plan = oracle.interleave_plan(g["new_len"], g["prefix_len"], g["C"])
    p = g["printed"]
    assert plan["order"][0] == p["rank0"]
    assert plan["order"][1] == p["rank1"]
    i5 = plan["order"][1].index(5)
    assert plan["req"][1][i5] == p["index5_request"]
    assert plan["pos"][1][i5] == p["index5_offset_in_request"]
    # the index does not reset at the request boundary
    assert plan["order"][2] == [2, 6] and plan["order"][3] == [3, 7]
    # positions keep their original values within each request
    assert plan["pos"][2] == [2, 1] and plan["req"][2] == [0, 1]


def test_consecutive_split_pairs_match_page():
    g = golden("consecutive_split_pairs_16tokens_4gpus.json")
    pairs = oracle.consecutive_split_pairs(g["n"], g["C"])
    assert pairs[0] == g["gpu0_pairs"] and pairs[-1] == g["gpu3_pairs"]
    assert pairs == [10, 26, 42, 58]
    # the long-prompt limit of last/first is 2C-1
    big = oracle.consecutive_split_pairs(4 * 4096, 4)
    assert abs(big[-1] / big[0] - g["ratio_formula_long_prompt"]) < 0.01


def brute_pairs(owner_of_token, C):
    """Pairs per rank by brute force: count (q, k) with k <= q."""
    out = [0] * C
    for qpos, r in enumerate(owner_of_token):
        for k in range(qpos + 1):
            out[r] += 1
    return out


def test_pair_counts_16_tokens_cp4_brute_force():
    zz = oracle.zigzag_plan([16], [0], 4)
    il = oracle.interleave_plan([16], [0], 4)
    for plan in (zz, il):
        owner = [None] * 16
        for r in range(4):
            for f in plan["order"][r]:
                owner[f] = r
        assert oracle.pairs_per_rank(plan) == brute_pairs(owner, 4)
    # zigzag balances exactly, interleave nearly
    assert oracle.pairs_per_rank(zz) == [34, 34, 34, 34]
    assert oracle.pairs_per_rank(il) == [28, 32, 36, 40]


def test_zigzag_block_units_equal_2C():
    # block b reads the b blocks before it plus half of itself: b + 1/2 units;
    # in units of (block queries x block keys) the exact pair count of block b
    # with blocks of size s is s*s*b + s*(s+1)/2.
    g = golden("long_prompt_counts.json")
    for C in (2, 4, 8):
        s = 1024
        plan = oracle.zigzag_plan([2 * C * s], [0], C)
        pairs = oracle.pairs_per_rank(plan)
        assert len(set(pairs)) == 1
        units = pairs[0] / (s * s)
        assert abs(units - 2 * C) < 2.0 / s
    assert g["zigzag_units_C4"] == 2 * 4


def test_long_prompt_closed_forms():
    g = golden("long_prompt_counts.json")
    n = g["n"]
    # about N^2/2 pairs for the whole prompt
    total = n * (n + 1) // 2
    assert round(total / 1e9, 1) == g["pairs_billion_rounded"]
    il = oracle.interleave_plan_np([n], [0], g["interleave_C"])
    pairs = [int((p + 1).sum()) for p in il["pos"]]
    assert sum(pairs) == total
    excess = (max(pairs) - total / g["interleave_C"]) / (total / g["interleave_C"]) * 100
    assert 0.005 < excess < 0.02  # "about 0.01%"


def test_maps_are_partitions_with_prefix_and_ragged_batch():
    rng = np.random.default_rng(0)
    for C in (1, 2, 3, 4, 8):
        new = [int(x) for x in rng.integers(0, 40, size=5)]
        pre = [int(x) for x in rng.integers(0, 30, size=5)]
        T = sum(new)
        for plan in (oracle.zigzag_plan(new, pre, C), oracle.interleave_plan(new, pre, C)):
            allf = sorted(f for r in range(C) for f in plan["order"][r])
            assert allf == list(range(T))
            # every query's position is prefix + its offset in its request
            starts = np.concatenate([[0], np.cumsum(new)[:-1]])
            for r in range(C):
                for f, j, p in zip(plan["order"][r], plan["req"][r], plan["pos"][r]):
                    assert starts[j] <= f < starts[j] + new[j]
                    assert p == pre[j] + (f - starts[j])


def test_zigzag_remainder_and_kv_lengths():
    # 19 tokens, C=4: 8 blocks of 2, the first 3 blocks get one more
    b = oracle.zigzag_block_bounds(19, 4)
    assert [e - s for s, e in b] == [3, 3, 3, 2, 2, 2, 2, 2]
    plan = oracle.zigzag_plan([19], [7], 4)
    for (r, j, which, blk, qs, ql, kvl) in plan["blocks"]:
        assert blk == (r if which == 0 else 7 - r)
        assert (qs, qs + ql) == b[blk]
        assert kvl == 7 + b[blk][1]  # reads end where the block ends, prefix included
    # fewer tokens than blocks: some blocks are empty
    b = oracle.zigzag_block_bounds(3, 4)
    assert [e - s for s, e in b] == [1, 1, 1, 0, 0, 0, 0, 0]


def test_interleave_np_matches_loop():
    rng = np.random.default_rng(1)
    for C in (1, 3, 8):
        new = [int(x) for x in rng.integers(1, 50, size=6)]
        pre = [int(x) for x in rng.integers(0, 20, size=6)]
        a = oracle.interleave_plan(new, pre, C)
        b = oracle.interleave_plan_np(new, pre, C)
        for r in range(C):
            assert list(a["order"][r]) == list(b["order"][r])
            assert list(a["req"][r]) == list(b["req"][r])
            assert list(a["pos"][r]) == list(b["pos"][r])


def test_decode_slot_map_matches_page():
    g = golden("decode_slot9_4gpus.json")
    shard, row = oracle.decode_shard_map(g["slot"] + 1, g["C"])
    assert shard[g["slot"]] == g["gpu"] and row[g["slot"]] == g["row"]
    # shards partition the tokens; shard r holds ceil((L - r)/C) rows
    for L in (0, 1, 5, 257):
        for C in (1, 4, 8):
            shard, row = oracle.decode_shard_map(L, C)
            for r in range(C):
                rows = [row[p] for p in range(L) if shard[p] == r]
                assert rows == list(range(len(rows)))
                assert len(rows) == max(0, -(-(L - r) // C))


# ------------------------------------------------------------------ fp8


def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = oracle.e4m3_decode(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ref[~nan], ours[~nan])
    assert oracle.e4m3_to_float(0x7E) == 448.0
    assert oracle.e4m3_to_float(0x01) == 2.0 ** -9


# ------------------------------------------------------------------ attention


def sdpa_causal_ref(q, k, v, pos, scale):
    """torch SDPA in fp64 with a boolean mask: key j readable iff j <= pos."""
    n, Hq, D = q.shape
    L, Hkv, _ = k.shape
    g = Hq // Hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)  # [Hq, n, D]
    kt = torch.from_numpy(k).repeat_interleave(g, dim=1).permute(1, 0, 2)
    vt = torch.from_numpy(v).repeat_interleave(g, dim=1).permute(1, 0, 2)
    mask = torch.arange(L)[None, :] <= torch.from_numpy(np.asarray(pos))[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    s = (qt @ kt.transpose(1, 2)) * scale
    s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


@pytest.mark.parametrize("Hq,Hkv,D,n,pre", [(4, 1, 8, 13, 0), (8, 2, 16, 11, 5), (6, 3, 4, 1, 0)])
def test_causal_rows_vs_torch_sdpa(Hq, Hkv, D, n, pre):
    rng = np.random.default_rng(Hq * 100 + n)
    L = pre + n
    q = rng.standard_normal((n, Hq, D))
    k = rng.standard_normal((L, Hkv, D))
    v = rng.standard_normal((L, Hkv, D))
    pos = np.arange(pre, pre + n)
    scale = 1 / math.sqrt(D)
    o, lse = oracle.causal_rows(q, k, v, pos, scale)
    o_ref, lse_ref = sdpa_causal_ref(q, k, v, pos, scale)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
@pytest.mark.parametrize("C", [1, 3, 4])
def test_prefill_reference_rank_order_vs_sdpa(strategy, C):
    """prefill_reference's rows, rank by rank in local order, against torch
    SDPA over each whole request (its prefix included): local row i of rank r
    is flattened new token f = order[r][i], whose request and position follow
    from the request lengths alone."""
    rng = np.random.default_rng(C * 7 + len(strategy))
    nl, pl = [37, 20, 1], [5, 0, 3]
    Hq, Hkv, D = 4, 2, 8
    T = sum(nl)
    q = rng.standard_normal((T, Hq, D))
    k = rng.standard_normal((sum(nl) + sum(pl), Hkv, D))
    v = rng.standard_normal((sum(nl) + sum(pl), Hkv, D))
    scale = 1 / math.sqrt(D)
    plan = oracle.zigzag_plan(nl, pl, C) if strategy == "zigzag" else oracle.interleave_plan_np(nl, pl, C)
    ref = oracle.prefill_reference(plan, nl, pl, q, k, v, scale)
    # whole-request SDPA, indexed by flattened new token
    want_o, want_l = np.zeros((T, Hq, D)), np.zeros((T, Hq))
    f0, kv0 = 0, 0
    for n, p_ in zip(nl, pl):
        pos = np.arange(p_, p_ + n)
        o_, l_ = sdpa_causal_ref(q[f0:f0 + n], k[kv0:kv0 + p_ + n], v[kv0:kv0 + p_ + n], pos, scale)
        want_o[f0:f0 + n], want_l[f0:f0 + n] = o_, l_
        f0 += n
        kv0 += p_ + n
    seen = []
    for r in range(C):
        local, o, lse = ref[r]
        f = np.asarray(plan["order"][r], dtype=np.int64)[local]
        np.testing.assert_allclose(o, want_o[f], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, want_l[f], rtol=1e-12, atol=1e-12)
        seen.extend(f.tolist())
    assert sorted(seen) == list(range(T))


def test_causal_rows_brute_force_python():
    """Pure-Python probability table on a tiny case (no numpy algebra)."""
    rng = np.random.default_rng(7)
    n, Hq, Hkv, D = 5, 2, 1, 3
    q = rng.standard_normal((n, Hq, D))
    k = rng.standard_normal((n, Hkv, D))
    v = rng.standard_normal((n, Hkv, D))
    o, lse = oracle.causal_rows(q, k, v, np.arange(n), 0.7)
    for i in range(n):
        for h in range(Hq):
            w = [math.exp(0.7 * sum(q[i, h, d] * k[j, 0, d] for d in range(D))) for j in range(i + 1)]
            Z = sum(w)
            for d in range(D):
                assert abs(o[i, h, d] - sum(w[j] * v[j, 0, d] for j in range(i + 1)) / Z) < 1e-12
            assert abs(lse[i, h] - math.log(Z)) < 1e-12


def test_single_key_and_identical_keys():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 2, 4))
    k = rng.standard_normal((1, 1, 4))
    v = rng.standard_normal((1, 1, 4))
    o, lse = oracle.causal_rows(q, k, v, [0], 0.5)
    for h in range(2):
        np.testing.assert_allclose(o[0, h], v[0, 0], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[0, h], 0.5 * q[0, h] @ k[0, 0], rtol=0, atol=1e-14)
    # n identical keys: O = mean(v), LSE = s + ln n
    n = 9
    k = np.repeat(k, n, axis=0)
    v = rng.standard_normal((n, 1, 4))
    o, lse = oracle.decode_attention(q[0], k, v, 0.5)
    for h in range(2):
        np.testing.assert_allclose(o[h], v[:, 0].mean(axis=0), atol=1e-14)
        np.testing.assert_allclose(lse[h], 0.5 * q[0, h] @ k[0, 0] + math.log(n), atol=1e-13)


def test_decode_attention_vs_torch_and_gqa_mapping():
    rng = np.random.default_rng(11)
    H, Hkv, D, L = 8, 2, 6, 37
    q = rng.standard_normal((H, D))
    k = rng.standard_normal((L, Hkv, D))
    v = rng.standard_normal((L, Hkv, D + 2))
    o, lse = oracle.decode_attention(q, k, v, 0.3)
    for h in range(H):
        kh = h // (H // Hkv)  # consecutive grouping
        s = torch.from_numpy(0.3 * (k[:, kh] @ q[h]))
        ref_lse = torch.logsumexp(s, 0).item()
        ref_o = (torch.softmax(s, 0) @ torch.from_numpy(v[:, kh])).numpy()
        assert abs(lse[h] - ref_lse) < 1e-12
        np.testing.assert_allclose(o[h], ref_o, atol=1e-12)
    # empty key set
    o, lse = oracle.decode_attention(q, k[:0], v[:0], 0.3)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_mla_cache_split():
    rng = np.random.default_rng(5)
    lat = rng.standard_normal((7, 576))
    sc = rng.random(7) + 0.5
    K, V = oracle.mla_cache_to_kv(lat, sc)
    assert K.shape == (7, 1, 576) and V.shape == (7, 1, 512)
    np.testing.assert_array_equal(K[:, 0, :512], V[:, 0])
    np.testing.assert_allclose(K[:, 0, 575], lat[:, 575] * sc)


# ------------------------------------------------------------------ merge


def test_figure8_merge_values():
    g = golden("figure8_merge.json")
    e = np.array(g["exp_scores"], dtype=np.float64)
    s = np.log(e)[None, :]  # scores whose exponentials are 4, 2, 1, 1
    v = np.eye(4)  # value j = unit vector j, so O = probabilities
    o, lse = oracle.softmax_attention(s, v)
    np.testing.assert_allclose(o[0], g["global_probs"], atol=1e-15)
    parts_o, parts_lse = [], []
    for toks, lp, ls in zip(g["gpu_tokens"], g["local_probs"], g["local_sums"]):
        op, lsep = oracle.softmax_attention(s[:, toks], v[toks])
        np.testing.assert_allclose(op[0][toks], lp, atol=1e-15)
        assert abs(lsep[0] - math.log(ls)) < 1e-15
        parts_o.append(op)
        parts_lse.append(lsep)
    o_m, lse_m = oracle.lse_merge(np.stack(parts_o), np.stack(parts_lse))
    np.testing.assert_allclose(o_m[0], g["global_probs"], atol=1e-15)
    assert abs(lse_m[0] - math.log(8)) < 1e-15
    # the scale of each GPU is exp(LSE_p - global LSE)
    for lsep, sc in zip(parts_lse, g["scales"]):
        assert abs(math.exp(lsep[0] - lse_m[0]) - sc) < 1e-15


def test_merge_over_every_two_way_partition_equals_unsharded():
    rng = np.random.default_rng(21)
    n, H, Dv = 10, 3, 5
    q = rng.standard_normal((H, 4)) * 2
    k = rng.standard_normal((n, 1, 4))
    v = rng.standard_normal((n, 1, Dv))
    o_full, lse_full = oracle.decode_attention(q, k, v, 1.0)
    for bits in itertools.product([0, 1], repeat=n):
        sel = np.array(bits, dtype=bool)
        parts = [oracle.decode_attention(q, k, v, 1.0, keys=np.nonzero(sel == b)[0]) for b in (0, 1)]
        o, lse = oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        np.testing.assert_allclose(o, o_full, atol=1e-13)
        np.testing.assert_allclose(lse, lse_full, atol=1e-13)


def test_merge_random_multiway_partitions_and_shards():
    rng = np.random.default_rng(22)
    for trial in range(20):
        L = int(rng.integers(1, 60))
        P = int(rng.integers(1, 9))
        q = rng.standard_normal((4, 8)) * 3
        k = rng.standard_normal((L, 2, 8))
        v = rng.standard_normal((L, 2, 7))
        o_full, lse_full = oracle.decode_attention(q, k, v, 0.5)
        owner = rng.integers(0, P, size=L)
        parts = [oracle.decode_attention(q, k, v, 0.5, keys=np.nonzero(owner == p)[0]) for p in range(P)]
        o, lse = oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        np.testing.assert_allclose(o, o_full, atol=1e-12)
        np.testing.assert_allclose(lse, lse_full, atol=1e-12)
        # the token-sharded partials (p mod C) merge to the same result
        po, pl = oracle.decode_shard_partials(q, k, v, P, 0.5)
        o2, l2 = oracle.lse_merge(po, pl)
        np.testing.assert_allclose(o2, o_full, atol=1e-12)
        np.testing.assert_allclose(l2, lse_full, atol=1e-12)


def test_merge_all_empty_and_vs_torch_logsumexp():
    o, lse = oracle.lse_merge(np.zeros((3, 2, 4)), np.full((3, 2), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    rng = np.random.default_rng(2)
    lp = rng.standard_normal((5, 6)) * 10
    lp[2, 3] = -np.inf
    op = rng.standard_normal((5, 6, 3))
    o, lse = oracle.lse_merge(op, lp)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.from_numpy(lp), dim=0).numpy(), atol=1e-12)


# ------------------------------------------------------------------ planted mistakes


def test_planted_mistakes_are_caught(monkeypatch):
    """Plant plausible mistakes in copies of oracle steps and check that the
    pins above would catch each of them."""
    g = golden("zigzag_cp4_16tokens.json")

    def wrong_pairing(new_len, prefix_len, C):  # rank r takes r and 2C-2-r
        out = [[] for _ in range(C)]
        bounds = oracle.zigzag_block_bounds(new_len[0], C)
        for r in range(C):
            for b in (r, (2 * C - 2 - r) % (2 * C)):
                out[r] += list(range(*bounds[b]))
        return out

    assert [sorted(o) for o in wrong_pairing([16], [0], 4)] != g["rank_tokens"]

    # a merge that drops the max shift overflows / a merge without weights is wrong
    f8 = golden("figure8_merge.json")
    s = np.log(np.array(f8["exp_scores"], float))[None, :]
    v = np.eye(4)
    parts = [oracle.softmax_attention(s[:, t], v[t]) for t in f8["gpu_tokens"]]
    naive = sum(p[0] for p in parts)  # "just add the results"
    assert not np.allclose(naive[0], f8["global_probs"])
    # a transposed operand in the scores is caught by the SDPA pin
    rng = np.random.default_rng(0)
    q = rng.standard_normal((6, 2, 6))
    k = rng.standard_normal((6, 1, 6))
    vv = rng.standard_normal((6, 1, 6))
    o_ref, _ = sdpa_causal_ref(q, k, vv, np.arange(6), 0.5)
    qT = np.ascontiguousarray(np.transpose(q, (2, 1, 0)))
    o_bad, _ = oracle.causal_rows(qT, k, vv, np.arange(6), 0.5)
    assert not np.allclose(o_bad, o_ref)
    # an off-by-one causal extent (reading keys < pos only) is caught
    with monkeypatch.context() as m:
        orig = oracle.causal_rows

        def shifted(q, k, v, pos, sc):
            return orig(q, k, v, np.maximum(np.asarray(pos) - 1, 0), sc)

        m.setattr(oracle, "causal_rows", shifted)
        o_bad, _ = oracle.causal_rows(q, k, vv, np.arange(6), 0.5)
        assert not np.allclose(o_bad, o_ref)


# ---------------------------------------------------------------- paged shard rows

def test_paged_rows_hand_example():
    """C = 2, one request of 5 tokens, pages of 2 rows.  Shard 0 holds tokens
    0, 2, 4 (rows 0, 1, 2) on pages [3, 1]; shard 1 holds tokens 1, 3 (rows
    0, 1) on page [0].  Pool row = page * 2 + row % 2:
    token 0 -> page 3 row 0 = 6, token 2 -> page 3 row 1 = 7,
    token 4 -> page 1 row 0 = 2, token 1 -> page 0 row 0 = 0,
    token 3 -> page 0 row 1 = 1."""
    got = oracle.paged_token_rows([5], 2, [[3, 1], [0, 0]], 2)
    assert got == [(0, 0, 6), (0, 1, 0), (0, 2, 7), (0, 3, 1), (0, 4, 2)]


def test_paged_rows_partition_and_contiguous_limit():
    rng = np.random.default_rng(5)
    ctx, C, ps = [0, 1, 77, 300, 129], 4, 8
    B = len(ctx)
    need = [[-(-len(range(r, L, C)) // ps) for L in ctx] for r in range(C)]
    maxp = max(max(n) for n in need)
    ids = rng.permutation(sum(sum(n) for n in need))
    table = np.full((C * B, maxp), -1)
    k = 0
    for r in range(C):
        for b in range(B):
            for i in range(need[r][b]):
                table[r * B + b, i] = ids[k]
                k += 1
    rows = oracle.paged_token_rows(ctx, C, table, ps)
    assert sorted((b, p) for b, p, _ in rows) == [(b, p) for b, L in enumerate(ctx) for p in range(L)]
    assert len({x for _, _, x in rows}) == len(rows)  # distinct pages -> distinct pool rows
    # one shard, one page as large as the request, page 0: the pool row is the token
    assert [x for _, _, x in oracle.paged_token_rows([40], 1, [[0]], 64)] == list(range(40))


def test_paged_rows_pin_catches_swapped_row_and_shard():
    """A planted mistake (shard p // C, row p mod C) moves tokens."""
    def wrong(ctx_len, C, table, ps):
        out = []
        for b, L in enumerate(ctx_len):
            for p in range(L):
                pair, i = (p // C) * len(ctx_len) + b, p % C
                out.append((b, p, int(table[pair][i // ps]) * ps + i % ps))
        return out
    assert wrong([5], 2, [[3, 1], [0, 0], [2, 2]], 2) != [(0, 0, 6), (0, 1, 0), (0, 2, 7), (0, 3, 1), (0, 4, 2)]


# ---------------------------------------------------------------- replicated window, designated rank

def _window_case(L=37, W=9, H=4, Hkv=2, D=16, seed=11):
    rng = np.random.default_rng(seed)
    q = rng.normal(size=(H, D))
    km, vm = rng.normal(size=(L, Hkv, D)), rng.normal(size=(L, Hkv, D))
    kw, vw = rng.normal(size=(W, Hkv, D)), rng.normal(size=(W, Hkv, D))
    return q, km, vm, kw, vw


def test_designated_window_counted_once():
    """[V4] §5.3: the window's mass is counted once, so the exact combine of
    the shards' partials is the attention over main cache + window."""
    q, km, vm, kw, vw = _window_case()
    scale = 0.3
    for C, d in [(1, 0), (4, 0), (4, 3), (5, 2)]:
        po, pl = oracle.designated_partials(q, km, vm, kw, vw, C, d, scale)
        o, lse = oracle.lse_merge(po, pl)
        fo, fl = oracle.decode_attention(q, np.concatenate([km, kw]), np.concatenate([vm, vw]), scale)
        assert np.allclose(o, fo, atol=1e-12) and np.allclose(lse, fl, atol=1e-12)
        # the other shards hold main-cache tokens only
        so, sl = oracle.decode_shard_partials(q, km, vm, C, scale)
        for r in range(C):
            if r != d:
                assert np.allclose(po[r], so[r]) and np.allclose(pl[r], sl[r])


def test_designated_window_pin_catches_double_count():
    """A planted mistake: every shard counts its copy of the window."""
    q, km, vm, kw, vw = _window_case()
    C, scale = 4, 0.3
    parts = [oracle.designated_partials(q, km, vm, kw, vw, C, r, scale) for r in range(C)]
    wrong_o = np.stack([parts[r][0][r] for r in range(C)])
    wrong_l = np.stack([parts[r][1][r] for r in range(C)])
    o, lse = oracle.lse_merge(wrong_o, wrong_l)
    fo, fl = oracle.decode_attention(q, np.concatenate([km, kw]), np.concatenate([vm, vw]), scale)
    assert not np.allclose(lse, fl, atol=1e-6)


def test_designated_window_empty_main_cache():
    q, km, vm, kw, vw = _window_case(L=0)
    po, pl = oracle.designated_partials(q, km, vm, kw, vw, 3, 1, 0.5)
    wo, wl = oracle.decode_attention(q, kw, vw, 0.5)
    assert np.allclose(po[1], wo) and np.allclose(pl[1], wl)
    assert np.isneginf(pl[0]).all() and np.isneginf(pl[2]).all() and not po[0].any()


# ------------------------------------------------------------------ contiguous DCP and query rows


def test_contiguous_map_dcp_example():
    """vLLM DCP post §4: a 200K-token request on four GPUs, each holding one
    50K range of positions (0-50K on GPU 0, 50K-100K on GPU 1, ...)."""
    shard, row = oracle.decode_shard_map_contiguous(200_000, 4)
    for r in range(4):
        lo, hi = 50_000 * r, 50_000 * (r + 1)
        assert shard[lo] == r and row[lo] == 0
        assert shard[hi - 1] == r and row[hi - 1] == 49_999
    assert np.bincount(shard).tolist() == [50_000] * 4


def test_contiguous_map_remainder_and_partition():
    """Reading: the first L mod C chunks hold one token more; every token is
    stored once and each shard's rows are 0, 1, ... in token order."""
    shard, row = oracle.decode_shard_map_contiguous(10, 4)
    assert shard == [0, 0, 0, 1, 1, 1, 2, 2, 3, 3]
    assert row == [0, 1, 2, 0, 1, 2, 0, 1, 0, 1]
    for L, C in [(0, 3), (1, 4), (7, 8), (129, 8), (1000, 7)]:
        shard, row = oracle.decode_shard_map_contiguous(L, C)
        counts = np.bincount(shard, minlength=C) if L else np.zeros(C, int)
        assert counts.max() - counts.min() <= 1
        assert all(shard[p] <= shard[p + 1] for p in range(L - 1))
        for r in range(C):
            assert [row[p] for p in range(L) if shard[p] == r] == list(range(counts[r]))


def _rows_case(L=11, s_q=3, H=4, D=16, seed=5):
    g = np.random.default_rng(seed)
    q_all = g.standard_normal((L, H, D))
    k = g.standard_normal((L, 1, D))
    v = g.standard_normal((L, 1, D))
    return q_all, k, v


@pytest.mark.parametrize("contiguous", [False, True])
def test_query_rows_match_causal_sdpa(contiguous):
    """The s_q query rows of a decode step are the request's last s_q
    positions: merged over the shards they equal the last s_q rows of
    torch's causal scaled_dot_product_attention over the whole request."""
    L, s_q, H, D = 11, 3, 4, 16
    q_all, k, v = _rows_case(L, s_q, H, D)
    scale = 0.37
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q_all).permute(1, 0, 2), torch.from_numpy(k[:, 0]).expand(H, L, D),
        torch.from_numpy(v[:, 0]).expand(H, L, D), is_causal=True, scale=scale).permute(1, 0, 2).numpy()
    for C in (1, 3, 4, 16):
        po, pl = oracle.query_rows_partials(q_all[L - s_q:], k, v, C, scale, contiguous=contiguous)
        o, lse = oracle.lse_merge(po, pl)
        assert np.allclose(o, ref[L - s_q:], atol=1e-12)
        # LSE: logsumexp of the row's causal scores, from torch
        s = torch.einsum("qhd,kd->qhk", torch.from_numpy(q_all[L - s_q:]), torch.from_numpy(k[:, 0])) * scale
        mask = torch.arange(L)[None, :] <= torch.arange(L - s_q, L)[:, None]
        want = torch.logsumexp(s.masked_fill(~mask[:, None, :], -math.inf), dim=-1).numpy()
        assert np.allclose(lse, want, atol=1e-12)


def test_query_rows_one_row_is_decode():
    L, H, D = 9, 2, 8
    q_all, k, v = _rows_case(L, 1, H, D, seed=9)
    po, pl = oracle.query_rows_partials(q_all[-1:], k, v, 4, 0.5)
    so, sl = oracle.decode_shard_partials(q_all[-1], k, v, 4, 0.5)
    assert np.allclose(po[:, 0], so) and np.allclose(pl[:, 0], sl)


def test_query_rows_pin_catches_off_by_one(monkeypatch):
    """A row that stops one token early (or reads one late) fails the SDPA pin."""
    L, s_q, H, D = 11, 3, 4, 16
    q_all, k, v = _rows_case(L, s_q, H, D)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q_all).permute(1, 0, 2), torch.from_numpy(k[:, 0]).expand(H, L, D),
        torch.from_numpy(v[:, 0]).expand(H, L, D), is_causal=True, scale=0.37).permute(1, 0, 2).numpy()
    real = oracle.decode_attention
    for shift in (-1, 1):
        def shifted(q, kc, vc, sm, keys=None, _s=shift):
            keys = np.asarray(keys)
            if len(keys):
                top = keys.max() + _s
                keys = np.arange(0, min(top, kc.shape[0] - 1) + 1)
            return real(q, kc, vc, sm, keys=keys)
        monkeypatch.setattr(oracle.cpattn_oracle, "decode_attention", shifted)
        po, pl = oracle.query_rows_partials(q_all[L - s_q:], k, v, 1, 0.37)
        o, _ = oracle.lse_merge(po, pl)
        monkeypatch.setattr(oracle.cpattn_oracle, "decode_attention", real)
        assert not np.allclose(o, ref[L - s_q:], atol=1e-6)


# ------------------------------------------------------------------ exact sharded top-k


def _global_topk(scores, k):
    """Brute force: every token ranked at once (higher score, then lower index)."""
    return sorted(sorted(range(len(scores)), key=lambda p: (-float(scores[p]), p))[:k])


@pytest.mark.parametrize("contiguous", [False, True])
def test_sharded_topk_equals_global_topk(contiguous):
    """[V4] §5.2: the union of the local top-k lists contains the global
    top-k, so merging them is exact — against brute force, ties included."""
    rng = np.random.default_rng(11)
    for L, C, k in [(1, 1, 1), (20, 4, 5), (37, 8, 1), (100, 3, 17), (64, 8, 64), (50, 7, 80)]:
        for ties in (False, True):
            s = rng.standard_normal(L).astype(np.float32)
            if ties:
                s = np.round(s * 2) / 2  # few distinct values, many ties
            got, local = oracle.sharded_topk(s, C, k, contiguous=contiguous)
            assert got == _global_topk(s, k)
            assert len(got) == min(k, L)
            shard, _ = (oracle.decode_shard_map_contiguous if contiguous else oracle.decode_shard_map)(L, C)
            for r, lst in enumerate(local):
                assert len(lst) == min(k, shard.count(r)) and all(shard[p] == r for p in lst)


def test_sharded_topk_tie_rule_and_all_selected():
    s = np.zeros(30, np.float32)
    assert oracle.sharded_topk(s, 4, 7)[0] == list(range(7))  # equal scores: lower index first
    s = np.arange(10, dtype=np.float32)
    assert oracle.sharded_topk(s, 3, 50)[0] == list(range(10))  # k >= L: everything
    assert oracle.sharded_topk(s, 3, 3)[0] == [7, 8, 9]


def test_sharded_topk_pin_catches_short_local_lists(monkeypatch):
    """Local lists cut to k / C (a plausible shortcut) lose exactness when the
    best tokens sit on one shard; the brute-force pin catches it."""
    L, C, k = 64, 4, 8
    s = np.zeros(L, np.float32)
    s[::C] = 10 + np.arange(L // C)  # shard 0 holds every high score
    got, _ = oracle.sharded_topk(s, C, k)
    assert got == _global_topk(s, k)
    # plant: each shard keeps only k // C candidates
    orig = oracle.cpattn_oracle.sharded_topk

    def planted(scores, C, k, contiguous=False):
        shard, _ = oracle.decode_shard_map(len(scores), C)
        better = lambda p: (-float(scores[p]), p)  # noqa: E731
        local = [sorted([p for p in range(len(scores)) if shard[p] == r], key=better)[:k // C]
                 for r in range(C)]
        return sorted(sorted([p for lst in local for p in lst], key=better)[:k]), local
    monkeypatch.setattr(oracle.cpattn_oracle, "sharded_topk", planted)
    assert oracle.cpattn_oracle.sharded_topk(s, C, k)[0] != _global_topk(s, k)
    monkeypatch.setattr(oracle.cpattn_oracle, "sharded_topk", orig)


def test_sparse_partials_merge_to_attention_over_selection():
    rng = np.random.default_rng(4)
    L, H, D = 40, 3, 8
    q = rng.standard_normal((H, D))
    k = rng.standard_normal((L, 1, D))
    v = rng.standard_normal((L, 1, D))
    s = rng.standard_normal(L).astype(np.float32)
    for C, kk, contiguous in [(1, 9, False), (4, 9, False), (4, 9, True), (8, 50, False)]:
        sel, _ = oracle.sharded_topk(s, C, kk, contiguous=contiguous)
        po, pl = oracle.sparse_partials(q, k, v, sel, C, 0.4, contiguous=contiguous)
        o, lse = oracle.lse_merge(po, pl)
        # against torch: softmax over the selected tokens only
        qs = torch.from_numpy(q)
        ks = torch.from_numpy(k[sel, 0])
        vs = torch.from_numpy(v[sel, 0])
        sc = qs @ ks.T * 0.4
        assert np.allclose(o, (torch.softmax(sc, -1) @ vs).numpy(), atol=1e-12)
        assert np.allclose(lse, torch.logsumexp(sc, -1).numpy(), atol=1e-12)
