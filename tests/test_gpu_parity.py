"""GPU parity: the CUDA library through its C ABI against the fp64 oracle.

Tolerances (written here, applied to every floating-point comparison):
  bf16 inputs, O:      max abs error <= 2e-2 and relative Frobenius <= 5e-3
  fp32 inputs (tiny):  held to the bf16 bound
  FP8-E4M3 cache, O:   max abs error <= 6e-2
  LSE:                 max abs error <= 1e-3
Shard maps, packing and plans: bit-exact.
"""

import math

import numpy as np
import pytest
import torch

import cp_workloads as W
import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL_BF16 = dict(max_abs=2e-2, rel_fro=5e-3)
TOL_FP8 = dict(max_abs=6e-2, rel_fro=None)
TOL_LSE = 1e-3


@pytest.fixture(scope="module")
def cp():
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")
    import __graft_entry__
    __graft_entry__.ensure_built()
    import context_long_attention_gb300 as cp
    return cp


def check_o(got, ref, max_abs, rel_fro, what="O"):
    g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    d = g - ref
    err = np.abs(d).max() if d.size else 0.0
    assert err <= max_abs, f"{what}: max abs err {err:.3e} > {max_abs}"
    if rel_fro is not None and d.size:
        nr = np.linalg.norm(ref)
        rf = np.linalg.norm(d) / nr if nr > 0 else np.linalg.norm(d)
        assert rf <= rel_fro, f"{what}: rel Frobenius err {rf:.3e} > {rel_fro}"


def check_lse(got, ref, tol=TOL_LSE):
    g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    assert np.array_equal(np.isneginf(g), np.isneginf(ref)), "LSE -inf pattern differs"
    fin = np.isfinite(ref)
    if fin.any():
        err = np.abs(g[fin] - ref[fin]).max()
        assert err <= tol, f"LSE max abs err {err:.3e} > {tol}"


def np64(t):
    return t.detach().to(torch.float64).cpu().numpy()


# ---------------------------------------------------------------- plans

PLAN_BATCHES = [([16], [0], 4), ([5, 3], [0, 0], 4), ([19], [7], 4), ([3], [2], 4),
                ([0, 9, 1, 33], [4, 0, 11, 2], 3), ([100, 1, 0, 57, 256], [0, 13, 5, 0, 1000], 8),
                ([1000], [0], 1), ([7, 7, 7], [0, 0, 0], 64)]


@pytest.mark.parametrize("new_len,prefix_len,C", PLAN_BATCHES)
def test_device_maps_bit_exact(cp, new_len, prefix_len, C):
    for strategy, ofn in ((cp.CP_ZIGZAG, oracle.zigzag_plan), (cp.CP_INTERLEAVE, oracle.interleave_plan)):
        plan = cp.cp_shard_plan(strategy, C, new_len, prefix_len, device=DEV)
        idx, qpos, qreq = (t.cpu().numpy() for t in plan.device_maps())
        ref = ofn(new_len, prefix_len, C)
        ro = plan.rank_off
        for r in range(C):
            sl = slice(ro[r], ro[r + 1])
            assert list(idx[sl]) == list(ref["order"][r])
            assert list(qpos[sl]) == list(ref["pos"][r])
            assert list(qreq[sl]) == list(ref["req"][r])
        # the device copy of the host part is identical
        hw = plan.host_words
        assert np.array_equal(plan.dev[:hw].cpu().numpy(), plan.host[:hw])


def test_device_maps_full_size(cp):
    z = W.WORKLOADS["zigzag"]
    lens = W.interleave_lengths()
    for strategy, nl, pl, C, ofn in (
            (cp.CP_ZIGZAG, z["new_len"], z["prefix_len"], z["C"], oracle.zigzag_plan),
            (cp.CP_INTERLEAVE, lens, [0] * len(lens), 8, oracle.interleave_plan_np)):
        plan = cp.cp_shard_plan(strategy, C, nl, pl, device=DEV)
        idx, qpos, qreq = (t.cpu().numpy() for t in plan.device_maps())
        ref = ofn(nl, pl, C)
        ro = plan.rank_off
        for r in range(C):
            sl = slice(ro[r], ro[r + 1])
            assert np.array_equal(idx[sl], np.asarray(ref["order"][r]))
            assert np.array_equal(qpos[sl], np.asarray(ref["pos"][r]))
            assert np.array_equal(qreq[sl], np.asarray(ref["req"][r]))


# ---------------------------------------------------------------- prefill


def prefill_vs_oracle(cp, strategy, new_len, prefix_len, C, Hq, Hkv, D, dtype, seed, rows=None,
                      tol=TOL_BF16, std=None, check_ranks=False, qkv=None):
    if qkv is None:
        q, k, v = W.prefill_inputs(new_len, prefix_len, Hq, Hkv, D, dtype, seed=seed, device=DEV, std=std)
    else:
        q, k, v = (x.to(DEV) for x in qkv)
    plan = cp.cp_shard_plan(strategy, C, new_len, prefix_len, device=DEV)
    scale = 1.0 / math.sqrt(D)
    o, lse = cp.cp_prefill_attn(plan, q, k, v, scale)
    cp.cp_device_error_check()
    ofn = oracle.zigzag_plan if strategy == cp.CP_ZIGZAG else oracle.interleave_plan_np
    ref_plan = ofn(new_len, prefix_len, C)
    ref = oracle.prefill_reference(ref_plan, new_len, prefix_len, np64(q), np64(k), np64(v), scale,
                                   rows=rows)
    ro = plan.rank_off
    for r in range(C):
        local, o_ref, l_ref = ref[r]
        rows_g = ro[r] + local
        check_o(o[rows_g], o_ref, what=f"rank {r} O", **tol)
        check_lse(lse[rows_g], l_ref)
    if check_ranks:  # a single rank's call gives that rank's rows, in local order
        for r in range(C):
            o_r, l_r = cp.cp_prefill_attn(plan, q, k, v, scale, rank=r)
            assert torch.equal(o_r, o[ro[r]:ro[r + 1]])
            assert torch.equal(l_r, lse[ro[r]:ro[r + 1]])
    return plan


def test_prefill_tiny_fp32(cp):
    w = W.WORKLOADS["tiny"]
    prefill_vs_oracle(cp, cp.CP_ZIGZAG, w["new_len"], w["prefix_len"], w["C"], w["Hq"], w["Hkv"],
                      w["D"], "fp32", W.SEEDS["tiny"], check_ranks=True)


@pytest.mark.parametrize("strategy", [0, 1])
@pytest.mark.parametrize("D", [64, 128])
def test_prefill_fp32_ragged_batch(cp, strategy, D):
    """fp32 inputs on the tf32 tensor-core prefill: ragged requests with and
    without a cached prefix, several 128-query M tiles and 128-key tiles,
    every rank's call alone; held to the bf16 bound."""
    prefill_vs_oracle(cp, strategy, [300, 1000, 77, 5], [0, 500, 13, 0], 4, 8, 2, D, "fp32",
                      seed=21 + D + strategy, check_ranks=True)


def test_prefill_fp32_sharp_scores(cp):
    prefill_vs_oracle(cp, cp.CP_ZIGZAG, [700, 333], [129, 0], 8, 16, 4, 64, "fp32", seed=98, std=0.35)


@pytest.mark.parametrize("strategy", [0, 1])
@pytest.mark.parametrize("D", [64, 128])
def test_prefill_bf16_ragged_batch(cp, strategy, D):
    prefill_vs_oracle(cp, strategy, [300, 1000, 77, 5], [0, 500, 13, 0], 4, 8, 2, D, "bf16",
                      seed=7 + D + strategy, check_ranks=True)


@pytest.mark.parametrize("strategy", [0, 1])
def test_prefill_bf16_sharp_scores(cp, strategy):
    # larger inputs give peaked softmax rows (scores of order 10)
    prefill_vs_oracle(cp, strategy, [700, 333], [129, 0], 8, 16, 4, 128, "bf16", seed=99,
                      std=0.35)


def scores_along_keys(T, KV, Hq, Hkv, D, slope, seed):
    """bf16 Q, K, V whose scores move linearly along the keys: q = 4u + noise,
    k_j = (b0 + slope j) u + noise for a unit vector u."""
    g = torch.Generator().manual_seed(seed)
    u = torch.randn(D, generator=g, dtype=torch.float64)
    u /= u.norm()
    b = (0.0 if slope > 0 else -slope * KV) + slope * torch.arange(KV, dtype=torch.float64)
    q = 4.0 * u + 0.3 * torch.randn(T, Hq, D, generator=g, dtype=torch.float64)
    k = b[:, None, None] * u + 0.3 * torch.randn(KV, Hkv, D, generator=g, dtype=torch.float64)
    v = torch.randn(KV, Hkv, D, generator=g, dtype=torch.float64)
    return tuple(x.to(torch.bfloat16) for x in (q, k, v))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("slope", [0.25, -0.25])
def test_prefill_bf16_scores_along_keys(cp, D, slope):
    """Rising scores pass the running max by far more than 2^8 on every KV
    tile (about 11 natural units per 128 keys at head dim 128), so every tile
    takes the softmax's exact path (maxima exchanged, O rescaled) after its
    speculative P; falling scores keep the first tile's max, so every later
    tile keeps its speculative P."""
    new_len, prefix_len = [1100, 300], [60, 0]
    qkv = scores_along_keys(1400, 1460, 4, 2, D, slope, seed=31 + D)
    prefill_vs_oracle(cp, cp.CP_ZIGZAG, new_len, prefix_len, 4, 4, 2, D, "bf16", seed=0, qkv=qkv)
    prefill_vs_oracle(cp, cp.CP_INTERLEAVE, new_len, prefix_len, 4, 4, 2, D, "bf16", seed=0, qkv=qkv)


def test_prefill_edge_cases(cp):
    # C=1 (textbook causal attention); fewer tokens than blocks; a single token
    prefill_vs_oracle(cp, cp.CP_ZIGZAG, [200], [0], 1, 4, 4, 64, "bf16", seed=3)
    prefill_vs_oracle(cp, cp.CP_ZIGZAG, [3, 1], [5, 0], 4, 4, 1, 64, "bf16", seed=4)
    prefill_vs_oracle(cp, cp.CP_INTERLEAVE, [1], [0], 8, 2, 2, 128, "fp32", seed=5)


@pytest.mark.parametrize("strategy", [0, 1])
def test_prefill_maximum_shards(cp, strategy):
    # C = 64, the shard limit: 128 zigzag blocks, most of a few tokens, some empty
    prefill_vs_oracle(cp, strategy, [300, 2000, 40], [0, 64, 7], 64, 8, 2, 128, "bf16", seed=21 + strategy)


@pytest.mark.parametrize("kind", ["fp8", "bf16", "gqa"])
def test_decode_maximum_shards(cp, kind):
    """C = 64, the shard limit: requests shorter than C leave shards empty."""
    ctx, C = [1, 63, 100, 5000], 64
    if kind == "gqa":
        q, k, v = W.gqa_decode_inputs(len(ctx), ctx, 16, 4, 128, "bf16", seed=22, device=DEV, std=0.3)
        gqa_decode_case(cp, q, k, v, ctx, C, 1.0 / math.sqrt(128), 9)
    else:
        fp8 = kind == "fp8"
        data = W.mla_decode_inputs(ctx, H=64, seed=23, device=DEV, fp8=fp8, bf16=not fp8)
        mla_decode_case(cp, data, C, fp8, 9)


def sample_rows(plan, per_rank=48, seed=0):
    """Each segment's first and last row, plus random rows, per rank."""
    rng = np.random.default_rng(seed)
    ro = plan.rank_off
    out = []
    for r in range(plan.C):
        n = int(ro[r + 1] - ro[r])
        pick = set()
        for s in plan.segments:
            if s[0] == r and s[5] > 0:
                pick.add(int(s[4] - ro[r]))
                pick.add(int(s[4] + s[5] - 1 - ro[r]))
        pick.update(int(x) for x in rng.integers(0, n, size=per_rank)) if n else None
        out.append(np.array(sorted(pick), dtype=np.int64))
    return out


def test_prefill_zigzag_full_size_sampled(cp):
    z = W.WORKLOADS["zigzag"]
    plan = cp.cp_shard_plan(cp.CP_ZIGZAG, z["C"], z["new_len"], z["prefix_len"], device=None)
    rows = sample_rows(plan, per_rank=24)
    prefill_vs_oracle(cp, cp.CP_ZIGZAG, z["new_len"], z["prefix_len"], z["C"], z["Hq"], z["Hkv"],
                      z["D"], "bf16", W.SEEDS["zigzag"], rows=rows)


# ---------------------------------------------------------------- merge


@pytest.mark.parametrize("P", [1, 3, 8, 64])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_lse_merge(cp, P, out_dtype):
    g = torch.Generator(device="cpu").manual_seed(P)
    N, H, Dv = 5, 4, 96
    o_part = torch.randn((P, N, H, Dv), generator=g)
    lse_part = torch.randn((P, N, H), generator=g) * 5
    if P > 1:
        lse_part[1, 0, :] = -math.inf  # an empty part
    lse_part[:, 2, 1] = -math.inf      # every part empty
    o_part[:, 2, 1] = 0
    o, lse = cp.cp_lse_merge(o_part.to(DEV), lse_part.to(DEV), out_dtype=out_dtype)
    o_ref, l_ref = oracle.lse_merge(o_part.double().numpy(), lse_part.double().numpy())
    tol = dict(max_abs=1e-5, rel_fro=1e-6) if out_dtype == torch.float32 else TOL_BF16
    check_o(o, o_ref, **tol)
    check_lse(lse, l_ref, 1e-5)


# ---------------------------------------------------------------- decode


def test_kv_shard_pack_bit_exact(cp):
    ctx = [0, 1, 5, 1000, 3, 257]
    C = 4
    data = W.mla_decode_inputs(ctx, H=2, seed=11, device=DEV)
    plan = cp.cp_decode_plan(C, ctx, n_workers=5, device=DEV)
    for kv, sc in ((data["kv_bf16"], None), (data["kv_fp8"], data["kv_scale"])):
        shards, scales = cp.cp_kv_shard_pack(plan, kv, sc)
        kvc = kv.cpu()
        base = np.concatenate([[0], np.cumsum(ctx)])
        for r in range(C):
            sh = shards[r].cpu()
            row = 0
            for b, L in enumerate(ctx):
                shard, rowmap = oracle.decode_shard_map(L, C)
                toks = [p for p in range(L) if shard[p] == r]
                assert [rowmap[p] for p in toks] == list(range(len(toks)))
                idx = torch.tensor([base[b] + p for p in toks], dtype=torch.long)
                got = sh[row:row + len(toks)]
                assert torch.equal(got.view(torch.uint8), kvc[idx].view(torch.uint8))
                if sc is not None:
                    assert torch.equal(scales[r].cpu()[row:row + len(toks)], sc.cpu()[idx])
                row += len(toks)
            assert row == sh.shape[0]


def gqa_decode_case(cp, q, kc, vc, ctx, C, scale, n_workers, dtype_tol=TOL_BF16):
    plan = cp.cp_decode_plan(C, ctx, n_workers=n_workers, device=DEV)
    sk, _ = cp.cp_kv_shard_pack(plan, kc)
    sv, _ = cp.cp_kv_shard_pack(plan, vc)
    o_part, lse_part = cp.cp_decode_attn(plan, cp.CP_DECODE_GQA, q, sk, sv, sm_scale=scale)
    o, lse = cp.cp_lse_merge(o_part, lse_part, out_dtype=torch.float32)
    cp.cp_device_error_check()
    base = np.concatenate([[0], np.cumsum(ctx)])
    qn, kn, vn = np64(q), np64(kc), np64(vc)
    for b, L in enumerate(ctx):
        kb, vb = kn[base[b]:base[b] + L], vn[base[b]:base[b] + L]
        po, pl = oracle.decode_shard_partials(qn[b], kb, vb, C, scale)
        for r in range(C):
            check_o(o_part[r, b], po[r], what=f"partial r{r} b{b}", **dtype_tol)
            check_lse(lse_part[r, b], pl[r])
        fo, fl = oracle.decode_attention(qn[b], kb, vb, scale)
        check_o(o[b], fo, what=f"merged b{b}", **dtype_tol)
        check_lse(lse[b], fl)


def test_decode_gqa_tiny(cp):
    t = W.tiny_inputs(device=DEV)
    w = W.WORKLOADS["tiny"]
    for nw in (0, 3, 64):
        gqa_decode_case(cp, t["dec_q"], t["dec_k"], t["dec_v"], t["ctx"], w["C"],
                        1.0 / math.sqrt(w["D"]), nw)


@pytest.mark.parametrize("Hq,Hkv,D,nw", [(16, 4, 128, 6), (8, 2, 64, 0), (32, 1, 64, 7), (64, 1, 128, 5)])
def test_decode_gqa_fp32(cp, Hq, Hkv, D, nw):
    """fp32 caches on the tf32 tensor-core GQA decode: ragged requests, empty
    shards, split pairs, 4 to 64 query columns per kv head; every shard's
    partial and the merge; held to the bf16 bound."""
    ctx = [0, 2, 300, 2100]
    q, k, v = W.gqa_decode_inputs(len(ctx), ctx, Hq, Hkv, D, "fp32", seed=Hq + D, device=DEV, std=0.3)
    gqa_decode_case(cp, q, k, v, ctx, 8, 1.0 / math.sqrt(D), nw)


def test_decode_gqa_bf16_ragged(cp):
    ctx = [0, 2, 300, 4100]
    q, k, v = W.gqa_decode_inputs(len(ctx), ctx, 16, 4, 128, "bf16", seed=12, device=DEV, std=0.3)
    gqa_decode_case(cp, q, k, v, ctx, 8, 1.0 / math.sqrt(128), 6)


@pytest.mark.parametrize("ctx,C,Hq,Hkv,D,nw", [([0, 2, 300, 4100], 4, 16, 4, 128, 6),
                                                ([1, 700, 2049], 8, 8, 2, 64, 0),
                                                ([3, 129, 5000], 8, 32, 1, 128, 7),
                                                ([0, 640, 3000], 4, 32, 2, 128, 0),
                                                ([257, 1000], 4, 64, 1, 128, 5)])
def test_decode_gqa_fp8(cp, ctx, C, Hq, Hkv, D, nw):
    """GQA over an E4M3 cache: codes with one scale per token for its K and
    V rows; every shard's partial and the merge against the oracle."""
    q, kc, vc, sc = W.gqa_decode_inputs_fp8(len(ctx), ctx, Hq, Hkv, D, seed=C + D, device=DEV, std=0.3)
    plan = cp.cp_decode_plan(C, ctx, n_workers=nw, device=DEV)
    sk, ss = cp.cp_kv_shard_pack(plan, kc, sc)
    sv, _ = cp.cp_kv_shard_pack(plan, vc)
    scale = 1.0 / math.sqrt(D)
    o_part, lse_part = cp.cp_decode_attn(plan, cp.CP_DECODE_GQA, q, sk, sv, shard_scale=ss, sm_scale=scale)
    o, lse = cp.cp_lse_merge(o_part, lse_part, out_dtype=torch.float32)
    cp.cp_device_error_check()
    s64 = sc.double().cpu().numpy()[:, None, None]
    kn = oracle.e4m3_decode(kc.cpu().numpy()) * s64
    vn = oracle.e4m3_decode(vc.cpu().numpy()) * s64
    qn = np64(q)
    base = np.concatenate([[0], np.cumsum(ctx)])
    for b, L in enumerate(ctx):
        kb, vb = kn[base[b]:base[b] + L], vn[base[b]:base[b] + L]
        po, pl = oracle.decode_shard_partials(qn[b], kb, vb, C, scale)
        for r in range(C):
            check_o(o_part[r, b], po[r], what=f"partial r{r} b{b}", **TOL_FP8)
            check_lse(lse_part[r, b], pl[r])
        fo, fl = oracle.decode_attention(qn[b], kb, vb, scale)
        check_o(o[b], fo, what=f"merged b{b}", **TOL_FP8)
        check_lse(lse[b], fl)


def mla_decode_case(cp, data, C, fp8, n_workers, check_reqs=None, H=64):
    ctx = data["ctx"]
    scale = 1.0 / math.sqrt(576)
    plan = cp.cp_decode_plan(C, ctx, n_workers=n_workers, device=DEV)
    if fp8:
        shards, scales = cp.cp_kv_shard_pack(plan, data["kv_fp8"], data["kv_scale"])
    else:
        shards, scales = cp.cp_kv_shard_pack(plan, data["kv_bf16"])
    o_part, lse_part = cp.cp_decode_attn(plan, cp.CP_DECODE_MLA, data["q"], shards,
                                         shard_scale=scales, sm_scale=scale)
    o, lse = cp.cp_lse_merge(o_part, lse_part, out_dtype=torch.bfloat16)
    cp.cp_device_error_check()
    tol = TOL_FP8 if fp8 else TOL_BF16
    base = np.concatenate([[0], np.cumsum(ctx)])
    qn = np64(data["q"])
    reqs = range(len(ctx)) if check_reqs is None else check_reqs
    for b in reqs:
        L = ctx[b]
        if fp8:
            codes = data["kv_fp8"][base[b]:base[b] + L].cpu().numpy()
            lat = oracle.e4m3_decode(codes)
            sc = data["kv_scale"][base[b]:base[b] + L].double().cpu().numpy()
            K, V = oracle.mla_cache_to_kv(lat, sc)
        else:
            K, V = oracle.mla_cache_to_kv(np64(data["kv_bf16"][base[b]:base[b] + L]))
        po, pl = oracle.decode_shard_partials(qn[b], K, V, C, scale)
        for r in range(C):
            check_o(o_part[r, b], po[r], what=f"partial r{r} b{b}", **tol)
            check_lse(lse_part[r, b], pl[r])
        fo, fl = oracle.decode_attention(qn[b], K, V, scale)
        check_o(o[b], fo, what=f"merged b{b}", **tol)
        check_lse(lse[b], fl)
    return o_part, lse_part


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("C,nw", [(8, 5), (1, 3), (4, 0)])
def test_decode_mla_ragged(cp, fp8, C, nw):
    ctx = [0, 1, 3, 129, 1000, 4097]
    data = W.mla_decode_inputs(ctx, H=64, seed=21 + C, device=DEV)
    mla_decode_case(cp, data, C, fp8, nw)


def test_decode_mla_sharp_scores(cp):
    ctx = [517, 2048]
    data = W.mla_decode_inputs(ctx, H=64, seed=31, device=DEV, q_std=3.0)
    for fp8 in (False, True):
        mla_decode_case(cp, data, 8, fp8, 4)


def test_decode_mla_fp8_scale_spread(cp):
    """FP8 cache whose per-token scales grow along each request by up to 2^6
    (so later tiles hold tokens with far larger scales than the first), with
    the same values: the latent is re-quantised with the larger scales, so its
    codes use less of the E4M3 range.  40 of the 64 head slots in use."""
    ctx = [3000, 700, 129]
    data = W.mla_decode_inputs(ctx, H=40, seed=41, device=DEV)
    g = torch.Generator().manual_seed(43)
    k = torch.cat([torch.clamp(torch.arange(L) * 7 // L + torch.randint(0, 2, (L,), generator=g), max=6)
                   for L in ctx]).to(torch.float32)
    scale = (data["kv_scale"].cpu() * torch.pow(2.0, k)).to(DEV)
    data["kv_fp8"] = (data["kv_bf16"].float() / scale[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    data["kv_scale"] = scale
    for C, nw in [(8, 3), (2, 0)]:
        mla_decode_case(cp, data, C, True, nw, H=40)


@pytest.mark.parametrize("fp8", [True, False])
def test_decode_mla_full_size_sampled(cp, fp8):
    w = W.WORKLOADS["mla"]
    data = W.mla_decode_inputs([w["ctx"]] * w["B"], H=w["H"], seed=W.SEEDS["mla"], device=DEV,
                               fp8=fp8, bf16=not fp8)
    mla_decode_case(cp, data, w["C"], fp8, 0, check_reqs=[0, 37, 63])
    del data
    torch.cuda.empty_cache()


def test_misaligned_pointer_rejected(cp):
    t = W.tiny_inputs(device=DEV)
    plan = cp.cp_shard_plan(cp.CP_ZIGZAG, 4, [256], [0], device=DEV)
    q = t["q"]
    bad = q.view(-1)[1:].view(-1)[: q.numel() - 1]
    o = torch.empty_like(q)
    lse = torch.empty((256, 8), device=DEV)
    import ctypes
    st = cp.lib.cp_prefill_attn(plan.host.ctypes.data_as(ctypes.c_void_p), ctypes.c_void_p(plan.dev.data_ptr()),
                                -1, cp.CP_FP32, ctypes.c_void_p(bad.data_ptr()), ctypes.c_void_p(t["k"].data_ptr()),
                                ctypes.c_void_p(t["v"].data_ptr()), 8, 2, 64, 0.125, ctypes.c_void_p(o.data_ptr()),
                                ctypes.c_void_p(lse.data_ptr()), None)
    assert st == cp.CpError(-1, "").status and b"aligned" in cp.lib.cp_last_error()


def test_prefill_interleave_full_size_sampled(cp):
    """The ragged interleave workload at full size (16 requests, 2^20 tokens,
    64 q / 8 kv heads); the oracle checks sampled rows of three requests
    (shortest, middle, longest): every rank's first and last query of the
    request plus one at random."""
    w = W.WORKLOADS["interleave"]
    lens = W.interleave_lengths()
    pre = [0] * len(lens)
    C, Hq, Hkv, D = w["C"], w["Hq"], w["Hkv"], w["D"]
    q, k, v = W.prefill_inputs(lens, pre, Hq, Hkv, D, "bf16", seed=W.SEEDS["interleave"], device=DEV)
    plan = cp.cp_shard_plan(cp.CP_INTERLEAVE, C, lens, pre, device=DEV)
    scale = 1.0 / math.sqrt(D)
    o, lse = cp.cp_prefill_attn(plan, q, k, v, scale)
    cp.cp_device_error_check()
    ref_plan = oracle.interleave_plan_np(lens, pre, C)
    order = np.argsort(lens)
    picks = [int(order[0]), int(order[len(order) // 2]), int(order[-1])]
    base = np.concatenate([[0], np.cumsum(lens)])
    rng = np.random.default_rng(3)
    ro = plan.rank_off
    for j in picks:
        L = lens[j]
        kj = np64(k[base[j]:base[j] + L])
        vj = np64(v[base[j]:base[j] + L])
        for r in range(C):
            local = np.nonzero(np.asarray(ref_plan["req"][r]) == j)[0]
            if len(local) == 0:
                continue
            sel = np.unique([local[0], local[-1], local[rng.integers(0, len(local))]])
            f = np.asarray(ref_plan["order"][r])[sel]
            pos = np.asarray(ref_plan["pos"][r])[sel]
            o_ref, l_ref = oracle.causal_rows(np64(q[torch.as_tensor(f, device=DEV)]), kj, vj, pos, scale)
            rows_g = torch.as_tensor(ro[r] + sel, device=DEV)
            check_o(o[rows_g], o_ref, what=f"req {j} rank {r}", **TOL_BF16)
            check_lse(lse[rows_g], l_ref)
        del kj, vj


def test_decode_mla_mixed_full_size_sampled(cp):
    """The mixed-length FP8 MLA workload at full size (128 requests, 1k..1M
    contexts, 8 shards); the oracle checks the shortest, the median and a
    ~200k-token request in full (all shards' partials and the merge)."""
    w = W.WORKLOADS["mla_mixed"]
    ctx = W.mixed_context_lengths()
    data = W.mla_decode_inputs(ctx, H=w["H"], seed=W.SEEDS["mla_mixed"], device=DEV, bf16=False)
    srt = np.argsort(ctx)
    near200k = int(np.argmin(np.abs(np.asarray(ctx) - 200000)))
    mla_decode_case(cp, data, w["C"], True, 0,
                    check_reqs=[int(srt[0]), int(srt[len(srt) // 2]), near200k])
    del data
    torch.cuda.empty_cache()
