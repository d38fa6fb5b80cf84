"""GPU parity of decode with a replicated local window and a designated
rank ("DeepSeek-V4 Attention Inference Systems" §5.1, §5.3): every shard
attends to its token-sharded main-cache rows; the window (each request's
last W uncompressed tokens, held by every rank) is attended once, as a
one-shard decode, and folded with cp_lse_fold into the designated shard's
partial only.  Partials and the merged result against the oracle."""

import math

import numpy as np
import pytest
import torch

import cp_workloads as W
import oracle
from test_gpu_parity import DEV, TOL_BF16, TOL_FP8, check_lse, check_o, cp, np64  # noqa: F401

pytestmark = pytest.mark.gpu


def run_window_decode(cp, mode, q, main, win, ctx, win_len, C, d, scale, nw=0):
    """main / win: (k, v, scale) token-ordered caches.  Returns o_part, lse_part
    [C, B, H, Dv] / [C, B, H] after the fold, and the merged (o, lse)."""
    plan = cp.cp_decode_plan(C, ctx, n_workers=nw, device=DEV)
    wplan = cp.cp_decode_plan(1, win_len, device=DEV)
    mk, mv, ms = main
    wk, wv, ws = win
    sk, ssc = cp.cp_kv_shard_pack(plan, mk, ms)
    wsk, wssc = cp.cp_kv_shard_pack(wplan, wk, ws)
    sv = cp.cp_kv_shard_pack(plan, mv)[0] if mv is not None else None
    wsv = cp.cp_kv_shard_pack(wplan, wv)[0] if wv is not None else None
    o_part, lse_part = cp.cp_decode_attn(plan, mode, q, sk, sv, shard_scale=ssc, sm_scale=scale)
    o_w, lse_w = cp.cp_decode_attn(wplan, mode, q, wsk, wsv, shard_scale=wssc, sm_scale=scale)
    cp.cp_lse_fold(o_part[d], lse_part[d], o_w[0], lse_w[0])
    o, lse = cp.cp_lse_merge(o_part, lse_part, out_dtype=torch.float32)
    cp.cp_device_error_check()
    return o_part, lse_part, o, lse


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("C,d", [(8, 3), (2, 0)])
def test_window_mla(cp, fp8, C, d):
    ctx = [0, 1, 129, 1000, 4097]
    win_len = [128, 5, 0, 128, 64]
    B = len(ctx)
    main = W.mla_decode_inputs(ctx, H=64, seed=71, device=DEV)
    win = W.mla_decode_inputs(win_len, H=64, seed=72, device=DEV)
    q = main["q"]
    scale = 1.0 / math.sqrt(576)
    if fp8:
        mt, wt = (main["kv_fp8"], None, main["kv_scale"]), (win["kv_fp8"], None, win["kv_scale"])
    else:
        mt, wt = (main["kv_bf16"], None, None), (win["kv_bf16"], None, None)
    o_part, lse_part, o, lse = run_window_decode(cp, cp.CP_DECODE_MLA, q, mt, wt, ctx, win_len, C, d,
                                                 scale, nw=5)
    tol = TOL_FP8 if fp8 else TOL_BF16
    mb = np.concatenate([[0], np.cumsum(ctx)])
    wb = np.concatenate([[0], np.cumsum(win_len)])
    qn = np64(q)

    def kv(data, base, b, L):
        if fp8:
            lat = oracle.e4m3_decode(data["kv_fp8"][base[b]:base[b] + L].cpu().numpy())
            return oracle.mla_cache_to_kv(lat, data["kv_scale"][base[b]:base[b] + L].double().cpu().numpy())
        return oracle.mla_cache_to_kv(np64(data["kv_bf16"][base[b]:base[b] + L]))

    for b in range(B):
        Km, Vm = kv(main, mb, b, ctx[b])
        Kw, Vw = kv(win, wb, b, win_len[b])
        po, pl = oracle.designated_partials(qn[b], Km, Vm, Kw, Vw, C, d, scale)
        for r in range(C):
            check_o(o_part[r, b], po[r], what=f"window partial r{r} b{b}", **tol)
            check_lse(lse_part[r, b], pl[r])
        fo, fl = oracle.decode_attention(qn[b], np.concatenate([Km, Kw]), np.concatenate([Vm, Vw]), scale)
        check_o(o[b], fo, what=f"window merged b{b}", **tol)
        check_lse(lse[b], fl)


def test_window_gqa(cp):
    ctx, win_len = [0, 300, 4100], [16, 0, 128]
    C, d, Hq, Hkv, D = 4, 1, 16, 4, 128
    q, mk, mv = W.gqa_decode_inputs(len(ctx), ctx, Hq, Hkv, D, "bf16", seed=81, device=DEV, std=0.3)
    _, wk, wv = W.gqa_decode_inputs(len(ctx), win_len, Hq, Hkv, D, "bf16", seed=82, device=DEV, std=0.3)
    scale = 1.0 / math.sqrt(D)
    o_part, lse_part, o, lse = run_window_decode(cp, cp.CP_DECODE_GQA, q, (mk, mv, None), (wk, wv, None),
                                                 ctx, win_len, C, d, scale)
    mb = np.concatenate([[0], np.cumsum(ctx)])
    wb = np.concatenate([[0], np.cumsum(win_len)])
    qn, mkn, mvn, wkn, wvn = np64(q), np64(mk), np64(mv), np64(wk), np64(wv)
    for b in range(len(ctx)):
        Km, Vm = mkn[mb[b]:mb[b] + ctx[b]], mvn[mb[b]:mb[b] + ctx[b]]
        Kw, Vw = wkn[wb[b]:wb[b] + win_len[b]], wvn[wb[b]:wb[b] + win_len[b]]
        po, pl = oracle.designated_partials(qn[b], Km, Vm, Kw, Vw, C, d, scale)
        for r in range(C):
            check_o(o_part[r, b], po[r], what=f"GQA window partial r{r} b{b}", **TOL_BF16)
            check_lse(lse_part[r, b], pl[r])
        fo, fl = oracle.decode_attention(qn[b], np.concatenate([Km, Kw]), np.concatenate([Vm, Vw]), scale)
        check_o(o[b], fo, what=f"GQA window merged b{b}", **TOL_BF16)
        check_lse(lse[b], fl)


def test_fold_empty_and_one_sided(cp):
    """Folding an empty partial changes nothing; folding into an empty one copies."""
    N, H, Dv = 3, 2, 8
    o = torch.randn(N, H, Dv, device=DEV)
    lse = torch.randn(N, H, device=DEV)
    o0, l0 = o.clone(), lse.clone()
    cp.cp_lse_fold(o, lse, torch.zeros_like(o), torch.full_like(lse, float("-inf")))
    assert torch.allclose(o, o0) and torch.allclose(lse, l0)
    e, el = torch.zeros_like(o), torch.full_like(lse, float("-inf"))
    cp.cp_lse_fold(e, el, o0, l0)
    assert torch.allclose(e, o0, atol=1e-6) and torch.allclose(el, l0, atol=1e-6)
    z, zl = torch.zeros_like(o), torch.full_like(lse, float("-inf"))
    cp.cp_lse_fold(z, zl, torch.zeros_like(o), torch.full_like(lse, float("-inf")))
    assert not z.any() and torch.isneginf(zl).all()
