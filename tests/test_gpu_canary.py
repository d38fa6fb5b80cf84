"""Canary-guarded outputs: every kernel writes through a view inside a
larger buffer whose guard regions hold a seeded byte pattern; after the
call the guards must be unchanged (no write outside the declared outputs)."""

import math

import pytest
import torch

import cp_workloads as W
from test_gpu_parity import DEV, cp  # noqa: F401

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes of guard on each side (a multiple of 16 keeps views aligned)


def guarded(shape, dtype, seed):
    """A view of `shape` in the middle of a byte buffer with random guards."""
    esz = torch.empty((), dtype=dtype).element_size()
    n = int(torch.tensor(shape).prod()) * esz
    g = torch.Generator(device=DEV).manual_seed(seed)
    buf = torch.randint(0, 256, (n + 2 * GUARD,), dtype=torch.uint8, device=DEV, generator=g)
    keep = buf.clone()
    view = buf[GUARD:GUARD + n].view(dtype).view(shape)
    return view, buf, keep


def check_guards(buf, keep, what):
    torch.cuda.synchronize()
    assert torch.equal(buf[:GUARD], keep[:GUARD]), f"{what}: wrote before its output"
    assert torch.equal(buf[-GUARD:], keep[-GUARD:]), f"{what}: wrote after its output"


def test_prefill_and_plan_guards(cp):
    nl, pl, C, Hq, Hkv, D = [1000, 77], [128, 0], 4, 8, 2, 128
    q, k, v = W.prefill_inputs(nl, pl, Hq, Hkv, D, "bf16", seed=1, device=DEV)
    plan = cp.cp_shard_plan(cp.CP_ZIGZAG, C, nl, pl, device=DEV)
    o, ob, ok = guarded((q.shape[0], Hq, D), torch.bfloat16, 2)
    lse, lb, lk = guarded((q.shape[0], Hq), torch.float32, 3)
    cp.cp_prefill_attn(plan, q, k, v, 1.0 / math.sqrt(D), out=o, lse=lse)
    cp.cp_device_error_check()
    check_guards(ob, ok, "prefill O")
    check_guards(lb, lk, "prefill LSE")
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("fp8", [True, False])
def test_decode_pack_merge_guards(cp, fp8):
    ctx, C, H = [1, 300, 1000], 8, 64
    data = W.mla_decode_inputs(ctx, H=H, seed=4, device=DEV, fp8=fp8, bf16=not fp8)
    plan = cp.cp_decode_plan_ex(C, ctx, n_workers=7, device=DEV)
    kv = data["kv_fp8"] if fp8 else data["kv_bf16"]
    rows = plan.shard_rows()
    shards, sb = [], []
    for r, n in enumerate(rows):
        t, b_, k_ = guarded((max(n, 1), 576), kv.dtype, 10 + r)
        shards.append(t[:n])
        sb.append((b_, k_))
    scales = None
    if fp8:
        scales, scb = [], []
        for r, n in enumerate(rows):
            t, b_, k_ = guarded((max(n, 1),), torch.float32, 30 + r)
            scales.append(t[:n])
            scb.append((b_, k_))
    cp.cp_kv_shard_pack(plan, kv, data.get("kv_scale"), shards=shards, shard_scales=scales)
    cp.cp_device_error_check()
    for r, (b_, k_) in enumerate(sb):
        torch.cuda.synchronize()
        assert torch.equal(b_[:GUARD], k_[:GUARD]), f"pack shard {r}: wrote before"
        end = GUARD + rows[r] * shards[r].element_size() * 576
        assert torch.equal(b_[end:], k_[end:]), f"pack shard {r}: wrote after"
    if fp8:
        for r, (b_, k_) in enumerate(scb):
            end = GUARD + rows[r] * 4
            assert torch.equal(b_[:GUARD], k_[:GUARD]) and torch.equal(b_[end:], k_[end:]), f"scale {r}"
    B = len(ctx)
    o_part, opb, opk = guarded((C, B, H, 512), torch.float32, 50)
    lse_part, lpb, lpk = guarded((C, B, H), torch.float32, 51)
    ws_bytes = cp.cp_decode_workspace_size(plan, H, 512)
    ws, wsb, wsk = guarded((max(ws_bytes, 16),), torch.uint8, 52)
    cp.cp_decode_attn(plan, cp.CP_DECODE_MLA, data["q"], shards, shard_scale=scales,
                      sm_scale=1.0 / 24, o_part=o_part, lse_part=lse_part, ws=ws)
    o, ob, okk = guarded((B, H, 512), torch.bfloat16, 53)
    lse, lb, lk = guarded((B, H), torch.float32, 54)
    cp.cp_lse_merge(o_part, lse_part, out=o, lse=lse)
    cp.cp_device_error_check()
    for (b_, k_), what in [((opb, opk), "o_part"), ((lpb, lpk), "lse_part"), ((wsb, wsk), "workspace"),
                           ((ob, okk), "merged O"), ((lb, lk), "merged LSE")]:
        check_guards(b_, k_, what)


@pytest.mark.parametrize("D,s_q,kv", [(128, 1, "bf16"), (64, 1, "bf16"), (128, 3, "bf16"), (128, 1, "fp8"),
                                       (128, 3, "fp8")])
def test_gqa_decode_guards(cp, D, s_q, kv):
    """The GQA decode (the tensor-core kernels for these shapes, bf16 and FP8
    caches) writes only its partials, their LSE and its workspace; split
    pairs use the workspace."""
    ctx, C, Hq, Hkv = [s_q, 300, 1000], 4, 8, 2
    B = len(ctx)
    plan = cp.cp_decode_plan_ex(C, ctx, s_q=s_q, n_workers=7, device=DEV)
    ss = None
    if kv == "fp8":
        q, kc, vc, sc = W.gqa_decode_inputs_fp8(B, ctx, Hq * s_q, Hkv, D, seed=15 + s_q, device=DEV, std=0.3)
        sk, ss = cp.cp_kv_shard_pack(plan, kc, sc)
        sv, _ = cp.cp_kv_shard_pack(plan, vc)
    else:
        q, k, v = W.gqa_decode_inputs(B, ctx, Hq * s_q, Hkv, D, "bf16", seed=5 + D + s_q, device=DEV, std=0.3)
        sk, _ = cp.cp_kv_shard_pack(plan, k)
        sv, _ = cp.cp_kv_shard_pack(plan, v)
    lead = (B, s_q) if s_q > 1 else (B,)
    qq = q.reshape(B, s_q, Hq, D) if s_q > 1 else q
    o_part, opb, opk = guarded((C, *lead, Hq, D), torch.float32, 60)
    lse_part, lpb, lpk = guarded((C, *lead, Hq), torch.float32, 61)
    ws_bytes = cp.cp_decode_workspace_size(plan, Hq, D)
    ws, wsb, wsk = guarded((max(ws_bytes, 16),), torch.uint8, 62)
    cp.cp_decode_attn(plan, cp.CP_DECODE_GQA, qq, sk, sv, shard_scale=ss, sm_scale=1.0 / math.sqrt(D),
                      o_part=o_part, lse_part=lse_part, ws=ws)
    cp.cp_device_error_check()
    for (b_, k_), what in [((opb, opk), "o_part"), ((lpb, lpk), "lse_part"), ((wsb, wsk), "workspace")]:
        check_guards(b_, k_, what)
    assert torch.isfinite(o_part).all()


def test_sparse_guards(cp):
    ctx, C, k = [5, 900, 3000], 4, 100
    plan = cp.cp_decode_plan_ex(C, ctx, n_workers=5, device=DEV)
    data = W.mla_decode_inputs(ctx, H=64, seed=6, device=DEV, bf16=False)
    sh, sc = cp.cp_kv_shard_pack(plan, data["kv_fp8"], data["kv_scale"])
    scores = W.index_scores(ctx, seed=7, device=DEV)
    base = [0, 5, 905]
    sn = scores.cpu()
    shard_scores = [torch.cat([sn[base[b] + r:base[b] + L:C] for b, L in enumerate(ctx)]).to(DEV)
                    for r in range(C)]
    B = len(ctx)
    sel, selb, selk = guarded((B, k), torch.int32, 60)
    cnt, cb, ck = guarded((B,), torch.int32, 61)
    ws_bytes = cp.cp_sparse_workspace_size(plan, k)
    ws, wsb, wsk = guarded((ws_bytes,), torch.uint8, 62)
    cp.cp_sparse_topk(plan, shard_scores, k, sel_ids=sel, sel_count=cnt, ws=ws)
    kp = cp.sparse_slot_rows(k)
    sel_kv, skb = zip(*[(lambda t: (t[0], (t[1], t[2])))(guarded((B * kp, 576), torch.uint8, 70 + r))
                        for r in range(C)])
    sel_sc, ssb = zip(*[(lambda t: (t[0], (t[1], t[2])))(guarded((B * kp,), torch.float32, 80 + r))
                        for r in range(C)])
    pc, pcb, pck = guarded((C * B,), torch.int32, 90)
    cp.cp_sparse_gather(plan, k, ws, sh, sc, list(sel_kv), list(sel_sc), pc)
    cp.cp_device_error_check()
    for (b_, k_), what in [((selb, selk), "sel_ids"), ((cb, ck), "sel_count"), ((wsb, wsk), "topk ws"),
                           ((pcb, pck), "pair_count")] + [(x, f"sel_kv {r}") for r, x in enumerate(skb)] + \
                          [(x, f"sel_scale {r}") for r, x in enumerate(ssb)]:
        check_guards(b_, k_, what)
