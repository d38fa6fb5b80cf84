"""Seeded synthetic workloads for context-parallel attention.

This module only draws inputs: sequence lengths, Q/K/V tensors and MLA latent
caches (bf16, or FP8-E4M3 with one fp32 scale per token).  It holds none of
the attention arithmetic, shard maps or merges, so both the CUDA library's
tests and the fp64 oracle can take their inputs from here.

Workloads (lengths in tokens; "1M" is 2**20):

* ``tiny``        1 request, 256-token prompt, GQA 8 q / 2 kv heads, head dim
                  64, fp32 values ~N(0,1)/sqrt(64), zigzag over 4 virtual
                  shards; then one decode step whose 257-token cache (the
                  prompt plus the decoded token itself) is split into 4
                  token-interleaved shards.
* ``zigzag``      1 request, 32,768 new tokens after a 4,096-token cached
                  prefix, GQA 32 q / 8 kv heads, head dim 128, bf16
                  ~N(0,1)/sqrt(128), zigzag over 8 virtual shards.
* ``interleave``  16 requests, bimodal lengths (47% log-uniform 512..64k,
                  53% log-uniform 64k..256k; total capped at 1M tokens),
                  GQA 64 q / 8 kv heads, head dim 128, bf16, interleave over
                  8 virtual shards, no prefix.
* ``mla``         64 requests x 131,072 cached tokens, 64 heads over one
                  576-dim latent (value = first 512 dims), bf16 or FP8 cache,
                  8 token-interleaved shards.
* ``mla_mixed``   128 requests, bimodal context lengths (18% log-uniform
                  1k..8k, 29% 8k..64k, 53% 64k..1M), FP8 cache, 8 shards.
* ``gqa_decode``  16 requests x 131,072 cached tokens, GQA 32 q / 8 kv
                  heads, head dim 128, bf16 ~N(0,1)/sqrt(128), 8
                  token-interleaved shards.

The long-context agentic traces the pages measure on are not available here;
these length mixes stand in for them.
"""

from __future__ import annotations

import math

import numpy as np
import torch

E4M3_MAX = 448.0

SEEDS = {"tiny": 1001, "zigzag": 1002, "interleave": 1003, "mla": 1004, "mla_mixed": 1005,
         "index": 1006, "gqa_decode": 1007}

WORKLOADS = {
    "tiny": dict(kind="prefill+decode", strategy="zigzag", new_len=[256], prefix_len=[0], C=4,
                 Hq=8, Hkv=2, D=64, dtype="fp32", decode_ctx=257),
    "zigzag": dict(kind="prefill", strategy="zigzag", new_len=[32768], prefix_len=[4096], C=8,
                   Hq=32, Hkv=8, D=128, dtype="bf16"),
    "interleave": dict(kind="prefill", strategy="interleave", new_len=None, prefix_len=None, C=8,
                       Hq=64, Hkv=8, D=128, dtype="bf16", R=16),
    "mla": dict(kind="decode", B=64, ctx=131072, H=64, Dqk=576, Dv=512, C=8),
    "mla_mixed": dict(kind="decode", B=128, ctx=None, H=64, Dqk=576, Dv=512, C=8, kv="fp8"),
    "gqa_decode": dict(kind="decode", B=16, ctx=131072, Hq=32, Hkv=8, D=128, C=8, kv="bf16"),
}


def log_uniform_int(rng: np.random.Generator, lo: float, hi: float) -> int:
    return int(round(math.exp(rng.uniform(math.log(lo), math.log(hi)))))


def interleave_lengths(seed: int = SEEDS["interleave"], R: int = 16, cap: int = 1 << 20) -> list[int]:
    """Bimodal ragged prompt lengths: class 'long' with probability 0.53
    (log-uniform 64k..256k), else 'short' (log-uniform 512..64k); if the
    total exceeds ``cap``, every length is scaled by cap/total (floor, >= 1)."""
    rng = np.random.default_rng(seed)
    lens = []
    for _ in range(R):
        if rng.random() < 0.53:
            lens.append(log_uniform_int(rng, 65536, 262144))
        else:
            lens.append(log_uniform_int(rng, 512, 65536))
    total = sum(lens)
    if total > cap:
        lens = [max(1, (x * cap) // total) for x in lens]
    return lens


def mixed_context_lengths(seed: int = SEEDS["mla_mixed"], B: int = 128) -> list[int]:
    """Decode context lengths: 18% log-uniform 1k..8k, 29% 8k..64k, 53%
    64k..1M (heavy tail)."""
    rng = np.random.default_rng(seed)
    lens = []
    for _ in range(B):
        u = rng.random()
        if u < 0.18:
            lens.append(log_uniform_int(rng, 1024, 8192))
        elif u < 0.47:
            lens.append(log_uniform_int(rng, 8192, 65536))
        else:
            lens.append(log_uniform_int(rng, 65536, 1 << 20))
    return lens


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, gen, device, std, dtype):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def torch_dtype(name: str):
    return {"fp32": torch.float32, "bf16": torch.bfloat16}[name]


def prefill_inputs(new_len, prefix_len, Hq, Hkv, D, dtype="bf16", seed=0, device="cpu",
                   std=None):
    """Q [T, Hq, D] in flattened new-token order, K and V
    [sum(prefix+new), Hkv, D] with each request's prefix then new tokens,
    requests back to back.  Values ~N(0,1) * std (default 1/sqrt(D))."""
    std = 1.0 / math.sqrt(D) if std is None else std
    T = int(sum(new_len))
    KV = int(sum(new_len) + sum(prefix_len))
    g = _gen(device, seed)
    dt = torch_dtype(dtype)
    q = _randn((T, Hq, D), g, device, std, dt)
    k = _randn((KV, Hkv, D), g, device, std, dt)
    v = _randn((KV, Hkv, D), g, device, std, dt)
    return q, k, v


def gqa_decode_inputs(B, ctx, Hq, Hkv, D, dtype="fp32", seed=0, device="cpu", std=None):
    """Decode query Q [B, Hq, D] and per-request caches K, V
    [sum(ctx), Hkv, D] in token order, requests back to back."""
    std = 1.0 / math.sqrt(D) if std is None else std
    g = _gen(device, seed)
    dt = torch_dtype(dtype)
    ctx = [int(c) for c in ctx] if not isinstance(ctx, int) else [ctx] * B
    q = _randn((B, Hq, D), g, device, std, dt)
    k = _randn((sum(ctx), Hkv, D), g, device, std, dt)
    v = _randn((sum(ctx), Hkv, D), g, device, std, dt)
    return q, k, v


def gqa_decode_inputs_fp8(B, ctx, Hq, Hkv, D, seed=0, device="cpu", std=None):
    """GQA decode inputs with an FP8 cache: Q [B, Hq, D] bf16, K and V codes
    [sum(ctx), Hkv, D] (uint8 E4M3) and one fp32 scale per token for both of
    its rows (amax over the token's K and V values / 448).  The codes quantise
    the bf16 K and V of gqa_decode_inputs with the same seed."""
    q, k, v = gqa_decode_inputs(B, ctx, Hq, Hkv, D, "bf16", seed=seed, device=device, std=std)
    T = k.shape[0]
    codes, scale = quantize_e4m3_per_token(torch.cat([k.reshape(T, -1), v.reshape(T, -1)], dim=1))
    kc = codes[:, :Hkv * D].reshape(T, Hkv, D).contiguous()
    vc = codes[:, Hkv * D:].reshape(T, Hkv, D).contiguous()
    return q, kc, vc, scale


def quantize_e4m3_per_token(x: torch.Tensor):
    """FP8-E4M3 codes and one fp32 scale per row: scale = amax/448 (1 for an
    all-zero row), code = round-to-nearest-even(x / scale).  Done once, at
    data generation; both the library and the oracle consume the bytes."""
    xf = x.float()
    amax = xf.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    codes = (xf / scale[..., None]).clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return codes.view(torch.uint8), scale.contiguous()


def mla_decode_inputs(ctx, H=64, Dqk=576, seed=0, device="cpu", q_std=1.0, kv_std=1.0,
                      fp8=True, bf16=True, chunk_rows=1 << 24):
    """MLA decode inputs: Q [B, H, Dqk] bf16 and the latent cache
    [sum(ctx), Dqk] in token order, requests back to back: bf16 and/or FP8
    codes (uint8) with a fp32 per-token scale.  The FP8 cache quantises the
    bf16 cache's values."""
    ctx = [int(c) for c in ctx]
    g = _gen(device, seed)
    B = len(ctx)
    q = _randn((B, H, Dqk), g, device, q_std, torch.bfloat16)
    N = sum(ctx)
    lat = torch.empty((N, Dqk), dtype=torch.bfloat16, device=device)
    codes = torch.empty((N, Dqk), dtype=torch.uint8, device=device) if fp8 else None
    scale = torch.empty((N,), dtype=torch.float32, device=device) if fp8 else None
    for s in range(0, N, chunk_rows):
        e = min(N, s + chunk_rows)
        lat[s:e] = _randn((e - s, Dqk), g, device, kv_std, torch.bfloat16)
        if fp8:
            codes[s:e], scale[s:e] = quantize_e4m3_per_token(lat[s:e])
    out = {"q": q, "ctx": ctx}
    if bf16:
        out["kv_bf16"] = lat
    else:
        del lat
    if fp8:
        out["kv_fp8"] = codes
        out["kv_scale"] = scale
    return out


def index_scores(ctx, seed=SEEDS["index"], device="cpu", ties=False):
    """Relevance scores of every cached token [sum(ctx)] fp32, token order,
    requests back to back: N(0, 1), or with ``ties`` rounded to multiples of
    1/2 (few distinct values, many equal scores).  They stand in for the
    output of a sparse-attention index scan, whose weights are not here."""
    g = _gen(device, seed)
    s = torch.randn((sum(int(c) for c in ctx),), generator=g, device=device, dtype=torch.float32)
    return torch.round(s * 2) / 2 if ties else s


def tiny_inputs(device="cpu", seed=SEEDS["tiny"]):
    """The tiny workload: prefill Q/K/V of a 256-token prompt (fp32), then the
    decode step of token 256, whose cache holds the 256 prompt entries plus
    its own key and value (257 entries, token order)."""
    w = WORKLOADS["tiny"]
    q, k, v = prefill_inputs(w["new_len"], w["prefix_len"], w["Hq"], w["Hkv"], w["D"], w["dtype"],
                             seed=seed, device=device)
    dq, dk, dv = gqa_decode_inputs(1, [1], w["Hq"], w["Hkv"], w["D"], w["dtype"], seed=seed + 1,
                                   device=device)
    return {"q": q, "k": k, "v": v, "dec_q": dq, "dec_k": torch.cat([k, dk]),
            "dec_v": torch.cat([v, dv]), "ctx": [w["decode_ctx"]]}
