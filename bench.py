#!/usr/bin/env python
"""Benchmark of context-parallel attention on GB300, one JSON line.

One step = one pass of the whole hot path over one batch of synthetic input:
  prefill  zigzag shard plan + causal GQA prefill over 8 virtual shards of a
           32,768-token prompt after a 4,096-token cached prefix (32 q / 8 kv
           heads, head dim 128, bf16) — the primary metric, TFLOP/s;
  decode   decode shard plan + split-KV MLA decode of 64 requests x 131,072
           cached tokens over 8 token shards (FP8-E4M3 latent cache with a
           per-token scale) + exact LSE merge — reported as KV HBM GB/s.
The token-shard packing of the decode cache happens once, before timing
(the prefill-to-decode hand-off).  Inputs are larger than L2 (129 MB), so no
flush is needed between steps.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
prefill workload on the host cores (there is no other implementation to run:
the pages describe serving systems, not a library).
Multi-GPU (torchrun): replicas only — every rank runs its own copy of the
step; the value is the work of all ranks over the slowest rank's time.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import cp_workloads as W  # noqa: E402

# DRAM bytes (read + write) per launch from the ncu captures summarised in
# profiles/; a figure is reported only while the kernel sources it was
# measured on are unchanged (SHA-1 of the kernel file and the shared PTX
# header).  The MLA decode captures ran 8 of the 64 requests and the GQA one 4
# of 16; their traffic scales with the tokens read.
PROFILED_TRAFFIC = {
    "prefill": {"src": ["context_long_attention_gb300/csrc/prefill_tc.cu",
                        "context_long_attention_gb300/csrc/tc_ptx.cuh"],
                "sha1": "98ac8718b240f5fd25a3280da4134f23934e585d", "bytes": 0.424714e9 + 0.244750e9},
    "decode_fp8": {"src": ["context_long_attention_gb300/csrc/decode_mla_fp8.cu",
                           "context_long_attention_gb300/csrc/tc_ptx.cuh"],
                   "sha1": "c9efc8882c264cf544b88b58756f4d6698949a1b",
                   "bytes_per_token": (0.610205e9 + 0.009656e9) / (8 * 131072)},
    "decode_bf16": {"src": ["context_long_attention_gb300/csrc/decode_mla_tc.cu",
                            "context_long_attention_gb300/csrc/tc_ptx.cuh"],
                    "sha1": "4998f17b89e397c6fa2724adb688bda380f3b834",
                    "bytes_per_token": (1.208675e9 + 0.010585e9) / (8 * 131072)},
    "decode_gqa": {"src": ["context_long_attention_gb300/csrc/decode_gqa_tc.cu",
                           "context_long_attention_gb300/csrc/tc_ptx.cuh"],
                   "sha1": "66afd4cc6ca2416d3262e0e21695f9dcf534f72c",
                   "bytes_per_token": (2.147824e9 + 0.006298e9) / (4 * 131072)},
    "decode_fp8_merged": {"src": ["context_long_attention_gb300/csrc/decode_mla_fp8.cu",
                                  "context_long_attention_gb300/csrc/tc_ptx.cuh"],
                          "sha1": "c9efc8882c264cf544b88b58756f4d6698949a1b",
                          "bytes_per_token": (0.609321e9 + 0.000153e9) / (8 * 131072)},
    "decode_gqa8": {"src": ["context_long_attention_gb300/csrc/decode_gqa_f8.cu",
                            "context_long_attention_gb300/csrc/tc_ptx.cuh"],
                    "sha1": "c19956b2693cf34223e556901c4c0d1891584060",
                    "bytes_per_token": (1.078127e9 + 0.006134e9) / (4 * 131072)},
}


def sources_sha1(paths):
    import hashlib
    h = hashlib.sha1()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(key, tokens=None):
    """DRAM bytes per launch from the committed ncu capture of this kernel,
    or None once the kernel's sources differ from the captured ones."""
    rec = PROFILED_TRAFFIC[key]
    if rec["sha1"] is None or any(not os.path.exists(os.path.join(ROOT, r)) for r in rec["src"]):
        return None
    if sources_sha1(rec["src"]) != rec["sha1"]:
        return None
    return rec["bytes"] if "bytes" in rec else rec["bytes_per_token"] * tokens


FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


WORKLOAD = ("zigzag prefill: 1 request, 32768 new tokens + 4096-token cached prefix, GQA 32q/8kv, "
            "D 128, bf16, CP=8 virtual shards; plus MLA decode: 64 x 131072 ctx, 64 heads, 576/512 "
            "FP8-E4M3 latent, DCP=8, LSE merge")

PREFILL_WORKLOADS = {
    "zigzag": "zigzag prefill: 1 request, 32768 new tokens + 4096-token cached prefix, GQA 32q/8kv, "
              "D 128, bf16, CP=8 virtual shards",
    "interleave": "interleave prefill: 16 ragged requests (bimodal log-uniform lengths, 2^20 tokens "
                  "in all), GQA 64q/8kv, D 128, bf16, CP=8 virtual shards",
}
DECODE_WORKLOADS = {
    "uniform": "MLA decode: 64 x 131072 ctx, 64 heads, 576/512 latent, DCP=8, LSE merge",
    "mixed": "MLA decode: 128 requests, bimodal log-uniform ctx 1k..1M (2.4e7 tokens), 64 heads, "
             "576/512 latent, DCP=8, LSE merge",
    "gqa": "GQA decode: 16 x 131072 ctx, 32 q / 8 kv heads, head dim 128, bf16 (or E4M3) cache, DCP=8, LSE merge",
}


def workload_name(args):
    if args.prefill_workload == "zigzag" and args.decode_workload == "uniform":
        return WORKLOAD
    return PREFILL_WORKLOADS[args.prefill_workload] + "; plus " + DECODE_WORKLOADS[args.decode_workload]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def prefill_flops(new_len, prefix_len, Hq, D):
    """4 * D * Hq per causal (query, key) pair; pairs = sum of query extents.
    Masked halves of diagonal tiles are not credited."""
    pairs = 0
    for n, p in zip(new_len, prefix_len):
        pairs += n * p + n * (n + 1) // 2
    return 4 * D * Hq * pairs, pairs


def gqa_decode_bytes(ctx, Hq, Hkv, D, fp8=False):
    """K and V rows read once (2 Hkv D values per token: bf16, or E4M3 codes
    plus one 4-byte scale), the bf16 query and the bf16 merged output."""
    B = len(ctx)
    per_tok = 2 * Hkv * D + 4 if fp8 else 2 * Hkv * D * 2
    return sum(ctx) * per_tok + 2 * B * Hq * D * 2


def decode_bytes(ctx, H, fp8=True):
    """KV rows read once (576 B + 4 B scale per token for FP8, 1,152 B for
    bf16), the bf16 query and the bf16 merged output."""
    per_tok = 580 if fp8 else 1152
    B = len(ctx)
    return sum(ctx) * per_tok + B * H * 576 * 2 + B * H * 512 * 2


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""

    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active," \
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown," \
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_rate(units_per_rank, total_ms, world):
    """Units processed by all ranks (every replica runs the same workload) per
    second of the slowest rank's time."""
    return world * units_per_rank / (total_ms / 1e3)


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- CPU oracle


def oracle_prefill_sample(workload="zigzag", rows_per_call=64, seed=0, budget_s=15.0):
    """The fp64 oracle on a bounded sample of a prefill workload, all heads:
    rows of rank 0's late zigzag block (the longest extents), or late rows of
    the interleave batch's longest request (its K/V and the sampled query rows
    drawn at that shape: a timing sample, not the GPU run's values).  Returns
    a dict: TFLOP/s, seconds, rows, cores, (query, key) pairs per second and
    the whole workload's time extrapolated from the sample."""
    import oracle
    z = W.WORKLOADS[workload]
    Hq, Hkv, D, C = z["Hq"], z["Hkv"], z["D"], z["C"]
    rng = np.random.default_rng(seed)
    if workload == "zigzag":
        nl, pl = z["new_len"], z["prefix_len"]
        q, k, v = W.prefill_inputs(nl, pl, Hq, Hkv, D, "bf16", seed=W.SEEDS["zigzag"], device="cpu")
        plan = oracle.zigzag_plan(nl, pl, C)
        n_late = len(plan["order"][0]) // 2
        L = nl[0] + pl[0]
        qd = q.double().numpy()

        def draw():
            li = n_late + rng.choice(n_late, size=rows_per_call, replace=False)
            return qd[np.asarray(plan["order"][0])[li]], np.asarray(plan["pos"][0])[li]
    else:
        nl = W.interleave_lengths()
        pl = [0] * len(nl)
        L = max(nl)
        g = torch.Generator().manual_seed(W.SEEDS[workload])
        sd = 1.0 / math.sqrt(D)
        k = (torch.randn((L, Hkv, D), generator=g) * sd).to(torch.bfloat16)
        v = (torch.randn((L, Hkv, D), generator=g) * sd).to(torch.bfloat16)

        def draw():
            qr = (torch.randn((rows_per_call, Hq, D), generator=g) * sd).to(torch.bfloat16)
            return qr.double().numpy(), rng.integers(L // 2, L, size=rows_per_call)
    k64 = k.double().numpy()[:L]
    v64 = v.double().numpy()[:L]
    done_pairs = 0
    done_rows = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s and done_rows < 64 * rows_per_call:
        qr, pos = draw()
        oracle.causal_rows(qr, k64, v64, pos, 1.0 / math.sqrt(D))
        done_pairs += int((pos + 1).sum())
        done_rows += rows_per_call
    dt = time.perf_counter() - t0
    flops, pairs = prefill_flops(nl, pl, Hq, D)
    rate = 4 * D * Hq * done_pairs / dt
    return {"tflops": rate / 1e12, "seconds": dt, "rows": done_rows, "cores": len(os.sched_getaffinity(0)),
            "pairs_per_s": Hq * done_pairs / dt, "full_s": flops / rate}


def oracle_decode_sample(ctx=None, workload="mla", fp8=True):
    """The fp64 oracle on one request of an MLA decode workload (64 heads):
    E4M3 decode of the cache (FP8) or its bf16 values, then attention over all
    of it.  Returns (decode KV GB/s, seconds, cores)."""
    import oracle
    m = W.WORKLOADS[workload]
    ctx = ctx or m["ctx"]
    d = W.mla_decode_inputs([ctx], H=m["H"], seed=W.SEEDS[workload], device="cpu", bf16=not fp8, fp8=fp8)
    t0 = time.perf_counter()
    if fp8:
        lat = oracle.e4m3_decode(d["kv_fp8"].numpy())
        K, V = oracle.mla_cache_to_kv(lat, d["kv_scale"].double().numpy())
    else:
        K, V = oracle.mla_cache_to_kv(d["kv_bf16"].double().numpy(), None)
    oracle.decode_attention(d["q"][0].double().numpy(), K, V, 1.0 / math.sqrt(m["Dqk"]))
    dt = time.perf_counter() - t0
    return decode_bytes([ctx], m["H"], fp8=fp8) / dt / 1e9, dt, len(os.sched_getaffinity(0))


def oracle_tiny():
    """The fp64 oracle on the whole tiny workload: the zigzag prefill of all 4
    shards and the 257-token decode.  Returns (seconds, cores)."""
    import oracle
    w = W.WORKLOADS["tiny"]
    t = W.tiny_inputs(device="cpu")
    f64 = lambda x: x.double().numpy()  # noqa: E731
    scale = 1.0 / math.sqrt(w["D"])
    t0 = time.perf_counter()
    plan = oracle.zigzag_plan(w["new_len"], w["prefix_len"], w["C"])
    oracle.prefill_reference(plan, w["new_len"], w["prefix_len"], f64(t["q"]), f64(t["k"]), f64(t["v"]), scale)
    oracle.decode_attention(f64(t["dec_q"][0]), f64(t["dec_k"]), f64(t["dec_v"]), scale)
    return time.perf_counter() - t0, len(os.sched_getaffinity(0))


def run_reference(args, world, rank):
    if rank != 0:
        return
    steps = []
    for i in range(args.warmup + args.steps):
        o = oracle_prefill_sample(rows_per_call=16, seed=i, budget_s=2.0)
        tf, dt, rows, cores = o["tflops"], o["seconds"], o["rows"], o["cores"]
        if i >= args.warmup:
            steps.append((tf, dt, rows))
    value = statistics.median(s[0] for s in steps)
    z = W.WORKLOADS["zigzag"]
    line = {
        "impl": "reference", "metric": "prefill causal-attn TFLOP/s", "value": value,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * statistics.median(s[1] for s in steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "timed": "prefill (oracle sample)",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{steps[0][2]} query rows x {z['Hq']} heads per step "
                                   "(rank 0's late zigzag block)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm


def sparse_leg(cp, args, dev, stream, ctx, m, fp8, dplan, shards, scales, dq, world, rank):
    """Top-k over per-token relevance scores on every shard, the exact merge,
    the owners' gather and attention over the selected rows, and the LSE merge,
    each stage timed with CUDA events; inputs resident in HBM."""
    if args.decode_paged or args.decode_rows > 1 or args.decode_layout != "round_robin":
        raise SystemExit("--sparse-k runs on the round-robin, one-row, per-shard cache")
    if args.decode_workload != "uniform" or ctx[0] % m["C"]:
        raise SystemExit("--sparse-k runs on the uniform MLA workload with contexts a multiple of C")
    k, C, B, L = args.sparse_k, m["C"], len(ctx), ctx[0]
    scores = W.index_scores(ctx, seed=W.SEEDS["index"] + rank, device=dev)
    st = scores.view(B, L // C, C)  # round robin: shard r holds tokens r, r + C, ...
    shard_scores = [st[:, :, r].contiguous().view(-1) for r in range(C)]
    del scores, st
    splan = cp.cp_sparse_plan(C, B, k, device=dev)
    sel_ids, sel_cnt, ws = cp.cp_sparse_topk(dplan, shard_scores, k)
    selk, selsc, pc = cp.cp_sparse_gather(dplan, k, ws, shards, scales)
    Hr, Dv = m["H"], m["Dv"]
    o_part = torch.empty((C, B, Hr, Dv), dtype=torch.float32, device=dev)
    lse_part = torch.empty((C, B, Hr), dtype=torch.float32, device=dev)
    o_dec = torch.empty((B, Hr, Dv), dtype=torch.bfloat16, device=dev)
    lse_dec = torch.empty((B, Hr), dtype=torch.float32, device=dev)
    dws = torch.empty(max(16, cp.cp_decode_workspace_size(splan, Hr, Dv)), dtype=torch.uint8, device=dev)
    mws = torch.empty(max(16, cp.cp_decode_merged_workspace_size(
        splan, cp.CP_DECODE_MLA, cp.CP_FP8_E4M3 if fp8 else cp.CP_BF16, Hr, Dv)), dtype=torch.uint8, device=dev)
    o_one = torch.empty_like(o_dec)
    lse_one = torch.empty_like(lse_dec)
    scale = 1.0 / math.sqrt(m["Dqk"])
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step(e, one_call):
        e[0].record(stream)
        cp.cp_sparse_topk(dplan, shard_scores, k, sel_ids, sel_cnt, ws)
        e[1].record(stream)
        cp.cp_sparse_gather(dplan, k, ws, shards, scales, selk, selsc, pc)
        e[2].record(stream)
        if one_call:  # the attention and the merge in one call
            cp.cp_sparse_decode_attn_merged(splan, pc, cp.CP_DECODE_MLA, dq, selk, sel_scale=selsc,
                                            sm_scale=scale, o=o_one, lse=lse_one, ws=mws)
        else:
            cp.cp_sparse_decode_attn(splan, pc, cp.CP_DECODE_MLA, dq, selk, sel_scale=selsc,
                                     sm_scale=scale, o_part=o_part, lse_part=lse_part, ws=dws)
        e[3].record(stream)
        if not one_call:
            cp.cp_lse_merge(o_part, lse_part, out=o_dec, lse=lse_dec)
        e[4].record(stream)

    def timed(one_call):
        for _ in range(max(3, args.warmup)):
            step([ev() for _ in range(5)], one_call)
        torch.cuda.synchronize(dev)
        cp.cp_device_error_check(dev)
        recs = [[ev() for _ in range(5)] for _ in range(args.steps)]
        barrier(world)
        for i in range(args.steps):
            step(recs[i], one_call)
        torch.cuda.synchronize(dev)
        barrier(world)
        cp.cp_device_error_check(dev)
        return [[r[i].elapsed_time(r[i + 1]) for r in recs] for i in range(4)]

    stage = timed(False)
    stage_one = timed(True)  # a loop of its own: the two paths do not share a step
    total = max_over_ranks(sum(sum(x) for x in stage), world)
    total_one = max_over_ranks(sum(sum(x) for x in stage_one), world)
    row = 580 if fp8 else 1152
    alg = 4 * sum(ctx) + B * k * row + B * Hr * 576 * 2 + B * Hr * 512 * 2
    return {"k": k, "workload": f"{B} x {L} tokens, C={C}, top-{k} of per-token fp32 scores, "
                                f"MLA {'FP8' if fp8 else 'bf16'} rows",
            "ms": {"topk": statistics.mean(stage[0]), "gather": statistics.mean(stage[1]),
                   "decode": statistics.mean(stage[2]), "merge": statistics.mean(stage[3]),
                   "decode_and_merge_one_call": statistics.mean(stage_one[2])},
            "value_one_call": whole_job_rate(alg * args.steps, total_one, world) / 1e9,
            "algorithmic_bytes_per_step": alg,
            "value": whole_job_rate(alg * args.steps, total, world) / 1e9, "unit": "GB/s",
            "note": "scores read once + selected rows once + Q + O over the time of all four stages; "
                    "value_one_call: top-k + gather + cp_sparse_decode_attn_merged"}


def time_region(dev, stream, world, step, steps, warmup):
    """W untimed steps, then K steps, each bracketed by CUDA events on the
    launch stream, between a barrier and a synchronize on both sides; clocks
    sampled by nvidia-smi meanwhile.  Returns (per-step records, clocks)."""
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    for _ in range(warmup):
        step(None)
    torch.cuda.synchronize(dev)
    recs = [None] * steps
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    for i in range(steps):
        recs[i] = step(ev)
    torch.cuda.synchronize(dev)
    barrier(world)
    return recs, clocks.stop()


def leg_prefill_interleave(cp, args, dev, stream, world, rank, peaks, peak_kind):
    """The ragged interleave prefill (16 requests, 2^20 tokens, 64 q / 8 kv
    heads): shard plan + prefill per step, against the sustained tensor peak
    (one launch lasts over a second)."""
    z = W.WORKLOADS["interleave"]
    nl = W.interleave_lengths()
    pl = [0] * len(nl)
    Hq, Hkv, D, C = z["Hq"], z["Hkv"], z["D"], z["C"]
    q, k, v = W.prefill_inputs(nl, pl, Hq, Hkv, D, "bf16", seed=W.SEEDS["interleave"] + rank, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((q.shape[0], Hq), dtype=torch.float32, device=dev)
    flops, _ = prefill_flops(nl, pl, Hq, D)
    scale = 1.0 / math.sqrt(D)

    def step(ev):
        e = [ev() for _ in range(3)] if ev else None
        if e:
            e[0].record(stream)
        plan = cp.cp_shard_plan(cp.CP_INTERLEAVE, C, nl, pl, device=dev)
        if e:
            e[1].record(stream)
        cp.cp_prefill_attn(plan, q, k, v, scale, out=o, lse=lse)
        if e:
            e[2].record(stream)
        return e

    steps = max(1, min(args.steps, args.leg_steps_long))
    recs, clk = time_region(dev, stream, world, step, steps, max(3, min(args.warmup, 3)))
    cp.cp_device_error_check(dev)
    plan_ms = [r[0].elapsed_time(r[1]) for r in recs]
    pre_ms = [r[1].elapsed_time(r[2]) for r in recs]
    total = max_over_ranks(sum(plan_ms) + sum(pre_ms), world)
    ach = flops / (statistics.mean(pre_ms) / 1e3) / 1e12
    peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    del q, k, v, o, lse
    torch.cuda.empty_cache()
    out = {"workload": PREFILL_WORKLOADS["interleave"], "lengths": {"requests": len(nl), "tokens": sum(nl),
                                                                  "median": int(statistics.median(nl))},
           "metric": "prefill causal-attn TFLOP/s", "unit": "TFLOP/s",
           "value": whole_job_rate(flops * steps, total, world) / 1e12,
           "steps": steps, "ms_plan": statistics.mean(plan_ms), "ms_prefill": statistics.mean(pre_ms),
           "flops_per_step": flops, "gpu_launches": 2 * steps,
           "roofline": {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                        "frac": ach / peak, "traffic": None,
                        "peak_kind": peak_kind + " sustained", "kernel": "prefill_tc_kernel<128>"},
           "clocks": clk}
    if not args.no_cpu and rank == 0:
        o_s = oracle_prefill_sample("interleave", rows_per_call=32, budget_s=args.cpu_budget)
        out["cpu_baseline"] = {
            "value": o_s["tflops"], "unit": "TFLOP/s", "cores": o_s["cores"], "kind": "oracle",
            "sample": f"{o_s['rows']} query rows x {Hq} heads, late rows of the longest request, fp64 "
                      f"numpy, {o_s['seconds']:.1f} s; the whole prefill extrapolates to "
                      f"{o_s['full_s']:.0f} s (extrapolated)"}
    return out


def leg_decode(cp, args, dev, stream, world, rank, peaks, peak_kind, workload, fp8, merged=False):
    """MLA decode of one of the decode workloads (plan + split-KV decode + LSE
    merge per step, or with merged: plan + cp_decode_attn_merged) from
    per-shard buffers packed once before timing."""
    m = W.WORKLOADS[workload]
    ctx = W.mixed_context_lengths() if workload == "mla_mixed" else [m["ctx"]] * m["B"]
    data = W.mla_decode_inputs(ctx, H=m["H"], seed=W.SEEDS[workload] + rank, device=dev,
                               bf16=not fp8, fp8=fp8)
    plan = cp.cp_decode_plan(m["C"], ctx, device=dev)
    if fp8:
        shards, scales = cp.cp_kv_shard_pack(plan, data["kv_fp8"], data["kv_scale"])
        del data["kv_fp8"], data["kv_scale"]
    else:
        shards, scales = cp.cp_kv_shard_pack(plan, data["kv_bf16"])
        del data["kv_bf16"]
    torch.cuda.empty_cache()
    dq = data["q"]
    B, H, Dv, C = len(ctx), m["H"], m["Dv"], m["C"]
    o_part = torch.empty((C, B, H, Dv), dtype=torch.float32, device=dev)
    lse_part = torch.empty((C, B, H), dtype=torch.float32, device=dev)
    o_dec = torch.empty((B, H, Dv), dtype=torch.bfloat16, device=dev)
    lse_dec = torch.empty((B, H), dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, cp.cp_decode_workspace_size(plan, H, Dv)), dtype=torch.uint8, device=dev)
    kv_code = cp.CP_FP8_E4M3 if fp8 else cp.CP_BF16
    ws_m = (torch.empty(max(16, cp.cp_decode_merged_workspace_size(plan, cp.CP_DECODE_MLA, kv_code, H, Dv)),
                        dtype=torch.uint8, device=dev) if merged else None)
    scale = 1.0 / math.sqrt(m["Dqk"])
    nbytes = decode_bytes(ctx, H, fp8=fp8)

    def step(ev):
        e = [ev() for _ in range(4)] if ev else None
        if e:
            e[0].record(stream)
        dp = cp.cp_decode_plan(C, ctx, device=dev)
        if e:
            e[3].record(stream)  # the plan is built and copied: the decode kernels start here
        if merged:
            cp.cp_decode_attn_merged(dp, cp.CP_DECODE_MLA, dq, shards, shard_scale=scales, sm_scale=scale,
                                     o=o_dec, lse=lse_dec, ws=ws_m)
        else:
            cp.cp_decode_attn(dp, cp.CP_DECODE_MLA, dq, shards, shard_scale=scales, sm_scale=scale,
                              o_part=o_part, lse_part=lse_part, ws=ws)
        if e:
            e[1].record(stream)
        if not merged:
            cp.cp_lse_merge(o_part, lse_part, out=o_dec, lse=lse_dec)
        if e:
            e[2].record(stream)
        return e

    steps = max(1, min(args.steps, args.leg_steps))
    recs, clk = time_region(dev, stream, world, step, steps, max(3, args.warmup))
    cp.cp_device_error_check(dev)
    dec_ms = [r[0].elapsed_time(r[1]) for r in recs]
    mrg_ms = [r[1].elapsed_time(r[2]) for r in recs]
    dk_ms = [r[3].elapsed_time(r[1]) for r in recs]  # the decode kernels alone, without the plan
    total = max_over_ranks(sum(dec_ms) + sum(mrg_ms), world)
    ach = nbytes / (statistics.mean(dk_ms) / 1e3) / 1e9
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    if merged:  # decode (+ the runs' parts merge, when a request is cut by a worker boundary)
        n_k = 1 + (1 if len(plan.merge_list) else 0) if fp8 else 2 + (1 if plan.n_split > 0 else 0)
    else:
        n_k = 2 + (1 if plan.n_split > 0 else 0)
    traffic_key = ("decode_fp8_merged" if merged else "decode_fp8") if fp8 else "decode_bf16"
    out = {"workload": (DECODE_WORKLOADS["mixed"] if workload == "mla_mixed" else DECODE_WORKLOADS["uniform"]),
           "api": ("cp_decode_attn_merged (ms_decode: decode and merge in one call)" if merged
                   else "cp_decode_attn + cp_lse_merge"),
           "kv": "fp8" if fp8 else "bf16", "metric": "decode KV HBM GB/s", "unit": "GB/s",
           "context": {"requests": B, "tokens": sum(ctx), "median": int(statistics.median(ctx)),
                       "min": min(ctx), "max": max(ctx)},
           "value": whole_job_rate(nbytes * steps, total, world) / 1e9, "steps": steps,
           "ms_decode": statistics.mean(dec_ms), "ms_decode_kernels": statistics.mean(dk_ms),
           "ms_merge": statistics.mean(mrg_ms),
           "merge_share": statistics.mean(mrg_ms) / (statistics.mean(dec_ms) + statistics.mean(mrg_ms)),
           "bytes_per_step": nbytes, "gpu_launches": n_k * steps,
           "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                        "traffic": (profiled_traffic(traffic_key, sum(ctx))
                                    if workload == "mla" and (fp8 or not merged) else None),
                        "peak_kind": peak_kind,
                        "kernel": "decode_mla_fp8_kernel" if fp8 else "decode_mla_tc_kernel"},
           "clocks": clk}
    del shards, scales, o_part, lse_part, o_dec, lse_dec, ws, ws_m, data
    torch.cuda.empty_cache()
    if not args.no_cpu and rank == 0 and not merged:  # the merged legs run the same workloads
        one = sorted(ctx)[len(ctx) // 2]  # the median request
        gbs, sec, cores = oracle_decode_sample(one, workload, fp8)
        out["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                               "sample": f"1 request of {one} {'FP8' if fp8 else 'bf16'} tokens (the "
                                         f"batch's median), 64 heads, fp64 numpy, {sec:.1f} s; the "
                                         f"whole batch extrapolates to {sec * sum(ctx) / one:.0f} s "
                                         "(extrapolated)"}
    return out


def leg_tiny(cp, args, dev, stream, world, rank):
    """The tiny workload as one step: zigzag plan + fp32 prefill over 4
    shards, decode plan + GQA decode of the 257-token cache over 4
    token-interleaved shards (packed before timing) + LSE merge."""
    w = W.WORKLOADS["tiny"]
    t = W.tiny_inputs(device=dev)
    scale = 1.0 / math.sqrt(w["D"])
    dplan = cp.cp_decode_plan(w["C"], t["ctx"], device=dev)
    sk, _ = cp.cp_kv_shard_pack(dplan, t["dec_k"])
    sv, _ = cp.cp_kv_shard_pack(dplan, t["dec_v"])
    pflops, _ = prefill_flops(w["new_len"], w["prefix_len"], w["Hq"], w["D"])
    dbytes = 2 * w["decode_ctx"] * w["Hkv"] * w["D"] * 4 + 2 * w["Hq"] * w["D"] * 4

    def step(ev):
        e = [ev() for _ in range(3)] if ev else None
        if e:
            e[0].record(stream)
        plan = cp.cp_shard_plan(cp.CP_ZIGZAG, w["C"], w["new_len"], w["prefix_len"], device=dev)
        cp.cp_prefill_attn(plan, t["q"], t["k"], t["v"], scale)
        if e:
            e[1].record(stream)
        dp = cp.cp_decode_plan(w["C"], t["ctx"], device=dev)
        op, lp = cp.cp_decode_attn(dp, cp.CP_DECODE_GQA, t["dec_q"], sk, sv, sm_scale=scale)
        cp.cp_lse_merge(op, lp, out_dtype=torch.float32)
        if e:
            e[2].record(stream)
        return e

    steps = max(1, min(args.steps, 50))
    recs, clk = time_region(dev, stream, world, step, steps, max(3, args.warmup))
    cp.cp_device_error_check(dev)
    pre = [r[0].elapsed_time(r[1]) for r in recs]
    dec = [r[1].elapsed_time(r[2]) for r in recs]
    total = max_over_ranks(sum(pre) + sum(dec), world)
    out = {"workload": "tiny: 256-token fp32 prompt, GQA 8q/2kv, D 64, zigzag CP=4; decode of the "
                       "257-token cache over 4 token-interleaved shards + LSE merge",
           "metric": "ms per step (prefill + decode)", "unit": "ms", "higher_is_better": False,
           "value": total / steps, "steps": steps,
           "ms_prefill": statistics.mean(pre), "ms_decode": statistics.mean(dec),
           "prefill_tflops": pflops / (statistics.mean(pre) / 1e3) / 1e12,
           "decode_gbs": dbytes / (statistics.mean(dec) / 1e3) / 1e9,
           "gpu_launches": 5 * steps, "clocks": clk,
           "note": "launch-bound: 2.7e8 FLOP and 0.26 MB per step; no roofline is meaningful at this size"}
    if not args.no_cpu and rank == 0:
        sec, cores = oracle_tiny()
        out["cpu_baseline"] = {"value": sec * 1e3, "unit": "ms", "cores": cores, "kind": "oracle",
                               "sample": "the whole tiny workload (prefill of all 4 shards + the decode), "
                                         "fp64 numpy"}
    return out


def decode_e2e(cp, args, dev, stream, world, ctx, m, dq, shards, scales, dscale, d_bytes):
    """The decode step end to end through the binding with host buffers:
    every step uploads the decode query from pinned host memory, builds the
    decode plan on the host and copies it up, runs the decode and the LSE
    merge, and reads the merged O and LSE back into pinned host memory.  The
    copies run on two copy streams with double-buffered device buffers, so
    step i + 1's upload and step i - 1's download overlap step i."""
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    B, H, Dv, C = len(ctx), m["H"], m["Dv"], m["C"]
    qh = dq.cpu().pin_memory()
    dqs = [torch.empty_like(dq) for _ in range(2)]
    o_part = torch.empty((C, B, H, Dv), dtype=torch.float32, device=dev)
    lse_part = torch.empty((C, B, H), dtype=torch.float32, device=dev)
    outs = [(torch.empty((B, H, Dv), dtype=torch.bfloat16, device=dev),
             torch.empty((B, H), dtype=torch.float32, device=dev)) for _ in range(2)]
    hosts = [(torch.empty((B, H, Dv), dtype=torch.bfloat16).pin_memory(),
              torch.empty((B, H), dtype=torch.float32).pin_memory()) for _ in range(2)]
    probe = cp.cp_decode_plan(C, ctx, device=dev)
    ws = torch.empty(max(16, cp.cp_decode_workspace_size(probe, H, Dv)), dtype=torch.uint8, device=dev)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(n):
        uploaded = [ev() for _ in range(n)]
        computed = [ev() for _ in range(n)]
        downloaded = [ev() for _ in range(n)]

        def upload(i):
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(computed[i - 2])
                dqs[i % 2].copy_(qh, non_blocking=True)
                uploaded[i].record(up)

        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            stream.wait_event(uploaded[i])
            if i >= 2:
                stream.wait_event(downloaded[i - 2])
            dp = cp.cp_decode_plan(C, ctx, device=dev)
            cp.cp_decode_attn(dp, cp.CP_DECODE_MLA, dqs[i % 2], shards, shard_scale=scales,
                              sm_scale=dscale, o_part=o_part, lse_part=lse_part, ws=ws)
            od, ld = outs[i % 2]
            cp.cp_lse_merge(o_part, lse_part, out=od, lse=ld)
            computed[i].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[i])
                hosts[i % 2][0].copy_(od, non_blocking=True)
                hosts[i % 2][1].copy_(ld, non_blocking=True)
                downloaded[i].record(down)
        stream.wait_event(downloaded[n - 1])

    run(3)
    torch.cuda.synchronize(dev)
    n = args.steps + 2
    barrier(world)
    clk = ClockSampler(dev.index if dev.index is not None else 0)
    clk.start()
    a, b = ev(), ev()
    a.record(stream)
    run(n)
    b.record(stream)
    torch.cuda.synchronize(dev)
    info = clk.stop()
    ms = max_over_ranks(a.elapsed_time(b), world)
    h2d = dq.numel() * dq.element_size() + probe.dev.numel() * 4
    d2h = B * H * Dv * 2 + B * H * 4
    return {"value": whole_job_rate(d_bytes * n, ms, world) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n, "clocks": info,
            "note": "query uploaded from pinned host memory and the plan built on the host and copied "
                    "up every step; merged O and LSE read back to pinned host memory; copies on two "
                    "copy streams overlap the neighbouring steps (double-buffered); the KV cache "
                    "stays resident"}


def run_ours(args, world, rank, local):
    import __graft_entry__
    if rank == 0:
        __graft_entry__.ensure_built()  # rebuilds a library older than its sources
    barrier(world)
    import context_long_attention_gb300 as cp

    dev = torch.device("cuda", local if world > 1 else 0)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_kind = load_peaks()
    do_pre = args.only in ("all", "prefill")
    do_dec = args.only in ("all", "decode")

    # ---- prefill inputs (zigzag: one long request; interleave: the ragged batch)
    zz = args.prefill_workload == "zigzag"
    z = W.WORKLOADS[args.prefill_workload]
    if zz:
        nl, pl, strategy = z["new_len"], z["prefix_len"], cp.CP_ZIGZAG
    else:
        nl = W.interleave_lengths()
        pl, strategy = [0] * len(nl), cp.CP_INTERLEAVE
    C, Hq, Hkv, D = z["C"], z["Hq"], z["Hkv"], z["D"]
    scale = 1.0 / math.sqrt(D)
    p_flops, _ = prefill_flops(nl, pl, Hq, D)
    if do_pre:
        q, k, v = W.prefill_inputs(nl, pl, Hq, Hkv, D, "bf16", seed=W.SEEDS[args.prefill_workload] + rank,
                                   device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((q.shape[0], Hq), dtype=torch.float32, device=dev)

    # ---- decode inputs (MLA latent cache, FP8 or bf16, or a GQA bf16 cache),
    # packed into token shards once
    dw = args.decode_workload
    gqa = dw == "gqa"
    uniform = dw == "uniform"
    m = W.WORKLOADS[{"uniform": "mla", "mixed": "mla_mixed", "gqa": "gqa_decode"}[dw]]
    if dw == "mixed":
        ctx = W.mixed_context_lengths()
        ctx = ctx[:args.decode_batch] if args.decode_batch else ctx
    else:
        ctx = [args.decode_ctx or m["ctx"]] * (args.decode_batch or m["B"])
    kv_kind = args.decode_kv or ("bf16" if gqa else "fp8")  # MLA defaults to FP8, GQA to bf16
    fp8 = kv_kind == "fp8"
    if gqa:
        if args.decode_paged or args.decode_rows > 1 or args.sparse_k:
            raise SystemExit("--decode-workload gqa times the one-row decode from per-shard buffers")
        d_bytes = gqa_decode_bytes(ctx, m["Hq"], m["Hkv"], m["D"], fp8=fp8)
        dscale = 1.0 / math.sqrt(m["D"])
    else:
        d_bytes = decode_bytes(ctx, m["H"], fp8=fp8)
        dscale = 1.0 / math.sqrt(m["Dqk"])
    n_dec_kernels = 0
    vshards = None
    if do_dec and gqa:
        Hr, Dv, s_q, pages, scales = m["Hq"], m["D"], 1, None, None
        layout = cp.CP_DCP_CONTIGUOUS if args.decode_layout == "contiguous" else cp.CP_DCP_ROUND_ROBIN
        B = len(ctx)
        if fp8:
            dq, kc, vc, kvs = W.gqa_decode_inputs_fp8(B, ctx, Hr, m["Hkv"], Dv, seed=W.SEEDS["gqa_decode"] + rank,
                                                      device=dev)
        else:
            dq, kc, vc = W.gqa_decode_inputs(B, ctx, Hr, m["Hkv"], Dv, "bf16",
                                             seed=W.SEEDS["gqa_decode"] + rank, device=dev)
            kvs = None
        dplan = cp.cp_decode_plan_ex(m["C"], ctx, layout=layout, s_q=1, device=dev)
        shards, scales = cp.cp_kv_shard_pack(dplan, kc, kvs)
        vshards, _ = cp.cp_kv_shard_pack(dplan, vc)
        del kc, vc
        lead = (B,)
    elif do_dec:
        Dv = m["Dv"]
        data = W.mla_decode_inputs(ctx, H=m["H"], seed=W.SEEDS["mla" if uniform else "mla_mixed"] + rank,
                                   device=dev,
                                   bf16=not fp8, fp8=fp8)
        layout = cp.CP_DCP_CONTIGUOUS if args.decode_layout == "contiguous" else cp.CP_DCP_ROUND_ROBIN
        s_q = args.decode_rows
        if s_q < 1 or m["H"] % s_q:
            raise SystemExit(f"--decode-rows must divide {m['H']}")
        Hr = m["H"] // s_q  # heads per query row: the s_q rows fill the kernels' 64 columns
        dplan = cp.cp_decode_plan_ex(m["C"], ctx, layout=layout, s_q=s_q, device=dev)
        kv, kv_scale = (data["kv_fp8"], data["kv_scale"]) if fp8 else (data["kv_bf16"], None)
        pages = None
        if args.decode_paged:
            # every (shard, request) pair's rows in pages of a shared pool, placed at random
            ps = args.decode_paged
            need = [-(-int(n) // ps) for n in dplan.pairs[:, 0]]
            ids = np.random.default_rng(W.SEEDS["mla"] + rank).permutation(sum(need))
            table = np.full((len(need), max(need)), -1, np.int32)
            k0 = 0
            for pr, n in enumerate(need):
                table[pr, :n] = ids[k0:k0 + n]
                k0 += n
            pages = cp.PageTable(table, ps, sum(need), device=dev)
            shards, scales = cp.cp_kv_shard_pack_paged(dplan, pages, kv, kv_scale)
        else:
            shards, scales = cp.cp_kv_shard_pack(dplan, kv, kv_scale)
        del kv, kv_scale, data["kv_fp8" if fp8 else "kv_bf16"]
        if fp8:
            del data["kv_scale"]
        B = len(ctx)
        dq = data["q"].reshape(B, s_q, Hr, m["Dqk"]) if s_q > 1 else data["q"]
        lead = (B, s_q) if s_q > 1 else (B,)
    if do_dec:
        o_part = torch.empty((m["C"], *lead, Hr, Dv), dtype=torch.float32, device=dev)
        lse_part = torch.empty((m["C"], *lead, Hr), dtype=torch.float32, device=dev)
        o_mrg = o_part.view(m["C"], B * s_q, Hr, Dv)
        lse_mrg = lse_part.view(m["C"], B * s_q, Hr)
        o_dec = torch.empty((B * s_q, Hr, Dv), dtype=torch.bfloat16, device=dev)
        lse_dec = torch.empty((B * s_q, Hr), dtype=torch.float32, device=dev)
        ws_bytes = cp.cp_decode_workspace_size(dplan, Hr, Dv)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        n_dec_kernels = 2 + (1 if dplan.n_split > 0 else 0)  # decode (+ split merge) + LSE merge
        if args.decode_merged:
            if args.decode_paged:
                raise SystemExit("--decode-merged takes per-shard buffers, not a paged pool")
            mode_code = cp.CP_DECODE_GQA if gqa else cp.CP_DECODE_MLA
            kv_code = cp.CP_FP8_E4M3 if fp8 else (cp.CP_FP32 if shards[0].dtype == torch.float32 else cp.CP_BF16)
            ws_m = torch.empty(max(16, cp.cp_decode_merged_workspace_size(dplan, mode_code, kv_code, Hr, Dv)),
                               dtype=torch.uint8, device=dev)
            merged_native = fp8 and not gqa
            # decode (+ the runs' merge), or decode (+ split merge) + LSE merge
            n_dec_kernels = (1 + (1 if len(dplan.merge_list) else 0)) if merged_native else n_dec_kernels
    torch.cuda.synchronize(dev)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step(rec):
        e0, e1, e2, e3, e4, e5 = rec
        e0.record(stream)
        if do_pre:
            plan = cp.cp_shard_plan(strategy, C, nl, pl, device=dev)
        e1.record(stream)
        if do_pre:
            cp.cp_prefill_attn(plan, q, k, v, scale, out=o, lse=lse)
        e2.record(stream)
        if do_dec:
            dp = cp.cp_decode_plan_ex(m["C"], ctx, layout=layout, s_q=s_q, device=dev)
        e5.record(stream)  # the decode plan is built and copied: the decode kernels start here
        if do_dec:
            if args.decode_merged:
                cp.cp_decode_attn_merged(dp, cp.CP_DECODE_GQA if gqa else cp.CP_DECODE_MLA, dq, shards,
                                         vshards if gqa else None, shard_scale=scales, sm_scale=dscale,
                                         o=o_dec.view(*lead, Hr, Dv), lse=lse_dec.view(*lead, Hr), ws=ws_m)
            elif pages is not None:
                cp.cp_decode_attn_paged(dp, pages, cp.CP_DECODE_MLA, dq, shards, scale_pool=scales,
                                        sm_scale=dscale, o_part=o_part, lse_part=lse_part, ws=ws)
            elif gqa:
                cp.cp_decode_attn(dp, cp.CP_DECODE_GQA, dq, shards, vshards, shard_scale=scales,
                                  sm_scale=dscale, o_part=o_part, lse_part=lse_part, ws=ws)
            else:
                cp.cp_decode_attn(dp, cp.CP_DECODE_MLA, dq, shards, shard_scale=scales,
                                  sm_scale=dscale, o_part=o_part, lse_part=lse_part, ws=ws)
        e3.record(stream)
        if do_dec and not args.decode_merged:
            cp.cp_lse_merge(o_mrg, lse_mrg, out=o_dec, lse=lse_dec)
        e4.record(stream)

    for _ in range(args.warmup):
        step([ev() for _ in range(6)])
    cp.cp_device_error_check(dev)
    torch.cuda.synchronize(dev)

    recs = [[ev() for _ in range(6)] for _ in range(args.steps)]
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    t_start, t_end = ev(), ev()
    t_start.record(stream)
    for i in range(args.steps):
        step(recs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clock_info = clocks.stop()
    cp.cp_device_error_check(dev)

    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    plan_ms = [r[0].elapsed_time(r[1]) for r in recs]
    pre_ms = [r[1].elapsed_time(r[2]) for r in recs]
    dec_ms = [r[2].elapsed_time(r[3]) for r in recs]
    dk_ms = [r[5].elapsed_time(r[3]) for r in recs]  # the decode kernels alone, without the plan
    mrg_ms = [r[3].elapsed_time(r[4]) for r in recs]
    # whole job: the work of all ranks over the slowest rank's time
    pre_total = max_over_ranks(sum(plan_ms) + sum(pre_ms), world)
    dec_total = max_over_ranks(sum(dec_ms) + sum(mrg_ms), world)
    value = whole_job_rate(p_flops * args.steps, pre_total, world) / 1e12 if do_pre else None
    dec_gbs = whole_job_rate(d_bytes * args.steps, dec_total, world) / 1e9 if do_dec else None

    # ---- end to end through the public API with host buffers (prefill).  Every
    # step copies its inputs from pinned host memory and its outputs back; the
    # copies run on two copy streams, double-buffered, so step i + 1's inputs
    # upload and step i - 1's outputs download while step i computes.
    e2e = None
    if do_pre and zz:
        qh = q.cpu().pin_memory()
        kh = k.cpu().pin_memory()
        vh = v.cpu().pin_memory()
        oh = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
        lh = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
        dev_in = [(torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)) for _ in range(2)]
        dev_out = [(torch.empty_like(o), torch.empty_like(lse)) for _ in range(2)]
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        n_e2e = args.steps + 2

        def run_e2e(n):
            uploaded = [ev() for _ in range(n)]
            computed = [ev() for _ in range(n)]
            downloaded = [ev() for _ in range(n)]

            def upload(i):
                with torch.cuda.stream(up):
                    if i >= 2:
                        up.wait_event(computed[i - 2])  # buffer i % 2 is free again
                    for d_, h_ in zip(dev_in[i % 2], (qh, kh, vh)):
                        d_.copy_(h_, non_blocking=True)
                    uploaded[i].record(up)

            upload(0)
            for i in range(n):
                if i + 1 < n:
                    upload(i + 1)
                stream.wait_event(uploaded[i])
                if i >= 2:
                    stream.wait_event(downloaded[i - 2])  # outputs i % 2 read back
                qd, kd, vd = dev_in[i % 2]
                od, ld = dev_out[i % 2]
                plan = cp.cp_shard_plan(cp.CP_ZIGZAG, C, nl, pl, device=dev)
                cp.cp_prefill_attn(plan, qd, kd, vd, scale, out=od, lse=ld)
                computed[i].record(stream)
                with torch.cuda.stream(down):
                    down.wait_event(computed[i])
                    oh[i % 2].copy_(od, non_blocking=True)
                    lh[i % 2].copy_(ld, non_blocking=True)
                    downloaded[i].record(down)
            stream.wait_event(downloaded[n - 1])

        # the copies' own rates, one upload and one download timed alone
        ca, cb, cc = ev(), ev(), ev()
        ca.record(up)
        with torch.cuda.stream(up):
            for d_, h_ in zip(dev_in[0], (qh, kh, vh)):
                d_.copy_(h_, non_blocking=True)
        cb.record(up)
        with torch.cuda.stream(up):
            oh[0].copy_(dev_out[0][0], non_blocking=True)
            lh[0].copy_(dev_out[0][1], non_blocking=True)
        cc.record(up)
        torch.cuda.synchronize(dev)
        h2d_bytes = q.numel() * 2 + k.numel() * 2 + v.numel() * 2
        d2h_bytes = o.numel() * 2 + lse.numel() * 4
        h2d_gbs = h2d_bytes / (ca.elapsed_time(cb) / 1e3) / 1e9
        d2h_gbs = d2h_bytes / (cb.elapsed_time(cc) / 1e3) / 1e9
        run_e2e(3)
        torch.cuda.synchronize(dev)
        barrier(world)
        e2e_clocks = ClockSampler(dev.index if dev.index is not None else 0)
        e2e_clocks.start()
        a, b = ev(), ev()
        a.record(stream)
        run_e2e(n_e2e)
        b.record(stream)
        torch.cuda.synchronize(dev)
        e2e_clock_info = e2e_clocks.stop()
        e2e_ms = max_over_ranks(a.elapsed_time(b), world)
        e2e = {"value": whole_job_rate(p_flops * n_e2e, e2e_ms, world) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d_bytes,
               "d2h_bytes_per_step": d2h_bytes,
               "copy_gbs": {"h2d": h2d_gbs, "d2h": d2h_gbs},
               "clocks": e2e_clock_info,
               "steps": n_e2e,
               "note": "pinned host buffers; uploads and downloads on two copy streams overlap "
                       "the neighbouring steps' compute (double-buffered)"}

    # ---- sparse decode with an exact sharded top-k (timed on its own)
    sparse = None
    if do_dec and args.sparse_k:
        sparse = sparse_leg(cp, args, dev, stream, ctx, m, fp8, dplan, shards, scales, dq, world, rank)

    # ---- the decode half end to end through the binding with host buffers
    dec_e2e = None
    default_decode = (do_dec and uniform and fp8 and not args.decode_paged and args.decode_rows == 1
                      and args.decode_layout == "round_robin" and not args.decode_ctx
                      and not args.decode_batch and not args.decode_merged)
    if default_decode:
        dec_e2e = decode_e2e(cp, args, dev, stream, world, ctx, m, dq, shards, scales, dscale, d_bytes)

    # ---- the other workloads, each timed on its own (the default line only)
    legs = None
    if args.legs and args.only == "all" and zz and default_decode and not args.sparse_k:
        del q, k, v, o, lse, shards, scales, o_part, lse_part, o_mrg, lse_mrg, o_dec, lse_dec, ws, dq
        if e2e is not None:
            del qh, kh, vh, oh, lh, dev_in, dev_out
        torch.cuda.empty_cache()
        legs = {"tiny": leg_tiny(cp, args, dev, stream, world, rank),
                "decode_bf16": leg_decode(cp, args, dev, stream, world, rank, peaks, peak_kind, "mla", False),
                "decode_mixed": leg_decode(cp, args, dev, stream, world, rank, peaks, peak_kind,
                                           "mla_mixed", True),
                "decode_merged": leg_decode(cp, args, dev, stream, world, rank, peaks, peak_kind, "mla", True,
                                            merged=True),
                "decode_mixed_merged": leg_decode(cp, args, dev, stream, world, rank, peaks, peak_kind,
                                                  "mla_mixed", True, merged=True),
                "prefill_interleave": leg_prefill_interleave(cp, args, dev, stream, world, rank, peaks,
                                                             peak_kind)}

    if rank != 0:
        return
    # the tensor peak: the burst figure, or the sustained one (under the power
    # cap) when the timed prefill work lasts more than a second
    sustained = do_pre and sum(pre_ms) > 1000.0
    peak_key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    peak = float(peaks.get(peak_key, FALLBACK_PEAKS[peak_key]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    roof = dec = None
    if do_pre:
        pre_avg = statistics.mean(pre_ms)
        achieved = p_flops / (pre_avg / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": profiled_traffic("prefill") if zz else None,
                "peak_kind": peak_kind + (" sustained" if sustained else " burst"),
                "kernel": "prefill_tc_kernel<128>"}
    if do_dec:
        dec_avg = statistics.mean(dec_ms)
        dec_ach = d_bytes / (statistics.mean(dk_ms) / 1e3) / 1e9  # per launch of the decode kernels
        dec = {"metric": "decode KV HBM GB/s", "value": dec_gbs, "unit": "GB/s",
               "kv": kv_kind,
               "mode": "gqa" if gqa else "mla",
               "cache": (f"paged, {args.decode_paged}-row pages placed at random"
                         if args.decode_paged else "one contiguous buffer per shard"),
               "layout": args.decode_layout,
               "query_rows": args.decode_rows,
               "api": ("cp_decode_attn_merged (ms_decode: decode and merge)" if args.decode_merged
                       else "cp_decode_attn + cp_lse_merge"),
               "ms_decode": dec_avg, "ms_decode_kernels": statistics.mean(dk_ms),
               "ms_merge": statistics.mean(mrg_ms),
               "merge_share": statistics.mean(mrg_ms) / (dec_avg + statistics.mean(mrg_ms)),
               "roofline": {"bound": "hbm", "achieved": dec_ach, "peak": hbm, "unit": "GB/s",
                            "frac": dec_ach / hbm,
                            "traffic": (None if args.decode_paged or args.decode_rows > 1
                                        or args.decode_layout != "round_robin" or not (uniform or gqa)
                                        else profiled_traffic(("decode_gqa" + ("8" if fp8 else ""))
                                                              if gqa else "decode_" + kv_kind,
                                                              sum(ctx))),
                            "peak_kind": peak_kind}}
        if dec_e2e is not None:
            dec["e2e"] = dec_e2e
    cpu = None
    if not args.no_cpu:
        o_s = oracle_prefill_sample(args.prefill_workload, rows_per_call=32, budget_s=12.0)
        where = ("rank 0's late zigzag block" if zz else "late rows of the interleave batch's longest request")
        cpu = {"value": o_s["tflops"], "unit": "TFLOP/s", "cores": o_s["cores"], "kind": "oracle",
               "sample": f"{o_s['rows']} query rows x {Hq} heads of {where}, fp64 numpy, "
                         f"{o_s['seconds']:.1f} s; {o_s['pairs_per_s']:.3g} (query, key) head pairs/s; "
                         f"the whole prefill extrapolates to {o_s['full_s']:.0f} s (extrapolated)"}
        if do_dec and uniform and fp8:
            dec_gbs_cpu, dec_s, _ = oracle_decode_sample()
            cpu["decode"] = {"value": dec_gbs_cpu, "unit": "GB/s",
                             "sample": f"1 of the {len(ctx)} requests (131,072 FP8 tokens, 64 heads), fp64 "
                                       f"numpy, {dec_s:.1f} s; the whole batch extrapolates to "
                                       f"{dec_s * len(ctx):.0f} s"}
    line = {
        "metric": "prefill causal-attn TFLOP/s",
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": workload_name(args),
            "timed": args.only,
            "prefill_flops_per_step": p_flops,
            "decode_bytes_per_step": d_bytes,
            "l2": ("inputs larger than L2 (K/V 151 MB, Q 268 MB, FP8 cache 4.9 GB); no flush"
                   if zz and uniform else "inputs larger than L2; no flush"),
            "parallelism": "virtual CP=8 on each GPU; replicas across GPUs",
        },
        "decode": dec,
        "sparse_decode": sparse,
        "ms_breakdown": {"plan": statistics.mean(plan_ms), "prefill": statistics.mean(pre_ms),
                         "decode": statistics.mean(dec_ms), "merge": statistics.mean(mrg_ms)},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * ((2 if do_pre else 0) + n_dec_kernels),
        "clocks": clock_info,
        "legs": legs,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only", choices=["all", "prefill", "decode"], default="all",
                    help="time one half of the step (for profiler captures)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--decode-kv", choices=["fp8", "bf16"], default=None,
                    help="decode cache type (default: fp8 for the MLA workloads, bf16 for gqa)")
    ap.add_argument("--decode-paged", type=int, default=0, metavar="PAGE_ROWS",
                    help="decode from a paged pool with pages of this many rows (multiple of 64), "
                         "placed at random; 0 = one contiguous buffer per shard")
    ap.add_argument("--decode-layout", choices=["round_robin", "contiguous"], default="round_robin",
                    help="decode token shards: token p on shard p mod C, or C contiguous chunks")
    ap.add_argument("--decode-rows", type=int, default=1, metavar="S_Q",
                    help="query rows per request (MTP); the 64 heads split into S_Q rows of 64/S_Q")
    ap.add_argument("--decode-merged", action="store_true",
                    help="time the decode through cp_decode_attn_merged (decode and merge in one call)")
    ap.add_argument("--sparse-k", type=int, default=0, metavar="K",
                    help="also time sparse decode over the exact sharded top-K of per-token scores")
    ap.add_argument("--prefill-workload", choices=list(PREFILL_WORKLOADS), default="zigzag",
                    help="zigzag: one 32k request after a 4k prefix (the default line); interleave: "
                         "16 ragged requests, 2^20 tokens (about 1.3 s per step)")
    ap.add_argument("--decode-workload", choices=list(DECODE_WORKLOADS), default="uniform",
                    help="uniform: MLA 64 x 131072 (the default line); mixed: MLA 128 requests, "
                         "1k..1M; gqa: GQA 16 x 131072, 32 q / 8 kv heads, head dim 128")
    ap.add_argument("--decode-ctx", type=int, default=0, metavar="L",
                    help="cached tokens per request for the uniform and gqa decode workloads (0: 131072)")
    ap.add_argument("--decode-batch", type=int, default=0,
                    help="requests in the decode batch (0: the workload's 64); for profiler captures")
    ap.add_argument("--no-legs", dest="legs", action="store_false",
                    help="skip the other workloads' legs of the default line (tiny, bf16 and mixed "
                         "MLA decode, interleave prefill)")
    ap.add_argument("--leg-steps", type=int, default=20, help="timed steps of the decode legs (at most --steps)")
    ap.add_argument("--leg-steps-long", type=int, default=3,
                    help="timed steps of the interleave prefill leg (1.3 s each; at most --steps)")
    ap.add_argument("--cpu-budget", type=float, default=8.0,
                    help="seconds of oracle time for each leg's CPU baseline sample")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
