"""CPU tests of the C ABI: the library loads, exports every declared entry
point, validates arguments, and its host-side planning matches the oracle's
enumerated shard maps bit for bit (no GPU needed: plans are built host-only)."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cp():
    import __graft_entry__
    __graft_entry__.ensure_built()
    import context_long_attention_gb300 as cp
    return cp


def declared_functions():
    with open(os.path.join(ROOT, "include", "cpattn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cp_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(cp):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(cp.lib, n), n
    assert cp.lib.cp_version() == 1


def test_noalloc_scratch_size_matches_header(cp):
    with open(os.path.join(ROOT, "include", "cpattn.h")) as f:
        m = re.search(r"#define CP_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", f.read())
    assert m, "CP_NOALLOC_SCRATCH_BYTES not found in the header"
    assert cp.lib.cp_noalloc_scratch_bytes() == int(m.group(1)) << int(m.group(2))
    assert cp._binding.NOALLOC_SCRATCH_BYTES == cp.lib.cp_noalloc_scratch_bytes()


def expand_segments(plan):
    """(f, pos, req) of every rank-major row, from the host segment table."""
    T = plan.T
    f = np.full(T, -1, np.int64)
    pos = np.full(T, -1, np.int64)
    req = np.full(T, -1, np.int64)
    for s in plan.segments:
        d = dict(zip(cp_fields(), s))
        for i in range(d["count"]):
            row = d["local_start"] + i
            f[row] = d["first_f"] + i * d["stride"]
            pos[row] = d["first_pos"] + i * d["stride"]
            req[row] = d["req"]
    return f, pos, req


def cp_fields():
    from context_long_attention_gb300._binding import SEG_FIELDS
    return SEG_FIELDS


BATCHES = [
    ([16], [0], 4),
    ([5, 3], [0, 0], 4),
    ([19], [7], 4),
    ([3], [2], 4),
    ([0, 9, 1, 33], [4, 0, 11, 2], 3),
    ([100, 1, 0, 57, 256], [0, 13, 5, 0, 1000], 8),
    ([1000], [0], 1),
    ([7, 7, 7], [0, 0, 0], 64),
]


@pytest.mark.parametrize("new_len,prefix_len,C", BATCHES)
def test_host_plan_matches_oracle(cp, new_len, prefix_len, C):
    for strategy, ofn in ((cp.CP_ZIGZAG, oracle.zigzag_plan), (cp.CP_INTERLEAVE, oracle.interleave_plan)):
        plan = cp.cp_shard_plan(strategy, C, new_len, prefix_len, device=None)
        ref = ofn(new_len, prefix_len, C)
        f, pos, req = expand_segments(plan)
        ro = plan.rank_off
        for r in range(C):
            sl = slice(ro[r], ro[r + 1])
            assert list(f[sl]) == list(ref["order"][r])
            assert list(pos[sl]) == list(ref["pos"][r])
            assert list(req[sl]) == list(ref["req"][r])
        if strategy == cp.CP_ZIGZAG:
            got = []
            for s in plan.segments:
                d = dict(zip(cp_fields(), s))
                got.append((d["rank"], d["req"], d["which"], d["block"], d["q_start"], d["count"], d["kv_len"]))
            assert sorted(got) == sorted(ref["blocks"])
        # tiles cover every query exactly once, in both orders
        for tiles in (plan.tiles, plan.tiles_by_rank):
            seen = np.zeros(plan.T, np.int64)
            for seg, off in tiles:
                d = dict(zip(cp_fields(), plan.segments[seg]))
                n = min(256, d["count"] - off)
                seen[d["local_start"] + off:d["local_start"] + off + n] += 1
            assert np.all(seen == 1)


def test_host_plan_full_size_workloads(cp):
    import cp_workloads as W
    z = W.WORKLOADS["zigzag"]
    plan = cp.cp_shard_plan(cp.CP_ZIGZAG, z["C"], z["new_len"], z["prefix_len"])
    ref = oracle.zigzag_plan(z["new_len"], z["prefix_len"], z["C"])
    got = sorted((int(s[0]), int(s[1]), int(s[3]), int(s[2]), int(s[8]), int(s[5]), int(s[10])) for s in plan.segments)
    assert got == sorted(ref["blocks"])
    # rank r: early kv_len = 4096 + 2048 (r+1), late = 4096 + 2048 (16 - r)
    for s in plan.segments:
        r, which, count, kvl = int(s[0]), int(s[3]), int(s[5]), int(s[10])
        assert count == 2048
        assert kvl == 4096 + 2048 * ((r + 1) if which == 0 else (16 - r))
    lens = W.interleave_lengths()
    plan = cp.cp_shard_plan(cp.CP_INTERLEAVE, 8, lens, [0] * len(lens))
    ref = oracle.interleave_plan_np(lens, [0] * len(lens), 8)
    f, pos, req = expand_segments_fast(plan)
    ro = plan.rank_off
    for r in range(8):
        sl = slice(ro[r], ro[r + 1])
        assert np.array_equal(f[sl], ref["order"][r])
        assert np.array_equal(pos[sl], ref["pos"][r])
        assert np.array_equal(req[sl], ref["req"][r])


def expand_segments_fast(plan):
    T = plan.T
    f = np.empty(T, np.int64)
    pos = np.empty(T, np.int64)
    req = np.empty(T, np.int64)
    for s in plan.segments:
        d = dict(zip(cp_fields(), (int(x) for x in s)))
        i = np.arange(d["count"])
        rows = d["local_start"] + i
        f[rows] = d["first_f"] + i * d["stride"]
        pos[rows] = d["first_pos"] + i * d["stride"]
        req[rows] = d["req"]
    return f, pos, req


@pytest.mark.parametrize("ctx,C,G", [([257], 4, 3), ([0, 1, 5, 1000, 3], 4, 7), ([131072] * 4, 8, 148),
                                     ([2, 2], 8, 4), ([300000, 1024, 70000], 8, 16)])
def test_decode_plan_matches_shard_map_and_covers_rows(cp, ctx, C, G):
    plan = cp.cp_decode_plan(C, ctx, n_workers=G, device=None)
    B = len(ctx)
    pairs = plan.pairs
    for r in range(C):
        off = 0
        for b in range(B):
            shard, row = oracle.decode_shard_map(ctx[b], C)
            rows = sum(1 for s in shard if s == r)
            p = pairs[r * B + b]
            assert p[0] == rows and p[1] == off and p[2] == ctx[b]
            off += rows
    covered = [np.zeros(int(p[0]), np.int64) for p in pairs]
    parts = {}
    for pair, rb, re_, part in plan.work:
        covered[pair][rb:re_] += 1
        parts.setdefault(int(pair), []).append(int(part))
        assert rb % 128 == 0
    for i, c in enumerate(covered):
        assert np.all(c == 1)
        ps = parts[i]
        if len(ps) == 1:
            assert ps == [-1] and pairs[i][3] == 1
        else:
            first = int(pairs[i][4])
            assert sorted(ps) == list(range(first, first + len(ps)))
    # balance: a worker's cost (its tiles plus ITEM_COST per nonempty item) is
    # within ITEM_COST + 1 of an even share of the total
    ITEM_COST = 2
    tiles, cost = [0] * G, [0] * G
    wo = plan.worker_off
    for w in range(G):
        for pair, rb, re_, part in plan.work[wo[w]:wo[w + 1]]:
            nt = (re_ - rb + 127) // 128
            tiles[w] += nt
            cost[w] += nt + (ITEM_COST if nt else 0)
    NT = sum((int(p[0]) + 127) // 128 for p in pairs)
    total = NT + ITEM_COST * sum(1 for p in pairs if p[0] > 0)
    assert sum(tiles) == NT
    assert max(abs(c - total / G) for c in cost) <= ITEM_COST + 1


def test_argument_validation(cp):
    with pytest.raises(cp.CpError, match="INVALID_ARG"):
        cp.cp_shard_plan(cp.CP_ZIGZAG, 0, [4], [0])
    with pytest.raises(cp.CpError, match="INVALID_ARG"):
        cp.cp_shard_plan(cp.CP_ZIGZAG, 65, [4], [0])
    with pytest.raises(cp.CpError, match="INVALID_ARG"):
        cp.cp_shard_plan(cp.CP_INTERLEAVE, 2, [4, -1], [0, 0])
    with pytest.raises(cp.CpError, match="INVALID_ARG"):
        cp.cp_shard_plan(7, 2, [4], [0])
    with pytest.raises(cp.CpError, match="INVALID_ARG"):
        cp.cp_decode_plan(4, [10, -2], n_workers=4)
    lib = cp.lib
    # null pointers and bad plans are rejected before any launch
    assert lib.cp_prefill_attn(None, None, -1, 0, None, None, None, 8, 2, 64, 0.1, None, None, None) == -1
    bogus = np.zeros(64, np.int32)
    st = lib.cp_decode_attn(bogus.ctypes.data_as(ctypes.c_void_p), None, 1, 0, None, None, None, None,
                            64, 1, 576, 512, 0.1, None, None, None, 0, None)
    assert st == -1 and b"magic" in lib.cp_last_error()
    assert lib.cp_lse_merge(0, 1, 1, 4, None, None, None, 0, None, None) == -1
    assert lib.cp_lse_merge(2, 1, 1, 6, None, None, None, 0, None, None) == -1


def test_paged_argument_validation(cp):
    """Page tables are checked on their host copy before any launch."""
    plan = cp.cp_decode_plan(2, [5, 0, 130], n_workers=3)  # shard rows [3, 0, 65] and [2, 0, 65]
    lib = cp.lib
    fake = ctypes.c_void_p(256)  # never dereferenced: every case fails before a launch
    good = np.array([[0, -1], [-1, -1], [1, 2], [3, -1], [-1, -1], [4, 5]], np.int32)

    def pack(table, max_pages, page_size, num_pages):
        t = np.ascontiguousarray(table, dtype=np.int32)
        return lib.cp_kv_shard_pack_paged(plan.host.ctypes.data_as(ctypes.c_void_p), fake, cp.CP_BF16, fake,
                                          None, 576, fake, None, t.ctypes.data_as(ctypes.c_void_p), fake,
                                          max_pages, page_size, num_pages, None)

    def decode(table, max_pages, page_size, num_pages):
        t = np.ascontiguousarray(table, dtype=np.int32)
        return lib.cp_decode_attn_paged(plan.host.ctypes.data_as(ctypes.c_void_p), fake, cp.CP_DECODE_MLA,
                                        cp.CP_BF16, fake, fake, None, None, t.ctypes.data_as(ctypes.c_void_p),
                                        fake, max_pages, page_size, num_pages, 64, 1, 576, 512, 0.04, fake,
                                        fake, None, 0, None)

    assert pack(good, 2, 96, 6) == -2 and b"multiple of 64" in lib.cp_last_error()
    bad = good.copy(); bad[5, 1] = 6
    assert pack(bad, 2, 64, 6) == -1 and b"outside [0, 6)" in lib.cp_last_error()
    assert decode(bad, 2, 64, 6) == -1 and b"outside [0, 6)" in lib.cp_last_error()
    assert pack(good[:, :1], 1, 64, 6) == -1 and b"needs 2 pages" in lib.cp_last_error()
    dup = good.copy(); dup[3, 0] = 1
    assert pack(dup, 2, 64, 6) == -1 and b"used twice" in lib.cp_last_error()
    assert decode(good, 2, 64, 0) == -1 and b"num_pages=0" in lib.cp_last_error()


@pytest.mark.parametrize("ctx,C", [([0, 1, 10, 129, 4100], 4), ([3, 8, 1000], 8), ([5], 1)])
def test_contiguous_decode_plan_matches_oracle_map(cp, ctx, C):
    """Pair rows and the row -> token map of a contiguous-layout plan against
    the oracle's enumeration of the chunks."""
    plan = cp.cp_decode_plan_ex(C, ctx, layout=cp.CP_DCP_CONTIGUOUS, n_workers=7, device=None)
    assert plan.layout == 1 and plan.query_rows == 1
    B = len(ctx)
    for r in range(C):
        off = 0
        for b in range(B):
            shard, row = oracle.decode_shard_map_contiguous(ctx[b], C)
            toks = [p for p in range(ctx[b]) if shard[p] == r]
            rows, row_off, L, _, _, tok0, step, _ = plan.pairs[r * B + b]
            assert rows == len(toks) and row_off == off and L == ctx[b]
            # row i holds token tok0 + i * step
            assert [tok0 + i * step for i in range(rows)] == toks
            off += rows
    covered = [np.zeros(int(p[0]), np.int64) for p in plan.pairs]
    for pair, rb, re_, _ in plan.work:
        covered[pair][rb:re_] += 1
    assert all(np.all(c == 1) for c in covered)


def test_round_robin_pairs_record_token_map(cp):
    ctx, C = [0, 7, 300], 4
    plan = cp.cp_decode_plan_ex(C, ctx, layout=cp.CP_DCP_ROUND_ROBIN, n_workers=5, device=None)
    for r in range(C):
        for b in range(len(ctx)):
            shard, _ = oracle.decode_shard_map(ctx[b], C)
            rows, _, _, _, _, tok0, step, _ = plan.pairs[r * len(ctx) + b]
            assert [tok0 + i * step for i in range(rows)] == [p for p in range(ctx[b]) if shard[p] == r]


def test_decode_plan_ex_validation(cp):
    with pytest.raises(cp.CpError):
        cp.cp_decode_plan_ex(4, [10], layout=2)
    for s_q in (0, 65):
        with pytest.raises(cp.CpError):
            cp.cp_decode_plan_ex(4, [100], s_q=s_q)
    with pytest.raises(cp.CpError):  # a request shorter than its query rows
        cp.cp_decode_plan_ex(4, [10, 2], s_q=3)
    plan = cp.cp_decode_plan_ex(4, [10, 3], s_q=3, n_workers=5)
    assert plan.query_rows == 3 and plan.layout == 0


def test_sparse_plan_and_argument_validation(cp):
    splan = cp.cp_sparse_plan(4, 3, 16, n_workers=5)
    assert splan.layout == cp.CP_DCP_SELECTED
    # every (shard, request) pair has room for kp = 128 rows at row b kp of its shard
    for r in range(4):
        for b in range(3):
            rows, row_off = splan.pairs[r * 3 + b, :2]
            assert rows == 128 and row_off == 128 * b
    assert cp.sparse_slot_rows(512) == 512 and cp.sparse_slot_rows(513) == 640
    for k in (0, 4097):
        with pytest.raises(cp.CpError, match="INVALID_ARG"):
            cp.cp_sparse_plan(4, 3, k, n_workers=5)
    with pytest.raises(cp.CpError, match="INVALID_ARG"):  # top-k runs on a cache plan
        cp.cp_sparse_workspace_size(splan, 16)
    with pytest.raises(cp.CpError, match="INVALID_ARG"):  # selection plans come from cp_sparse_plan
        cp.cp_decode_plan_ex(4, [10], layout=cp.CP_DCP_SELECTED, n_workers=5)
    mtp = cp.cp_decode_plan_ex(4, [10, 12], s_q=2, n_workers=5)
    with pytest.raises(cp.CpError, match="UNSUPPORTED"):
        cp.cp_sparse_workspace_size(mtp, 8)
    plan = cp.cp_decode_plan_ex(4, [10, 12], n_workers=5)
    assert cp.cp_sparse_workspace_size(plan, 8) >= 4 * 2 * 8 * 8
