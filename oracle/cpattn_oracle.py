"""fp64 CPU oracle for context-parallel attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code, table or
helper with the CUDA library; the only thing both sides share is the seeded
input generator module ``cp_workloads``, which holds no attention arithmetic.

Every function is the plain definition from the pages, written out in fp64
with numpy (a matrix product is the only library primitive used as a step).
There is no tiling, no online softmax and no reordering beyond the
definitions.  Sources, cited by page title and section:

* [CTX]  "How GPUs Share a Long Context During LLM Inference"
         (vincentzed.com/writing/context-parallelism)
* [SGL]  SGLang documentation, "Prefill context parallelism" page
         (docs.sglang.io/docs/advanced_features/prefill_cp)
* [V4]   "DeepSeek-V4 Attention Inference Systems", §5 "Decode CP: Shard
         Cache, Do Not Reconstruct It"
* [GLM]  vLLM blog "GLM-5.3 Part 2: PCP, DCP and Hybrid HiSparse on 16 H200",
         footnote 1 (MLA: QK over 576 dims, PV over 512)

Readings taken where the pages are silent:

* zigzag remainder: the first ``n mod 2C`` blocks (in block order) get one
  extra token ([SGL] "early blocks receive the remainder");
* zigzag local order per rank: request by request, block r then block 2C-1-r;
* interleave local order: ascending flattened index, no padding;
* GQA head mapping: consecutive groups, q head h reads kv head h // (Hq/Hkv);
* LSE is the natural log; an empty key set has O = 0 and LSE = -inf;
* MLA value = the first 512 of the 576 latent dims ([GLM] footnote 1);
* FP8: one fp32 scale per cached token for all its dims.
"""

from __future__ import annotations

import math

import numpy as np

# --------------------------------------------------------------------------
# Shard maps (integer work): enumeration straight from the rule text.
# --------------------------------------------------------------------------


def zigzag_block_bounds(n_new: int, C: int) -> list[tuple[int, int]]:
    """[start, end) of each of the 2C contiguous blocks of one request.

    [SGL] "Zigzag strategy": split the request's newly extended tokens into
    2C contiguous blocks; early blocks receive the remainder.
    """
    nb = 2 * C
    base, rem = divmod(n_new, nb)
    bounds = []
    start = 0
    for b in range(nb):
        size = base + (1 if b < rem else 0)
        bounds.append((start, start + size))
        start += size
    assert start == n_new
    return bounds


def zigzag_plan(new_len, prefix_len, C: int) -> dict:
    """Zigzag shard map for a batch.

    [CTX] §2.3 "Zigzag": 2C blocks, GPU r takes block r and block 2C-1-r;
    [SGL] "Zigzag strategy": the split restarts for every request, and the
    metadata records q and kv lengths of the early and late block including
    the cached prefix ([CTX] §2.3: both blocks still read the cached part; a
    block's reads end at its last token).

    Returns a dict with
      ``order[r]``   flattened new-token indices owned by rank r, local order;
      ``req[r]``, ``pos[r]``  request id and position (prefix included) of
                     each owned query; its causal extent is pos + 1;
      ``blocks``     list of (rank, req, which, block, q_start, q_len, kv_len)
                     with which = 0 for the early block, 1 for the late one,
                     q_start an offset into the request's new tokens and
                     kv_len = prefix + block end.
    """
    R = len(new_len)
    owner_of_block = {}
    for b in range(2 * C):
        # rank r owns blocks r and 2C-1-r
        for r in range(C):
            if b == r or b == 2 * C - 1 - r:
                owner_of_block[b] = r
    order = [[] for _ in range(C)]
    req = [[] for _ in range(C)]
    pos = [[] for _ in range(C)]
    blocks = []
    q_base = 0
    for j in range(R):
        n, pre = int(new_len[j]), int(prefix_len[j])
        bounds = zigzag_block_bounds(n, C)
        for r in range(C):
            mine = [b for b in range(2 * C) if owner_of_block[b] == r]
            mine.sort()  # early block first
            for which, b in enumerate(mine):
                s, e = bounds[b]
                blocks.append((r, j, which, b, s, e - s, pre + e))
                for t in range(s, e):
                    order[r].append(q_base + t)
                    req[r].append(j)
                    pos[r].append(pre + t)
        q_base += n
    return {"order": order, "req": req, "pos": pos, "blocks": blocks}


def interleave_plan(new_len, prefix_len, C: int) -> dict:
    """Interleave (striped) shard map for a batch.

    [SGL] "Interleave strategy": rank r receives flattened token indices
    r, r+C, r+2C, ...; the index runs across the batch's new tokens and does
    not reset at request boundaries; position ids keep their original value.
    [CTX] §2.4 "Interleave" gives the same rule for one request.

    Returns ``order``, ``req`` and ``pos`` as :func:`zigzag_plan` does.
    """
    R = len(new_len)
    owner_req = []
    owner_pos = []
    for j in range(R):
        for t in range(int(new_len[j])):
            owner_req.append(j)
            owner_pos.append(int(prefix_len[j]) + t)
    T = len(owner_req)
    order = [[] for _ in range(C)]
    req = [[] for _ in range(C)]
    pos = [[] for _ in range(C)]
    for f in range(T):
        r = f % C
        order[r].append(f)
        req[r].append(owner_req[f])
        pos[r].append(owner_pos[f])
    return {"order": order, "req": req, "pos": pos}


def interleave_plan_np(new_len, prefix_len, C: int) -> dict:
    """Same map as :func:`interleave_plan`, enumerated with numpy arrays.

    Used for batches of about a million tokens, where a Python loop over
    every token is slow.  The rule is the same: owner = f mod C, local order
    ascending f.  Tests check that both versions agree on small batches.
    """
    new_len = np.asarray(new_len, dtype=np.int64)
    prefix_len = np.asarray(prefix_len, dtype=np.int64)
    T = int(new_len.sum())
    f = np.arange(T, dtype=np.int64)
    req_of_f = np.repeat(np.arange(len(new_len), dtype=np.int64), new_len)
    start_of_req = np.concatenate([[0], np.cumsum(new_len)[:-1]])
    pos_of_f = prefix_len[req_of_f] + (f - start_of_req[req_of_f])
    order, req, pos = [], [], []
    for r in range(C):
        sel = f[f % C == r]
        order.append(sel)
        req.append(req_of_f[sel])
        pos.append(pos_of_f[sel])
    return {"order": order, "req": req, "pos": pos}


def consecutive_split_pairs(n: int, C: int) -> list[int]:
    """Causal (query, key) pairs per GPU when n tokens are cut into C
    consecutive pieces ([CTX] §2.2 "Why consecutive pieces don't work")."""
    piece = n // C
    out = []
    for r in range(C):
        lo, hi = r * piece, (r + 1) * piece if r < C - 1 else n
        out.append(sum(p + 1 for p in range(lo, hi)))
    return out


def pairs_per_rank(plan: dict) -> list[int]:
    """Sum of causal extents (pos + 1) of each rank's queries ([CTX] §1.2)."""
    return [int(sum(int(p) + 1 for p in plan["pos"][r])) for r in range(len(plan["pos"]))]


def decode_shard_map(ctx_len: int, C: int) -> tuple[list[int], list[int]]:
    """Owner shard and row of every cached token of one request.

    [CTX] §3.1 "Storing each token once": token p goes to GPU p mod C, at
    row p // C of that GPU; [V4] §5 owner(j) = j mod P.
    """
    shard, row = [], []
    for p in range(ctx_len):
        shard.append(p % C)
        row.append(p // C)
    return shard, row


def decode_shard_map_contiguous(ctx_len: int, C: int) -> tuple[list[int], list[int]]:
    """Owner shard and row of every cached token when each shard holds one
    chunk of consecutive positions.

    vLLM's Decode Context Parallelism post, §4 "What is DCP?": each GPU keeps
    the cache of a contiguous range of token positions (its example puts a
    200K-token request on four GPUs, 50K positions each).  Where L is not a
    multiple of C the reading taken is that the first L mod C chunks hold one
    token more.  Enumerated: walk the tokens in order and fill chunk r to its
    size before starting chunk r + 1.
    """
    sizes = [ctx_len // C + (1 if r < ctx_len % C else 0) for r in range(C)]
    shard, row = [], []
    r, i = 0, 0
    for _ in range(ctx_len):
        while i == sizes[r]:
            r, i = r + 1, 0
        shard.append(r)
        row.append(i)
        i += 1
    return shard, row


def paged_token_rows(ctx_len, C: int, page_table, page_size: int) -> list[tuple[int, int, int]]:
    """Pool row of every cached token when the shards' rows are kept in pages.

    [CTX] §3.1: token p of a request lives on shard p mod C at row p // C;
    serving caches keep a shard's rows in fixed-size pages ([V4] §9.2).  Here
    row i of the pair (shard r, request b) — pair index r * B + b — sits at
    row i mod page_size of page page_table[pair][i // page_size], so its
    pool row is page * page_size + i mod page_size.
    Returns (request, token position, pool row) for every token.
    """
    B = len(ctx_len)
    out = []
    for b, L in enumerate(ctx_len):
        shard, row = decode_shard_map(int(L), C)
        for p in range(int(L)):
            pair = shard[p] * B + b
            i = row[p]
            page = int(page_table[pair][i // page_size])
            out.append((b, p, page * page_size + i % page_size))
    return out


# --------------------------------------------------------------------------
# FP8 E4M3 decoding, bit by bit from the OCP 8-bit floating point format.
# --------------------------------------------------------------------------


def e4m3_to_float(code: int) -> float:
    """Value of one E4M3 byte: 1 sign bit, 4 exponent bits (bias 7), 3
    mantissa bits; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN;
    there is no infinity."""
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        mag = (m / 8.0) * 2.0 ** (-6)
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


E4M3_TABLE = np.array([e4m3_to_float(c) for c in range(256)], dtype=np.float64)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Elementwise decode of a uint8 array through the 256-entry table."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


# --------------------------------------------------------------------------
# Attention: the plain definition, two passes, fp64.
# --------------------------------------------------------------------------


def softmax_attention(s: np.ndarray, v: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """O and LSE of rows of scores ``s`` [n, L] over values ``v`` [L, Dv].

    [CTX] §1.1: probabilities are the softmax of the scores and the output
    sums the values weighted by them; [CTX] §3.3 and [V4] §5: LSE is the log
    of the sum of exponentiated scores.  Entries of ``s`` that are -inf are
    keys the row does not read.  Two passes: the max, then the sums.
    """
    s = np.asarray(s, dtype=np.float64)
    n = s.shape[0]
    m = np.max(s, axis=1, initial=-np.inf)
    o = np.zeros((n, v.shape[1]), dtype=np.float64)
    lse = np.full(n, -np.inf, dtype=np.float64)
    live = np.isfinite(m)
    if np.any(live):
        e = np.exp(s[live] - m[live, None])
        z = e.sum(axis=1)
        o[live] = (e @ v) / z[:, None]
        lse[live] = m[live] + np.log(z)
    return o, lse


def causal_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, pos: np.ndarray,
                sm_scale: float) -> tuple[np.ndarray, np.ndarray]:
    """Causal GQA attention for query rows of one request.

    q [n, Hq, D]; k, v [L, Hkv, D] (the request's whole cache: prefix and new
    tokens in position order); pos[i] = position of query i, which reads keys
    0..pos[i] ([CTX] §1.1: up to and including itself).  Query head h reads
    kv head h // (Hq/Hkv).  Returns O [n, Hq, D] and LSE [n, Hq] in fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, Hq, D = q.shape
    L, Hkv, _ = k.shape
    g = Hq // Hkv
    pos = np.asarray(pos, dtype=np.int64)
    assert pos.max(initial=-1) < L
    mask = np.arange(L)[None, :] > pos[:, None]  # True where the key is later
    o = np.zeros((n, Hq, v.shape[2]), dtype=np.float64)
    lse = np.zeros((n, Hq), dtype=np.float64)
    for h in range(Hq):
        kh = h // g
        s = sm_scale * (q[:, h, :] @ k[:, kh, :].T)
        s[mask] = -np.inf
        o[:, h, :], lse[:, h] = softmax_attention(s, v[:, kh, :])
    return o, lse


def prefill_reference(plan: dict, new_len, prefix_len, q: np.ndarray, k: np.ndarray,
                      v: np.ndarray, sm_scale: float, ranks=None, rows=None):
    """Per-rank prefill outputs in each rank's local order.

    q [T, Hq, D] in flattened new-token order; k, v [sum(prefix+new), Hkv, D]
    with each request's prefix then new tokens, requests back to back.  With
    virtual shards the all-gather of keys and values is the identity
    ([CTX] §2.1), so every owned query reads its request's full causal
    history.  ``rows`` optionally selects local rows per rank (sampling).
    Returns {rank: (local_rows, O, LSE)}.
    """
    new_len = [int(x) for x in new_len]
    prefix_len = [int(x) for x in prefix_len]
    kv_base = np.concatenate([[0], np.cumsum(np.add(new_len, prefix_len))]).astype(np.int64)
    C = len(plan["order"])
    ranks = range(C) if ranks is None else ranks
    out = {}
    for r in ranks:
        order = np.asarray(plan["order"][r], dtype=np.int64)
        req = np.asarray(plan["req"][r], dtype=np.int64)
        pos = np.asarray(plan["pos"][r], dtype=np.int64)
        local = np.arange(len(order)) if rows is None else np.asarray(rows[r], dtype=np.int64)
        Hq, D = q.shape[1], q.shape[2]
        o = np.zeros((len(local), Hq, v.shape[2]))
        lse = np.zeros((len(local), Hq))
        for j in np.unique(req[local]) if len(local) else []:
            sel = np.nonzero(req[local] == j)[0]
            li = local[sel]
            L = prefix_len[j] + new_len[j]
            kj = k[kv_base[j]:kv_base[j] + L]
            vj = v[kv_base[j]:kv_base[j] + L]
            oj, lj = causal_rows(q[order[li]], kj, vj, pos[li], sm_scale)
            o[sel], lse[sel] = oj, lj
        out[r] = (local, o, lse)
    return out


def decode_scores(q: np.ndarray, kcache: np.ndarray, sm_scale: float) -> np.ndarray:
    """Scores of one request's decode query against its cached keys.

    q [H, Dqk]; kcache [L, Hkv, Dqk].  Head h reads kv head h // (H/Hkv).
    Returns s [H, L].
    """
    q = np.asarray(q, dtype=np.float64)
    kc = np.asarray(kcache, dtype=np.float64)
    H = q.shape[0]
    g = H // kc.shape[1]
    s = np.empty((H, kc.shape[0]))
    for h in range(H):
        s[h] = sm_scale * (kc[:, h // g, :] @ q[h])
    return s


def decode_attention(q: np.ndarray, kcache: np.ndarray, vcache: np.ndarray, sm_scale: float,
                     keys=None) -> tuple[np.ndarray, np.ndarray]:
    """One decode query against a set of cached tokens (all of them, or the
    subset ``keys``).  [CTX] §1.2: the decode step has one query row per
    request; §3.2: a shard runs the same attention over only its tokens.

    q [H, Dqk]; kcache [L, Hkv, Dqk]; vcache [L, Hkv, Dv].
    Returns O [H, Dv], LSE [H]; an empty key set gives O = 0, LSE = -inf.
    """
    H = q.shape[0]
    if keys is not None:
        kcache = kcache[keys]
        vcache = vcache[keys]
    Dv = vcache.shape[2]
    if kcache.shape[0] == 0:
        return np.zeros((H, Dv)), np.full(H, -np.inf)
    s = decode_scores(q, kcache, sm_scale)
    g = H // kcache.shape[1]
    o = np.empty((H, Dv))
    lse = np.empty(H)
    vc = np.asarray(vcache, dtype=np.float64)
    for h in range(H):
        oh, lh = softmax_attention(s[h:h + 1], vc[:, h // g, :])
        o[h], lse[h] = oh[0], lh[0]
    return o, lse


def mla_cache_to_kv(latent: np.ndarray, scale: np.ndarray | None = None, dv: int = 512):
    """MLA cache rows as (K, V) for the attention definition above.

    latent [L, 576]: one latent entry per token shared by all heads
    ([CTX] §1.3; one KV "head").  K is the whole entry and V its first 512
    dims ([GLM] footnote 1: QK over 576 dims, PV over 512).  ``scale`` is the
    per-token fp32 dequantisation factor of an FP8 cache (None for bf16).
    Returns K [L, 1, 576], V [L, 1, dv].
    """
    x = np.asarray(latent, dtype=np.float64)
    if scale is not None:
        x = x * np.asarray(scale, dtype=np.float64)[:, None]
    return x[:, None, :], x[:, None, :dv]


def lse_merge(o_parts: np.ndarray, lse_parts: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Exact combine of partial attention results.

    [V4] §5: with per-part max m_p, local sum l_p and unnormalised output
    u_p, the global result is m = max_p m_p, Z = sum_p e^{m_p - m} l_p,
    o = sum_p e^{m_p - m} u_p / Z.  Written with the normalised partial
    output O_p = u_p / l_p and LSE_p = m_p + ln l_p ([CTX] §3.3), the weights
    become e^{LSE_p - g} with g = max_p LSE_p.  Parts with LSE = -inf carry
    no weight; if every part is empty, O = 0 and LSE = -inf.

    o_parts [P, ..., Dv], lse_parts [P, ...] -> O [..., Dv], LSE [...].
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    g = np.max(lse_parts, axis=0)
    fin = np.isfinite(g)
    g_safe = np.where(fin, g, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - g_safe[None]), 0.0)
    z = w.sum(axis=0)
    o = np.where(fin[..., None], (w[..., None] * o_parts).sum(axis=0) / np.where(fin, z, 1.0)[..., None], 0.0)
    lse = np.where(fin, g_safe + np.log(np.where(fin, z, 1.0)), -np.inf)
    return o, lse


def decode_shard_partials(q: np.ndarray, kcache: np.ndarray, vcache: np.ndarray, C: int,
                          sm_scale: float) -> tuple[np.ndarray, np.ndarray]:
    """Per-shard partial (O_r, LSE_r) of one request's decode step when its
    cache is sharded by token p -> shard p mod C ([CTX] §3.1, §3.4 step 3).
    Returns O [C, H, Dv], LSE [C, H]."""
    L = kcache.shape[0]
    shard, _ = decode_shard_map(L, C)
    shard = np.asarray(shard)
    outs, lses = [], []
    for r in range(C):
        o, lse = decode_attention(q, kcache, vcache, sm_scale, keys=np.nonzero(shard == r)[0])
        outs.append(o)
        lses.append(lse)
    return np.stack(outs), np.stack(lses)


def query_rows_partials(q_rows: np.ndarray, kcache: np.ndarray, vcache: np.ndarray, C: int,
                        sm_scale: float, contiguous: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """Per-shard partials of one request with several query rows.

    [V4] §2.2: multi-token prediction or speculative decoding gives a decode
    step a small number s_q of query rows per request instead of one.  The
    reading taken: the rows are the request's last s_q positions, so row i
    stands at position L - s_q + i and reads the tokens 0 .. L - s_q + i
    (causal among themselves, as in prefill).  Shard r's key set for row i is
    its own tokens (round robin, or contiguous chunks) up to that position.

    q_rows [s_q, H, Dqk]; caches as decode_attention.
    Returns O [C, s_q, H, Dv], LSE [C, s_q, H].
    """
    L, s_q = kcache.shape[0], q_rows.shape[0]
    shard, _ = (decode_shard_map_contiguous if contiguous else decode_shard_map)(L, C)
    shard = np.asarray(shard)
    outs = np.empty((C, s_q, q_rows.shape[1], vcache.shape[2]))
    lses = np.empty((C, s_q, q_rows.shape[1]))
    for r in range(C):
        for i in range(s_q):
            last = L - s_q + i  # the row's own position
            keys = [p for p in range(L) if shard[p] == r and p <= last]
            outs[r, i], lses[r, i] = decode_attention(q_rows[i], kcache, vcache, sm_scale,
                                                      keys=np.asarray(keys, dtype=np.int64))
    return outs, lses


def sharded_topk(scores, C: int, k: int, contiguous: bool = False):
    """Exact global top-k from shard-local top-k lists.

    [V4] §5.2, steps 2-4: each rank scores only its own tokens, keeps a local
    top-k list of (score, token), and the at most C k candidates are merged
    into the global top-k; the union of the local lists contains the global
    top-k, so the merge is exact.  [CTX] §4.1 describes the same exchange of
    best candidates when the index is split with the cache.  Order: higher
    score first; equal scores by lower token index (reading: the pages only
    ask for deterministic ties).

    scores [L] (the index scan's output per token).  Returns the selected
    token indices in increasing order and the C local lists.
    """
    L = len(scores)
    shard, _ = (decode_shard_map_contiguous if contiguous else decode_shard_map)(L, C)
    better = lambda p: (-float(scores[p]), p)  # noqa: E731
    local = []
    for r in range(C):
        mine = [p for p in range(L) if shard[p] == r]
        local.append(sorted(mine, key=better)[:k])
    candidates = [p for lst in local for p in lst]
    chosen = sorted(candidates, key=better)[:k]
    return sorted(chosen), local


def sparse_partials(q: np.ndarray, kcache: np.ndarray, vcache: np.ndarray, selected, C: int,
                    sm_scale: float, contiguous: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """[V4] §5.2, steps 5-7: the selected tokens go to the shards that store
    them and each shard attends to its own selected tokens; the partials
    combine exactly.  Returns O [C, H, Dv], LSE [C, H]."""
    L = kcache.shape[0]
    shard, _ = (decode_shard_map_contiguous if contiguous else decode_shard_map)(L, C)
    outs, lses = [], []
    for r in range(C):
        keys = np.asarray([p for p in selected if shard[p] == r], dtype=np.int64)
        o, lse = decode_attention(q, kcache, vcache, sm_scale, keys=keys)
        outs.append(o)
        lses.append(lse)
    return np.stack(outs), np.stack(lses)


def designated_partials(q: np.ndarray, kmain: np.ndarray, vmain: np.ndarray, kwin: np.ndarray,
                        vwin: np.ndarray, C: int, designated: int,
                        sm_scale: float) -> tuple[np.ndarray, np.ndarray]:
    """Per-shard partials when a local window is replicated on every shard.

    [V4] §5.1, §5.3: each rank attends to the main-cache entries it owns
    (token p on shard p mod C); the small local window is held by every rank,
    but only the designated rank includes it in its partial softmax, so its
    probability mass is counted once in the exact combine.  Shard r's key set
    is {main tokens p : p mod C = r}, plus every window row when r is the
    designated rank.  Returns O [C, H, Dv], LSE [C, H] (empty: 0, -inf).
    """
    L = kmain.shape[0]
    shard, _ = decode_shard_map(L, C)
    shard = np.asarray(shard)
    outs, lses = [], []
    for r in range(C):
        keys = [kmain[shard == r]]
        vals = [vmain[shard == r]]
        if r == designated:
            keys.append(kwin)
            vals.append(vwin)
        o, lse = decode_attention(q, np.concatenate(keys, axis=0), np.concatenate(vals, axis=0),
                                  sm_scale)
        outs.append(o)
        lses.append(lse)
    return np.stack(outs), np.stack(lses)

