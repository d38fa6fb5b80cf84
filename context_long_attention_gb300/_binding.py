"""ctypes binding of libcpattn.so (argument marshalling only)."""

from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "_lib", "libcpattn.so")

CP_ZIGZAG, CP_INTERLEAVE = 0, 1
CP_BF16, CP_FP32, CP_FP8_E4M3 = 0, 1, 2
CP_DECODE_GQA, CP_DECODE_MLA = 0, 1
CP_DCP_ROUND_ROBIN, CP_DCP_CONTIGUOUS, CP_DCP_SELECTED = 0, 1, 2
_STATUS = {0: "CP_OK", -1: "CP_ERR_INVALID_ARG", -2: "CP_ERR_UNSUPPORTED", -3: "CP_ERR_CUDA",
           -4: "CP_ERR_DEVICE_TIMEOUT", -5: "CP_ERR_WORKSPACE"}
MAX_SHARDS = 64
HEADER_WORDS = 24
SEG_WORDS, PAIR_WORDS, WORK_WORDS = 12, 8, 4
HEADER_FIELDS = ["magic", "kind", "C", "R", "T", "KV", "n_seg", "n_tiles", "off_rank", "off_req",
                 "off_seg", "off_tiles", "off_rtile", "off_idx", "off_qpos", "off_qreq",
                 "host_words", "dev_words", "n_parts", "tile_rows", "n_split", "layout", "s_q",
                 "off_run"]
SEG_FIELDS = ["rank", "req", "block", "which", "local_start", "count", "first_f", "stride",
              "q_start", "first_pos", "kv_len", "kv_base"]


class CpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


if not os.path.exists(lib_path):
    raise ImportError(f"{lib_path} is missing: build it with __graft_entry__.build()")
if os.path.isdir(os.path.join(_HERE, "csrc")):
    from . import _build
    if _build.is_stale():
        raise ImportError(f"{lib_path} was built from other sources than the ones in "
                          f"{os.path.join(_HERE, 'csrc')}: rebuild it with __graft_entry__.build()")
lib = ctypes.CDLL(lib_path)

_vp, _i, _sz, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
_szp = ctypes.POINTER(ctypes.c_size_t)
_SIGS = {
    "cp_last_error": (ctypes.c_char_p, []),
    "cp_version": (_i, []),
    "cp_device_error_check": (_i, [_vp]),
    "cp_plan_size": (_i, [_i, _i, _i, _vp, _vp, _szp, _szp]),
    "cp_shard_plan": (_i, [_i, _i, _i, _vp, _vp, _vp, _sz, _vp, _sz, _vp]),
    "cp_prefill_attn": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _i, _i, _i, _f, _vp, _vp, _vp]),
    "cp_decode_plan_size": (_i, [_i, _i, _vp, _i, _szp, _szp]),
    "cp_decode_plan": (_i, [_i, _i, _vp, _i, _vp, _sz, _vp, _sz, _vp]),
    "cp_decode_plan_ex_size": (_i, [_i, _i, _vp, _i, _i, _i, _szp, _szp]),
    "cp_decode_plan_ex": (_i, [_i, _i, _vp, _i, _i, _i, _vp, _sz, _vp, _sz, _vp]),
    "cp_kv_shard_pack": (_i, [_vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _vp]),
    "cp_decode_workspace_size": (_i, [_vp, _i, _i, _szp]),
    "cp_decode_attn": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _vp, _vp,
                            _vp, _sz, _vp]),
    "cp_decode_merged_workspace_size": (_i, [_vp, _i, _i, _i, _i, _szp]),
    "cp_decode_attn_merged": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _vp, _i,
                                   _vp, _vp, _sz, _vp]),
    "cp_lse_merge": (_i, [_i, _i, _i, _i, _vp, _vp, _vp, _i, _vp, _vp]),
    "cp_lse_fold": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "cp_decode_attn_noalloc": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _vp,
                                    _vp, _vp]),
    "cp_noalloc_scratch_bytes": (_sz, []),
    "cp_kv_shard_pack_paged": (_i, [_vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i,
                                    _vp]),
    "cp_decode_attn_paged": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i,
                                  _i, _i, _i, _f, _vp, _vp, _vp, _sz, _vp]),
    "cp_sparse_workspace_size": (_i, [_vp, _i, _szp]),
    "cp_sparse_topk": (_i, [_vp, _vp, _vp, _i, _vp, _vp, _vp, _sz, _vp]),
    "cp_sparse_gather": (_i, [_vp, _vp, _i, _vp, _sz, _i, _vp, _vp, _i, _vp, _vp, _vp, _vp]),
    "cp_sparse_plan_size": (_i, [_i, _i, _i, _i, _szp, _szp]),
    "cp_sparse_plan": (_i, [_i, _i, _i, _i, _vp, _sz, _vp, _sz, _vp]),
    "cp_sparse_decode_attn": (_i, [_vp, _vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f,
                                   _vp, _vp, _vp, _sz, _vp]),
    "cp_sparse_decode_attn_merged": (_i, [_vp, _vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f,
                                          _vp, _i, _vp, _vp, _sz, _vp]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args
NOALLOC_SCRATCH_BYTES = int(lib.cp_noalloc_scratch_bytes())


def _check(status: int):
    if status != 0:
        raise CpError(status, lib.cp_last_error().decode())


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return CP_BF16
    if t.dtype == torch.float32:
        return CP_FP32
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return CP_FP8_E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _need_cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("tensors must be on a CUDA device")
            if not t.is_contiguous():
                raise ValueError("tensors must be contiguous")


class _Plan:
    def __init__(self, host: np.ndarray, dev: torch.Tensor | None):
        self.host = host  # int32 words (host part)
        self.dev = dev    # int32 device words, or None for a host-only plan
        self.header = {k: int(v) for k, v in zip(HEADER_FIELDS, host[:len(HEADER_FIELDS)])}

    def __getattr__(self, k):
        h = self.__dict__.get("header", {})
        if k in h:
            return h[k]
        raise AttributeError(k)

    def words(self, off, n):
        return self.host[off:off + n]


class PrefillPlan(_Plan):
    """A prefill shard plan (zigzag or interleave)."""

    @property
    def rank_off(self):
        return self.words(self.off_rank, self.C + 1)

    @property
    def requests(self):
        return self.words(self.off_req, 4 * self.R).reshape(self.R, 4)

    @property
    def segments(self):
        return self.words(self.off_seg, SEG_WORDS * self.n_seg).reshape(self.n_seg, SEG_WORDS)

    @property
    def tiles(self):
        return self.words(self.off_tiles, 2 * self.n_tiles).reshape(-1, 2)

    @property
    def rank_tile_off(self):
        return self.words(self.off_rtile, self.C + 1)

    @property
    def tiles_by_rank(self):
        return self.words(self.off_rtile + self.C + 1, 2 * self.n_tiles).reshape(-1, 2)

    def device_maps(self):
        """(idx, qpos, qreq) int32 device tensors of length T."""
        d = self.dev
        return (d[self.off_idx:self.off_idx + self.T], d[self.off_qpos:self.off_qpos + self.T],
                d[self.off_qreq:self.off_qreq + self.T])

    def rank_rows(self, rank: int) -> int:
        return self.T if rank < 0 else int(self.rank_off[rank + 1] - self.rank_off[rank])


class DecodePlan(_Plan):
    """A decode token-shard plan with its split-KV schedule."""

    @property
    def pairs(self):
        P = self.C * self.R
        return self.words(self.off_rank, PAIR_WORDS * P).reshape(P, PAIR_WORDS)

    @property
    def worker_off(self):
        return self.words(self.off_req, self.n_tiles + 1)

    @property
    def work(self):
        return self.words(self.off_seg, WORK_WORDS * self.n_seg).reshape(-1, WORK_WORDS)

    @property
    def requests(self):
        return self.words(self.off_tiles, 2 * self.R).reshape(self.R, 2)

    @property
    def split_pairs(self):
        return self.words(self.off_rtile, self.n_split)

    @property
    def run_out(self):
        """Per work item, for the merged-output decode: -1 the run goes on to
        the worker's next item; -2 the last item of a run holding its whole
        request; k >= 0 the last item of a partial run, written to part slot
        k; -3 an empty pair's item."""
        return self.words(self.off_run + 2, self.n_seg)

    @property
    def merge_list(self):
        """[m, 3]: (request, first part slot, parts) of the requests merged from parts."""
        n = int(self.words(self.off_run + 1, 1)[0])
        return self.words(self.off_run + 2 + self.n_seg, 3 * n).reshape(n, 3)

    @property
    def n_merge_parts(self):
        return int(self.words(self.off_run, 1)[0])

    def shard_rows(self):
        p = self.pairs
        return [int(p[r * self.R:(r + 1) * self.R, 0].sum()) for r in range(self.C)]

    @property
    def query_rows(self):
        """Query rows per request (s_q; 1 unless planned for MTP)."""
        return max(1, self.header.get("s_q", 1))


def cp_plan_size(strategy: int, C: int, new_len, prefix_len):
    nl, pl = _i32(new_len), _i32(prefix_len)
    hb, db = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib.cp_plan_size(strategy, C, len(nl), _np_ptr(nl), _np_ptr(pl), ctypes.byref(hb),
                            ctypes.byref(db)))
    return hb.value, db.value


def cp_shard_plan(strategy: int, C: int, new_len, prefix_len=None, device=None) -> PrefillPlan:
    """Builds a prefill shard plan.  With ``device=None`` only the host part
    is computed (no CUDA call); otherwise the plan is copied to ``device`` and
    the per-query maps are filled there by a kernel on the current stream."""
    nl = _i32(new_len)
    pl = _i32(prefix_len if prefix_len is not None else np.zeros_like(nl))
    hb, db = cp_plan_size(strategy, C, nl, pl)
    host = np.zeros(hb // 4, dtype=np.int32)
    dev = None
    if device is not None:
        dev = torch.empty(db // 4, dtype=torch.int32, device=device)
    _check(lib.cp_shard_plan(strategy, C, len(nl), _np_ptr(nl), _np_ptr(pl), _np_ptr(host), hb,
                             _ptr(dev), db, _stream(dev.device) if dev is not None else None))
    return PrefillPlan(host, dev)


def cp_prefill_attn(plan: PrefillPlan, q, k, v, sm_scale=None, rank: int = -1, out=None,
                    lse=None):
    """Causal GQA prefill for the queries of ``rank`` (-1: all ranks,
    rank-major).  q [T, Hq, D]; k, v [KV, Hkv, D]; returns (o, lse)."""
    _need_cuda(q, k, v, out, lse)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    rows = plan.rank_rows(rank)
    if out is None:
        out = torch.empty((rows, Hq, D), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((rows, Hq), dtype=torch.float32, device=q.device)
    _check(lib.cp_prefill_attn(_np_ptr(plan.host), _ptr(plan.dev), rank, _dtype_code(q), _ptr(q),
                               _ptr(k), _ptr(v), Hq, Hkv, D, float(sm_scale), _ptr(out), _ptr(lse),
                               _stream(q.device)))
    return out, lse


def cp_decode_plan(C: int, ctx_len, n_workers: int = 0, device=None) -> DecodePlan:
    cl = _i32(ctx_len)
    hb, db = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib.cp_decode_plan_size(C, len(cl), _np_ptr(cl), n_workers, ctypes.byref(hb),
                                   ctypes.byref(db)))
    host = np.zeros(hb.value // 4, dtype=np.int32)
    dev = None
    if device is not None:
        dev = torch.empty(db.value // 4, dtype=torch.int32, device=device)
    _check(lib.cp_decode_plan(C, len(cl), _np_ptr(cl), n_workers, _np_ptr(host), hb.value,
                              _ptr(dev), db.value, _stream(dev.device) if dev is not None else None))
    return DecodePlan(host, dev)


def cp_decode_plan_ex(C: int, ctx_len, layout: int = 0, s_q: int = 1, n_workers: int = 0,
                      device=None) -> DecodePlan:
    """cp_decode_plan with a shard layout (CP_DCP_ROUND_ROBIN or
    CP_DCP_CONTIGUOUS) and s_q query rows per request."""
    cl = _i32(ctx_len)
    hb, db = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib.cp_decode_plan_ex_size(C, len(cl), _np_ptr(cl), layout, s_q, n_workers,
                                      ctypes.byref(hb), ctypes.byref(db)))
    host = np.zeros(hb.value // 4, dtype=np.int32)
    dev = None
    if device is not None:
        dev = torch.empty(db.value // 4, dtype=torch.int32, device=device)
    _check(lib.cp_decode_plan_ex(C, len(cl), _np_ptr(cl), layout, s_q, n_workers, _np_ptr(host),
                                 hb.value, _ptr(dev), db.value,
                                 _stream(dev.device) if dev is not None else None))
    return DecodePlan(host, dev)


def _decode_shapes(plan, q):
    """(lead, H, Dqk) of a decode query: lead = (B,) or (B, s_q) for MTP plans."""
    s_q = plan.query_rows
    if s_q > 1:
        B, sq, H, Dqk = q.shape
        if sq != s_q:
            raise ValueError(f"q has {sq} query rows, the plan {s_q}")
        return (B, s_q), H, Dqk
    B, H, Dqk = q.shape
    return (B,), H, Dqk


def _ptr_array(ts):
    arr = (ctypes.c_void_p * max(1, len(ts)))()
    for i, t in enumerate(ts):
        arr[i] = None if t is None else t.data_ptr()
    return arr


def cp_kv_shard_pack(plan: DecodePlan, kv, kv_scale=None, shards=None, shard_scales=None):
    """Gathers a token-ordered cache kv [T, ...] into C token shards.
    Returns (shards, shard_scales) — lists of C tensors."""
    _need_cuda(kv, kv_scale)
    if kv.dtype == torch.float8_e4m3fn:
        kv = kv.view(torch.uint8)
    row_elems = int(np.prod(kv.shape[1:]))
    rows = plan.shard_rows()
    if shards is None:
        shards = [torch.empty((n, *kv.shape[1:]), dtype=kv.dtype, device=kv.device) for n in rows]
    if kv_scale is not None and shard_scales is None:
        shard_scales = [torch.empty((n,), dtype=torch.float32, device=kv.device) for n in rows]
    _need_cuda(*shards)
    sarr = _ptr_array(shards)
    scarr = _ptr_array(shard_scales) if kv_scale is not None else None
    _check(lib.cp_kv_shard_pack(_np_ptr(plan.host), _ptr(plan.dev), _dtype_code(kv), _ptr(kv),
                                _ptr(kv_scale), row_elems, sarr, scarr, _stream(kv.device)))
    return shards, (shard_scales if kv_scale is not None else None)


class PageTable:
    """A paged decode cache's page table: int32 [C * R][max_pages] page ids
    (row i of pair (shard r, request b) is row i % page_size of page
    table[r * R + b][i // page_size]), kept as a host array and a device copy."""

    def __init__(self, table, page_size: int, num_pages: int, device=None):
        self.host = np.ascontiguousarray(np.asarray(table, dtype=np.int32))
        assert self.host.ndim == 2
        self.max_pages = int(self.host.shape[1])
        self.page_size = int(page_size)
        self.num_pages = int(num_pages)
        self.dev = torch.from_numpy(self.host).to(device) if device is not None else None

    @property
    def pool_rows(self) -> int:
        return self.num_pages * self.page_size


def cp_kv_shard_pack_paged(plan: DecodePlan, pages: PageTable, kv, kv_scale=None, pool=None,
                           scale_pool=None):
    """Gathers a token-ordered cache kv [T, ...] into a paged pool
    [pool_rows, ...].  Returns (pool, scale_pool)."""
    _need_cuda(kv, kv_scale)
    if kv.dtype == torch.float8_e4m3fn:
        kv = kv.view(torch.uint8)
    row_elems = int(np.prod(kv.shape[1:]))
    if pool is None:
        pool = torch.empty((pages.pool_rows, *kv.shape[1:]), dtype=kv.dtype, device=kv.device)
    if kv_scale is not None and scale_pool is None:
        scale_pool = torch.empty((pages.pool_rows,), dtype=torch.float32, device=kv.device)
    _check(lib.cp_kv_shard_pack_paged(_np_ptr(plan.host), _ptr(plan.dev), _dtype_code(kv), _ptr(kv),
                                      _ptr(kv_scale), row_elems, _ptr(pool),
                                      _ptr(scale_pool) if kv_scale is not None else None,
                                      _np_ptr(pages.host), _ptr(pages.dev), pages.max_pages,
                                      pages.page_size, pages.num_pages, _stream(kv.device)))
    return pool, (scale_pool if kv_scale is not None else None)


def cp_decode_attn_paged(plan: DecodePlan, pages: PageTable, mode: int, q, k_pool, v_pool=None,
                         scale_pool=None, sm_scale=None, o_part=None, lse_part=None, ws=None):
    """cp_decode_attn over a paged pool (k_pool [pool_rows, 576] for MLA, or
    k_pool / v_pool [pool_rows, Hkv, D] for GQA)."""
    lead, H, Dqk = _decode_shapes(plan, q)
    _need_cuda(q, k_pool)
    kp = k_pool.view(torch.uint8) if k_pool.dtype == torch.float8_e4m3fn else k_pool
    kv_dtype = _dtype_code(kp)
    if mode == CP_DECODE_MLA:
        Hkv, Dv = 1, 512
    else:
        Hkv, Dv = kp.shape[1], Dqk
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(Dqk)
    C = plan.C
    if o_part is None:
        o_part = torch.empty((C, *lead, H, Dv), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((C, *lead, H), dtype=torch.float32, device=q.device)
    need = cp_decode_workspace_size(plan, H, Dv)
    if ws is None and need:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib.cp_decode_attn_paged(_np_ptr(plan.host), _ptr(plan.dev), mode, kv_dtype, _ptr(q),
                                    _ptr(kp), _ptr(v_pool), _ptr(scale_pool), _np_ptr(pages.host),
                                    _ptr(pages.dev), pages.max_pages, pages.page_size,
                                    pages.num_pages, H, Hkv, Dqk, Dv, float(sm_scale), _ptr(o_part),
                                    _ptr(lse_part), _ptr(ws), ws_bytes, _stream(q.device)))
    return o_part, lse_part


def cp_decode_workspace_size(plan: DecodePlan, H: int, Dv: int) -> int:
    b = ctypes.c_size_t()
    _check(lib.cp_decode_workspace_size(_np_ptr(plan.host), H, Dv, ctypes.byref(b)))
    return b.value


def cp_decode_attn(plan: DecodePlan, mode: int, q, shard_k, shard_v=None, shard_scale=None,
                   sm_scale=None, o_part=None, lse_part=None, ws=None):
    """Per-shard partial decode attention.  MLA: q [B, H, 576] bf16,
    shard_k[r] [rows_r, 576] bf16 or fp8 codes (+ shard_scale[r]).
    GQA: q [B, Hq, D], shard_k[r]/shard_v[r] [rows_r, Hkv, D] bf16 or fp32 (q
    of the same type), or E4M3 codes with shard_scale[r] [rows_r] fp32, one
    scale per token for its K and V rows (q bf16).
    Returns (o_part [C, B, H, Dv] fp32, lse_part [C, B, H] fp32).  With an
    MTP plan (s_q > 1) q is [B, s_q, H, Dqk] and the outputs [C, B, s_q, ...]."""
    lead, H, Dqk = _decode_shapes(plan, q)
    _need_cuda(q, *[t for t in shard_k if t is not None])
    sk = [t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t for t in shard_k]
    kv_dtype = _dtype_code(sk[0]) if sk else CP_BF16
    if mode == CP_DECODE_MLA:
        Hkv, Dv = 1, 512
    else:
        Hkv, Dv = sk[0].shape[1], Dqk
        want_q = torch.float32 if kv_dtype == CP_FP32 else torch.bfloat16
        if q.dtype != want_q:
            raise TypeError(f"GQA decode over this cache takes a {want_q} query, got {q.dtype}")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(Dqk)
    C = plan.C
    if o_part is None:
        o_part = torch.empty((C, *lead, H, Dv), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((C, *lead, H), dtype=torch.float32, device=q.device)
    need = cp_decode_workspace_size(plan, H, Dv)
    if ws is None and need:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib.cp_decode_attn(_np_ptr(plan.host), _ptr(plan.dev), mode, kv_dtype, _ptr(q),
                              _ptr_array(sk), _ptr_array(shard_v) if shard_v is not None else None,
                              _ptr_array(shard_scale) if shard_scale is not None else None,
                              H, Hkv, Dqk, Dv, float(sm_scale), _ptr(o_part), _ptr(lse_part),
                              _ptr(ws), ws_bytes, _stream(q.device)))
    return o_part, lse_part


def cp_decode_merged_workspace_size(plan: DecodePlan, mode: int, kv_dtype: int, H: int, Dv: int) -> int:
    b = ctypes.c_size_t()
    _check(lib.cp_decode_merged_workspace_size(_np_ptr(plan.host), mode, kv_dtype, H, Dv, ctypes.byref(b)))
    return b.value


def cp_decode_attn_merged(plan: DecodePlan, mode: int, q, shard_k, shard_v=None, shard_scale=None,
                          sm_scale=None, out_dtype=torch.bfloat16, o=None, lse=None, ws=None):
    """cp_decode_attn and the LSE merge of its partials in one call: returns
    (o [B, H, Dv] out_dtype, lse [B, H] fp32); with an MTP plan (s_q > 1)
    q is [B, s_q, H, Dqk] and the outputs [B, s_q, ...].  MLA over an FP8
    cache accumulates each worker's items of one request together and writes
    partials only for requests cut by a worker boundary."""
    lead, H, Dqk = _decode_shapes(plan, q)
    _need_cuda(q, *[t for t in shard_k if t is not None], o, lse)
    sk = [t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t for t in shard_k]
    kv_dtype = _dtype_code(sk[0]) if sk else CP_BF16
    if mode == CP_DECODE_MLA:
        Hkv, Dv = 1, 512
    else:
        Hkv, Dv = sk[0].shape[1], Dqk
        want_q = torch.float32 if kv_dtype == CP_FP32 else torch.bfloat16
        if q.dtype != want_q:
            raise TypeError(f"GQA decode over this cache takes a {want_q} query, got {q.dtype}")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(Dqk)
    if o is None:
        o = torch.empty((*lead, H, Dv), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((*lead, H), dtype=torch.float32, device=q.device)
    need = cp_decode_merged_workspace_size(plan, mode, kv_dtype, H, Dv)
    if ws is None and need:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib.cp_decode_attn_merged(_np_ptr(plan.host), _ptr(plan.dev), mode, kv_dtype, _ptr(q),
                                     _ptr_array(sk), _ptr_array(shard_v) if shard_v is not None else None,
                                     _ptr_array(shard_scale) if shard_scale is not None else None,
                                     H, Hkv, Dqk, Dv, float(sm_scale), _ptr(o), _dtype_code(o), _ptr(lse),
                                     _ptr(ws), ws_bytes, _stream(q.device)))
    return o, lse


def cp_decode_attn_noalloc(plan: DecodePlan, mode: int, q, shard_k, shard_v=None,
                           shard_scale=None, sm_scale=None, o_part=None, lse_part=None):
    """cp_decode_attn without a workspace argument: the split-KV scratch is a
    fixed library-owned device array (NOALLOC_SCRATCH_BYTES).  Calls must not
    overlap on the GPU."""
    lead, H, Dqk = _decode_shapes(plan, q)
    _need_cuda(q, *[t for t in shard_k if t is not None])
    sk = [t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t for t in shard_k]
    kv_dtype = _dtype_code(sk[0]) if sk else CP_BF16
    if mode == CP_DECODE_MLA:
        Hkv, Dv = 1, 512
    else:
        Hkv, Dv = sk[0].shape[1], Dqk
        want_q = torch.float32 if kv_dtype == CP_FP32 else torch.bfloat16
        if q.dtype != want_q:
            raise TypeError(f"GQA decode over this cache takes a {want_q} query, got {q.dtype}")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(Dqk)
    C = plan.C
    if o_part is None:
        o_part = torch.empty((C, *lead, H, Dv), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((C, *lead, H), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):  # the library uses the current device's array
        _check(lib.cp_decode_attn_noalloc(
            _np_ptr(plan.host), _ptr(plan.dev), mode, kv_dtype, _ptr(q), _ptr_array(sk),
            _ptr_array(shard_v) if shard_v is not None else None,
            _ptr_array(shard_scale) if shard_scale is not None else None, H, Hkv, Dqk, Dv,
            float(sm_scale), _ptr(o_part), _ptr(lse_part), _stream(q.device)))
    return o_part, lse_part


def cp_lse_merge(o_part, lse_part, out_dtype=torch.bfloat16, out=None, lse=None):
    """Exact LSE merge over the leading dim: o_part [P, N, H, Dv],
    lse_part [P, N, H] -> (o [N, H, Dv], lse [N, H])."""
    _need_cuda(o_part, lse_part, out, lse)
    P, N, H, Dv = o_part.shape
    if out is None:
        out = torch.empty((N, H, Dv), dtype=out_dtype, device=o_part.device)
    if lse is None:
        lse = torch.empty((N, H), dtype=torch.float32, device=o_part.device)
    _check(lib.cp_lse_merge(P, N, H, Dv, _ptr(o_part), _ptr(lse_part), _ptr(out),
                            _dtype_code(out), _ptr(lse), _stream(o_part.device)))
    return out, lse


def cp_lse_fold(o, lse, o_add, lse_add):
    """(o, lse) <- exact combine of (o, lse) and (o_add, lse_add), in place;
    o, o_add [N, H, Dv] fp32 contiguous, lse, lse_add [N, H] fp32."""
    _need_cuda(o, lse, o_add, lse_add)
    for t in (o, lse, o_add, lse_add):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("cp_lse_fold takes contiguous fp32 tensors")
    N, H, Dv = o.shape
    _check(lib.cp_lse_fold(N, H, Dv, _ptr(o), _ptr(lse), _ptr(o_add), _ptr(lse_add),
                           _stream(o.device)))
    return o, lse


def cp_device_error_check(device=None):
    _check(lib.cp_device_error_check(_stream(device)))


# ---------------------------------------------------------------- sparse decode

def cp_sparse_workspace_size(plan: DecodePlan, k: int) -> int:
    b = ctypes.c_size_t()
    _check(lib.cp_sparse_workspace_size(_np_ptr(plan.host), k, ctypes.byref(b)))
    return b.value


def cp_sparse_topk(plan: DecodePlan, shard_scores, k: int, sel_ids=None, sel_count=None, ws=None):
    """Exact sharded top-k: shard_scores[r] fp32 [rows_r] (the plan's rows).
    Returns (sel_ids [B, k] int32 ascending, -1 padded; sel_count [B]; ws),
    ws holding the candidates for cp_sparse_gather."""
    dev = next(t.device for t in shard_scores if t is not None)
    _need_cuda(*[t for t in shard_scores if t is not None])
    B = plan.R
    if sel_ids is None:
        sel_ids = torch.empty((B, k), dtype=torch.int32, device=dev)
    if sel_count is None:
        sel_count = torch.empty((B,), dtype=torch.int32, device=dev)
    need = cp_sparse_workspace_size(plan, k)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
    _check(lib.cp_sparse_topk(_np_ptr(plan.host), _ptr(plan.dev), _ptr_array(shard_scores), k,
                              _ptr(sel_ids), _ptr(sel_count), _ptr(ws), ws.numel(), _stream(dev)))
    return sel_ids, sel_count, ws


def sparse_slot_rows(k: int) -> int:
    """Rows per (shard, request) slot of a selection buffer: k rounded up to 128."""
    return (k + 127) // 128 * 128


def cp_sparse_gather(plan: DecodePlan, k: int, ws, shard_kv, shard_scale=None, sel_kv=None,
                     sel_scale=None, pair_count=None):
    """Packs each owner's selected rows (after cp_sparse_topk with the same
    plan, k, ws) into selection buffers [B kp, ...] (kp = sparse_slot_rows(k));
    returns
    (sel_kv list, sel_scale list or None, pair_count [C * B])."""
    sk = [t.view(torch.uint8) if t is not None and t.dtype == torch.float8_e4m3fn else t
          for t in shard_kv]
    ref = next(t for t in sk if t is not None)
    _need_cuda(*[t for t in sk if t is not None])
    C, B = plan.C, plan.R
    kp = sparse_slot_rows(k)
    if sel_kv is None:
        sel_kv = [torch.empty((B * kp, *ref.shape[1:]), dtype=ref.dtype, device=ref.device)
                  for _ in range(C)]
    if shard_scale is not None and sel_scale is None:
        sel_scale = [torch.empty((B * kp,), dtype=torch.float32, device=ref.device) for _ in range(C)]
    if pair_count is None:
        pair_count = torch.empty((C * B,), dtype=torch.int32, device=ref.device)
    row_elems = int(np.prod(ref.shape[1:]))
    _check(lib.cp_sparse_gather(_np_ptr(plan.host), _ptr(plan.dev), k, _ptr(ws), ws.numel(),
                                _dtype_code(ref), _ptr_array(sk),
                                _ptr_array(shard_scale) if shard_scale is not None else None,
                                row_elems, _ptr_array(sel_kv),
                                _ptr_array(sel_scale) if sel_scale is not None else None,
                                _ptr(pair_count), _stream(ref.device)))
    return sel_kv, sel_scale, pair_count


def cp_sparse_plan(C: int, B: int, k: int, n_workers: int = 0, device=None) -> DecodePlan:
    """The decode plan over selection buffers with room for k rows per pair."""
    hb, db = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib.cp_sparse_plan_size(C, B, k, n_workers, ctypes.byref(hb), ctypes.byref(db)))
    host = np.zeros(hb.value // 4, dtype=np.int32)
    dev = None
    if device is not None:
        dev = torch.empty(db.value // 4, dtype=torch.int32, device=device)
    _check(lib.cp_sparse_plan(C, B, k, n_workers, _np_ptr(host), hb.value, _ptr(dev), db.value,
                              _stream(dev.device) if dev is not None else None))
    return DecodePlan(host, dev)


def cp_sparse_decode_attn(plan: DecodePlan, pair_count, mode: int, q, sel_k, sel_v=None,
                          sel_scale=None, sm_scale=None, o_part=None, lse_part=None, ws=None):
    """cp_decode_attn over the selection buffers (plan from cp_sparse_plan)."""
    B, H, Dqk = q.shape
    sk = [t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t for t in sel_k]
    _need_cuda(q, pair_count, *sk)
    kv_dtype = _dtype_code(sk[0])
    if mode == CP_DECODE_MLA:
        Hkv, Dv = 1, 512
    else:
        Hkv, Dv = sk[0].shape[1], Dqk
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(Dqk)
    C = plan.C
    if o_part is None:
        o_part = torch.empty((C, B, H, Dv), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((C, B, H), dtype=torch.float32, device=q.device)
    need = cp_decode_workspace_size(plan, H, Dv)
    if ws is None and need:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib.cp_sparse_decode_attn(_np_ptr(plan.host), _ptr(plan.dev), _ptr(pair_count), mode,
                                     kv_dtype, _ptr(q), _ptr_array(sk),
                                     _ptr_array(sel_v) if sel_v is not None else None,
                                     _ptr_array(sel_scale) if sel_scale is not None else None,
                                     H, Hkv, Dqk, Dv, float(sm_scale), _ptr(o_part), _ptr(lse_part),
                                     _ptr(ws), ws_bytes, _stream(q.device)))
    return o_part, lse_part


def cp_sparse_decode_attn_merged(plan: DecodePlan, pair_count, mode: int, q, sel_k, sel_v=None,
                                 sel_scale=None, sm_scale=None, out_dtype=torch.bfloat16, o=None, lse=None,
                                 ws=None):
    """cp_sparse_decode_attn and the LSE merge of its partials in one call:
    returns (o [B, H, Dv] out_dtype, lse [B, H] fp32)."""
    B, H, Dqk = q.shape
    sk = [t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t for t in sel_k]
    _need_cuda(q, pair_count, *sk, o, lse)
    kv_dtype = _dtype_code(sk[0])
    if mode == CP_DECODE_MLA:
        Hkv, Dv = 1, 512
    else:
        Hkv, Dv = sk[0].shape[1], Dqk
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(Dqk)
    if o is None:
        o = torch.empty((B, H, Dv), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    need = cp_decode_merged_workspace_size(plan, mode, kv_dtype, H, Dv)
    if ws is None and need:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib.cp_sparse_decode_attn_merged(_np_ptr(plan.host), _ptr(plan.dev), _ptr(pair_count), mode,
                                            kv_dtype, _ptr(q), _ptr_array(sk),
                                            _ptr_array(sel_v) if sel_v is not None else None,
                                            _ptr_array(sel_scale) if sel_scale is not None else None,
                                            H, Hkv, Dqk, Dv, float(sm_scale), _ptr(o), _dtype_code(o), _ptr(lse),
                                            _ptr(ws), ws_bytes, _stream(q.device)))
    return o, lse


# ---------------------------------------------------------------- NVTX ranges
# With CPATTN_NVTX=1 every public entry point runs inside an NVTX range of
# its own name, so a timeline profiler shows the path's steps (plan, prefill,
# pack, decode, merge, ...) on the host and the launch rows they issue.
if os.environ.get("CPATTN_NVTX") == "1":
    import functools

    def _ranged(fn):
        @functools.wraps(fn)
        def wrapper(*args, **kwargs):
            torch.cuda.nvtx.range_push(fn.__name__)
            try:
                return fn(*args, **kwargs)
            finally:
                torch.cuda.nvtx.range_pop()
        return wrapper

    for _n, _f in list(globals().items()):
        if _n.startswith("cp_") and callable(_f):
            globals()[_n] = _ranged(_f)
