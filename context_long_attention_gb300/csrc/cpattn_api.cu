// C-ABI entry points: argument validation, host-side planning and launches.
//
// Planning follows the shard rules of "How GPUs Share a Long Context During
// LLM Inference" (§2.3 Zigzag, §2.4 Interleave, §3.1 Storing each token
// once) and the SGLang "Prefill context parallelism" page (Zigzag strategy,
// Interleave strategy).  The per-token arrays of a prefill plan are filled on
// the device (plan_kernels.cu); everything else here is O(requests x shards).
#include <algorithm>
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "internal.h"

using namespace cpattn;

namespace {

thread_local std::string g_err;

cp_status fail(cp_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

cp_status ok() {
  g_err.clear();
  return CP_OK;
}

cp_status cuda_fail(cudaError_t e, const char* what) {
  return fail(CP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int align4(int w) { return (w + 3) & ~3; }

// Status words of the bounded waits, one copy per device.
__device__ unsigned g_cp_status[4];

// ------------------------------------------------------------------ prefill plan

struct PrefillBuild {
  std::vector<int32_t> words;  // host part
  int dev_words = 0;
};

cp_status check_batch(int C, int R, const int32_t* new_len, const int32_t* prefix_len,
                      long long* T_out, long long* KV_out) {
  if (C < 1 || C > CP_MAX_SHARDS) return fail(CP_ERR_INVALID_ARG, "C=%d outside [1, %d]", C, CP_MAX_SHARDS);
  if (R < 1) return fail(CP_ERR_INVALID_ARG, "R=%d must be >= 1", R);
  if (!new_len || !prefix_len) return fail(CP_ERR_INVALID_ARG, "new_len/prefix_len is NULL");
  long long T = 0, KV = 0;
  for (int j = 0; j < R; ++j) {
    if (new_len[j] < 0 || prefix_len[j] < 0)
      return fail(CP_ERR_INVALID_ARG, "request %d has a negative length", j);
    T += new_len[j];
    KV += (long long)new_len[j] + prefix_len[j];
  }
  if (KV >= (1LL << 31) - 1) return fail(CP_ERR_INVALID_ARG, "total K/V rows %lld >= 2^31", KV);
  *T_out = T;
  *KV_out = KV;
  return CP_OK;
}

cp_status build_prefill_plan(cp_strategy strategy, int C, int R, const int32_t* new_len,
                             const int32_t* prefix_len, PrefillBuild* out) {
  if (strategy != CP_ZIGZAG && strategy != CP_INTERLEAVE)
    return fail(CP_ERR_INVALID_ARG, "unknown strategy %d", (int)strategy);
  long long T = 0, KV = 0;
  cp_status st = check_batch(C, R, new_len, prefix_len, &T, &KV);
  if (st != CP_OK) return st;

  std::vector<cp_req_desc> req(R);
  {
    int q = 0, kv = 0;
    for (int j = 0; j < R; ++j) {
      req[j] = {new_len[j], prefix_len[j], q, kv};
      q += new_len[j];
      kv += new_len[j] + prefix_len[j];
    }
  }
  // Segments, rank-major, in each rank's local order.
  std::vector<cp_seg_desc> seg;
  std::vector<int32_t> rank_off(C + 1, 0);
  int local = 0;
  for (int r = 0; r < C; ++r) {
    rank_off[r] = local;
    for (int j = 0; j < R; ++j) {
      const int n = new_len[j], pre = prefix_len[j];
      if (strategy == CP_ZIGZAG) {
        // 2C blocks; the first n mod 2C get one extra token; rank r takes
        // block r (early) and block 2C-1-r (late).
        const int nb = 2 * C, base = n / nb, rem = n % nb;
        for (int which = 0; which < 2; ++which) {
          const int b = which == 0 ? r : nb - 1 - r;
          const int start = b * base + std::min(b, rem);
          const int size = base + (b < rem ? 1 : 0);
          cp_seg_desc s;
          s.rank = r;
          s.req = j;
          s.block = b;
          s.which = which;
          s.local_start = local;
          s.count = size;
          s.first_f = req[j].q_base + start;
          s.stride = 1;
          s.q_start = start;
          s.first_pos = pre + start;
          s.kv_len = pre + start + size;  // reads end where the block ends
          s.kv_base = req[j].kv_base;
          seg.push_back(s);
          local += size;
        }
      } else {
        // Flattened index f owned by rank r iff f mod C == r.
        const int qb = req[j].q_base;
        const int f0 = qb + ((r - qb) % C + C) % C;
        const int count = f0 < qb + n ? (qb + n - 1 - f0) / C + 1 : 0;
        cp_seg_desc s;
        s.rank = r;
        s.req = j;
        s.block = -1;
        s.which = 0;
        s.local_start = local;
        s.count = count;
        s.first_f = f0;
        s.stride = C;
        s.q_start = f0 - qb;
        s.first_pos = pre + (f0 - qb);
        s.kv_len = count > 0 ? s.first_pos + (count - 1) * C + 1 : 0;
        s.kv_base = req[j].kv_base;
        seg.push_back(s);
        local += count;
      }
    }
  }
  rank_off[C] = local;

  // 128-query tiles; longest-first order (by the keys the last query reads).
  struct TileKey {
    cp_tile_desc t;
    long long work;
    int rank;
  };
  std::vector<TileKey> tiles;
  for (int i = 0; i < (int)seg.size(); ++i) {
    const cp_seg_desc& s = seg[i];
    for (int off = 0; off < s.count; off += kPrefillTileRows) {
      const int nrow = std::min(kPrefillTileRows, s.count - off);
      const long long kv_hi = (long long)s.first_pos + (long long)(off + nrow - 1) * s.stride + 1;
      tiles.push_back({{i, off}, kv_hi * nrow, s.rank});
    }
  }
  std::vector<TileKey> by_work = tiles;
  std::stable_sort(by_work.begin(), by_work.end(),
                   [](const TileKey& a, const TileKey& b) { return a.work > b.work; });
  std::vector<TileKey> by_rank = tiles;
  std::stable_sort(by_rank.begin(), by_rank.end(), [](const TileKey& a, const TileKey& b) {
    return a.rank != b.rank ? a.rank < b.rank : a.work > b.work;
  });
  std::vector<int32_t> rank_tile_off(C + 1, 0);
  for (const TileKey& t : by_rank) rank_tile_off[t.rank + 1]++;
  for (int r = 0; r < C; ++r) rank_tile_off[r + 1] += rank_tile_off[r];

  const int n_seg = (int)seg.size(), n_tiles = (int)tiles.size();
  cp_plan_header h;
  memset(&h, 0, sizeof(h));
  h.magic = CP_PLAN_MAGIC;
  h.kind = strategy == CP_ZIGZAG ? 0 : 1;
  h.C = C;
  h.R = R;
  h.T = (int32_t)T;
  h.KV = (int32_t)KV;
  h.n_seg = n_seg;
  h.n_tiles = n_tiles;
  int w = align4(kHeaderWords);
  h.off_rank = w;
  w = align4(w + C + 1);
  h.off_req = w;
  w = align4(w + 4 * R);
  h.off_seg = w;
  w = align4(w + kSegWords * n_seg);
  h.off_tiles = w;
  w = align4(w + 2 * n_tiles);
  h.off_rtile = w;
  w = align4(w + (C + 1) + 2 * n_tiles);
  h.host_words = w;
  h.off_idx = w;
  w = align4(w + (int)T);
  h.off_qpos = w;
  w = align4(w + (int)T);
  h.off_qreq = w;
  w = align4(w + (int)T);
  h.dev_words = w;
  h.tile_rows = kPrefillTileRows;

  out->words.assign(h.host_words, 0);
  int32_t* W = out->words.data();
  memcpy(W, &h, sizeof(h));
  memcpy(W + h.off_rank, rank_off.data(), 4 * (C + 1));
  memcpy(W + h.off_req, req.data(), sizeof(cp_req_desc) * R);
  if (n_seg) memcpy(W + h.off_seg, seg.data(), sizeof(cp_seg_desc) * n_seg);
  for (int i = 0; i < n_tiles; ++i) {
    W[h.off_tiles + 2 * i] = by_work[i].t.seg;
    W[h.off_tiles + 2 * i + 1] = by_work[i].t.q_off;
  }
  memcpy(W + h.off_rtile, rank_tile_off.data(), 4 * (C + 1));
  for (int i = 0; i < n_tiles; ++i) {
    W[h.off_rtile + C + 1 + 2 * i] = by_rank[i].t.seg;
    W[h.off_rtile + C + 1 + 2 * i + 1] = by_rank[i].t.q_off;
  }
  out->dev_words = h.dev_words;
  return CP_OK;
}

// ------------------------------------------------------------------ decode plan

struct DecodeBuild {
  std::vector<int32_t> words;
};

cp_status sm_count(int* n) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
  return CP_OK;
}

cp_status build_decode_plan(int C, int B, const int32_t* ctx_len, int layout, int s_q,
                            int n_workers, DecodeBuild* out) {
  if (C < 1 || C > CP_MAX_SHARDS) return fail(CP_ERR_INVALID_ARG, "C=%d outside [1, %d]", C, CP_MAX_SHARDS);
  if (B < 1) return fail(CP_ERR_INVALID_ARG, "B=%d must be >= 1", B);
  if (!ctx_len) return fail(CP_ERR_INVALID_ARG, "ctx_len is NULL");
  if (n_workers < 0) return fail(CP_ERR_INVALID_ARG, "n_workers=%d < 0", n_workers);
  if (layout != CP_DCP_ROUND_ROBIN && layout != CP_DCP_CONTIGUOUS && layout != CP_DCP_SELECTED)
    return fail(CP_ERR_INVALID_ARG, "layout=%d is not a cp_dcp_layout", layout);
  if (s_q < 1 || s_q > 64) return fail(CP_ERR_INVALID_ARG, "s_q=%d outside [1, 64]", s_q);
  long long total = 0;
  for (int b = 0; b < B; ++b) {
    if (ctx_len[b] < 0) return fail(CP_ERR_INVALID_ARG, "ctx_len[%d] < 0", b);
    if (s_q > 1 && ctx_len[b] < s_q)
      return fail(CP_ERR_INVALID_ARG, "ctx_len[%d]=%d < s_q=%d query rows", b, ctx_len[b], s_q);
    total += ctx_len[b];
  }
  if (total >= (1LL << 31) - 1) return fail(CP_ERR_INVALID_ARG, "total tokens %lld >= 2^31", total);
  int G = n_workers;
  if (G == 0) {
    cp_status st = sm_count(&G);
    if (st != CP_OK) return st;
  }
  const int P = C * B, TR = kDecodeTileRows;
  std::vector<cp_pair_desc> pair(P);
  std::vector<long long> tile_start(P + 1, 0);
  for (int r = 0; r < C; ++r) {
    int off = 0;
    for (int b = 0; b < B; ++b) {
      const int L = ctx_len[b];
      int rows, tok0, step;
      if (layout == CP_DCP_ROUND_ROBIN) {  // tokens p = r, r + C, ...
        rows = L > r ? (L - r + C - 1) / C : 0;
        tok0 = r;
        step = C;
      } else if (layout == CP_DCP_CONTIGUOUS) {  // one chunk; the first L mod C one token longer
        const int q = L / C, m = L % C;
        rows = q + (r < m ? 1 : 0);
        tok0 = r * q + std::min(r, m);
        step = 1;
      } else {  // selection buffer: room for L rows per pair, the count known on the device
        rows = L;
        tok0 = 0;
        step = 1;
      }
      cp_pair_desc& d = pair[r * B + b];
      memset(&d, 0, sizeof(d));
      d.rows = rows;
      d.row_off = off;
      d.ctx_len = L;
      d.first_part = -1;
      d.tok0 = tok0;
      d.tok_step = step;
      off += rows;
    }
  }
  // The schedule walks the pairs request by request (shards 0..C-1 of
  // request 0, then of request 1, ...), so that consecutive items of a worker
  // share a request and the MLA kernels keep its query in shared memory.
  auto walk = [&](int s) { return (s % C) * B + s / C; };  // walk position -> pair index
  for (int i = 0; i < P; ++i) tile_start[i + 1] = tile_start[i] + (pair[walk(i)].rows + TR - 1) / TR;
  const long long NT = tile_start[P];

  // Worker ranges balance a cost: every tile, plus kDecodeItemCost tiles for
  // each nonempty pair (a work item's fixed work: its query, the first tile's
  // fill, the epilogue and the partial's write), so that many short pairs do
  // not pile up on one worker.  A cut that falls in a pair's fixed cost moves
  // to the pair's start; one inside its tiles splits the pair there.
  std::vector<long long> cost_start(P + 1, 0);
  for (int i = 0; i < P; ++i) {
    const long long nt = tile_start[i + 1] - tile_start[i];
    cost_start[i + 1] = cost_start[i] + (nt > 0 ? kDecodeItemCost + nt : 0);
  }
  const long long total_cost = cost_start[P];
  std::vector<long long> cut(G + 1, NT);  // worker w: tiles [cut[w], cut[w + 1])
  {
    int i = 0;
    for (int wkr = 0; wkr < G; ++wkr) {
      const long long x = total_cost * wkr / G;
      while (i < P && cost_start[i + 1] <= x) ++i;
      if (i == P) break;
      cut[wkr] = tile_start[i] + std::max(0LL, x - cost_start[i] - kDecodeItemCost);
    }
  }

  // Contiguous tile ranges per worker, cut at pair boundaries into items.
  std::vector<std::vector<cp_work_desc>> per_worker(G);
  int p = 0;
  for (int wkr = 0; wkr < G; ++wkr) {
    const long long t0 = cut[wkr], t1 = cut[wkr + 1];
    long long t = t0;
    while (t < t1) {
      while (tile_start[p + 1] <= t) ++p;
      const long long pend = std::min(t1, tile_start[p + 1]);
      cp_work_desc wd;
      wd.pair = walk(p);
      wd.row_begin = (int)((t - tile_start[p]) * TR);
      wd.row_end = (int)std::min<long long>(pair[walk(p)].rows, (pend - tile_start[p]) * TR);
      wd.part = -1;
      per_worker[wkr].push_back(wd);
      t = pend;
    }
  }
  // Empty pairs still produce (O = 0, LSE = -inf).
  int rr = 0;
  for (int i = 0; i < P; ++i)
    if (pair[i].rows == 0) {
      per_worker[rr % G].push_back({i, 0, 0, -1});
      ++rr;
    }
  std::vector<cp_work_desc> work;
  std::vector<int32_t> worker_off(G + 1, 0);
  for (int wkr = 0; wkr < G; ++wkr) {
    worker_off[wkr] = (int)work.size();
    work.insert(work.end(), per_worker[wkr].begin(), per_worker[wkr].end());
  }
  worker_off[G] = (int)work.size();
  for (const cp_work_desc& wd : work) pair[wd.pair].n_parts++;
  int n_parts = 0;
  std::vector<int32_t> split;
  for (int i = 0; i < P; ++i)
    if (pair[i].n_parts > 1) {
      pair[i].first_part = n_parts;
      n_parts += pair[i].n_parts;
      split.push_back(i);
    }
  std::vector<int> next(P, 0);
  for (cp_work_desc& wd : work)
    if (pair[wd.pair].n_parts > 1) wd.part = pair[wd.pair].first_part + next[wd.pair]++;

  const int n_work = (int)work.size();

  // Runs for the merged-output decode: within a worker, the consecutive items
  // (of nonempty pairs) of one request.  A run that holds all of its request's
  // nonempty items writes the request's result; the others write parts, which
  // a merge combines.  A request's parts are consecutive slots, in worker order.
  std::vector<int32_t> run_out(n_work, -3);  // -3: an empty pair's item (nothing to do)
  std::vector<int> req_items(B, 0), req_parts(B, 0), run_req, run_last, run_n;
  for (const cp_work_desc& wd : work)
    if (pair[wd.pair].rows > 0) req_items[wd.pair % B]++;
  for (int wkr = 0; wkr < G; ++wkr) {
    int cur = -1;  // this worker's open run
    for (int i = worker_off[wkr]; i < worker_off[wkr + 1]; ++i) {
      if (pair[work[i].pair].rows == 0) continue;
      const int b = work[i].pair % B;
      if (cur >= 0 && run_req[cur] == b) {
        run_out[run_last[cur]] = -1;  // the run goes on to item i
        run_last[cur] = i;
        run_n[cur]++;
      } else {
        cur = (int)run_req.size();
        run_req.push_back(b);
        run_last.push_back(i);
        run_n.push_back(1);
      }
      run_out[i] = -2;  // provisionally the last item of a complete run
    }
  }
  for (size_t k = 0; k < run_req.size(); ++k)
    if (run_n[k] < req_items[run_req[k]]) req_parts[run_req[k]]++;
  std::vector<int> req_first(B, 0), req_next(B, 0);
  std::vector<int32_t> merge_list;  // {request, first part slot, parts}
  int n_mparts = 0;
  for (int b = 0; b < B; ++b) {
    req_first[b] = n_mparts;
    n_mparts += req_parts[b];
    if (req_parts[b] > 0 || req_items[b] == 0) {  // parts to merge, or no rows at all (O = 0, LSE = -inf)
      merge_list.push_back(b);
      merge_list.push_back(req_first[b]);
      merge_list.push_back(req_parts[b]);
    }
  }
  for (size_t k = 0; k < run_req.size(); ++k)
    if (run_n[k] < req_items[run_req[k]]) {
      const int b = run_req[k];
      run_out[run_last[k]] = req_first[b] + req_next[b]++;
    }
  const int n_mlist = (int)merge_list.size() / 3;

  cp_plan_header h;
  memset(&h, 0, sizeof(h));
  h.magic = CP_PLAN_MAGIC;
  h.kind = 2;
  h.C = C;
  h.R = B;
  h.T = (int32_t)total;
  h.n_seg = n_work;
  h.n_tiles = G;
  h.n_parts = n_parts;
  h.n_split = (int)split.size();
  h.tile_rows = TR;
  h.layout = layout;
  h.s_q = s_q;
  int w = align4(kHeaderWords);
  h.off_rank = w;
  w = align4(w + kPairWords * P);
  h.off_req = w;
  w = align4(w + G + 1);
  h.off_seg = w;
  w = align4(w + kWorkWords * n_work);
  h.off_tiles = w;
  w = align4(w + 2 * B);
  h.off_rtile = w;
  w = align4(w + (int)split.size());
  h.off_run = w;
  w = align4(w + 2 + n_work + 3 * n_mlist);
  h.host_words = w;
  h.dev_words = w;
  out->words.assign(w, 0);
  int32_t* W = out->words.data();
  memcpy(W, &h, sizeof(h));
  W[h.off_run] = n_mparts;
  W[h.off_run + 1] = n_mlist;
  if (n_work) memcpy(W + h.off_run + 2, run_out.data(), 4 * n_work);
  if (n_mlist) memcpy(W + h.off_run + 2 + n_work, merge_list.data(), 4 * merge_list.size());
  memcpy(W + h.off_rank, pair.data(), sizeof(cp_pair_desc) * P);
  memcpy(W + h.off_req, worker_off.data(), 4 * (G + 1));
  if (n_work) memcpy(W + h.off_seg, work.data(), sizeof(cp_work_desc) * n_work);
  long long tok = 0;
  for (int b = 0; b < B; ++b) {
    W[h.off_tiles + 2 * b] = ctx_len[b];
    W[h.off_tiles + 2 * b + 1] = (int32_t)tok;
    tok += ctx_len[b];
  }
  if (!split.empty()) memcpy(W + h.off_rtile, split.data(), 4 * split.size());
  return CP_OK;
}

cp_status read_header(const void* host_plan, int want_kind, cp_plan_header* h) {
  if (!host_plan) return fail(CP_ERR_INVALID_ARG, "host_plan is NULL");
  memcpy(h, host_plan, sizeof(*h));
  if (h->magic != CP_PLAN_MAGIC) return fail(CP_ERR_INVALID_ARG, "host_plan is not a plan (bad magic)");
  if (want_kind == 2 && h->kind != 2) return fail(CP_ERR_INVALID_ARG, "expected a decode plan");
  if (want_kind != 2 && h->kind == 2) return fail(CP_ERR_INVALID_ARG, "expected a prefill plan");
  return CP_OK;
}

cp_status copy_plan(const std::vector<int32_t>& words, void* host_plan, size_t host_bytes,
                    void* dev_plan, size_t dev_bytes, size_t dev_need, cudaStream_t s) {
  const size_t hb = words.size() * 4;
  if (!host_plan) return fail(CP_ERR_INVALID_ARG, "host_plan is NULL");
  if (host_bytes < hb) return fail(CP_ERR_INVALID_ARG, "host_bytes %zu < %zu needed", host_bytes, hb);
  memcpy(host_plan, words.data(), hb);
  if (!dev_plan) return CP_OK;  // host-only planning
  if (!aligned16(dev_plan)) return fail(CP_ERR_INVALID_ARG, "dev_plan is not 16-byte aligned");
  if (dev_bytes < dev_need) return fail(CP_ERR_INVALID_ARG, "dev_bytes %zu < %zu needed", dev_bytes, dev_need);
  cudaError_t e = cudaMemcpyAsync(dev_plan, host_plan, hb, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "plan copy");
  return CP_OK;
}

size_t elem_size(cp_dtype d) { return d == CP_FP32 ? 4 : d == CP_BF16 ? 2 : 1; }

}  // namespace

namespace cpattn {
cp_status report_error(cp_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

unsigned* device_status_ptr() {
  static unsigned* ptrs[256] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return nullptr;
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_cp_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned*>(p);
  }
  return ptrs[dev];
}
}  // namespace cpattn

// ====================================================================== decode helpers

namespace {

long long pair_rows_of_shard(const cp_plan_header& h, const int32_t* W, int r) {
  long long rows = 0;
  for (int b = 0; b < h.R; ++b) rows += W[h.off_rank + kPairWords * (r * h.R + b)];
  return rows;
}

// Page table checks on its host copy: page size, pages per pair, page ids
// in range and, when the call writes the pool, no page used twice.
cp_status check_pages(const cp_plan_header& h, const int32_t* W, const int32_t* host_table,
                      int max_pages, int page_size, int num_pages, bool distinct, RowMap* rm,
                      const int32_t* dev_table) {
  if (!host_table || !dev_table) return fail(CP_ERR_INVALID_ARG, "page table (host and device copies) is NULL");
  if (!aligned16(dev_table)) return fail(CP_ERR_INVALID_ARG, "device page table is not 16-byte aligned");
  if (page_size < 64 || page_size % 64) return fail(CP_ERR_UNSUPPORTED, "page_size=%d is not a positive multiple of 64", page_size);
  if (max_pages < 1 || num_pages < 1) return fail(CP_ERR_INVALID_ARG, "max_pages=%d, num_pages=%d must be >= 1", max_pages, num_pages);
  const long long pool_rows = (long long)num_pages * page_size;
  if (pool_rows > 0x7FFFFF00LL) return fail(CP_ERR_UNSUPPORTED, "pool of %lld rows is too large", pool_rows);
  std::vector<uint8_t> used(distinct ? (size_t)num_pages : 0, 0);
  for (int pr = 0; pr < h.C * h.R; ++pr) {
    const int rows = W[h.off_rank + kPairWords * pr];
    const int need = (rows + page_size - 1) / page_size;
    if (need > max_pages)
      return fail(CP_ERR_INVALID_ARG, "pair %d needs %d pages > max_pages=%d", pr, need, max_pages);
    for (int i = 0; i < need; ++i) {
      const int pg = host_table[(size_t)pr * max_pages + i];
      if (pg < 0 || pg >= num_pages)
        return fail(CP_ERR_INVALID_ARG, "pair %d page %d: id %d outside [0, %d)", pr, i, pg, num_pages);
      if (distinct) {
        if (used[pg]) return fail(CP_ERR_INVALID_ARG, "page %d is used twice", pg);
        used[pg] = 1;
      }
    }
  }
  rm->table = dev_table;
  rm->max_pages = max_pages;
  rm->page_size = page_size;
  rm->pool_rows = pool_rows;
  return ok();
}

cp_status check_decode_shapes(cp_decode_mode mode, cp_dtype kv_dtype, bool has_v, bool has_scale,
                              int Hq, int Hkv, int Dqk, int Dv, float sm_scale, int s_q) {
  if (!(sm_scale > 0.f)) return fail(CP_ERR_INVALID_ARG, "sm_scale must be > 0");
  if (mode != CP_DECODE_MLA && mode != CP_DECODE_GQA) return fail(CP_ERR_INVALID_ARG, "bad mode");
  if (mode == CP_DECODE_MLA) {
    if (Dqk != 576 || Dv != 512 || Hkv != 1) return fail(CP_ERR_UNSUPPORTED, "MLA needs Dqk=576, Dv=512, Hkv=1");
    if (Hq < 1 || Hq * s_q > 64)
      return fail(CP_ERR_UNSUPPORTED, "MLA Hq=%d x s_q=%d query rows outside [1, 64]", Hq, s_q);
    if (kv_dtype != CP_BF16 && kv_dtype != CP_FP8_E4M3) return fail(CP_ERR_UNSUPPORTED, "MLA cache must be bf16 or fp8");
    if (has_v) return fail(CP_ERR_INVALID_ARG, "MLA takes values from the latent: shard_v must be NULL");
    if ((kv_dtype == CP_FP8_E4M3) != has_scale)
      return fail(CP_ERR_INVALID_ARG, "shard_scale is required for fp8 and only for fp8");
  } else {
    if (Dqk != Dv || Dqk % 32 || Dqk < 32 || Dqk > 256) return fail(CP_ERR_UNSUPPORTED, "GQA needs Dqk == Dv, a multiple of 32 up to 256");
    if (Hq < 1 || Hkv < 1 || Hq % Hkv) return fail(CP_ERR_INVALID_ARG, "Hq=%d must be a multiple of Hkv=%d", Hq, Hkv);
    if (kv_dtype != CP_BF16 && kv_dtype != CP_FP32 && kv_dtype != CP_FP8_E4M3)
      return fail(CP_ERR_UNSUPPORTED, "GQA cache must be bf16, fp32 or fp8");
    if (!has_v) return fail(CP_ERR_INVALID_ARG, "GQA needs shard_v");
    if ((kv_dtype == CP_FP8_E4M3) != has_scale)
      return fail(CP_ERR_INVALID_ARG, "shard_scale is required for fp8 and only for fp8");
  }
  return ok();
}

// Workspace check, kernel dispatch and the split-pair merge shared by the
// contiguous and the paged decode.
cp_status run_decode(const cp_plan_header& h, const void* dev_plan, cp_decode_mode mode,
                     cp_dtype kv_dtype, const void* q, const ShardPtrs& K, const ShardPtrs& V,
                     const ScalePtrs& S, const long long* shard_rows, const RowMap& rm, int Hq,
                     int Hkv, int Dqk, int Dv, float sm_scale, float* o_part, float* lse_part,
                     void* ws, size_t ws_bytes, void* stream, const int32_t* pair_count = nullptr) {
  const int Hc = Hq * plan_s_q(h);  // query rows x heads: the kernels' head columns
  size_t need = (size_t)h.n_parts * Hc * (Dv + 1) * sizeof(float);
  if (ws_bytes < need || (need && !ws)) return fail(CP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  if (need && !aligned16(ws)) return fail(CP_ERR_INVALID_ARG, "ws is not 16-byte aligned");
  float* ws_o = (float*)ws;
  float* ws_lse = ws_o ? ws_o + (size_t)h.n_parts * Hc * Dv : nullptr;
  cudaStream_t s = (cudaStream_t)stream;
  const bool mla = mode == CP_DECODE_MLA;
  const int32_t* plan = (const int32_t*)dev_plan;
  cudaError_t e;
  if (mla && kv_dtype == CP_FP8_E4M3)
    e = launch_decode_mla_fp8(plan, h, q, K, S, shard_rows, rm, Hq, sm_scale, o_part, lse_part, ws_o, ws_lse,
                              pair_count, wait_limit_ns(), s);
  else if (mla)
    e = launch_decode_mla_tc(plan, h, q, K, shard_rows, rm, Hq, sm_scale, o_part, lse_part, ws_o, ws_lse,
                             pair_count, wait_limit_ns(), s);
  else if (kv_dtype == CP_FP8_E4M3 && gqa_f8_supported(Hq, Hkv, Dqk, Dv, plan_s_q(h), rm.table != nullptr))
    e = launch_decode_gqa_f8(plan, h, q, K, V, S, shard_rows, Hq, Hkv, sm_scale, o_part, lse_part, ws_o, ws_lse,
                             pair_count, wait_limit_ns(), s);
  else if (gqa_tc_supported(kv_dtype, Hq, Hkv, Dqk, Dv, plan_s_q(h)))
    e = launch_decode_gqa_tc(plan, h, q, K, V, shard_rows, rm, Hq, Hkv, Dqk, sm_scale, o_part, lse_part, ws_o,
                             ws_lse, pair_count, wait_limit_ns(), s);
  else if (kv_dtype == CP_FP32 && gqa_tf32_supported(Hq, Hkv, Dqk, Dv, plan_s_q(h), rm.table != nullptr))
    e = launch_decode_gqa_tf32(plan, h, q, K, V, Hq, Hkv, Dqk, sm_scale, o_part, lse_part, ws_o, ws_lse,
                               pair_count, s);
  else  // paged fp32 or FP8 pools, other head dims, more query columns per kv head: CUDA cores
    e = launch_decode_simt(plan, h, kv_dtype, q, K, V, S, rm, Hq, Hkv, Dqk, Dv, sm_scale, o_part, lse_part,
                           ws_o, ws_lse, pair_count, s);
  if (e != cudaSuccess) return cuda_fail(e, "decode kernel");
  if (h.n_split) {
    e = launch_decode_fixup((const int32_t*)dev_plan, h, Hc, Dv, ws_o, ws_lse, o_part, lse_part, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode split merge kernel");
  }
  return ok();
}

// The decode and the merge of its partials into o / lse: over an MLA cache
// (FP8 or bf16) a worker's items of one request accumulate as one run (the
// plan's run table) and only runs cut by a worker boundary leave parts; GQA
// caches write the per-shard partials into the workspace and merge them there.
cp_status run_decode_merged(const cp_plan_header& h, const int32_t* W, const void* dev_plan, cp_decode_mode mode,
                            cp_dtype kv_dtype, const void* q, const ShardPtrs& K, const ShardPtrs& V,
                            const ScalePtrs& S, const long long* shard_rows, int Hq, int Hkv, int Dqk, int Dv,
                            float sm_scale, void* o, cp_dtype o_dtype, float* lse, void* ws, size_t ws_bytes,
                            void* stream, const int32_t* pair_count) {
  RowMap rm;
  memset(&rm, 0, sizeof(rm));
  cudaStream_t s = (cudaStream_t)stream;
  const int Hc = Hq * plan_s_q(h);
  const bool bf16 = o_dtype == CP_BF16;
  if (mode == CP_DECODE_MLA) {
    // runs accumulate in the kernel; only the runs cut by a worker boundary leave parts
    const int n_mparts = W[h.off_run], n_list = W[h.off_run + 1];
    float* ws_o = (float*)ws;
    float* ws_lse = ws_o ? ws_o + (size_t)n_mparts * Hc * Dv : nullptr;
    const int32_t* plan = (const int32_t*)dev_plan;
    const MergedOut mo = {plan + h.off_run + 2, o, bf16, lse};
    cudaError_t e = kv_dtype == CP_FP8_E4M3
                        ? launch_decode_mla_fp8(plan, h, q, K, S, shard_rows, rm, Hq, sm_scale, nullptr, nullptr,
                                                ws_o, ws_lse, pair_count, wait_limit_ns(), s, &mo)
                        : launch_decode_mla_tc(plan, h, q, K, shard_rows, rm, Hq, sm_scale, nullptr, nullptr, ws_o,
                                               ws_lse, pair_count, wait_limit_ns(), s, &mo);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel");
    e = launch_merge_runs(plan, h, n_list, Hc, Dv, ws_o, ws_lse, o, bf16, lse, s);
    if (e != cudaSuccess) return cuda_fail(e, "merge of the runs' parts");
    return ok();
  }
  // other caches: the per-shard partials in the workspace, then their merge
  float* o_part = (float*)ws;
  float* lse_part = o_part + (size_t)h.C * h.R * Hc * Dv;
  const size_t part_bytes = ((size_t)h.C * h.R * Hc * (Dv + 1) * sizeof(float) + 15) / 16 * 16;
  const cp_status st = run_decode(h, dev_plan, mode, kv_dtype, q, K, V, S, shard_rows, rm, Hq, Hkv, Dqk, Dv,
                                  sm_scale, o_part, lse_part, (uint8_t*)ws + part_bytes, ws_bytes - part_bytes,
                                  stream, pair_count);
  if (st != CP_OK) return st;
  const cudaError_t e = launch_lse_merge(h.C, h.R, Hc, Dv, o_part, lse_part, o, bf16, lse, s);
  if (e != cudaSuccess) return cuda_fail(e, "LSE merge kernel");
  return ok();
}


}  // namespace

// ====================================================================== C ABI

extern "C" {

const char* cp_last_error(void) { return g_err.c_str(); }

int cp_version(void) { return CPATTN_VERSION; }

cp_status cp_device_error_check(void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned st[4] = {0, 0, 0, 0};
  e = cudaMemcpyFromSymbol(st, g_cp_status, sizeof(st));
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  if (st[0]) {
    unsigned zero[4] = {0, 0, 0, 0};
    cudaMemcpyToSymbol(g_cp_status, zero, sizeof(zero));
    return fail(CP_ERR_DEVICE_TIMEOUT, "kernel %u gave up a bounded wait at site %u (block %u)",
                st[1], st[2], st[3]);
  }
  return ok();
}

cp_status cp_plan_size(cp_strategy strategy, int C, int R, const int32_t* new_len,
                       const int32_t* prefix_len, size_t* host_bytes, size_t* dev_bytes) {
  if (!host_bytes || !dev_bytes) return fail(CP_ERR_INVALID_ARG, "size outputs are NULL");
  PrefillBuild b;
  cp_status st = build_prefill_plan(strategy, C, R, new_len, prefix_len, &b);
  if (st != CP_OK) return st;
  *host_bytes = b.words.size() * 4;
  *dev_bytes = (size_t)b.dev_words * 4;
  return ok();
}

cp_status cp_shard_plan(cp_strategy strategy, int C, int R, const int32_t* new_len,
                        const int32_t* prefix_len, void* host_plan, size_t host_bytes,
                        void* dev_plan, size_t dev_bytes, void* stream) {
  PrefillBuild b;
  cp_status st = build_prefill_plan(strategy, C, R, new_len, prefix_len, &b);
  if (st != CP_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  st = copy_plan(b.words, host_plan, host_bytes, dev_plan, dev_bytes, (size_t)b.dev_words * 4, s);
  if (st != CP_OK || !dev_plan) return st == CP_OK ? ok() : st;
  cp_plan_header h;
  memcpy(&h, b.words.data(), sizeof(h));
  cudaError_t e = launch_plan_maps((const int32_t*)dev_plan, h.n_seg, h.off_seg, h.off_idx,
                                   h.off_qpos, h.off_qreq, s);
  if (e != cudaSuccess) return cuda_fail(e, "plan map kernel");
  return ok();
}

cp_status cp_prefill_attn(const void* host_plan, const void* dev_plan, int rank, cp_dtype dtype,
                          const void* q, const void* k, const void* v, int Hq, int Hkv, int D,
                          float sm_scale, void* o, float* lse, void* stream) {
  cp_plan_header h;
  cp_status st = read_header(host_plan, 0, &h);
  if (st != CP_OK) return st;
  if (!dev_plan || !q || !k || !v || !o || !lse) return fail(CP_ERR_INVALID_ARG, "a pointer argument is NULL");
  if (!aligned16(dev_plan) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(CP_ERR_INVALID_ARG, "a device pointer is not 16-byte aligned");
  if (rank < -1 || rank >= h.C) return fail(CP_ERR_INVALID_ARG, "rank=%d outside [-1, %d)", rank, h.C);
  if (Hq < 1 || Hkv < 1 || Hq % Hkv) return fail(CP_ERR_INVALID_ARG, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  if (dtype != CP_BF16 && dtype != CP_FP32) return fail(CP_ERR_UNSUPPORTED, "prefill dtype must be bf16 or fp32");
  if (D < 32 || D > 128 || D % 32) return fail(CP_ERR_UNSUPPORTED, "head dim D=%d: need a multiple of 32 in [32, 128]", D);
  if (!(sm_scale > 0.f)) return fail(CP_ERR_INVALID_ARG, "sm_scale must be > 0");
  const int32_t* W = (const int32_t*)host_plan;
  const int row_begin = rank < 0 ? 0 : W[h.off_rank + rank];
  const int n_rows = rank < 0 ? h.T : W[h.off_rank + rank + 1] - W[h.off_rank + rank];
  if (n_rows == 0) return ok();
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  if (dtype == CP_BF16) {
    if (D != 64 && D != 128) return fail(CP_ERR_UNSUPPORTED, "bf16 prefill needs D in {64, 128}, got %d", D);
    // Test hook for failure detection: with CPATTN_TEST_STALL=1 one bounded
    // wait in the kernel waits for a barrier nothing arrives at.
    const char* stall = getenv("CPATTN_TEST_STALL");
    e = launch_prefill_tc((const int32_t*)dev_plan, W, h, rank, q, k, v, Hq, Hkv, D, sm_scale, o,
                          lse, stall && stall[0] == '1', s);
  } else if (prefill_tf32_supported(D)) {
    e = launch_prefill_tf32((const int32_t*)dev_plan, W, h, rank, q, k, v, Hq, Hkv, D, sm_scale, o, lse, s);
  } else {  // fp32 at head dims 32 and 96: CUDA cores
    e = launch_prefill_simt((const int32_t*)dev_plan, h, rank, row_begin, n_rows, false, q, k, v,
                            Hq, Hkv, D, sm_scale, o, lse, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "prefill kernel");
  return ok();
}

cp_status cp_decode_plan_size(int C, int B, const int32_t* ctx_len, int n_workers,
                              size_t* host_bytes, size_t* dev_bytes) {
  if (!host_bytes || !dev_bytes) return fail(CP_ERR_INVALID_ARG, "size outputs are NULL");
  DecodeBuild b;
  cp_status st = build_decode_plan(C, B, ctx_len, CP_DCP_ROUND_ROBIN, 1, n_workers, &b);
  if (st != CP_OK) return st;
  *host_bytes = *dev_bytes = b.words.size() * 4;
  return ok();
}

cp_status cp_decode_plan_ex_size(int C, int B, const int32_t* ctx_len, cp_dcp_layout layout, int s_q,
                                 int n_workers, size_t* host_bytes, size_t* dev_bytes) {
  if (!host_bytes || !dev_bytes) return fail(CP_ERR_INVALID_ARG, "size outputs are NULL");
  if (layout == CP_DCP_SELECTED) return fail(CP_ERR_INVALID_ARG, "selection plans come from cp_sparse_plan");
  DecodeBuild b;
  cp_status st = build_decode_plan(C, B, ctx_len, (int)layout, s_q, n_workers, &b);
  if (st != CP_OK) return st;
  *host_bytes = *dev_bytes = b.words.size() * 4;
  return ok();
}

cp_status cp_decode_plan_ex(int C, int B, const int32_t* ctx_len, cp_dcp_layout layout, int s_q,
                            int n_workers, void* host_plan, size_t host_bytes, void* dev_plan,
                            size_t dev_bytes, void* stream) {
  if (layout == CP_DCP_SELECTED) return fail(CP_ERR_INVALID_ARG, "selection plans come from cp_sparse_plan");
  DecodeBuild b;
  cp_status st = build_decode_plan(C, B, ctx_len, (int)layout, s_q, n_workers, &b);
  if (st != CP_OK) return st;
  st = copy_plan(b.words, host_plan, host_bytes, dev_plan, dev_bytes, b.words.size() * 4,
                 (cudaStream_t)stream);
  return st == CP_OK ? ok() : st;
}

cp_status cp_decode_plan(int C, int B, const int32_t* ctx_len, int n_workers, void* host_plan,
                         size_t host_bytes, void* dev_plan, size_t dev_bytes, void* stream) {
  DecodeBuild b;
  cp_status st = build_decode_plan(C, B, ctx_len, CP_DCP_ROUND_ROBIN, 1, n_workers, &b);
  if (st != CP_OK) return st;
  st = copy_plan(b.words, host_plan, host_bytes, dev_plan, dev_bytes, b.words.size() * 4,
                 (cudaStream_t)stream);
  return st == CP_OK ? ok() : st;
}

cp_status cp_kv_shard_pack(const void* host_plan, const void* dev_plan, cp_dtype dtype,
                           const void* kv, const float* kv_scale, int row_elems,
                           void* const* shard_kv, float* const* shard_scale, void* stream) {
  cp_plan_header h;
  cp_status st = read_header(host_plan, 2, &h);
  if (st != CP_OK) return st;
  if (!dev_plan || !kv || !shard_kv) return fail(CP_ERR_INVALID_ARG, "a pointer argument is NULL");
  if (dtype != CP_BF16 && dtype != CP_FP32 && dtype != CP_FP8_E4M3) return fail(CP_ERR_INVALID_ARG, "bad dtype");
  if (row_elems < 1) return fail(CP_ERR_INVALID_ARG, "row_elems=%d < 1", row_elems);
  const size_t rb = (size_t)row_elems * elem_size(dtype);
  if (rb % 16) return fail(CP_ERR_UNSUPPORTED, "row bytes %zu not a multiple of 16", rb);
  if ((kv_scale == nullptr) != (shard_scale == nullptr))
    return fail(CP_ERR_INVALID_ARG, "kv_scale and shard_scale must both be given or both NULL");
  if (!aligned16(kv) || !aligned16(dev_plan)) return fail(CP_ERR_INVALID_ARG, "kv/dev_plan not 16-byte aligned");
  MutShardPtrs dst;
  MutScalePtrs dsc;
  memset(&dst, 0, sizeof(dst));
  memset(&dsc, 0, sizeof(dsc));
  const int32_t* W = (const int32_t*)host_plan;
  for (int r = 0; r < h.C; ++r) {
    long long rows_r = 0;
    for (int b = 0; b < h.R; ++b) rows_r += W[h.off_rank + kPairWords * (r * h.R + b)];
    dst.p[r] = shard_kv[r];
    if (rows_r > 0 && (!shard_kv[r] || !aligned16(shard_kv[r])))
      return fail(CP_ERR_INVALID_ARG, "shard_kv[%d] is NULL or misaligned", r);
    if (shard_scale) {
      dsc.p[r] = shard_scale[r];
      if (rows_r > 0 && !shard_scale[r]) return fail(CP_ERR_INVALID_ARG, "shard_scale[%d] is NULL", r);
    }
  }
  if (h.T == 0) return ok();
  RowMap rm;
  memset(&rm, 0, sizeof(rm));
  cudaError_t e = launch_kv_pack((const int32_t*)dev_plan, h, (int)elem_size(dtype), kv, kv_scale,
                                 row_elems, dst, dsc, kv_scale != nullptr, rm, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kv pack kernel");
  return ok();
}

cp_status cp_decode_workspace_size(const void* host_plan, int H, int Dv, size_t* bytes) {
  cp_plan_header h;
  cp_status st = read_header(host_plan, 2, &h);
  if (st != CP_OK) return st;
  if (!bytes || H < 1 || Dv < 1) return fail(CP_ERR_INVALID_ARG, "bad arguments");
  *bytes = (size_t)h.n_parts * H * plan_s_q(h) * (Dv + 1) * sizeof(float);
  return ok();
}

cp_status cp_decode_attn(const void* host_plan, const void* dev_plan, cp_decode_mode mode,
                         cp_dtype kv_dtype, const void* q, const void* const* shard_k,
                         const void* const* shard_v, const float* const* shard_scale, int Hq,
                         int Hkv, int Dqk, int Dv, float sm_scale, float* o_part, float* lse_part,
                         void* ws, size_t ws_bytes, void* stream) {
  cp_plan_header h;
  cp_status st = read_header(host_plan, 2, &h);
  if (st != CP_OK) return st;
  if (!dev_plan || !q || !shard_k || !o_part || !lse_part) return fail(CP_ERR_INVALID_ARG, "a pointer argument is NULL");
  if (!aligned16(dev_plan) || !aligned16(q) || !aligned16(o_part) || !aligned16(lse_part))
    return fail(CP_ERR_INVALID_ARG, "a device pointer is not 16-byte aligned");
  st = check_decode_shapes(mode, kv_dtype, shard_v != nullptr, shard_scale != nullptr, Hq, Hkv, Dqk,
                           Dv, sm_scale, plan_s_q(h));
  if (st != CP_OK) return st;
  ShardPtrs K, V;
  ScalePtrs S;
  memset(&K, 0, sizeof(K));
  memset(&V, 0, sizeof(V));
  memset(&S, 0, sizeof(S));
  const int32_t* W = (const int32_t*)host_plan;
  long long shard_rows[CP_MAX_SHARDS] = {0};
  for (int r = 0; r < h.C; ++r) {
    const long long rows_r = pair_rows_of_shard(h, W, r);
    shard_rows[r] = rows_r;
    K.p[r] = shard_k[r];
    if (rows_r > 0 && (!shard_k[r] || !aligned16(shard_k[r]))) return fail(CP_ERR_INVALID_ARG, "shard_k[%d] NULL or misaligned", r);
    if (shard_v) {
      V.p[r] = shard_v[r];
      if (rows_r > 0 && (!shard_v[r] || !aligned16(shard_v[r]))) return fail(CP_ERR_INVALID_ARG, "shard_v[%d] NULL or misaligned", r);
    }
    if (shard_scale) {
      S.p[r] = shard_scale[r];
      if (rows_r > 0 && !shard_scale[r]) return fail(CP_ERR_INVALID_ARG, "shard_scale[%d] is NULL", r);
    }
  }
  RowMap rm;
  memset(&rm, 0, sizeof(rm));
  return run_decode(h, dev_plan, mode, kv_dtype, q, K, V, S, shard_rows, rm, Hq, Hkv, Dqk, Dv,
                    sm_scale, o_part, lse_part, ws, ws_bytes, stream);
}

cp_status cp_decode_merged_workspace_size(const void* host_plan, cp_decode_mode mode, cp_dtype kv_dtype, int H,
                                          int Dv, size_t* bytes) {
  cp_plan_header h;
  cp_status st = read_header(host_plan, 2, &h);
  if (st != CP_OK) return st;
  if (!bytes || H < 1 || Dv < 1) return fail(CP_ERR_INVALID_ARG, "bad arguments");
  if (h.off_run <= 0) return fail(CP_ERR_INVALID_ARG, "the plan has no run table");
  const size_t Hc = (size_t)H * plan_s_q(h);
  const int32_t* W = (const int32_t*)host_plan;
  if (mode == CP_DECODE_MLA)  // the runs' parts
    *bytes = (size_t)W[h.off_run] * Hc * (Dv + 1) * sizeof(float);
  else  // the per-shard partials, then the split-KV scratch
    *bytes = ((size_t)h.C * h.R * Hc * (Dv + 1) * sizeof(float) + 15) / 16 * 16 +
             (size_t)h.n_parts * Hc * (Dv + 1) * sizeof(float);
  return ok();
}

cp_status cp_decode_attn_merged(const void* host_plan, const void* dev_plan, cp_decode_mode mode,
                                cp_dtype kv_dtype, const void* q, const void* const* shard_k,
                                const void* const* shard_v, const float* const* shard_scale, int Hq, int Hkv,
                                int Dqk, int Dv, float sm_scale, void* o, cp_dtype o_dtype, float* lse, void* ws,
                                size_t ws_bytes, void* stream) {
  cp_plan_header h;
  cp_status st = read_header(host_plan, 2, &h);
  if (st != CP_OK) return st;
  if (!dev_plan || !q || !shard_k || !o || !lse) return fail(CP_ERR_INVALID_ARG, "a pointer argument is NULL");
  if (!aligned16(dev_plan) || !aligned16(q) || !aligned16(o) || !aligned16(lse))
    return fail(CP_ERR_INVALID_ARG, "a device pointer is not 16-byte aligned");
  if (o_dtype != CP_BF16 && o_dtype != CP_FP32) return fail(CP_ERR_INVALID_ARG, "o_dtype must be bf16 or fp32");
  if (h.off_run <= 0) return fail(CP_ERR_INVALID_ARG, "the plan has no run table");
  if (h.layout == CP_DCP_SELECTED) return fail(CP_ERR_INVALID_ARG, "a selection plan goes to cp_sparse_decode_attn");
  st = check_decode_shapes(mode, kv_dtype, shard_v != nullptr, shard_scale != nullptr, Hq, Hkv, Dqk, Dv, sm_scale,
                           plan_s_q(h));
  if (st != CP_OK) return st;
  size_t need = 0;
  st = cp_decode_merged_workspace_size(host_plan, mode, kv_dtype, Hq, Dv, &need);
  if (st != CP_OK) return st;
  if (ws_bytes < need || (need && !ws)) return fail(CP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  if (need && !aligned16(ws)) return fail(CP_ERR_INVALID_ARG, "ws is not 16-byte aligned");
  ShardPtrs K, V;
  ScalePtrs S;
  memset(&K, 0, sizeof(K));
  memset(&V, 0, sizeof(V));
  memset(&S, 0, sizeof(S));
  const int32_t* W = (const int32_t*)host_plan;
  long long shard_rows[CP_MAX_SHARDS] = {0};
  for (int r = 0; r < h.C; ++r) {
    const long long rows_r = pair_rows_of_shard(h, W, r);
    shard_rows[r] = rows_r;
    K.p[r] = shard_k[r];
    if (rows_r > 0 && (!shard_k[r] || !aligned16(shard_k[r]))) return fail(CP_ERR_INVALID_ARG, "shard_k[%d] NULL or misaligned", r);
    if (shard_v) {
      V.p[r] = shard_v[r];
      if (rows_r > 0 && (!shard_v[r] || !aligned16(shard_v[r]))) return fail(CP_ERR_INVALID_ARG, "shard_v[%d] NULL or misaligned", r);
    }
    if (shard_scale) {
      S.p[r] = shard_scale[r];
      if (rows_r > 0 && !shard_scale[r]) return fail(CP_ERR_INVALID_ARG, "shard_scale[%d] is NULL", r);
    }
  }
  return run_decode_merged(h, (const int32_t*)host_plan, dev_plan, mode, kv_dtype, q, K, V, S, shard_rows, Hq,
                           Hkv, Dqk, Dv, sm_scale, o, o_dtype, lse, ws, ws_bytes, stream, nullptr);
}

cp_status cp_decode_attn_paged(const void* host_plan, const void* dev_plan, cp_decode_mode mode,
                               cp_dtype kv_dtype, const void* q, const void* k_pool,
                               const void* v_pool, const float* scale_pool,
                               const int32_t* host_page_table, const int32_t* dev_page_table,
                               int max_pages, int page_size, int num_pages, int Hq, int Hkv,
                               int Dqk, int Dv, float sm_scale, float* o_part, float* lse_part,
                               void* ws, size_t ws_bytes, void* stream) {
  cp_plan_header h;
  cp_status st = read_header(host_plan, 2, &h);
  if (st != CP_OK) return st;
  if (!dev_plan || !q || !k_pool || !o_part || !lse_part) return fail(CP_ERR_INVALID_ARG, "a pointer argument is NULL");
  if (!aligned16(dev_plan) || !aligned16(q) || !aligned16(o_part) || !aligned16(lse_part) ||
      !aligned16(k_pool) || (v_pool && !aligned16(v_pool)))
    return fail(CP_ERR_INVALID_ARG, "a device pointer is not 16-byte aligned");
  st = check_decode_shapes(mode, kv_dtype, v_pool != nullptr, scale_pool != nullptr, Hq, Hkv, Dqk,
                           Dv, sm_scale, plan_s_q(h));
  if (st != CP_OK) return st;
  RowMap rm;
  st = check_pages(h, (const int32_t*)host_plan, host_page_table, max_pages, page_size, num_pages,
                   false, &rm, dev_page_table);
  if (st != CP_OK) return st;
  ShardPtrs K, V;
  ScalePtrs S;
  long long shard_rows[CP_MAX_SHARDS] = {0};
  for (int r = 0; r < CP_MAX_SHARDS; ++r) {  // every shard reads the one pool
    K.p[r] = k_pool;
    V.p[r] = v_pool;
    S.p[r] = scale_pool;
    if (r < h.C) shard_rows[r] = pair_rows_of_shard(h, (const int32_t*)host_plan, r);
  }
  return run_decode(h, dev_plan, mode, kv_dtype, q, K, V, S, shard_rows, rm, Hq, Hkv, Dqk, Dv,
                    sm_scale, o_part, lse_part, ws, ws_bytes, stream);
}

cp_status cp_kv_shard_pack_paged(const void* host_plan, const void* dev_plan, cp_dtype dtype,
                                 const void* kv, const float* kv_scale, int row_elems, void* pool,
                                 float* scale_pool, const int32_t* host_page_table,
                                 const int32_t* dev_page_table, int max_pages, int page_size,
                                 int num_pages, void* stream) {
  cp_plan_header h;
  cp_status st = read_header(host_plan, 2, &h);
  if (st != CP_OK) return st;
  if (!dev_plan || !kv || !pool) return fail(CP_ERR_INVALID_ARG, "a pointer argument is NULL");
  if (dtype != CP_BF16 && dtype != CP_FP32 && dtype != CP_FP8_E4M3) return fail(CP_ERR_INVALID_ARG, "bad dtype");
  if (row_elems < 1) return fail(CP_ERR_INVALID_ARG, "row_elems=%d < 1", row_elems);
  const size_t rb = (size_t)row_elems * elem_size(dtype);
  if (rb % 16) return fail(CP_ERR_UNSUPPORTED, "row bytes %zu not a multiple of 16", rb);
  if ((kv_scale == nullptr) != (scale_pool == nullptr))
    return fail(CP_ERR_INVALID_ARG, "kv_scale and scale_pool must both be given or both NULL");
  if (!aligned16(kv) || !aligned16(dev_plan) || !aligned16(pool))
    return fail(CP_ERR_INVALID_ARG, "kv/pool/dev_plan not 16-byte aligned");
  RowMap rm;
  st = check_pages(h, (const int32_t*)host_plan, host_page_table, max_pages, page_size, num_pages,
                   true, &rm, dev_page_table);
  if (st != CP_OK) return st;
  MutShardPtrs dst;
  MutScalePtrs dsc;
  for (int r = 0; r < CP_MAX_SHARDS; ++r) {
    dst.p[r] = pool;
    dsc.p[r] = scale_pool;
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (h.T > 0) {
    cudaError_t e = launch_kv_pack((const int32_t*)dev_plan, h, (int)elem_size(dtype), kv, kv_scale,
                                   row_elems, dst, dsc, kv_scale != nullptr, rm, s);
    if (e != cudaSuccess) return cuda_fail(e, "kv pack kernel");
  }
  cudaError_t e = launch_page_tail_zero((const int32_t*)dev_plan, h, rb, pool, scale_pool, rm, s);
  if (e != cudaSuccess) return cuda_fail(e, "page tail kernel");
  return ok();
}

cp_status cp_lse_merge(int P, int N, int H, int Dv, const float* o_part, const float* lse_part,
                       void* o, cp_dtype o_dtype, float* lse, void* stream) {
  if (P < 1 || P > CP_MAX_SHARDS) return fail(CP_ERR_INVALID_ARG, "P=%d outside [1, %d]", P, CP_MAX_SHARDS);
  if (N < 0 || H < 1 || Dv < 4 || Dv % 4) return fail(CP_ERR_INVALID_ARG, "bad shape N=%d H=%d Dv=%d", N, H, Dv);
  if (!o_part || !lse_part || !o) return fail(CP_ERR_INVALID_ARG, "a pointer argument is NULL");
  if (!aligned16(o_part) || !aligned16(o)) return fail(CP_ERR_INVALID_ARG, "o_part/o not 16-byte aligned");
  if (o_dtype != CP_BF16 && o_dtype != CP_FP32) return fail(CP_ERR_UNSUPPORTED, "merge output must be bf16 or fp32");
  if (N == 0) return ok();
  cudaError_t e = launch_lse_merge(P, N, H, Dv, o_part, lse_part, o, o_dtype == CP_BF16, lse,
                                   (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "merge kernel");
  return ok();
}

cp_status cp_lse_fold(int N, int H, int Dv, float* o, float* lse, const float* o_add,
                      const float* lse_add, void* stream) {
  if (N < 0 || H < 1 || Dv < 1) return fail(CP_ERR_INVALID_ARG, "bad shape N=%d H=%d Dv=%d", N, H, Dv);
  if (!o || !lse || !o_add || !lse_add) return fail(CP_ERR_INVALID_ARG, "a pointer argument is NULL");
  if (N == 0) return ok();
  cudaError_t e = launch_lse_fold(N, H, Dv, o, lse, o_add, lse_add, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "fold kernel");
  return ok();
}

// ---------------------------------------------------------------- sparse decode

namespace {
constexpr int kMaxTopK = 4096;

struct TopkWs {
  uint64_t* cand_keys;  // [C * B][k]
  uint64_t* thresh;     // [B]
  uint64_t* range;      // [C * B]
  int32_t* cand_n;      // [C * B]
};
size_t topk_ws_bytes(const cp_plan_header& h, int k) {
  const size_t P = (size_t)h.C * h.R;
  return P * k * 8 + (size_t)h.R * 8 + P * 8 + ((P * 4 + 15) / 16) * 16;
}
TopkWs topk_ws(const cp_plan_header& h, int k, void* ws) {
  TopkWs w;
  const size_t P = (size_t)h.C * h.R;
  w.cand_keys = static_cast<uint64_t*>(ws);
  w.thresh = w.cand_keys + P * k;
  w.range = w.thresh + h.R;
  w.cand_n = reinterpret_cast<int32_t*>(w.range + P);
  return w;
}
cp_status check_topk_args(const cp_plan_header& h, int k) {
  if (k < 1 || k > kMaxTopK) return fail(CP_ERR_INVALID_ARG, "k=%d outside [1, %d]", k, kMaxTopK);
  if (h.layout == CP_DCP_SELECTED) return fail(CP_ERR_INVALID_ARG, "top-k runs on a cache plan, not a selection plan");
  if (plan_s_q(h) != 1) return fail(CP_ERR_UNSUPPORTED, "sparse decode takes one query row per request");
  return ok();
}
}  // namespace

cp_status cp_sparse_plan_size(int C, int B, int k, int n_workers, size_t* host_bytes,
                              size_t* dev_bytes) {
  if (!host_bytes || !dev_bytes) return fail(CP_ERR_INVALID_ARG, "size outputs are NULL");
  if (k < 1 || k > kMaxTopK) return fail(CP_ERR_INVALID_ARG, "k=%d outside [1, %d]", k, kMaxTopK);
  if (B < 1) return fail(CP_ERR_INVALID_ARG, "B=%d must be >= 1", B);
  std::vector<int32_t> cap(B, (k + kDecodeTileRows - 1) / kDecodeTileRows * kDecodeTileRows);
  DecodeBuild b;
  cp_status st = build_decode_plan(C, B, cap.data(), CP_DCP_SELECTED, 1, n_workers, &b);
  if (st != CP_OK) return st;
  *host_bytes = *dev_bytes = b.words.size() * 4;
  return ok();
}

cp_status cp_sparse_plan(int C, int B, int k, int n_workers, void* host_plan, size_t host_bytes,
                         void* dev_plan, size_t dev_bytes, void* stream) {
  if (k < 1 || k > kMaxTopK) return fail(CP_ERR_INVALID_ARG, "k=%d outside [1, %d]", k, kMaxTopK);
  if (B < 1) return fail(CP_ERR_INVALID_ARG, "B=%d must be >= 1", B);
  std::vector<int32_t> cap(B, (k + kDecodeTileRows - 1) / kDecodeTileRows * kDecodeTileRows);
  DecodeBuild b;
  cp_status st = build_decode_plan(C, B, cap.data(), CP_DCP_SELECTED, 1, n_workers, &b);
  if (st != CP_OK) return st;
  st = copy_plan(b.words, host_plan, host_bytes, dev_plan, dev_bytes, b.words.size() * 4,
                 (cudaStream_t)stream);
  return st == CP_OK ? ok() : st;
}

cp_status cp_sparse_workspace_size(const void* host_plan, int k, size_t* bytes) {
  cp_plan_header h;
  cp_status st = read_header(host_plan, 2, &h);
  if (st != CP_OK) return st;
  if (!bytes) return fail(CP_ERR_INVALID_ARG, "bytes is NULL");
  st = check_topk_args(h, k);
  if (st != CP_OK) return st;
  *bytes = topk_ws_bytes(h, k);
  return ok();
}

cp_status cp_sparse_topk(const void* host_plan, const void* dev_plan, const float* const* shard_scores,
                         int k, int32_t* sel_ids, int32_t* sel_count, void* ws, size_t ws_bytes,
                         void* stream) {
  cp_plan_header h;
  cp_status st = read_header(host_plan, 2, &h);
  if (st != CP_OK) return st;
  st = check_topk_args(h, k);
  if (st != CP_OK) return st;
  if (!dev_plan || !shard_scores || !sel_ids || !sel_count || !ws)
    return fail(CP_ERR_INVALID_ARG, "a pointer argument is NULL");
  if (!aligned16(ws) || !aligned16(dev_plan)) return fail(CP_ERR_INVALID_ARG, "ws/dev_plan not 16-byte aligned");
  if (ws_bytes < topk_ws_bytes(h, k))
    return fail(CP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, topk_ws_bytes(h, k));
  ScorePtrs sc;
  memset(&sc, 0, sizeof(sc));
  const int32_t* W = (const int32_t*)host_plan;
  for (int r = 0; r < h.C; ++r) {
    sc.p[r] = shard_scores[r];
    if (pair_rows_of_shard(h, W, r) > 0 && !shard_scores[r])
      return fail(CP_ERR_INVALID_ARG, "shard_scores[%d] is NULL", r);
  }
  int max_rows = 0;
  for (int i = 0; i < h.C * h.R; ++i) max_rows = std::max(max_rows, W[h.off_rank + kPairWords * i]);
  const TopkWs w = topk_ws(h, k, ws);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e =
      launch_topk_local((const int32_t*)dev_plan, h, sc, k, max_rows, w.cand_keys, w.cand_n, w.range, s);
  if (e != cudaSuccess) return cuda_fail(e, "local top-k kernel");
  e = launch_topk_merge((const int32_t*)dev_plan, h, k, w.cand_keys, w.cand_n, w.range, w.thresh, sel_ids,
                        sel_count, s);
  if (e != cudaSuccess) return cuda_fail(e, "top-k merge kernel");
  return ok();
}

cp_status cp_sparse_gather(const void* host_plan, const void* dev_plan, int k, const void* ws,
                           size_t ws_bytes, cp_dtype dtype, const void* const* shard_kv,
                           const float* const* shard_scale, int row_elems, void* const* sel_kv,
                           float* const* sel_scale, int32_t* pair_count, void* stream) {
  cp_plan_header h;
  cp_status st = read_header(host_plan, 2, &h);
  if (st != CP_OK) return st;
  st = check_topk_args(h, k);
  if (st != CP_OK) return st;
  if (!dev_plan || !ws || !shard_kv || !sel_kv || !pair_count)
    return fail(CP_ERR_INVALID_ARG, "a pointer argument is NULL");
  if (ws_bytes < topk_ws_bytes(h, k))
    return fail(CP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, topk_ws_bytes(h, k));
  if (dtype != CP_BF16 && dtype != CP_FP32 && dtype != CP_FP8_E4M3) return fail(CP_ERR_INVALID_ARG, "bad dtype");
  if (row_elems < 1) return fail(CP_ERR_INVALID_ARG, "row_elems=%d < 1", row_elems);
  const size_t rb = (size_t)row_elems * elem_size(dtype);
  if (rb % 16) return fail(CP_ERR_UNSUPPORTED, "row bytes %zu not a multiple of 16", rb);
  if ((shard_scale == nullptr) != (sel_scale == nullptr))
    return fail(CP_ERR_INVALID_ARG, "shard_scale and sel_scale must both be given or both NULL");
  ShardPtrs src;
  ScalePtrs ssc;
  MutShardPtrs dst;
  MutScalePtrs dsc;
  memset(&src, 0, sizeof(src));
  memset(&ssc, 0, sizeof(ssc));
  memset(&dst, 0, sizeof(dst));
  memset(&dsc, 0, sizeof(dsc));
  const int32_t* W = (const int32_t*)host_plan;
  for (int r = 0; r < h.C; ++r) {
    const bool used = pair_rows_of_shard(h, W, r) > 0;
    src.p[r] = shard_kv[r];
    dst.p[r] = sel_kv[r];
    if (used && (!shard_kv[r] || !aligned16(shard_kv[r]))) return fail(CP_ERR_INVALID_ARG, "shard_kv[%d] NULL or misaligned", r);
    if (!sel_kv[r] || !aligned16(sel_kv[r])) return fail(CP_ERR_INVALID_ARG, "sel_kv[%d] NULL or misaligned", r);
    if (shard_scale) {
      ssc.p[r] = shard_scale[r];
      dsc.p[r] = sel_scale[r];
      if ((used && !shard_scale[r]) || !sel_scale[r]) return fail(CP_ERR_INVALID_ARG, "scale pointer %d is NULL", r);
    }
  }
  const TopkWs w = topk_ws(h, k, const_cast<void*>(ws));
  cudaError_t e = launch_sparse_gather((const int32_t*)dev_plan, h, k, w.cand_keys, w.cand_n, w.thresh,
                                       src, ssc, (int)rb, dst, dsc, shard_scale != nullptr, pair_count,
                                       (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "sparse gather kernel");
  return ok();
}

cp_status cp_sparse_decode_attn(const void* host_plan, const void* dev_plan, const int32_t* pair_count,
                                cp_decode_mode mode, cp_dtype kv_dtype, const void* q,
                                const void* const* sel_k, const void* const* sel_v,
                                const float* const* sel_scale, int Hq, int Hkv, int Dqk, int Dv,
                                float sm_scale, float* o_part, float* lse_part, void* ws,
                                size_t ws_bytes, void* stream) {
  cp_plan_header h;
  cp_status st = read_header(host_plan, 2, &h);
  if (st != CP_OK) return st;
  if (h.layout != CP_DCP_SELECTED) return fail(CP_ERR_INVALID_ARG, "needs a selection plan (cp_sparse_plan)");
  if (!dev_plan || !q || !sel_k || !o_part || !lse_part || !pair_count)
    return fail(CP_ERR_INVALID_ARG, "a pointer argument is NULL");
  if (!aligned16(dev_plan) || !aligned16(q) || !aligned16(o_part) || !aligned16(lse_part))
    return fail(CP_ERR_INVALID_ARG, "a device pointer is not 16-byte aligned");
  st = check_decode_shapes(mode, kv_dtype, sel_v != nullptr, sel_scale != nullptr, Hq, Hkv, Dqk, Dv,
                           sm_scale, 1);
  if (st != CP_OK) return st;
  ShardPtrs K, V;
  ScalePtrs S;
  memset(&K, 0, sizeof(K));
  memset(&V, 0, sizeof(V));
  memset(&S, 0, sizeof(S));
  long long shard_rows[CP_MAX_SHARDS] = {0};
  for (int r = 0; r < h.C; ++r) {
    shard_rows[r] = pair_rows_of_shard(h, (const int32_t*)host_plan, r);
    K.p[r] = sel_k[r];
    if (!sel_k[r] || !aligned16(sel_k[r])) return fail(CP_ERR_INVALID_ARG, "sel_k[%d] NULL or misaligned", r);
    if (sel_v) {
      V.p[r] = sel_v[r];
      if (!sel_v[r] || !aligned16(sel_v[r])) return fail(CP_ERR_INVALID_ARG, "sel_v[%d] NULL or misaligned", r);
    }
    if (sel_scale) {
      S.p[r] = sel_scale[r];
      if (!sel_scale[r]) return fail(CP_ERR_INVALID_ARG, "sel_scale[%d] is NULL", r);
    }
  }
  RowMap rm;
  memset(&rm, 0, sizeof(rm));
  return run_decode(h, dev_plan, mode, kv_dtype, q, K, V, S, shard_rows, rm, Hq, Hkv, Dqk, Dv,
                    sm_scale, o_part, lse_part, ws, ws_bytes, stream, pair_count);
}

cp_status cp_sparse_decode_attn_merged(const void* host_plan, const void* dev_plan, const int32_t* pair_count,
                                       cp_decode_mode mode, cp_dtype kv_dtype, const void* q,
                                       const void* const* sel_k, const void* const* sel_v,
                                       const float* const* sel_scale, int Hq, int Hkv, int Dqk, int Dv,
                                       float sm_scale, void* o, cp_dtype o_dtype, float* lse, void* ws,
                                       size_t ws_bytes, void* stream) {
  cp_plan_header h;
  cp_status st = read_header(host_plan, 2, &h);
  if (st != CP_OK) return st;
  if (h.layout != CP_DCP_SELECTED) return fail(CP_ERR_INVALID_ARG, "needs a selection plan (cp_sparse_plan)");
  if (!dev_plan || !q || !sel_k || !o || !lse || !pair_count)
    return fail(CP_ERR_INVALID_ARG, "a pointer argument is NULL");
  if (!aligned16(dev_plan) || !aligned16(q) || !aligned16(o) || !aligned16(lse))
    return fail(CP_ERR_INVALID_ARG, "a device pointer is not 16-byte aligned");
  if (o_dtype != CP_BF16 && o_dtype != CP_FP32) return fail(CP_ERR_INVALID_ARG, "o_dtype must be bf16 or fp32");
  if (h.off_run <= 0) return fail(CP_ERR_INVALID_ARG, "the plan has no run table");
  st = check_decode_shapes(mode, kv_dtype, sel_v != nullptr, sel_scale != nullptr, Hq, Hkv, Dqk, Dv, sm_scale, 1);
  if (st != CP_OK) return st;
  size_t need = 0;
  st = cp_decode_merged_workspace_size(host_plan, mode, kv_dtype, Hq, Dv, &need);
  if (st != CP_OK) return st;
  if (ws_bytes < need || (need && !ws)) return fail(CP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  if (need && !aligned16(ws)) return fail(CP_ERR_INVALID_ARG, "ws is not 16-byte aligned");
  ShardPtrs K, V;
  ScalePtrs S;
  memset(&K, 0, sizeof(K));
  memset(&V, 0, sizeof(V));
  memset(&S, 0, sizeof(S));
  long long shard_rows[CP_MAX_SHARDS] = {0};
  for (int r = 0; r < h.C; ++r) {
    shard_rows[r] = pair_rows_of_shard(h, (const int32_t*)host_plan, r);
    K.p[r] = sel_k[r];
    if (!sel_k[r] || !aligned16(sel_k[r])) return fail(CP_ERR_INVALID_ARG, "sel_k[%d] NULL or misaligned", r);
    if (sel_v) {
      V.p[r] = sel_v[r];
      if (!sel_v[r] || !aligned16(sel_v[r])) return fail(CP_ERR_INVALID_ARG, "sel_v[%d] NULL or misaligned", r);
    }
    if (sel_scale) {
      S.p[r] = sel_scale[r];
      if (!sel_scale[r]) return fail(CP_ERR_INVALID_ARG, "sel_scale[%d] is NULL", r);
    }
  }
  return run_decode_merged(h, (const int32_t*)host_plan, dev_plan, mode, kv_dtype, q, K, V, S, shard_rows, Hq,
                           Hkv, Dqk, Dv, sm_scale, o, o_dtype, lse, ws, ws_bytes, stream, pair_count);
}

}  // extern "C"
