// Exact sharded top-k selection for sparse decode, and the owner-side gather
// of the selected cache rows ("DeepSeek-V4 Attention Inference Systems" §5.2;
// "How GPUs Share a Long Context During LLM Inference" §4.1, the split index).
//
// Each shard scores only the tokens it stores; the scores of one request's
// tokens on shard r are the pair (r, b) rows of a decode plan, in the plan's
// shard layout.  The steps, as the pages order them:
//   local top-k   every (shard, request) pair keeps its k best tokens;
//   merge         the at most C k candidates of a request give the exact
//                 global top-k (the union of the local lists contains it);
//   route         every owner takes the selected tokens it stores and packs
//                 their cache rows, in token order, into a selection buffer
//                 that the decode kernels read like a shard (with a count).
// Order: higher score first, and between equal scores the lower token index
// (a deterministic tie rule).  Both are one 64-bit key,
//   key = ordered(score) << 32 | (2^32 - 1 - token),
// so "the k best" is "the k largest keys" and every key is distinct; the
// k-th largest key is found by an 8-pass radix select (8 bits a pass).
#include <cuda_runtime.h>

#include "internal.h"

namespace cpattn {
namespace {

constexpr int kThreads = 512;  // 16 warps: the select's loops are latency-bound
constexpr int kMaxTopK = 4096;  // largest k (the API rejects more)
constexpr unsigned kFull = 0xffffffffu;

// float -> uint32 that increases with the float (NaN excluded; -0 ranks as +0).
__device__ __forceinline__ uint32_t ordered_bits(float f) {
  if (f == 0.f) return 0x80000000u;
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint64_t token_key(float score, int token) {
  return ((uint64_t)ordered_bits(score) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)token);
}

__device__ __forceinline__ int key_token(uint64_t key) {
  return (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}

constexpr int kWarps = kThreads / 32;
constexpr int kSmallKeys = 2048;  // keys the select finishes on in shared memory (a power of two)
constexpr int kStageScores = 32768;  // a pair's scores staged in shared memory up to this many
constexpr int kStageKeys = 16384;    // a request's candidates staged in shared memory up to this many

// Ordered compaction: calls emit(i, j) for every i in [0, n) with pred(i), j
// counting those before i; returns their number.  Each warp takes one
// contiguous segment of [0, n) in steps of 32 (coalesced, conflict-free in
// shared memory): a counting pass, one scan of the warps' totals, a writing
// pass.  All threads of the block call it; warp_cnt is kWarps ints.
template <typename Pred, typename Emit>
__device__ int block_compact(int n, Pred pred, Emit emit, int* warp_cnt) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = (n + kWarps - 1) / kWarps;
  const int s0 = min(n, warp * seg), s1 = min(n, s0 + seg);
  int cnt = 0;
  for (int b = s0; b < s1; b += 32) cnt += __popc(__ballot_sync(kFull, b + lane < s1 && pred(b + lane)));
  if (lane == 0) warp_cnt[warp] = cnt;
  __syncthreads();
  int at = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int c = warp_cnt[w];
    at += w < warp ? c : 0;
    tot += c;
  }
  for (int b = s0; b < s1; b += 32) {
    const bool f = b + lane < s1 && pred(b + lane);
    const unsigned bal = __ballot_sync(kFull, f);
    if (f) emit(b + lane, at + __popc(bal & ((1u << lane) - 1u)));
    at += __popc(bal);
  }
  __syncthreads();
  return tot;
}

// Unordered collection of the i in [0, n) with pred(i) into out[]: one shared
// counter, one atomic per warp and step.  Returns the number (all threads).
template <typename Pred, typename Get>
__device__ int block_collect(int n, Pred pred, Get value, uint64_t* out, int* counter) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) *counter = 0;
  __syncthreads();
  for (int b = 0; b < n; b += blockDim.x) {
    const int i = b + threadIdx.x;
    const bool f = i < n && pred(i);
    const unsigned bal = __ballot_sync(kFull, f);
    int base = 0;
    if (lane == 0 && bal) base = atomicAdd(counter, __popc(bal));
    base = __shfl_sync(kFull, base, 0);
    if (f) out[base + __popc(bal & ((1u << lane) - 1u))] = value(i);
  }
  __syncthreads();
  return *counter;
}

// Bytes of the merge's token list in shared memory, padded to 16 so that the
// 64-bit keys staged after it stay aligned.
__host__ __device__ __forceinline__ size_t ids_bytes(int kpow2) {
  return ((size_t)kpow2 * sizeof(int32_t) + 15) & ~(size_t)15;
}

constexpr int kTopBins = 4096;  // the first pass splits on the key's top 12 bits

// Shared scratch of the radix select.
struct __align__(16) SelectSmem {
  uint32_t hist[kTopBins];
  uint32_t pick[4];
  int small_n;
  int warp_cnt[kWarps];
  int seg_cnt[kWarps];
  uint64_t small[kSmallKeys];
};

// Finds, among the NB bins of hist taken from the top, the one that holds
// rank `want` (1-based): pick = {bin, keys in higher bins, keys in it}.  Each
// thread owns NB / blockDim consecutive bins (one, or none, when NB is
// smaller than the block); one block-wide scan.
template <int NB>
__device__ void pick_bin(const uint32_t* hist, int want, uint32_t* pick, int* warp_cnt) {
  constexpr int PER = NB >= kThreads ? NB / kThreads : 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int top = NB - 1 - PER * (int)threadIdx.x;  // this thread's highest bin (< 0: none)
  uint32_t c[PER], sum = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    c[j] = top - j >= 0 ? hist[top - j] : 0u;
    sum += c[j];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t v = __shfl_up_sync(kFull, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_cnt[warp] = (int)incl;
  __syncthreads();
  uint32_t before = 0;
  for (int w = 0; w < warp; ++w) before += (uint32_t)warp_cnt[w];
  const uint32_t excl = before + incl - sum;
  if (excl < (uint32_t)want && (uint32_t)want <= excl + sum) {
    uint32_t above = excl;
    int j = 0;
    for (; j < PER - 1 && above + c[j] < (uint32_t)want; ++j) above += c[j];
    pick[0] = (uint32_t)(top - j);
    pick[1] = above;
    pick[2] = c[j];
  }
  __syncthreads();
}

// The k-th largest (k >= 1) of n distinct keys get(0..n-1), n >= k.  A first
// pass over the keys' top 12 bits finds the bin holding rank k; 8-bit passes
// then fix the lower bits, over all n keys until the keys still in play fit
// in shared memory (kSmallKeys; they are then collected once) and over those
// from there on.  All threads of the block call it.
template <typename Get, typename Top>
__device__ uint64_t kth_largest(int n, int k, Get get, Top top12, SelectSmem& sm) {
  // top12(i) == get(i) >> 52, possibly cheaper
  for (int i = threadIdx.x; i < kTopBins; i += blockDim.x) sm.hist[i] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) atomicAdd(&sm.hist[top12(i)], 1u);
  __syncthreads();
  pick_bin<kTopBins>(sm.hist, k, sm.pick, sm.warp_cnt);
  uint64_t prefix = (uint64_t)sm.pick[0] << 52, mask = 0xFFFull << 52;
  int want = k - (int)sm.pick[1];
  int in_bin = (int)sm.pick[2];
  int m = -1;  // keys collected in sm.small, once they fit
  for (int shift = 44;; shift = shift >= 8 ? shift - 8 : 0) {
    if (m < 0 && in_bin <= kSmallKeys) {
      const uint32_t bin12 = (uint32_t)(prefix >> 52);
      m = shift == 44 ? block_collect(n, [&](int i) { return top12(i) == bin12; }, get, sm.small,
                                      &sm.small_n)
                      : block_collect(n, [&](int i) { return (get(i) & mask) == prefix; }, get,
                                      sm.small, &sm.small_n);
    }
    for (int i = threadIdx.x; i < 256; i += blockDim.x) sm.hist[i] = 0;
    __syncthreads();
    const int cnt = m < 0 ? n : m;
    for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
      const uint64_t key = m < 0 ? get(i) : sm.small[i];
      if ((key & mask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    pick_bin<256>(sm.hist, want, sm.pick, sm.warp_cnt);
    prefix = (prefix & ~(255ull << shift)) | ((uint64_t)sm.pick[0] << shift);
    mask |= 255ull << shift;
    want -= (int)sm.pick[1];
    in_bin = (int)sm.pick[2];
    if (shift == 0) return prefix;  // all 64 bits fixed
  }
}

// Sorts a[0, m) (m <= kSmallKeys) in decreasing order, padding to a power
// of two with zeros (every key is > 0).
__device__ void sort_desc_small(uint64_t* a, int m) {
  int mp = 1;
  while (mp < m) mp <<= 1;
  for (int i = m + threadIdx.x; i < mp; i += blockDim.x) a[i] = 0;
  __syncthreads();
  for (int size = 2; size <= mp; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < mp; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const bool down = (i & size) == 0;
          const uint64_t x = a[i], y = a[j];
          if ((x < y) == down) {
            a[i] = y;
            a[j] = x;
          }
        }
      }
      __syncthreads();
    }
}

// The want-th largest (1-based) of a[0, m), m <= blockDim: a bitonic sort
// with one key per thread, through shuffles for strides below 32 and through
// a (reused) for the larger ones, so that only those stages meet a barrier.
__device__ uint64_t kth_of_small(uint64_t* a, int m, int want) {
  const int t = threadIdx.x;
  int mp = 32;
  while (mp < m) mp <<= 1;
  uint64_t v = t < m ? a[t] : 0ull;  // keys are > 0: the padding sorts last
  __syncthreads();
  for (int size = 2; size <= mp; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      uint64_t o;
      if (stride >= 32) {
        a[t] = v;
        __syncthreads();
        o = a[t ^ stride];
        __syncthreads();
      } else {
        o = __shfl_xor_sync(kFull, v, stride);
      }
      const bool desc = (t & size) == 0, lower = (t & stride) == 0;
      v = desc == lower ? (v > o ? v : o) : (v < o ? v : o);
    }
  a[t] = v;
  __syncthreads();
  return a[want - 1];
}

// The staged path of a pair's local top-k: stages the scores with a
// histogram of their top 12 bits, finds the bin holding rank k, collects that
// bin (at most kSmallKeys keys) while counting, per warp segment, the keys
// above it, sorts the bin for the k-th key, and writes the candidates in
// token order: three passes over the scores.  Returns false (scores staged,
// nothing written) when the bin is larger (many equal scores).
template <typename Get, typename Top>
__device__ bool local_topk_staged(int n, int k, const float* sc, float* staged, Get get, Top top12,
                                  uint64_t* out, SelectSmem& sm, const cp_pair_desc& pd,
                                  int32_t* n_out) {
  for (int i = threadIdx.x; i < kTopBins; i += blockDim.x) sm.hist[i] = 0;
  __syncthreads();
#pragma unroll 8
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const float f = __ldg(sc + i);
    staged[i] = f;
    atomicAdd(&sm.hist[ordered_bits(f) >> 20], 1u);
  }
  __syncthreads();
  pick_bin<kTopBins>(sm.hist, k, sm.pick, sm.warp_cnt);
  const uint32_t bin = sm.pick[0];
  const int want = k - (int)sm.pick[1];
  if ((int)sm.pick[2] > kSmallKeys) return false;
  // warp w classifies keys [w seg, (w + 1) seg) in steps of 32
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = (n + kWarps * 32 - 1) / (kWarps * 32) * 32;
  const int s0 = min(n, warp * seg), s1 = min(n, s0 + seg);
  if (threadIdx.x == 0) sm.small_n = 0;
  __syncthreads();
  int above = 0;
#pragma unroll 4
  for (int b = s0; b < s1; b += 32) {
    const int i = b + lane;
    const uint32_t t = i < s1 ? top12(i) : 0u;
    above += __popc(__ballot_sync(kFull, i < s1 && t > bin));
    const bool in = i < s1 && t == bin;
    const unsigned bal = __ballot_sync(kFull, in);
    if (bal) {
      int base = 0;
      if (lane == 0) base = atomicAdd(&sm.small_n, __popc(bal));
      base = __shfl_sync(kFull, base, 0);
      if (in) sm.small[base + __popc(bal & ((1u << lane) - 1u))] = get(i);
    }
  }
  if (lane == 0) sm.seg_cnt[warp] = above;
  __syncthreads();
  const int m = sm.small_n;
  // the bin's keys that make it, counted into their warps' segments
  uint64_t thresh;
  if (m <= kThreads) {
    const uint64_t mine = threadIdx.x < m ? sm.small[threadIdx.x] : 0ull;
    thresh = kth_of_small(sm.small, m, want);
    if (mine >= thresh && threadIdx.x < m)
      atomicAdd(&sm.seg_cnt[((key_token(mine) - pd.tok0) / pd.tok_step) / seg], 1);
  } else {
    sort_desc_small(sm.small, m);
    thresh = sm.small[want - 1];
    for (int j = threadIdx.x; j < m; j += blockDim.x) {
      const uint64_t key = sm.small[j];
      if (key >= thresh) atomicAdd(&sm.seg_cnt[((key_token(key) - pd.tok0) / pd.tok_step) / seg], 1);
    }
  }
  __syncthreads();
  int at = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int c = sm.seg_cnt[w];
    at += w < warp ? c : 0;
    tot += c;
  }
  const uint32_t th_hi = (uint32_t)(thresh >> 32), th_lo = (uint32_t)thresh;
#pragma unroll 4
  for (int b = s0; b < s1; b += 32) {
    const int i = b + lane;
    bool keep = false;
    if (i < s1) {
      const uint32_t hi = ordered_bits(staged[i]);
      keep = hi > th_hi || (hi == th_hi && 0xFFFFFFFFu - (uint32_t)(pd.tok0 + i * pd.tok_step) >= th_lo);
    }
    const unsigned bal = __ballot_sync(kFull, keep);
    if (keep) out[at + __popc(bal & ((1u << lane) - 1u))] = get(i);
    at += __popc(bal);
  }
  if (threadIdx.x == 0) *n_out = tot;
  return true;
}

// Local top-k of every (shard, request) pair: candidate keys in token order.
__global__ void __launch_bounds__(kThreads)
    topk_local_kernel(const int32_t* __restrict__ plan, int B, int off_pair,
                      ScorePtrs scores, int k, int stage_cap, uint64_t* __restrict__ cand_keys,
                      int32_t* __restrict__ cand_n) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelectSmem& sm = *reinterpret_cast<SelectSmem*>(smem_raw);
  const int pair = blockIdx.x;
  const cp_pair_desc pd = reinterpret_cast<const cp_pair_desc*>(plan + off_pair)[pair];
  const int r = pair / B;
  const int n = pd.rows;
  const float* sc = scores.p[r] + pd.row_off;
  // Every pass reads the pair's scores: stage them in shared memory once,
  // eight independent loads in flight per thread (the passes would otherwise
  // wait out an L2 round trip per element).
  float* staged = reinterpret_cast<float*>(smem_raw + sizeof(SelectSmem));
  const bool st = n <= stage_cap && n > k;  // staged by the fast path below
  auto score = [&](int i) { return st ? staged[i] : __ldg(sc + i); };
  auto get = [&](int i) { return token_key(score(i), pd.tok0 + i * pd.tok_step); };
  auto top12 = [&](int i) { return ordered_bits(score(i)) >> 20; };
  uint64_t* out = cand_keys + (long long)pair * k;
  if (st && n > k && local_topk_staged(n, k, sc, staged, get, top12, out, sm, pd, cand_n + pair)) return;
  const uint64_t thresh = n > k ? kth_largest(n, k, get, top12, sm) : 0ull;
  // the candidates in token order (the comparison split into two 32-bit halves)
  const uint32_t th_hi = (uint32_t)(thresh >> 32), th_lo = (uint32_t)thresh;
  auto keep = [&](int i) {
    const uint32_t hi = ordered_bits(score(i));
    return hi > th_hi || (hi == th_hi && 0xFFFFFFFFu - (uint32_t)(pd.tok0 + i * pd.tok_step) >= th_lo);
  };
  const int got = block_compact(n, keep, [&](int i, int j) { out[j] = get(i); }, sm.warp_cnt);
  if (threadIdx.x == 0) cand_n[pair] = got;
}

// Merge of one request's candidates: the global k-th key (the selection
// threshold) and the selected tokens in increasing order.
__global__ void __launch_bounds__(kThreads)
    topk_merge_kernel(int C, int B, int k, int kpow2, const uint64_t* __restrict__ cand_keys,
                      const int32_t* __restrict__ cand_n, int stage_cap, uint64_t* __restrict__ thresh,
                      int32_t* __restrict__ sel_ids, int32_t* __restrict__ sel_count) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelectSmem& sm = *reinterpret_cast<SelectSmem*>(smem_raw);
  int32_t* ids = reinterpret_cast<int32_t*>(smem_raw + sizeof(SelectSmem));  // kpow2 entries
  __shared__ int start[CP_MAX_SHARDS + 1];
  __shared__ int n_sel;
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    int s = 0;
    for (int r = 0; r < C; ++r) {
      start[r] = s;
      s += cand_n[r * B + b];
    }
    start[C] = s;
    n_sel = 0;
  }
  __syncthreads();
  const int N = start[C];
  auto get_global = [&](int i) {
    int r = 0;
    while (start[r + 1] <= i) ++r;
    return cand_keys[(long long)(r * B + b) * k + (i - start[r])];
  };
  // stage the candidates in shared memory when they fit (see topk_local_kernel)
  uint64_t* staged = reinterpret_cast<uint64_t*>(smem_raw + sizeof(SelectSmem) + ids_bytes(kpow2));
  const bool st = N <= stage_cap;
  if (st) {
    // stage the candidates with a histogram of their top 12 bits
    for (int i = threadIdx.x; i < kTopBins; i += blockDim.x) sm.hist[i] = 0;
    __syncthreads();
    for (int r = 0; r < C; ++r) {
      const uint64_t* src = cand_keys + (long long)(r * B + b) * k;
      const int n_r = start[r + 1] - start[r];
#pragma unroll 8
      for (int i = threadIdx.x; i < n_r; i += blockDim.x) {
        const uint64_t key = src[i];
        staged[start[r] + i] = key;
        atomicAdd(&sm.hist[key >> 52], 1u);
      }
    }
    __syncthreads();
  }
  auto get = [&](int i) { return st ? staged[i] : get_global(i); };
  auto top12 = [&](int i) { return (uint32_t)(get(i) >> 52); };
  uint64_t t = 0;
  bool found = N <= k;  // then every candidate is selected (t = 0)
  if (!found && st) {
    // the bin of rank k, collected and sorted when it is small (else the general path)
    pick_bin<kTopBins>(sm.hist, k, sm.pick, sm.warp_cnt);
    const uint32_t bin = sm.pick[0];
    const int want = k - (int)sm.pick[1];
    if ((int)sm.pick[2] <= kThreads) {
      const int m = block_collect(N, [&](int i) { return top12(i) == bin; }, get, sm.small, &sm.small_n);
      t = kth_of_small(sm.small, m, want);
      found = true;
    }
  }
  if (!found) t = kth_largest(N, k, get, top12, sm);
  for (int i = threadIdx.x; i < kpow2; i += blockDim.x) ids[i] = 0x7FFFFFFF;
  __syncthreads();
  const int got = block_compact(
      N, [&](int i) { return get(i) >= t; }, [&](int i, int j) { ids[j] = key_token(get(i)); },
      sm.warp_cnt);
  if (threadIdx.x == 0) n_sel = got;
  __syncthreads();
  // bitonic sort of the selected token indices, ascending
  for (int size = 2; size <= kpow2; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < kpow2; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          const int a = ids[i], c = ids[j];
          if ((a > c) == up) {
            ids[i] = c;
            ids[j] = a;
          }
        }
      }
      __syncthreads();
    }
  const int cnt = n_sel;
  for (int i = threadIdx.x; i < k; i += blockDim.x) sel_ids[(long long)b * k + i] = i < cnt ? ids[i] : -1;
  if (threadIdx.x == 0) {
    sel_count[b] = cnt;
    thresh[b] = t;
  }
}

// Owner side: pair (r, b) packs the cache rows of its selected tokens, in
// token order, at rows b kp .. b kp + count - 1 of shard r's selection
// buffer (kp = k rounded up to the decode tile of 128 rows), and zeroes the
// rows from there to the next multiple of 128: the decode reads whole tiles,
// and a row past the count enters its products with weight 0, which must not
// meet a NaN there.
__global__ void __launch_bounds__(kThreads)
    sparse_gather_kernel(const int32_t* __restrict__ plan, int B, int off_pair, int k, int kp,
                         const uint64_t* __restrict__ cand_keys, const int32_t* __restrict__ cand_n,
                         const uint64_t* __restrict__ thresh, ShardPtrs src, ScalePtrs src_scale,
                         int row_vec, MutShardPtrs dst, MutScalePtrs dst_scale, int has_scale,
                         int32_t* __restrict__ pair_count) {
  __shared__ int warp_cnt[kWarps];
  __shared__ int rows[kMaxTopK];  // source rows of this pair's selected tokens, in token order
  const int pair = blockIdx.x;
  const int r = pair / B, b = pair % B;
  const cp_pair_desc pd = reinterpret_cast<const cp_pair_desc*>(plan + off_pair)[pair];
  const int n = cand_n[pair];
  const uint64_t t = thresh[b];
  const uint64_t* keys = cand_keys + (long long)pair * k;
  const int count = block_compact(
      n, [&](int i) { return keys[i] >= t; },
      [&](int i, int j) { rows[j] = (key_token(keys[i]) - pd.tok0) / pd.tok_step; }, warp_cnt);
  // 16-byte pieces of all the selected rows, spread over the block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint4* sbase = static_cast<const uint4*>(src.p[r]);
  uint4* dbase = static_cast<uint4*>(dst.p[r]) + (long long)b * kp * row_vec;
  const int pieces = count * row_vec;
#pragma unroll 4
  for (int c = threadIdx.x; c < pieces; c += blockDim.x) {
    const int j = c / row_vec, q = c - j * row_vec;
    dbase[c] = __ldg(sbase + ((long long)pd.row_off + rows[j]) * row_vec + q);
  }
  if (has_scale)
    for (int j = threadIdx.x; j < count; j += blockDim.x)
      dst_scale.p[r][(long long)b * kp + j] = src_scale.p[r][(long long)pd.row_off + rows[j]];
  const int pad_end = min(kp, (count + kDecodeTileRows - 1) / kDecodeTileRows * kDecodeTileRows);
  for (int j = count + warp; j < pad_end; j += kWarps) {
    const long long drow = (long long)b * kp + j;
    uint4* dp = static_cast<uint4*>(dst.p[r]) + drow * row_vec;
    for (int c = lane; c < row_vec; c += 32) dp[c] = make_uint4(0, 0, 0, 0);
    if (has_scale && lane == 0) dst_scale.p[r][drow] = 0.f;
  }
  if (threadIdx.x == 0) pair_count[pair] = count;
}

}  // namespace

cudaError_t launch_topk_local(const int32_t* dev_plan, const cp_plan_header& h, const ScorePtrs& scores,
                              int k, int max_pair_rows, uint64_t* cand_keys, int32_t* cand_n,
                              cudaStream_t s) {
  const int pairs = h.C * h.R;
  // room to stage the longest pair's scores, up to kStageScores (longer pairs read from L2)
  const int cap = max_pair_rows < kStageScores ? max_pair_rows : kStageScores;
  const int smem = (int)sizeof(SelectSmem) + cap * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(topk_local_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  topk_local_kernel<<<pairs, kThreads, smem, s>>>(dev_plan, h.R, h.off_rank, scores, k, cap, cand_keys,
                                                  cand_n);
  return cudaGetLastError();
}

cudaError_t launch_topk_merge(const cp_plan_header& h, int k, const uint64_t* cand_keys,
                              const int32_t* cand_n, uint64_t* thresh, int32_t* sel_ids,
                              int32_t* sel_count, cudaStream_t s) {
  int kpow2 = 1;
  while (kpow2 < k) kpow2 <<= 1;
  const int cap = h.C * k < kStageKeys ? h.C * k : kStageKeys;
  const size_t smem = sizeof(SelectSmem) + ids_bytes(kpow2) + (size_t)cap * sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  topk_merge_kernel<<<h.R, kThreads, smem, s>>>(h.C, h.R, k, kpow2, cand_keys, cand_n, cap, thresh,
                                                 sel_ids, sel_count);
  return cudaGetLastError();
}

cudaError_t launch_sparse_gather(const int32_t* dev_plan, const cp_plan_header& h, int k,
                                 const uint64_t* cand_keys, const int32_t* cand_n,
                                 const uint64_t* thresh, const ShardPtrs& src,
                                 const ScalePtrs& src_scale, int row_bytes, const MutShardPtrs& dst,
                                 const MutScalePtrs& dst_scale, bool has_scale, int32_t* pair_count,
                                 cudaStream_t s) {
  const int pairs = h.C * h.R;
  const int kp = (k + kDecodeTileRows - 1) / kDecodeTileRows * kDecodeTileRows;
  sparse_gather_kernel<<<pairs, kThreads, 0, s>>>(dev_plan, h.R, h.off_rank, k, kp, cand_keys, cand_n,
                                                  thresh, src, src_scale, row_bytes / 16, dst,
                                                  dst_scale, has_scale ? 1 : 0, pair_count);
  return cudaGetLastError();
}

}  // namespace cpattn
