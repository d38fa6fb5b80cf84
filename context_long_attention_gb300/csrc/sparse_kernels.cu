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
// k-th largest key is found by a radix select: a 4,096-bin first pass, then
// 8-bit passes over the keys of the bin that holds rank k.
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

// The least float f with ordered_bits(f) >= v: codes up to -inf's (those
// below it belong to no number) give -inf, codes above +inf's give NaN, which
// no comparison passes.
__device__ __forceinline__ float from_ordered(uint32_t v) {
  if (v <= 0x007FFFFFu) return -INFINITY;
  return __uint_as_float((v & 0x80000000u) ? (v & 0x7FFFFFFFu) : ~v);
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

// Exclusive scan of one count per thread across the block: returns the sum
// of the counts of the threads before this one, *total the sum of all.  All
// threads call it; warp_cnt (kWarps ints) must be free on entry, and stays in
// use until the block's next barrier.
__device__ int block_excl_scan(int c, int* warp_cnt, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = c;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_cnt[warp] = incl;
  __syncthreads();
  int at = incl - c, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int v = warp_cnt[w];
    at += w < warp ? v : 0;
    tot += v;
  }
  *total = tot;
  return at;
}

constexpr int kTopBins = 4096;  // the first pass splits on the key's top 12 bits

// Shared scratch of the radix select.
struct __align__(16) SelectSmem {
  uint32_t hist[kTopBins];
  uint32_t pick[4];
  uint32_t top_bin;  // highest non-empty bin of a first-pass histogram
  uint32_t umax;
  int small_n;
  int few_n;
  int ids_n;
  int warp_cnt[kWarps];
  uint64_t small[kSmallKeys];
  uint64_t few[32];
  uint64_t result;
};

// Bit words of a staged pair's scores: one bit per score, the scores shifted
// by up to 3 places and covered in groups of 128 (two such arrays: the
// scores above the rank-k bin, and those in it).
constexpr int kStageWords = (kStageScores + 3 + 127) / 128 * 4;

// Finds, among the NB bins of hist taken from the top, the one that holds
// rank `want` (1-based): pick = {bin, keys in higher bins, keys in it}, and
// (top_bin given) the highest bin holding a key.  Each
// thread owns NB / blockDim consecutive bins (one, or none, when NB is
// smaller than the block); one block-wide scan.
template <int NB>
__device__ void pick_bin(const uint32_t* hist, int want, uint32_t* pick, int* warp_cnt,
                         uint32_t* top_bin = nullptr) {
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
    uint32_t above = excl, in_bin = 0;
    int jsel = -1;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      if (jsel < 0 && (j == PER - 1 || above + c[j] >= (uint32_t)want)) {
        jsel = j;
        in_bin = c[j];
      } else if (jsel < 0) {
        above += c[j];
      }
    }
    pick[0] = (uint32_t)(top - jsel);
    pick[1] = above;
    pick[2] = in_bin;
  }
  if (top_bin && excl == 0 && sum > 0) {  // the first thread from the top with a key
    int jt = -1;
#pragma unroll
    for (int j = 0; j < PER; ++j)
      if (jt < 0 && c[j] > 0) jt = j;
    *top_bin = (uint32_t)(top - jt);
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
  pick_bin<kTopBins>(sm.hist, k, sm.pick, sm.warp_cnt, &sm.top_bin);
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

// The want-th largest (1 <= want <= m) of m distinct keys a[0, m), m <=
// kSmallKeys, that agree on the bits `mask` selects (= prefix): 8-bit radix
// passes from bit sh down narrow the keys still in play to at most 32, which
// one warp sorts with shuffles.  All threads of the block call it.
__device__ uint64_t kth_refine(const uint64_t* a, int m, int want, uint64_t prefix, uint64_t mask, int sh,
                               SelectSmem& sm) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) sm.few_n = 0;
  __syncthreads();
  for (int in_play = m; in_play > 32; sh = sh >= 8 ? sh - 8 : 0) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) sm.hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < m; i += blockDim.x) {
      const uint64_t key = a[i];
      if ((key & mask) == prefix) atomicAdd(&sm.hist[(key >> sh) & 255u], 1u);
    }
    __syncthreads();
    pick_bin<256>(sm.hist, want, sm.pick, sm.warp_cnt);
    prefix = (prefix & ~(255ull << sh)) | ((uint64_t)sm.pick[0] << sh);
    mask |= 255ull << sh;
    want -= (int)sm.pick[1];
    in_play = (int)sm.pick[2];
    if (sh == 0) break;  // all 64 bits fixed (one key)
  }
  for (int i = threadIdx.x; i < m; i += blockDim.x) {
    const uint64_t key = a[i];
    if ((key & mask) == prefix) sm.few[atomicAdd(&sm.few_n, 1)] = key;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    // bitonic sort of the <= 32 keys in play, decreasing (the padding, 0, sorts last)
    uint64_t v = lane < sm.few_n ? sm.few[lane] : 0ull;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const uint64_t o = __shfl_xor_sync(kFull, v, stride);
        const bool desc = (lane & size) == 0, lower = (lane & stride) == 0;
        v = desc == lower ? (v > o ? v : o) : (v < o ? v : o);
      }
    if (lane == want - 1) sm.result = v;
  }
  __syncthreads();
  return sm.result;
}

// The staged path of a pair's local top-k (k < n <= the staging room).
// Score i is kept at stg[i] = staged[i + pad], pad in [0, 3] chosen so that
// the source's 16-byte groups land on 16-byte groups of shared memory; the
// passes work in that shifted index j = i + pad, four scores a thread, over
// whole groups of 128 (the places before pad and past pad + n hold NaN, which
// no comparison passes).
//   pass 1  stage the scores with a histogram of their top 12 bits; the bin
//           holding rank k is found from it;
//   pass 2  one bit per score above the bin and one per score in it (float
//           comparisons against the bin's bounds); the bin's keys are
//           collected from their bits, its want-th key is the threshold, and
//           the bin's keys at or above it join the first bits;
//   pass 3  the marked scores' keys written in token order (a scan of the
//           bit words' counts gives each thread its place).
// Returns false (scores staged, nothing written) when the bin holds more than
// kSmallKeys keys (many equal scores).
__device__ bool local_topk_staged(int n, int k, const float* sc, float* staged, uint32_t* bits, uint64_t* out,
                                  SelectSmem& sm, const cp_pair_desc& pd, int32_t* n_out, uint64_t* range_out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int head = (int)((16u - ((uint32_t)(uintptr_t)sc & 15u)) & 15u) >> 2;  // scores before a 16-byte boundary
  const int pad = (4 - head) & 3;
  const int J = pad + n, Q = (J + 127) >> 7;  // groups of 128 shifted indices
  uint32_t* in_bits = bits + kStageWords;
  float* stg = staged + pad;
  for (int i = threadIdx.x; i < kTopBins; i += blockDim.x) sm.hist[i] = 0;
  for (int j = threadIdx.x; j < pad; j += blockDim.x) staged[j] = __uint_as_float(0x7FFFFFFFu);
  for (int j = J + threadIdx.x; j < 128 * Q; j += blockDim.x) staged[j] = __uint_as_float(0x7FFFFFFFu);
  __syncthreads();
  const int h = min(head, n);
  const int nv = (n - h) >> 2;
  const float4* src4 = reinterpret_cast<const float4*>(sc + h);
  float4* dst4 = reinterpret_cast<float4*>(stg + h);  // pad + h is a multiple of 4 whenever nv > 0
#pragma unroll 8
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    const float4 f = __ldg(src4 + v);
    dst4[v] = f;
    atomicAdd(&sm.hist[ordered_bits(f.x) >> 20], 1u);
    atomicAdd(&sm.hist[ordered_bits(f.y) >> 20], 1u);
    atomicAdd(&sm.hist[ordered_bits(f.z) >> 20], 1u);
    atomicAdd(&sm.hist[ordered_bits(f.w) >> 20], 1u);
  }
  {  // the scalars before and after the groups of four (at most 3 each)
    const int rest = h + 4 * nv;
    int i = -1;
    if ((int)threadIdx.x < h) i = threadIdx.x;
    else if ((int)threadIdx.x - h < n - rest) i = rest + (int)threadIdx.x - h;
    if (i >= 0) {
      const float f = __ldg(sc + i);
      stg[i] = f;
      atomicAdd(&sm.hist[ordered_bits(f) >> 20], 1u);
    }
  }
  __syncthreads();
  pick_bin<kTopBins>(sm.hist, k, sm.pick, sm.warp_cnt, &sm.top_bin);
  const uint32_t bin = sm.pick[0];
  const int want = k - (int)sm.pick[1];
  if ((int)sm.pick[2] > kSmallKeys) return false;
  // the bin's scores are [f_lo, f_hi) (f_hi NaN for the top bin: nothing above it)
  const float f_lo = from_ordered(bin << 20);
  const float f_hi = bin + 1 < (uint32_t)kTopBins ? from_ordered((bin + 1) << 20) : __uint_as_float(0x7FFFFFFFu);
  const float4* s4 = reinterpret_cast<const float4*>(staged);
  for (int q = warp; q < Q; q += kWarps) {
    const float4 f = s4[32 * q + lane];
    const uint32_t up = (f.x >= f_hi ? 1u : 0u) | (f.y >= f_hi ? 2u : 0u) | (f.z >= f_hi ? 4u : 0u) |
                        (f.w >= f_hi ? 8u : 0u);
    const uint32_t at_least = (f.x >= f_lo ? 1u : 0u) | (f.y >= f_lo ? 2u : 0u) | (f.z >= f_lo ? 4u : 0u) |
                              (f.w >= f_lo ? 8u : 0u);
    // lanes 8w .. 8w + 7 hold the 32 bits of word 4q + w
    const int sh4 = 4 * (lane & 7);
    uint32_t wa = up << sh4, wb = (at_least & ~up) << sh4;
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) {
      wa |= __shfl_xor_sync(kFull, wa, d);
      wb |= __shfl_xor_sync(kFull, wb, d);
    }
    if ((lane & 7) == 0) {
      bits[4 * q + (lane >> 3)] = wa;
      in_bits[4 * q + (lane >> 3)] = wb;
    }
  }
  __syncthreads();
  // the bin's keys, collected in index order from their bits (thread t takes words [t per, (t + 1) per))
  const int W = 4 * Q;
  const int per = (W + (int)blockDim.x - 1) / (int)blockDim.x;
  const int w0 = min(W, (int)threadIdx.x * per), w1 = min(W, w0 + per);
  {
    int c = 0;
    for (int w = w0; w < w1; ++w) c += __popc(in_bits[w]);
    int m_all;
    int at = block_excl_scan(c, sm.warp_cnt, &m_all);
    for (int w = w0; w < w1; ++w)
      for (uint32_t word = in_bits[w]; word; word &= word - 1u) {
        const int j = 32 * w + __ffs(word) - 1;
        if (at < kSmallKeys) sm.small[at] = token_key(staged[j], pd.tok0 + (j - pad) * pd.tok_step);
        ++at;
      }
    if (threadIdx.x == 0) sm.small_n = min(m_all, kSmallKeys);  // m_all is the bin's count, at most kSmallKeys
  }
  __syncthreads();
  const int m = sm.small_n;
  const uint64_t thresh = kth_refine(sm.small, m, want, (uint64_t)bin << 52, 0xFFFull << 52, 44, sm);
  for (int i = threadIdx.x; i < m; i += blockDim.x) {
    const uint64_t key = sm.small[i];
    if (key >= thresh) {
      const int j = (key_token(key) - pd.tok0) / pd.tok_step + pad;
      atomicOr(&bits[j >> 5], 1u << (j & 31));
    }
  }
  __syncthreads();
  // pass 3
  int c = 0;
  for (int w = w0; w < w1; ++w) c += __popc(bits[w]);
  int tot;
  int at = block_excl_scan(c, sm.warp_cnt, &tot);
  for (int w = w0; w < w1; ++w) {
    for (uint32_t word = bits[w]; word; word &= word - 1u) {
      const int j = 32 * w + __ffs(word) - 1;
      if (at < k) out[at] = token_key(staged[j], pd.tok0 + (j - pad) * pd.tok_step);
      ++at;
    }
  }
  if (threadIdx.x == 0) {
    *n_out = min(tot, k);  // tot is k: the keys above the bin and the bin's want best
    *range_out = (uint64_t)((sm.top_bin << 20) | 0xFFFFFu) << 32 | (uint32_t)(thresh >> 32);
  }
  return true;
}

// Local top-k of every (shard, request) pair: candidate keys in token order,
// and the pair's score range for the merge: range = hi << 32 | lo, hi at or
// above every candidate's ordered score, lo the ordered score of the k-th key
// when the pair had more than k rows (else 0, no bound).
__global__ void __launch_bounds__(kThreads)
    topk_local_kernel(const int32_t* __restrict__ plan, int B, int off_pair,
                      ScorePtrs scores, int k, int stage_cap, uint64_t* __restrict__ cand_keys,
                      int32_t* __restrict__ cand_n, uint64_t* __restrict__ range) {
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
  uint32_t* bits = reinterpret_cast<uint32_t*>(smem_raw + sizeof(SelectSmem));
  float* staged = reinterpret_cast<float*>(smem_raw + sizeof(SelectSmem) + 2 * kStageWords * sizeof(uint32_t));
  const bool st = n <= stage_cap && n > k;  // staged by the fast path below
  const int pad = (4 - ((int)((16u - ((uint32_t)(uintptr_t)sc & 15u)) & 15u) >> 2)) & 3;
  auto score = [&](int i) { return st ? staged[pad + i] : __ldg(sc + i); };
  auto get = [&](int i) { return token_key(score(i), pd.tok0 + i * pd.tok_step); };
  auto top12 = [&](int i) { return ordered_bits(score(i)) >> 20; };
  uint64_t* out = cand_keys + (long long)pair * k;
  if (st && local_topk_staged(n, k, sc, staged, bits, out, sm, pd, cand_n + pair, range + pair)) return;
  uint64_t thresh = 0;
  uint32_t hi;
  if (n > k) {
    thresh = kth_largest(n, k, get, top12, sm);
    hi = (sm.top_bin << 20) | 0xFFFFFu;
  } else {  // every row is a candidate: the largest ordered score
    if (threadIdx.x == 0) sm.umax = 0;
    __syncthreads();
    uint32_t m = 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) m = max(m, ordered_bits(score(i)));
    m = __reduce_max_sync(kFull, m);
    if ((threadIdx.x & 31) == 0) atomicMax(&sm.umax, m);
    __syncthreads();
    hi = sm.umax;
  }
  // the candidates in token order (the comparison split into two 32-bit halves)
  const uint32_t th_hi = (uint32_t)(thresh >> 32), th_lo = (uint32_t)thresh;
  auto keep = [&](int i) {
    const uint32_t u = ordered_bits(score(i));
    return u > th_hi || (u == th_hi && 0xFFFFFFFFu - (uint32_t)(pd.tok0 + i * pd.tok_step) >= th_lo);
  };
  const int got = block_compact(n, keep, [&](int i, int j) { out[j] = get(i); }, sm.warp_cnt);
  if (threadIdx.x == 0) {
    cand_n[pair] = got;
    range[pair] = (uint64_t)hi << 32 | th_hi;
  }
}

// Merge of one request's candidates: the global k-th key (the selection
// threshold) and the selected tokens in increasing order.
//
// The threshold.  A shard that had more than k rows sent k candidates, all at
// or above its k-th key, so the global k-th key is at least the largest of
// those shards' k-th keys; lo, its ordered score, bounds the keys in play from
// below, and hi, the largest of the shards' upper bounds, from above.  The
// first histogram cuts [lo, hi] into kTopBins equal slices (a shift of u - lo)
// as the candidates are staged, so that the bin holding rank k is narrow even
// when the candidates share their top bits.  A second pass marks the
// candidates of the bins above it (one bit each) and collects the keys of that
// bin, whose want-th key (kth_refine) is the threshold.  A bin of more than
// kSmallKeys keys (many equal scores) goes to the general radix select, and
// the marks are then the keys at or above its result.
// The order.  The selected tokens are set as bits of a bitmap over token
// indices (kSortTokens of them at a time, in the histogram's words), whose
// scan gives every token its place: no sort.
constexpr int kSortTokens = kTopBins * 32;
constexpr int kMergeBatch = 16;  // candidate loads a thread keeps in flight

__global__ void __launch_bounds__(kThreads)
    topk_merge_kernel(const int32_t* __restrict__ plan, int off_pair, int C, int B, int k,
                      const uint64_t* __restrict__ cand_keys, const int32_t* __restrict__ cand_n,
                      const uint64_t* __restrict__ range, int stage_cap, uint64_t* __restrict__ thresh,
                      int32_t* __restrict__ sel_ids, int32_t* __restrict__ sel_count) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelectSmem& sm = *reinterpret_cast<SelectSmem*>(smem_raw);
  // marks of the selected candidates (one bit each): their own words when
  // the candidates are staged, else the unused staging room
  uint32_t* marks_st = reinterpret_cast<uint32_t*>(smem_raw + sizeof(SelectSmem));
  uint64_t* staged = reinterpret_cast<uint64_t*>(smem_raw + sizeof(SelectSmem) + kStageKeys / 8);
  __shared__ int start[CP_MAX_SHARDS + 1];  // shard r's candidates: [start[r], start[r + 1])
  __shared__ uint32_t lo_s, hi_s;
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int total = C * k;
  // entry idx of the flattened [C][k] lists is row idx - r k of shard r =
  // idx / k (a float estimate, corrected: no divide, no branch); entries past
  // a shard's count lie in the workspace too and are loaded but not used
  const float inv_k = 1.0f / (float)k;
  auto shard_of = [&](int idx) {
    int r = (int)((float)idx * inv_k);
    r -= r * k > idx ? 1 : 0;
    r += (r + 1) * k <= idx ? 1 : 0;
    return r;
  };
  auto load_batch = [&](int base, uint64_t (&kv)[kMergeBatch]) {
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const int idx = base + u * (int)blockDim.x + (int)threadIdx.x;
      const int r = shard_of(idx);
      kv[u] = idx < total ? __ldg(cand_keys + (long long)(r * B + b) * k + (idx - r * k)) : 0ull;
    }
  };
  uint64_t kv[kMergeBatch];
  load_batch(0, kv);  // in flight while warp 0 reads the shards' counts
  if (threadIdx.x < 32) {  // warp 0: the shards' counts (a scan) and ranges, two shards a lane
    int n0 = 0, n1 = 0;
    uint64_t g0 = 0, g1 = 0;
    if (lane < C) {
      n0 = cand_n[lane * B + b];
      g0 = range[lane * B + b];
    }
    if (lane + 32 < C) {
      n1 = cand_n[(lane + 32) * B + b];
      g1 = range[(lane + 32) * B + b];
    }
    int i0 = n0, i1 = n1;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v0 = __shfl_up_sync(kFull, i0, d), v1 = __shfl_up_sync(kFull, i1, d);
      if (lane >= d) {
        i0 += v0;
        i1 += v1;
      }
    }
    const int tot0 = __shfl_sync(kFull, i0, 31);
    if (lane < C) start[lane] = i0 - n0;
    if (lane + 32 < C) start[lane + 32] = tot0 + i1 - n1;
    if (lane == 31) start[C] = tot0 + i1;
    // hi: the largest bound; lo: the largest k-th key (0: no bound from that shard)
    const uint32_t hi = __reduce_max_sync(kFull, max(n0 ? (uint32_t)(g0 >> 32) : 0u, n1 ? (uint32_t)(g1 >> 32) : 0u));
    const uint32_t lo = __reduce_max_sync(kFull, max(n0 ? (uint32_t)g0 : 0u, n1 ? (uint32_t)g1 : 0u));
    if (lane == 0) {
      lo_s = lo;  // 0 when no shard bounds it: every candidate in play
      hi_s = max(hi, lo);
      sm.small_n = 0;
    }
  }
  for (int i = threadIdx.x; i < kTopBins; i += blockDim.x) sm.hist[i] = 0;
  __syncthreads();
  const int N = start[C];
  const uint32_t lo = lo_s;
  const int sh = max(0, 32 - __clz(hi_s - lo) - 12);  // (hi - lo) >> sh < kTopBins
  auto bin_of = [&](uint32_t u) { return min((u - lo) >> sh, (uint32_t)kTopBins - 1u); };
  const bool st = N <= stage_cap;
  const bool select = N > k;  // else every candidate is selected (threshold 0)
  // pass 1: stage the candidates (when they fit), counting those in play
  for (int base = 0; base < total; base += kMergeBatch * (int)blockDim.x) {
    if (base > 0) load_batch(base, kv);
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const int idx = base + u * (int)blockDim.x + (int)threadIdx.x;
      if (idx < total) {
        const int r = shard_of(idx);
        const int i = idx - r * k;
        if (i < start[r + 1] - start[r]) {
          if (st) staged[start[r] + i] = kv[u];
          const uint32_t u32 = (uint32_t)(kv[u] >> 32);
          if (select && u32 >= lo) atomicAdd(&sm.hist[bin_of(u32)], 1u);
        }
      }
    }
  }
  __syncthreads();
  auto get_global = [&](int i) {
    int r = 0;
    while (start[r + 1] <= i) ++r;
    return cand_keys[(long long)(r * B + b) * k + (i - start[r])];
  };
  auto get = [&](int i) { return st ? staged[i] : get_global(i); };
  uint32_t* marks = st ? marks_st : reinterpret_cast<uint32_t*>(staged);
  const int n_words = (N + 31) >> 5;
  // marks of whole warps of 32 candidates: mark(i, key) says whether key (candidate i) is selected
  auto mark_pass = [&](auto key_at, auto mark) {
    for (int i = threadIdx.x; i < 32 * n_words; i += blockDim.x) {
      const uint64_t key = i < N ? key_at(i) : 0ull;
      const unsigned bal = __ballot_sync(kFull, i < N && mark(i, key));
      if (lane == 0) marks[i >> 5] = bal;
    }
  };
  uint64_t t = 0;
  int m = 0;  // the rank-k bin's keys in sm.small (selected when >= t)
  bool done = false;
  if (select) {
    pick_bin<kTopBins>(sm.hist, k, sm.pick, sm.warp_cnt);
    const uint32_t bin = sm.pick[0];
    const int want = k - (int)sm.pick[1];
    if ((int)sm.pick[2] <= kSmallKeys) {
      // pass 2: marks for the bins above, the bin's keys to small
      auto above = [&](int, uint64_t key) {
        const uint32_t u = (uint32_t)(key >> 32);
        if (u < lo) return false;
        const uint32_t bi = bin_of(u);
        if (bi == bin) sm.small[atomicAdd(&sm.small_n, 1)] = key;  // a few keys
        return bi > bin;
      };
      if (st) mark_pass([&](int i) { return staged[i]; }, above);
      else mark_pass(get_global, above);
      __syncthreads();
      m = sm.small_n;
      t = kth_refine(sm.small, m, want, 0ull, 0ull, 56, sm);
      done = true;
    } else {
      t = kth_largest(N, k, get, [&](int i) { return (uint32_t)(get(i) >> 52); }, sm);
    }
  }
  if (!done) {  // every key at or above t
    __syncthreads();  // marks may alias the staging room the select just read
    auto at_least = [&](int, uint64_t key) { return key >= t; };
    if (st) mark_pass([&](int i) { return staged[i]; }, at_least);
    else mark_pass(get_global, at_least);
  }
  __syncthreads();
  // the selected tokens in increasing order, kSortTokens token indices at a time
  const int L = reinterpret_cast<const cp_pair_desc*>(plan + off_pair)[b].ctx_len;  // tokens are < L
  uint32_t* bmp = sm.hist;
  int32_t* out = sel_ids + (long long)b * k;
  int placed = 0;
  for (int t0 = 0; t0 < L; t0 += kSortTokens) {
    const int words = (min(L - t0, kSortTokens) + 31) >> 5;
    for (int w = threadIdx.x; w < words; w += blockDim.x) bmp[w] = 0;
    __syncthreads();
    auto set = [&](int tok) {
      tok -= t0;
      if (tok >= 0 && tok < kSortTokens) atomicOr(&bmp[tok >> 5], 1u << (tok & 31));
    };
    for (int w = threadIdx.x; w < n_words; w += blockDim.x)
      for (uint32_t word = marks[w]; word; word &= word - 1u) set(key_token(get(32 * w + __ffs(word) - 1)));
    for (int j = threadIdx.x; j < m; j += blockDim.x)
      if (sm.small[j] >= t) set(key_token(sm.small[j]));
    __syncthreads();
    const int per = (words + (int)blockDim.x - 1) / (int)blockDim.x;
    const int w0 = min(words, (int)threadIdx.x * per), w1 = min(words, w0 + per);
    int c = 0;
    for (int w = w0; w < w1; ++w) c += __popc(bmp[w]);
    int tot;
    int at = placed + block_excl_scan(c, sm.warp_cnt, &tot);
    for (int w = w0; w < w1; ++w)
      for (uint32_t word = bmp[w]; word; word &= word - 1u) {
        if (at < k) out[at] = t0 + 32 * w + __ffs(word) - 1;
        ++at;
      }
    placed += tot;
    __syncthreads();
  }
  const int cnt = min(placed, k);  // k when the request has more than k candidates, else all of them
  for (int i = cnt + threadIdx.x; i < k; i += blockDim.x) out[i] = -1;
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
                              int k, int max_pair_rows, uint64_t* cand_keys, int32_t* cand_n, uint64_t* range,
                              cudaStream_t s) {
  const int pairs = h.C * h.R;
  // room to stage the longest pair's scores, up to kStageScores (longer pairs read from L2)
  const int cap = max_pair_rows < kStageScores ? max_pair_rows : kStageScores;
  const int smem = (int)sizeof(SelectSmem) + 2 * kStageWords * (int)sizeof(uint32_t) +
                   (cap + 3 + 127) / 128 * 128 * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(topk_local_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  topk_local_kernel<<<pairs, kThreads, smem, s>>>(dev_plan, h.R, h.off_rank, scores, k, cap, cand_keys,
                                                  cand_n, range);
  return cudaGetLastError();
}

cudaError_t launch_topk_merge(const int32_t* dev_plan, const cp_plan_header& h, int k, const uint64_t* cand_keys,
                              const int32_t* cand_n, const uint64_t* range, uint64_t* thresh, int32_t* sel_ids,
                              int32_t* sel_count, cudaStream_t s) {
  const int cap = h.C * k < kStageKeys ? h.C * k : kStageKeys;
  // the staging room doubles as the marks when the candidates do not fit
  // (C k / 32 words <= kStageKeys * 2 words since C k <= 64 x 4096)
  const size_t smem = sizeof(SelectSmem) + kStageKeys / 8 + (size_t)kStageKeys * sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  topk_merge_kernel<<<h.R, kThreads, smem, s>>>(dev_plan, h.off_rank, h.C, h.R, k, cand_keys, cand_n, range,
                                                 cap, thresh, sel_ids, sel_count);
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
