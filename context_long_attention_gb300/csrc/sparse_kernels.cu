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

constexpr int kThreads = 256;
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

// The k-th largest (k >= 1) of n distinct keys get(0..n-1), n >= k, by radix
// select from the top byte down.  All threads of the block call it.
template <typename Get>
__device__ uint64_t kth_largest(int n, int k, Get get, uint32_t* hist, uint32_t* pick) {
  uint64_t prefix = 0, mask = 0;
  int want = k;  // rank still sought among the keys matching the prefix
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const uint64_t key = get(i);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l counts bins 255 - 8l .. 248 - 8l (from the top); a scan over
      // the lanes finds the bin holding the wanted rank
      const int lane = threadIdx.x;
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        sum += c[j];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint32_t v = __shfl_up_sync(kFull, incl, d);
        if (lane >= d) incl += v;
      }
      const uint32_t excl = incl - sum;
      if (excl < (uint32_t)want && (uint32_t)want <= incl) {
        uint32_t above = excl;
        int bin = 255 - 8 * lane;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (above + c[j] >= (uint32_t)want) {
            bin = 255 - 8 * lane - j;
            break;
          }
          above += c[j];
        }
        pick[0] = (uint32_t)bin;
        pick[1] = above;  // keys with this prefix in higher bins
      }
    }
    __syncthreads();
    prefix |= (uint64_t)pick[0] << shift;
    mask |= (uint64_t)255u << shift;
    want -= (int)pick[1];
    __syncthreads();
  }
  return prefix;
}

// Exclusive prefix sum over the block of one int per thread (256 threads).
__device__ int block_exclusive_sum(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, d);
    if (lane >= d) incl += t;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kThreads / 32 ? warp_sums[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int t = __shfl_up_sync(kFull, w, d);
      if (lane >= d) w += t;
    }
    if (lane < kThreads / 32) warp_sums[lane] = w;  // inclusive over warps
    if (lane == kThreads / 32 - 1) *total = w;
  }
  __syncthreads();
  const int before = warp == 0 ? 0 : warp_sums[warp - 1];
  const int r = before + incl - v;
  __syncthreads();
  return r;
}

// Local top-k of every (shard, request) pair: candidate keys in token order.
__global__ void __launch_bounds__(kThreads)
    topk_local_kernel(const int32_t* __restrict__ plan, int B, int off_pair,
                      ScorePtrs scores, int k, uint64_t* __restrict__ cand_keys,
                      int32_t* __restrict__ cand_n) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t pick[2];
  __shared__ int warp_sums[kThreads / 32];
  __shared__ int total;
  const int pair = blockIdx.x;
  const cp_pair_desc pd = reinterpret_cast<const cp_pair_desc*>(plan + off_pair)[pair];
  const int r = pair / B;
  const int n = pd.rows;
  const float* sc = scores.p[r] + pd.row_off;
  auto get = [&](int i) { return token_key(__ldg(sc + i), pd.tok0 + i * pd.tok_step); };
  const uint64_t thresh = n > k ? kth_largest(n, k, get, hist, pick) : 0ull;
  // ordered compaction: thread t takes rows [t per, (t + 1) per)
  const int per = (n + kThreads - 1) / kThreads;
  const int i0 = min(n, threadIdx.x * per), i1 = min(n, i0 + per);
  int mine = 0;
  for (int i = i0; i < i1; ++i) mine += get(i) >= thresh;
  int at = block_exclusive_sum(mine, warp_sums, &total);
  uint64_t* out = cand_keys + (long long)pair * k;
  for (int i = i0; i < i1; ++i) {
    const uint64_t key = get(i);
    if (key >= thresh) out[at++] = key;
  }
  if (threadIdx.x == 0) cand_n[pair] = total;
}

// Merge of one request's candidates: the global k-th key (the selection
// threshold) and the selected tokens in increasing order.
__global__ void __launch_bounds__(kThreads)
    topk_merge_kernel(int C, int B, int k, int kpow2, const uint64_t* __restrict__ cand_keys,
                      const int32_t* __restrict__ cand_n, uint64_t* __restrict__ thresh,
                      int32_t* __restrict__ sel_ids, int32_t* __restrict__ sel_count) {
  extern __shared__ int32_t ids[];  // kpow2 entries
  __shared__ uint32_t hist[256];
  __shared__ uint32_t pick[2];
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
  auto get = [&](int i) {
    int r = 0;
    while (start[r + 1] <= i) ++r;
    return cand_keys[(long long)(r * B + b) * k + (i - start[r])];
  };
  const uint64_t t = N > k ? kth_largest(N, k, get, hist, pick) : 0ull;
  for (int i = threadIdx.x; i < kpow2; i += blockDim.x) ids[i] = 0x7FFFFFFF;
  __syncthreads();
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    const uint64_t key = get(i);
    if (key >= t) ids[atomicAdd(&n_sel, 1)] = key_token(key);
  }
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
  __shared__ int warp_sums[kThreads / 32];
  __shared__ int total;
  __shared__ int rows[1024];  // source rows of this pair's selected tokens (chunk)
  const int pair = blockIdx.x;
  const int r = pair / B, b = pair % B;
  const cp_pair_desc pd = reinterpret_cast<const cp_pair_desc*>(plan + off_pair)[pair];
  const int n = cand_n[pair];
  const uint64_t t = thresh[b];
  const uint64_t* keys = cand_keys + (long long)pair * k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int base = 0;  // selected rows written so far
  for (int c0 = 0; c0 < n; c0 += 1024) {
    const int cn = min(1024, n - c0);
    const int per = (cn + kThreads - 1) / kThreads;
    const int i0 = min(cn, threadIdx.x * per), i1 = min(cn, i0 + per);
    int mine = 0;
    for (int i = i0; i < i1; ++i) mine += keys[c0 + i] >= t;
    int at = block_exclusive_sum(mine, warp_sums, &total);
    for (int i = i0; i < i1; ++i) {
      const uint64_t key = keys[c0 + i];
      if (key >= t) rows[at++] = (key_token(key) - pd.tok0) / pd.tok_step;
    }
    __syncthreads();
    const int got = total;
    // one warp per row: 16-byte copies
    for (int j = warp; j < got; j += kThreads / 32) {
      const long long srow = (long long)pd.row_off + rows[j];
      const long long drow = (long long)b * kp + base + j;
      const uint4* s = static_cast<const uint4*>(src.p[r]) + srow * row_vec;
      uint4* d = static_cast<uint4*>(dst.p[r]) + drow * row_vec;
      for (int c = lane; c < row_vec; c += 32) d[c] = s[c];
      if (has_scale && lane == 0) dst_scale.p[r][drow] = src_scale.p[r][srow];
    }
    base += got;
    __syncthreads();
  }
  const int pad_end = min(kp, (base + kDecodeTileRows - 1) / kDecodeTileRows * kDecodeTileRows);
  for (int j = base + warp; j < pad_end; j += kThreads / 32) {
    const long long drow = (long long)b * kp + j;
    uint4* d = static_cast<uint4*>(dst.p[r]) + drow * row_vec;
    for (int c = lane; c < row_vec; c += 32) d[c] = make_uint4(0, 0, 0, 0);
    if (has_scale && lane == 0) dst_scale.p[r][drow] = 0.f;
  }
  if (threadIdx.x == 0) pair_count[pair] = base;
}

}  // namespace

cudaError_t launch_topk_local(const int32_t* dev_plan, const cp_plan_header& h, const ScorePtrs& scores,
                              int k, uint64_t* cand_keys, int32_t* cand_n, cudaStream_t s) {
  const int pairs = h.C * h.R;
  topk_local_kernel<<<pairs, kThreads, 0, s>>>(dev_plan, h.R, h.off_rank, scores, k, cand_keys, cand_n);
  return cudaGetLastError();
}

cudaError_t launch_topk_merge(const cp_plan_header& h, int k, const uint64_t* cand_keys,
                              const int32_t* cand_n, uint64_t* thresh, int32_t* sel_ids,
                              int32_t* sel_count, cudaStream_t s) {
  int kpow2 = 1;
  while (kpow2 < k) kpow2 <<= 1;
  const size_t smem = (size_t)kpow2 * sizeof(int32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  topk_merge_kernel<<<h.R, kThreads, smem, s>>>(h.C, h.R, k, kpow2, cand_keys, cand_n, thresh,
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
