// Index maps, token-shard packing and the exact log-sum-exp merge.
//
// * plan_map_kernel: per-query arrays of a prefill plan (flattened index,
//   position, request) from its segments — zigzag blocks or interleave runs
//   ("How GPUs Share a Long Context During LLM Inference", §2.3-2.4).
// * kv_pack_kernel: token p of a request -> shard p mod C, row p / C (§3.1),
//   into the shard's buffer or, paged, into the pool row its page table gives.
// * lse_merge_kernel / decode_fixup_kernel / lse_fold_kernel: O = sum_p w_p O_p / sum_p w_p
//   with w_p = exp(LSE_p - max LSE) (§3.3; "DeepSeek-V4 Attention Inference
//   Systems" §5), one warp per (row, head, 128 output dims), 128-bit loads.
#include <cuda_bf16.h>

#include "internal.h"

namespace cpattn {
namespace {

__global__ void plan_map_kernel(int32_t* __restrict__ plan, int off_seg, int off_idx, int off_qpos,
                                int off_qreq) {
  const cp_seg_desc s = reinterpret_cast<const cp_seg_desc*>(plan + off_seg)[blockIdx.x];
  int32_t* idx = plan + off_idx;
  int32_t* qpos = plan + off_qpos;
  int32_t* qreq = plan + off_qreq;
  for (int i = threadIdx.x; i < s.count; i += blockDim.x) {
    const int row = s.local_start + i;
    idx[row] = s.first_f + i * s.stride;
    qpos[row] = s.first_pos + i * s.stride;
    qreq[row] = s.req;
  }
}

// One warp per token row.  The request of token t is the last b with
// first_token[b] <= t (requests of length 0 share their start with the next).
__global__ void kv_pack_kernel(const int32_t* __restrict__ plan, int C, int B, int T,
                               int off_pair, int off_req, const uint4* __restrict__ kv,
                               const float* __restrict__ kv_scale, int row_vec,
                               MutShardPtrs dst, MutScalePtrs dst_scale, int has_scale,
                               RowMap rm, int layout) {
  const int warps = blockDim.x >> 5;
  const long long t = (long long)blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int32_t* req = plan + off_req;  // [B][2] {ctx_len, first token}
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (req[2 * mid + 1] <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int p = (int)(t - req[2 * b + 1]);
  int r, i;  // shard and shard row of token p
  if (layout == CP_DCP_ROUND_ROBIN) {
    r = p % C;
    i = p / C;
  } else {  // chunks of q + 1 tokens for shards r < m, then of q tokens
    const int L = req[2 * b], q = L / C, m = L % C, big = m * (q + 1);
    r = p < big ? p / (q + 1) : m + (p - big) / q;
    i = p < big ? p % (q + 1) : (p - big) % q;
  }
  const cp_pair_desc* pair = reinterpret_cast<const cp_pair_desc*>(plan + off_pair);
  const long long row = map_row(rm, r * B + b, pair[r * B + b].row_off, i);
  const uint4* src = kv + t * row_vec;
  uint4* out = static_cast<uint4*>(dst.p[r]) + row * row_vec;
  for (int c = lane; c < row_vec; c += 32) out[c] = src[c];
  if (has_scale && lane == 0) dst_scale.p[r][row] = kv_scale[t];
}

// Paged caches: one block per pair zeroes rows [rows, pages x page_size) of
// the pair's last page (and their scales).
__global__ void page_tail_zero_kernel(const int32_t* __restrict__ plan, int off_pair,
                                      int row_vec, uint4* __restrict__ pool,
                                      float* __restrict__ scale_pool, RowMap rm) {
  const cp_pair_desc pd = reinterpret_cast<const cp_pair_desc*>(plan + off_pair)[blockIdx.x];
  if (pd.rows == 0) return;
  const int end = (pd.rows + rm.page_size - 1) / rm.page_size * rm.page_size;
  for (int i = pd.rows + threadIdx.y; i < end; i += blockDim.y) {
    const long long row = map_row(rm, blockIdx.x, 0, i);
    for (int c = threadIdx.x; c < row_vec; c += blockDim.x) pool[row * row_vec + c] = make_uint4(0, 0, 0, 0);
    if (scale_pool && threadIdx.x == 0) scale_pool[row] = 0.f;
  }
}

// Merge of P parts for one (row, head), parts at o + p*ostride, l + p*lstride:
// kSlices slices of 128 output dims from dim 4 * c0 (a launch over few rows
// gives each warp one slice, so that the warps fill the SMs), and the LSE with
// the slice at dim 0.  Any P: a warp takes the parts 32 at a time, lane u
// holding part p0 + u's weight; the sums take the parts in order.
//
// A merge is a short chain of dependent loads (LSEs, then weights, then the
// sums) and its time is their latency, so the loads in flight per warp set
// its speed: kBatch parts x kSlices slices at once, and the first batch goes
// out beside the LSEs, before the weights are known (a row whose weight turns
// out 0 is not summed; every part slot below P lies in the buffer).
constexpr int kMergeSlice = 32;  // float4 columns of a slice
template <int kSlices, int kBatch>
__device__ __forceinline__ void merge_row(int P, const float* __restrict__ o, long long ostride,
                                          const float* __restrict__ l, long long lstride, int Dv, int c0,
                                          float* out_f32, __nv_bfloat16* out_bf16, float* out_lse) {
  const int lane = threadIdx.x & 31;
  auto col = [&](int sl) { return c0 + kMergeSlice * sl + lane; };
  auto active = [&](int sl) { return col(sl) < Dv / 4; };  // lanes past the row's end skip loads and stores
  auto row = [&](int p, int sl) { return reinterpret_cast<const float4*>(o + (long long)p * ostride)[col(sl)]; };
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 x[kBatch][kSlices];
#pragma unroll
  for (int k = 0; k < kBatch; ++k)
#pragma unroll
    for (int sl = 0; sl < kSlices; ++sl) x[k][sl] = k < P && active(sl) ? row(k, sl) : zero;
  float g = -INFINITY;
  for (int p = lane; p < P; p += 32) g = fmaxf(g, l[p * lstride]);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) g = fmaxf(g, __shfl_xor_sync(0xffffffffu, g, d));
  const bool any = g != -INFINITY;
  auto weight = [&](int p) {  // part p's weight exp(LSE_p - max), 0 for an empty part or p >= P
    const float lp = p < P ? l[p * lstride] : -INFINITY;
    return (any && lp != -INFINITY) ? expf(lp - g) : 0.f;
  };
  // the weights of parts lane and lane + 32, once; parts past 64 (a pair cut
  // over more than 64 workers, a request over more than 64 runs) are weighed
  // again where they are summed
  const float w0 = weight(lane), w1 = weight(lane + 32);
  float z = w0 + w1;
  for (int p0 = 64; p0 < P; p0 += 32) z += weight(p0 + lane);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
  const float inv = any ? 1.f / z : 0.f;
  // every lane runs every iteration (the weights travel by warp shuffles)
  float4 acc[kSlices];
#pragma unroll
  for (int sl = 0; sl < kSlices; ++sl) acc[sl] = zero;
  for (int p0 = 0; p0 < P; p0 += 32) {
    const float wl = p0 == 0 ? w0 : p0 == 32 ? w1 : weight(p0 + lane);
    const int np = min(32, P - p0);
    for (int u0 = 0; u0 < np; u0 += kBatch) {
      float w[kBatch];
      const bool loaded = p0 + u0 == 0;  // the first batch is in x already
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        w[k] = __shfl_sync(0xffffffffu, wl, (u0 + k) & 31);
        const bool use = u0 + k < np && w[k] != 0.f;
        if (!loaded)
#pragma unroll
          for (int sl = 0; sl < kSlices; ++sl) x[k][sl] = use && active(sl) ? row(p0 + u0 + k, sl) : zero;
        if (!use) w[k] = 0.f;
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (w[k] != 0.f) {
#pragma unroll
          for (int sl = 0; sl < kSlices; ++sl) {
            acc[sl].x += w[k] * x[k][sl].x;
            acc[sl].y += w[k] * x[k][sl].y;
            acc[sl].z += w[k] * x[k][sl].z;
            acc[sl].w += w[k] * x[k][sl].w;
          }
        }
      }
    }
  }
#pragma unroll
  for (int sl = 0; sl < kSlices; ++sl) {
    float4 a4 = acc[sl];
    a4.x *= inv;
    a4.y *= inv;
    a4.z *= inv;
    a4.w *= inv;
    if (!active(sl)) continue;
    if (out_f32) {
      reinterpret_cast<float4*>(out_f32)[col(sl)] = a4;
    } else {
      __nv_bfloat162 a = __floats2bfloat162_rn(a4.x, a4.y);
      __nv_bfloat162 b = __floats2bfloat162_rn(a4.z, a4.w);
      uint2 u;
      u.x = *reinterpret_cast<unsigned*>(&a);
      u.y = *reinterpret_cast<unsigned*>(&b);
      reinterpret_cast<uint2*>(out_bf16)[col(sl)] = u;
    }
  }
  if (out_lse && c0 == 0 && lane == 0) *out_lse = any ? g + logf(z) : -INFINITY;
}

__global__ void lse_merge_kernel(int P, long long NH, int Dv, const float* __restrict__ o_part,
                                 const float* __restrict__ lse_part, void* __restrict__ o,
                                 int o_bf16, float* __restrict__ lse) {
  const long long i = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (i >= NH) return;
  float* of = o_bf16 ? nullptr : static_cast<float*>(o) + i * Dv;
  __nv_bfloat16* ob = o_bf16 ? static_cast<__nv_bfloat16*>(o) + i * Dv : nullptr;
  merge_row<1, 8>(P, o_part + i * Dv, NH * Dv, lse_part + i, NH, Dv, blockIdx.y * kMergeSlice, of, ob,
            lse ? lse + i : nullptr);
}

// (O, LSE) <- the exact combine of (O, LSE) and (O', LSE'), in place; one warp
// per (row, head).  Two empty partials stay O = 0, LSE = -inf.
__global__ void lse_fold_kernel(long long NH, int Dv, float* __restrict__ o, float* __restrict__ lse,
                                const float* __restrict__ o_add, const float* __restrict__ lse_add) {
  const long long i = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (i >= NH) return;
  const int lane = threadIdx.x & 31;
  const float l0 = lse[i], l1 = lse_add[i];
  const float g = fmaxf(l0, l1);
  float a0 = 0.f, a1 = 0.f, lg = -INFINITY;
  if (g != -INFINITY) {
    const float w0 = l0 == -INFINITY ? 0.f : expf(l0 - g);
    const float w1 = l1 == -INFINITY ? 0.f : expf(l1 - g);
    const float z = w0 + w1;
    a0 = w0 / z;
    a1 = w1 / z;
    lg = g + logf(z);
  }
  float* od = o + i * Dv;
  const float* oa = o_add + i * Dv;
  for (int c = lane; c < Dv; c += 32) od[c] = a0 * od[c] + a1 * oa[c];
  __syncwarp();
  if (lane == 0) lse[i] = lg;
}

// Requests of a merged decode whose result comes from parts: one warp per
// (listed request, head, 128 dims) combines the request's parts [first, first + n)
// (n = 0, a request with no rows: O = 0, LSE = -inf).
__global__ void merge_runs_kernel(const int32_t* __restrict__ list, int n_list, int H, int Dv,
                                  const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                                  void* __restrict__ o, int o_bf16, float* __restrict__ lse) {
  const long long i = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (i >= (long long)n_list * H) return;
  const int m = (int)(i / H), h = (int)(i % H);
  const int b = list[3 * m], first = list[3 * m + 1], n = list[3 * m + 2];
  const long long ob = (long long)b * H + h;
  float* of = o_bf16 ? nullptr : static_cast<float*>(o) + ob * Dv;
  __nv_bfloat16* obf = o_bf16 ? static_cast<__nv_bfloat16*>(o) + ob * Dv : nullptr;
  merge_row<1, 8>(n, ws_o + ((long long)first * H + h) * Dv, (long long)H * Dv, ws_lse + (long long)first * H + h, H,
            Dv, blockIdx.y * kMergeSlice, of, obf, lse + ob);
}

// A split pair holds few parts (2 or 3 at most worker counts): a warp takes
// kSlices slices of its row, so that each warp has kBatch x kSlices loads in
// flight and the launch fewer rounds of the load chain.
template <int kSlices, int kBatch>
__global__ void decode_fixup_kernel(const int32_t* __restrict__ plan, int B, int off_pair,
                                    int off_split, int n_split, int H, int Dv,
                                    const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                                    float* __restrict__ o_part, float* __restrict__ lse_part) {
  const long long i = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (i >= (long long)n_split * H) return;
  const int s = (int)(i / H), h = (int)(i % H);
  const int pair = plan[off_split + s];
  const cp_pair_desc d = reinterpret_cast<const cp_pair_desc*>(plan + off_pair)[pair];
  const long long ob = (long long)pair * H + h;
  merge_row<kSlices, kBatch>(d.n_parts, ws_o + ((long long)d.first_part * H + h) * Dv, (long long)H * Dv,
                             ws_lse + (long long)d.first_part * H + h, H, Dv, blockIdx.y * kSlices * kMergeSlice,
                             o_part + ob * Dv, nullptr, lse_part + ob);
}

// the groups of kSlices 128-dim slices of a row of Dv dims
unsigned merge_slices(int Dv, int kSlices = 1) {
  return (unsigned)((Dv / 4 + kSlices * kMergeSlice - 1) / (kSlices * kMergeSlice));
}

}  // namespace

cudaError_t launch_plan_maps(const int32_t* dev_plan, int n_seg, int off_seg, int off_idx,
                             int off_qpos, int off_qreq, cudaStream_t s) {
  if (n_seg == 0) return cudaSuccess;
  plan_map_kernel<<<n_seg, 256, 0, s>>>(const_cast<int32_t*>(dev_plan), off_seg, off_idx, off_qpos,
                                        off_qreq);
  return cudaGetLastError();
}

cudaError_t launch_kv_pack(const int32_t* dev_plan, const cp_plan_header& h, int elem_bytes,
                           const void* kv, const float* kv_scale, int row_elems,
                           const MutShardPtrs& dst, const MutScalePtrs& dst_scale, bool has_scale,
                           const RowMap& rm, cudaStream_t s) {
  const int row_vec = row_elems * elem_bytes / 16;
  const int warps = 8;
  const long long blocks = ((long long)h.T + warps - 1) / warps;
  kv_pack_kernel<<<(unsigned)blocks, warps * 32, 0, s>>>(dev_plan, h.C, h.R, h.T, h.off_rank,
                                                         h.off_tiles, static_cast<const uint4*>(kv),
                                                         kv_scale, row_vec, dst, dst_scale,
                                                         has_scale ? 1 : 0, rm, h.layout);
  return cudaGetLastError();
}

cudaError_t launch_page_tail_zero(const int32_t* dev_plan, const cp_plan_header& h,
                                  size_t row_bytes, void* pool, float* scale_pool,
                                  const RowMap& rm, cudaStream_t s) {
  const int pairs = h.C * h.R;
  if (pairs == 0) return cudaSuccess;
  page_tail_zero_kernel<<<pairs, dim3(32, 8), 0, s>>>(dev_plan, h.off_rank, (int)(row_bytes / 16),
                                                     static_cast<uint4*>(pool), scale_pool, rm);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(int P, int N, int H, int Dv, const float* o_part,
                             const float* lse_part, void* o, bool o_bf16, float* lse,
                             cudaStream_t s) {
  const long long NH = (long long)N * H;
  const int warps = 8;
  const long long blocks = (NH + warps - 1) / warps;
  const dim3 grid((unsigned)blocks, merge_slices(Dv));
  lse_merge_kernel<<<grid, warps * 32, 0, s>>>(P, NH, Dv, o_part, lse_part, o, o_bf16 ? 1 : 0, lse);
  return cudaGetLastError();
}

cudaError_t launch_merge_runs(const int32_t* dev_plan, const cp_plan_header& h, int n_list, int H, int Dv,
                              const float* ws_o, const float* ws_lse, void* o, bool o_bf16, float* lse,
                              cudaStream_t s) {
  if (n_list == 0) return cudaSuccess;
  const long long warps_needed = (long long)n_list * H;
  const int warps = 8;
  const long long blocks = (warps_needed + warps - 1) / warps;
  const int32_t* list = dev_plan + h.off_run + 2 + h.n_seg;
  const dim3 grid((unsigned)blocks, merge_slices(Dv));
  merge_runs_kernel<<<grid, warps * 32, 0, s>>>(list, n_list, H, Dv, ws_o, ws_lse, o, o_bf16 ? 1 : 0, lse);
  return cudaGetLastError();
}

cudaError_t launch_lse_fold(int N, int H, int Dv, float* o, float* lse, const float* o_add,
                            const float* lse_add, cudaStream_t s) {
  const long long NH = (long long)N * H;
  const int warps = 8;
  const long long blocks = (NH + warps - 1) / warps;
  lse_fold_kernel<<<(unsigned)blocks, warps * 32, 0, s>>>(NH, Dv, o, lse, o_add, lse_add);
  return cudaGetLastError();
}

cudaError_t launch_decode_fixup(const int32_t* dev_plan, const cp_plan_header& h, int H, int Dv,
                                const float* ws_o, const float* ws_lse, float* o_part,
                                float* lse_part, cudaStream_t s) {
  const long long n = (long long)h.n_split * H;
  if (n == 0) return cudaSuccess;
  const int warps = 8;
  const unsigned blocks = (unsigned)((n + warps - 1) / warps);
  if (Dv >= 4 * 4 * kMergeSlice)  // rows of 512 dims and more: four slices per warp
    decode_fixup_kernel<4, 4><<<dim3(blocks, merge_slices(Dv, 4)), warps * 32, 0, s>>>(
        dev_plan, h.R, h.off_rank, h.off_rtile, h.n_split, H, Dv, ws_o, ws_lse, o_part, lse_part);
  else
    decode_fixup_kernel<1, 8><<<dim3(blocks, merge_slices(Dv)), warps * 32, 0, s>>>(
        dev_plan, h.R, h.off_rank, h.off_rtile, h.n_split, H, Dv, ws_o, ws_lse, o_part, lse_part);
  return cudaGetLastError();
}

}  // namespace cpattn
