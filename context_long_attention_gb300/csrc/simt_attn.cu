// CUDA-core attention kernels: the fp32 prefill path and the GQA split-KV decode.
//
// Both compute the attention definition of "How GPUs Share a Long Context
// During LLM Inference" §1.1 (a query reads every key up to and including
// itself; softmax of the scaled scores weights the values) with a running
// (max, sum) so that one pass over the keys gives O and LSE (§3.3).
// One warp owns one (query row, head); lane l holds dims l, l+32, ... so that
// every key/value row is read with coalesced loads.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.h"

namespace cpattn {
namespace {

__device__ __forceinline__ float ld_elem(const float* p, long long i) { return p[i]; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16* p, long long i) {
  return __bfloat162float(p[i]);
}
// E4M3 codes (the caller's scale applies separately), converted by CUDA's own
// fp8 type
__device__ __forceinline__ float ld_elem(const __nv_fp8_e4m3* p, long long i) { return float(p[i]); }
__device__ __forceinline__ void st_elem(float* p, long long i, float x) { p[i] = x; }
__device__ __forceinline__ void st_elem(__nv_bfloat16* p, long long i, float x) {
  p[i] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) x += __shfl_xor_sync(0xffffffffu, x, d);
  return x;
}

// Running softmax state of one warp-owned row; NV value dims per lane.
template <int NV>
struct RowState {
  float m = -INFINITY, l = 0.f, acc[NV];
  __device__ RowState() {
#pragma unroll
    for (int e = 0; e < NV; ++e) acc[e] = 0.f;
  }
  // Adds one key with score s and value dims v[] (this lane's share).
  __device__ __forceinline__ void add(float s, const float (&v)[NV]) {
    const float mn = fmaxf(m, s);
    const float corr = expf(m - mn);  // m = -inf on the first key: corr = 0
    const float p = expf(s - mn);
    l = l * corr + p;
#pragma unroll
    for (int e = 0; e < NV; ++e) acc[e] = acc[e] * corr + p * v[e];
    m = mn;
  }
};

// ------------------------------------------------------------------ prefill

template <typename T, int ND>
__global__ void prefill_simt_kernel(const int32_t* __restrict__ plan, int off_req, int off_idx,
                                    int off_qpos, int off_qreq, int row_begin, int local_rows,
                                    const T* __restrict__ q, const T* __restrict__ k,
                                    const T* __restrict__ v, int Hq, int Hkv, float sm_scale,
                                    T* __restrict__ o, float* __restrict__ lse) {
  constexpr int D = ND * 32;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (h >= Hq) return;
  const int i = row_begin + blockIdx.x;  // rank-major row
  const int f = plan[off_idx + i], pos = plan[off_qpos + i], j = plan[off_qreq + i];
  const cp_req_desc rq = reinterpret_cast<const cp_req_desc*>(plan + off_req)[j];
  const int g = h / (Hq / Hkv);
  float qv[ND];
#pragma unroll
  for (int e = 0; e < ND; ++e) qv[e] = ld_elem(q, ((long long)f * Hq + h) * D + lane + 32 * e);
  RowState<ND> st;
  for (int t = 0; t <= pos; ++t) {
    const long long kr = ((long long)(rq.kv_base + t) * Hkv + g) * D + lane;
    float part = 0.f, vv[ND];
#pragma unroll
    for (int e = 0; e < ND; ++e) {
      part += qv[e] * ld_elem(k, kr + 32 * e);
      vv[e] = ld_elem(v, kr + 32 * e);
    }
    st.add(sm_scale * warp_sum(part), vv);
  }
  const long long out_row = local_rows ? (long long)blockIdx.x : (long long)i;
  const float inv = 1.f / st.l;
#pragma unroll
  for (int e = 0; e < ND; ++e) st_elem(o, (out_row * Hq + h) * D + lane + 32 * e, st.acc[e] * inv);
  if (lane == 0) lse[out_row * Hq + h] = st.m + logf(st.l);
}

// ------------------------------------------------------------------ decode

// GQA split-KV decode: a warp owns one (query head, work item) and walks the
// item's shard rows; ND dims per lane (D / 32).  The shapes the tensor-core
// GQA kernel does not take land here: fp32 caches, E4M3 caches (codes with one
// fp32 scale per token for its K and V rows: k = code_k scale, v = code_v
// scale), other head dims.  TQ is the query's type, T the cache's.
template <typename TQ, typename T, int ND>
__global__ void decode_gqa_simt_kernel(const int32_t* __restrict__ plan, int B, int off_pair,
                                       int off_worker, int off_work, const TQ* __restrict__ q,
                                       ShardPtrs kp, ShardPtrs vp, ScalePtrs sc, RowMap rm, int Hq, int Hkv,
                                       int s_q, float sm_scale, const int32_t* __restrict__ pair_count,
                                       float* __restrict__ o_part, float* __restrict__ lse_part,
                                       float* __restrict__ ws_o, float* __restrict__ ws_lse) {
  constexpr int D = ND * 32;
  const int lane = threadIdx.x & 31;
  // Column h = query row qi x Hq + head: a request's s_q query rows side by side.
  const int Hc = Hq * s_q;
  const int h = blockIdx.y * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (h >= Hc) return;
  const int qi = h / Hq;
  const int g = (h % Hq) / (Hq / Hkv);
  const int w0 = plan[off_worker + blockIdx.x], w1 = plan[off_worker + blockIdx.x + 1];
  const cp_pair_desc* pairs = reinterpret_cast<const cp_pair_desc*>(plan + off_pair);
  const cp_work_desc* work = reinterpret_cast<const cp_work_desc*>(plan + off_work);
  for (int wi = w0; wi < w1; ++wi) {
    const cp_work_desc wd = work[wi];
    const int r = wd.pair / B, b = wd.pair % B;
    const cp_pair_desc pd = pairs[wd.pair];
    float qv[ND];
#pragma unroll
    for (int e = 0; e < ND; ++e) qv[e] = ld_elem(q, ((long long)b * Hc + h) * D + lane + 32 * e);
    // Query row qi reads the tokens up to position L - s_q + qi: the pair's
    // rows hold tokens tok0 + i tok_step in increasing order, so a prefix.
    const int lim = pd.ctx_len - s_q + qi;
    const int n_valid = lim < pd.tok0 ? 0 : min(pd.rows, (lim - pd.tok0) / pd.tok_step + 1);
    const int row_end = min(min(wd.row_end, n_valid), pair_count ? pair_count[wd.pair] : wd.row_end);
    const T* kb = static_cast<const T*>(kp.p[r]);
    const T* vb = static_cast<const T*>(vp.p[r]);
    const float* scr = sc.p[r];  // per-row scales of an E4M3 cache, else nullptr
    RowState<ND> st;
    for (int row = wd.row_begin; row < row_end; ++row) {
      const long long cr = map_row(rm, wd.pair, pd.row_off, row);
      const long long kr = (cr * Hkv + g) * D + lane;
      const float rs = scr ? __ldg(scr + cr) : 1.f;
      float part = 0.f, vv[ND];
#pragma unroll
      for (int e = 0; e < ND; ++e) {
        part += qv[e] * ld_elem(kb, kr + 32 * e);
        vv[e] = ld_elem(vb, kr + 32 * e) * rs;
      }
      st.add(sm_scale * rs * warp_sum(part), vv);
    }
    float* ob;
    float* lb;
    if (wd.part < 0) {
      ob = o_part + ((long long)wd.pair * Hc + h) * D;
      lb = lse_part + (long long)wd.pair * Hc + h;
    } else {
      ob = ws_o + ((long long)wd.part * Hc + h) * D;
      lb = ws_lse + (long long)wd.part * Hc + h;
    }
    const bool empty = st.l == 0.f;
    const float inv = empty ? 0.f : 1.f / st.l;
#pragma unroll
    for (int e = 0; e < ND; ++e) ob[lane + 32 * e] = st.acc[e] * inv;
    if (lane == 0) *lb = empty ? -INFINITY : st.m + logf(st.l);
  }
}

template <typename T, int ND>
cudaError_t prefill_simt_t(const int32_t* plan, const cp_plan_header& h, int rank, int row_begin,
                           int n_rows, const void* q, const void* k, const void* v, int Hq,
                           int Hkv, float sm_scale, void* o, float* lse, cudaStream_t s) {
  const int warps = 4;
  dim3 grid(n_rows, (Hq + warps - 1) / warps);
  prefill_simt_kernel<T, ND><<<grid, warps * 32, 0, s>>>(
      plan, h.off_req, h.off_idx, h.off_qpos, h.off_qreq, row_begin, rank >= 0 ? 1 : 0,
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), Hq, Hkv,
      sm_scale, static_cast<T*>(o), lse);
  return cudaGetLastError();
}

template <typename TQ, typename T, int ND>
cudaError_t decode_gqa_t(const int32_t* plan, const cp_plan_header& h, const void* q,
                         const ShardPtrs& k, const ShardPtrs& v, const ScalePtrs& sc, const RowMap& rm,
                         int Hq, int Hkv, float sm_scale,
                         float* o_part, float* lse_part, float* ws_o, float* ws_lse,
                         const int32_t* pair_count, cudaStream_t s) {
  const int warps = 4;
  const int s_q = plan_s_q(h);
  dim3 grid(h.n_tiles, (Hq * s_q + warps - 1) / warps);
  decode_gqa_simt_kernel<TQ, T, ND><<<grid, warps * 32, 0, s>>>(
      plan, h.R, h.off_rank, h.off_req, h.off_seg, static_cast<const TQ*>(q), k, v, sc, rm, Hq, Hkv,
      s_q, sm_scale, pair_count, o_part, lse_part, ws_o, ws_lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_simt(const int32_t* plan, const cp_plan_header& h, int rank,
                                int row_begin, int n_rows, bool bf16, const void* q,
                                const void* k, const void* v, int Hq, int Hkv, int D,
                                float sm_scale, void* o, float* lse, cudaStream_t s) {
#define CP_PREFILL_CASE(ND)                                                                     \
  case ND:                                                                                      \
    return bf16 ? prefill_simt_t<__nv_bfloat16, ND>(plan, h, rank, row_begin, n_rows, q, k, v, \
                                                    Hq, Hkv, sm_scale, o, lse, s)               \
                : prefill_simt_t<float, ND>(plan, h, rank, row_begin, n_rows, q, k, v, Hq, Hkv, \
                                            sm_scale, o, lse, s);
  switch (D / 32) {
    CP_PREFILL_CASE(1)
    CP_PREFILL_CASE(2)
    CP_PREFILL_CASE(3)
    CP_PREFILL_CASE(4)
    default:
      return cudaErrorInvalidValue;
  }
#undef CP_PREFILL_CASE
}

cudaError_t launch_decode_simt(const int32_t* plan, const cp_plan_header& h,
                               cp_dtype kv_dtype, const void* q, const ShardPtrs& k,
                               const ShardPtrs& v, const ScalePtrs& sc, const RowMap& rm, int Hq,
                               int Hkv, int Dqk, int Dv, float sm_scale, float* o_part, float* lse_part,
                               float* ws_o, float* ws_lse, const int32_t* pair_count,
                               cudaStream_t s) {
  (void)Dv;
  ScalePtrs none;
  for (int r = 0; r < CP_MAX_SHARDS; ++r) none.p[r] = nullptr;
#define CP_GQA_CASE(ND)                                                                              \
  case ND:                                                                                           \
    return kv_dtype == CP_BF16                                                                       \
               ? decode_gqa_t<__nv_bfloat16, __nv_bfloat16, ND>(plan, h, q, k, v, none, rm, Hq, Hkv, \
                                                                sm_scale, o_part, lse_part, ws_o,    \
                                                                ws_lse, pair_count, s)               \
           : kv_dtype == CP_FP8_E4M3                                                                 \
               ? decode_gqa_t<__nv_bfloat16, __nv_fp8_e4m3, ND>(plan, h, q, k, v, sc, rm, Hq, Hkv,   \
                                                                sm_scale, o_part, lse_part, ws_o,    \
                                                                ws_lse, pair_count, s)               \
               : decode_gqa_t<float, float, ND>(plan, h, q, k, v, none, rm, Hq, Hkv, sm_scale,      \
                                                o_part, lse_part, ws_o, ws_lse, pair_count, s);
  switch (Dqk / 32) {
    CP_GQA_CASE(1)
    CP_GQA_CASE(2)
    CP_GQA_CASE(3)
    CP_GQA_CASE(4)
    CP_GQA_CASE(5)
    CP_GQA_CASE(6)
    CP_GQA_CASE(7)
    CP_GQA_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef CP_GQA_CASE
}

}  // namespace cpattn
