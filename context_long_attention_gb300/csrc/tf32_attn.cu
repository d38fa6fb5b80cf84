// Attention over fp32 inputs on the tcgen05 tensor cores (kind::tf32): the
// causal prefill and the GQA split-KV decode.
//
// The computation is the attention of "How GPUs Share a Long Context During
// LLM Inference" §1.1 (a query reads every key up to and including its own
// position; the softmax of the scaled scores weights the values), per shard:
// the prefill for the queries a virtual shard owns (§2.3 zigzag blocks, §2.4
// interleave runs), the decode as one partial (O, natural-log LSE) per work
// item of a (shard, request) pair, merged later exactly (§3.1-3.4).
//
// The products read their operands as tf32 (the fp32 values with a 10-bit
// mantissa) and accumulate in fp32; the softmax, O and LSE are fp32.  Every
// operand is K-major with a 128-byte swizzle (32 fp32 a row of a swizzle
// atom): the threads load the K and V tiles with plain loads and write V
// transposed (each dim's row of keys), so the tensor core never reads a
// transposed fp32 operand.  One pass per KV tile, synchronous: load, QK^T,
// softmax, P.V.  These kernels serve the fp32 path (not the bf16 and FP8
// bandwidth paths), so they keep the work order plain.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "tc_ptx.cuh"

namespace cpattn {
namespace {
using namespace tc;

constexpr int kRows = 128;  // MMA M: queries (prefill) or KV rows (decode) per tile
constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Instruction descriptor, kind::tf32 (A and B format code 2), fp32 accumulation,
// both operands K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D[tmem] (+)= A[smem] . B[smem], tf32
__device__ __forceinline__ void mma_ss_tf32(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
// D[tmem] (+)= A[tmem] . B[smem], tf32
__device__ __forceinline__ void mma_ts_tf32(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc));
}
// Byte offset of element (row, k) of a K-major fp32 operand of R rows, stored
// as 32-element chunks [R rows][128 B] with a 128-byte swizzle.
__device__ __forceinline__ int kmaj(int R, int row, int k) {
  const int byte = (k & 31) * 4;
  return (k >> 5) * R * 128 + row * 128 + ((((byte >> 4) ^ (row & 7))) << 4) + (byte & 15);
}
// Descriptor start-address step of K-step kk (8 elements) of such an operand.
__device__ __forceinline__ uint64_t kstep(int R, int kk) {
  return (uint64_t)((((kk >> 2) * R * 128) + (kk & 3) * 32) >> 4);
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ void report_timeout(unsigned* status, unsigned site, volatile int* abort) {
  *abort = 1;
  if (atomicCAS(status, 0u, 1u) == 0u) {
    status[1] = kKernTf32;
    status[2] = site;
    status[3] = blockIdx.x;
    __threadfence();
  }
}
// Issues the products of one step from warp 0 (one elected lane) and commits
// them to `bar`; every thread then waits for them.  False if the wait gave up.
template <typename F>
__device__ __forceinline__ bool run_mma(int warp, uint32_t bar, int& phase, unsigned long long wait_ns,
                                        volatile int* abort, F&& issue) {
  if (warp == 0) {
    tc_fence_after();
    if (elect_one()) {
      issue();
      mma_commit(bar);
    }
    __syncwarp();
  }
  const bool got = mbar_wait(bar, phase & 1, wait_ns, abort);
  ++phase;
  tc_fence_after();
  return __syncthreads_and(got);
}

// ------------------------------------------------------------------ prefill

struct PrefillParams {
  const int32_t* plan;
  int off_seg, tile_list, n_tiles, row_sub;
  const float* q;  // [T][Hq][D]
  const float* k;  // [KV][Hkv][D]
  const float* v;
  float* o;        // [rows][Hq][D]
  float* lse;      // [rows][Hq]
  int Hq, Hkv, group, KV;
  float scale_log2;
  unsigned* status;
  unsigned long long wait_ns;
};

// One CTA = one plan tile (up to 256 consecutive queries of one segment) x one
// query head, as two 128-query M tiles one after the other; thread i = query
// row i of the M tile = TMEM lane i.  TMEM: S (and P over it) in columns
// [0, 128), O in [128, 128 + D).
template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_tf32_kernel(const PrefillParams p) {
  constexpr int kTileBytes = kRows * D * 4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                // [128 queries x D], K-major
  uint8_t* sK = smem + kTileBytes;   // [128 keys x D], K-major
  uint8_t* sVt = sK + kTileBytes;    // V^T [D dims x 128 keys], K-major
  __shared__ __align__(8) uint64_t bar_mma, bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ volatile int zero_flag;  // never set: the drain ignores the abort flag

  const int tid = threadIdx.x, warp = tid >> 5;
  const int tile_i = blockIdx.x / p.Hq, h = blockIdx.x % p.Hq;
  const cp_tile_desc td = reinterpret_cast<const cp_tile_desc*>(p.plan + p.tile_list)[tile_i];
  const cp_seg_desc sg = reinterpret_cast<const cp_seg_desc*>(p.plan + p.off_seg)[td.seg];
  const int g = h / p.group;
  if (tid == 0) {
    mbar_init(smem_u32(&bar_mma), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    abort_flag = 0;
    zero_flag = 0;
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
  const uint32_t bar = smem_u32(&bar_mma);
  const uint32_t idS = idesc_tf32(kRows, kRows), idO = idesc_tf32(kRows, D);
  const uint64_t dQ = smem_desc(smem_u32(sQ), 16, 1024, 2);
  const uint64_t dK = smem_desc(smem_u32(sK), 16, 1024, 2);
  const uint64_t dVt = smem_desc(smem_u32(sVt), 16, 1024, 2);
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  int phase = 0;
  bool ok = true;
  for (int t = 0; t < 2 && ok; ++t) {
    const int rows = min(kRows, sg.count - td.q_off - kRows * t);
    if (rows <= 0) break;
    const int qrow = td.q_off + kRows * t + tid;  // query of this thread within the segment
    const bool valid = tid < rows;
    const int pos = valid ? sg.first_pos + qrow * sg.stride : -1;  // reads keys [0, pos]
    const int nkv = (sg.first_pos + (td.q_off + kRows * t + rows - 1) * sg.stride + kRows) / kRows;
    {  // Q row -> sQ
      const long long f = (long long)sg.first_f + (long long)qrow * sg.stride;
      const float4* src = reinterpret_cast<const float4*>(p.q + (f * p.Hq + h) * D);
#pragma unroll 4
      for (int c = 0; c < D / 4; ++c)
        *reinterpret_cast<float4*>(sQ + kmaj(kRows, tid, 4 * c)) = valid ? __ldg(src + c) : zero4;
    }
    float m = -INFINITY, l = 0.f;  // running max (log2 units of the scaled score) and sum
    for (int j = 0; j < nkv && ok; ++j) {
      {  // key 128 j + tid: its K row, and its V row into column tid of V^T
        const long long kr = (long long)sg.kv_base + kRows * j + tid;
        const bool in = kr < p.KV;  // keys past the tensor read zeros (they are masked)
        const float4* ks = reinterpret_cast<const float4*>(p.k + (kr * p.Hkv + g) * D);
        const float4* vs = reinterpret_cast<const float4*>(p.v + (kr * p.Hkv + g) * D);
#pragma unroll 4
        for (int c = 0; c < D / 4; ++c) {
          *reinterpret_cast<float4*>(sK + kmaj(kRows, tid, 4 * c)) = in ? __ldg(ks + c) : zero4;
          const float4 vv = in ? __ldg(vs + c) : zero4;
          *reinterpret_cast<float*>(sVt + kmaj(D, 4 * c + 0, tid)) = vv.x;
          *reinterpret_cast<float*>(sVt + kmaj(D, 4 * c + 1, tid)) = vv.y;
          *reinterpret_cast<float*>(sVt + kmaj(D, 4 * c + 2, tid)) = vv.z;
          *reinterpret_cast<float*>(sVt + kmaj(D, 4 * c + 3, tid)) = vv.w;
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      // S = Q K^T
      if (!run_mma(warp, bar, phase, p.wait_ns, &abort_flag, [&] {
#pragma unroll
            for (int kk = 0; kk < D / 8; ++kk)
              mma_ss_tf32(tmem, dQ + kstep(kRows, kk), dK + kstep(kRows, kk), idS, kk > 0 ? 1u : 0u);
          })) {
        if (tid == 0) report_timeout(p.status, 1, &abort_flag);
        ok = false;
        break;
      }
      // the row's scores, keys past its position masked; P = 2^(u - m) over S
      uint32_t sr[kRows];
#pragma unroll
      for (int c = 0; c < kRows / 32; ++c)
        tmem_ld32(lane_addr + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
      tmem_ld_wait();
      const int kb = kRows * j;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kRows; ++c) {
        const float u = kb + c <= pos ? __uint_as_float(sr[c]) * p.scale_log2 : -INFINITY;
        sr[c] = __float_as_uint(u);
        mx = fmaxf(mx, u);
      }
      const float m_new = fmaxf(m, mx);
      const float alpha = m == -INFINITY ? 0.f : ex2(m - m_new);  // 1 when the max did not move
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O holds the earlier tiles (their P.V completed): scale this row
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(lane_addr + kRows + 32 * c, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          tmem_st32(lane_addr + kRows + 32 * c, r);
        }
      }
      l *= alpha;
      m = m_new;
#pragma unroll
      for (int c = 0; c < kRows; ++c) {
        const float u = __uint_as_float(sr[c]);
        const float pc = u == -INFINITY ? 0.f : ex2(u - m);
        l += pc;
        sr[c] = __float_as_uint(pc);
      }
#pragma unroll
      for (int c = 0; c < kRows / 32; ++c)
        tmem_st32(lane_addr + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
      tmem_st_wait();
      tc_fence_before();
      __syncthreads();
      // O (+)= P V, P read from TMEM
      if (!run_mma(warp, bar, phase, p.wait_ns, &abort_flag, [&] {
#pragma unroll
            for (int kk = 0; kk < kRows / 8; ++kk)
              mma_ts_tf32(tmem + kRows, tmem + 8 * kk, dVt + kstep(D, kk), idO, (j > 0 || kk > 0) ? 1u : 0u);
          })) {
        if (tid == 0) report_timeout(p.status, 2, &abort_flag);
        ok = false;
        break;
      }
    }
    if (!ok) break;
    // epilogue: O / l and LSE
    const long long out_row = (long long)sg.local_start + qrow - p.row_sub;
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(lane_addr + kRows + 32 * c, r);
      tmem_ld_wait();
      if (valid) {
        float4* dst = reinterpret_cast<float4*>(p.o + (out_row * p.Hq + h) * D + 32 * c);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          dst[e] = make_float4(__uint_as_float(r[4 * e]) * inv, __uint_as_float(r[4 * e + 1]) * inv,
                               __uint_as_float(r[4 * e + 2]) * inv, __uint_as_float(r[4 * e + 3]) * inv);
      }
    }
    if (valid) p.lse[out_row * p.Hq + h] = l > 0.f ? (m + lg2(l)) * kLn2 : -INFINITY;
    tc_fence_before();
    __syncthreads();  // the next M tile rewrites sQ and TMEM
    tc_fence_after();
  }
  // Never free TMEM under a running product (a wait that gave up leaves one).
  if (warp == 0) {
    if (elect_one()) mma_commit(smem_u32(&bar_drain));
    __syncwarp();
    mbar_wait(smem_u32(&bar_drain), 0, 1000000000ull, &zero_flag);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------------ GQA decode

struct DecodeParams {
  const int32_t* plan;
  int B, off_pair, off_worker, off_work;
  const float* q;  // [B][s_q][Hq][D]
  ShardPtrs k, v;  // per shard [rows][Hkv][D]
  int Hq, Hkv, G, s_q, Hc, ncols;
  float scale_log2;
  float* o_part;
  float* lse_part;
  float* ws_o;
  float* ws_lse;
  const int32_t* pair_count;
  unsigned* status;
  unsigned long long wait_ns;
};

// One CTA = one decode worker; a unit is (work item, kv head g), whose n =
// qi G + i query columns are padded to NP; thread t = KV row t of a tile =
// TMEM lane t, and in the epilogue dim row t of O^T.  Products transposed so
// that M = 128:
//   S^T [128 rows x NP]  = K_g tile [128 x D] . Q_g^T
//   O^T [128 dims x NP] += V_g tile^T [128 x 128 rows] . P^T
// (dims past D are a zero block of V^T).  TMEM: S^T in [0, NP), O^T in [NP, 2 NP).
template <int D, int NP>
__global__ void __launch_bounds__(kThreads, 1) decode_gqa_tf32_kernel(const DecodeParams p) {
  constexpr int kKBytes = kRows * D * 4;       // K tile
  constexpr int kVtBytes = kRows * kRows * 4;  // V^T, 128 dim rows (zero past D)
  constexpr int kQBytes = NP * D * 4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sK = smem;                  // [128 rows x D], K-major
  uint8_t* sVt = sK + kKBytes;         // [128 dims x 128 rows], K-major
  uint8_t* sQ = sVt + kVtBytes;        // [NP columns x D], K-major
  uint8_t* sP = sQ + kQBytes;          // P^T as [NP columns x 128 rows], K-major
  __shared__ __align__(8) uint64_t bar_mma, bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ volatile int zero_flag;  // never set: the drain ignores the abort flag
  __shared__ float sM[NP];        // running max per column (log2 units)
  __shared__ float sAlpha[NP];    // this tile's rescale per column; in the epilogue 1 / sum
  __shared__ float sRed[4][NP];   // per-warp column maxima, then column sums
  __shared__ int sCol[NP];        // output column of unit column n for kv head 0

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(smem_u32(&bar_mma), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    abort_flag = 0;
    zero_flag = 0;
    mbar_init_fence();
  }
  if (tid < NP) sCol[tid] = (tid / p.G) * p.Hq + tid % p.G;
  // V^T dims past D and query columns past the unit's stay zero
  for (int i = tid; i < kVtBytes / 16; i += kThreads) reinterpret_cast<uint4*>(sVt)[i] = make_uint4(0, 0, 0, 0);
  for (int i = tid; i < kQBytes / 16; i += kThreads) reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
  const uint32_t bar = smem_u32(&bar_mma);
  const uint32_t idS = idesc_tf32(kRows, NP), idO = idesc_tf32(kRows, NP);
  const uint64_t dK = smem_desc(smem_u32(sK), 16, 1024, 2);
  const uint64_t dVt = smem_desc(smem_u32(sVt), 16, 1024, 2);
  const uint64_t dQ = smem_desc(smem_u32(sQ), 16, 1024, 2);
  const uint64_t dP = smem_desc(smem_u32(sP), 16, 1024, 2);
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  const cp_pair_desc* pairs = reinterpret_cast<const cp_pair_desc*>(p.plan + p.off_pair);
  const cp_work_desc* work = reinterpret_cast<const cp_work_desc*>(p.plan + p.off_work);
  const int w0 = p.plan[p.off_worker + blockIdx.x], w1 = p.plan[p.off_worker + blockIdx.x + 1];
  int phase = 0;
  bool ok = true;
  for (int wi = w0; wi < w1 && ok; ++wi) {
    const cp_work_desc wd = work[wi];
    const cp_pair_desc pd = pairs[wd.pair];
    const int r = wd.pair / p.B, b = wd.pair % p.B;
    const int row_end = p.pair_count ? min(wd.row_end, max(wd.row_begin, __ldg(p.pair_count + wd.pair)))
                                     : wd.row_end;
    const int nrows = row_end - wd.row_begin;
    const int ntiles = (nrows + kRows - 1) / kRows;
    float* out_o = wd.part < 0 ? p.o_part + (long long)wd.pair * p.Hc * D : p.ws_o + (long long)wd.part * p.Hc * D;
    float* out_l = wd.part < 0 ? p.lse_part + (long long)wd.pair * p.Hc : p.ws_lse + (long long)wd.part * p.Hc;
    if (ntiles == 0) {  // empty shard: O = 0, LSE = -inf
      for (int i = tid; i < p.Hc * D; i += kThreads) out_o[i] = 0.f;
      for (int i = tid; i < p.Hc; i += kThreads) out_l[i] = -INFINITY;
      continue;
    }
    const long long row0 = (long long)pd.row_off + wd.row_begin;
    const float* kb = static_cast<const float*>(p.k.p[r]);
    const float* vb = static_cast<const float*>(p.v.p[r]);
    // token of row t of tile j: tok_t + j tok_j; masked for the columns of the
    // query rows that come before it (several query rows per request)
    const int tok_j = kRows * pd.tok_step;
    const int tok_t = pd.tok0 + (wd.row_begin + tid) * pd.tok_step;
    const int lim = pd.ctx_len - p.s_q;
    for (int kh = 0; kh < p.Hkv && ok; ++kh) {
      // ---- the unit's query columns -> sQ (every product of the previous unit completed)
      for (int i = tid; i < p.ncols * (D / 4); i += kThreads) {
        const int n = i / (D / 4), c = i % (D / 4);
        const int qi = n / p.G, hh = kh * p.G + n % p.G;
        const float4 v = __ldg(reinterpret_cast<const float4*>(p.q + (((long long)b * p.s_q + qi) * p.Hq + hh) * D) + c);
        *reinterpret_cast<float4*>(sQ + kmaj(NP, n, 4 * c)) = v;
      }
      if (tid < NP) sM[tid] = -INFINITY;
      float l[NP];
#pragma unroll
      for (int n = 0; n < NP; ++n) l[n] = 0.f;
      for (int j = 0; j < ntiles && ok; ++j) {
        const int row = j * kRows + tid;
        const bool valid = row < nrows;
        {  // row t's K -> sK, its V -> column t of V^T (rows past the item read nothing)
          const long long sr = row0 + row;
          const float4* ks = reinterpret_cast<const float4*>(kb + (sr * p.Hkv + kh) * D);
          const float4* vs = reinterpret_cast<const float4*>(vb + (sr * p.Hkv + kh) * D);
#pragma unroll 4
          for (int c = 0; c < D / 4; ++c) {
            *reinterpret_cast<float4*>(sK + kmaj(kRows, tid, 4 * c)) = valid ? __ldg(ks + c) : zero4;
            const float4 vv = valid ? __ldg(vs + c) : zero4;
            *reinterpret_cast<float*>(sVt + kmaj(kRows, 4 * c + 0, tid)) = vv.x;
            *reinterpret_cast<float*>(sVt + kmaj(kRows, 4 * c + 1, tid)) = vv.y;
            *reinterpret_cast<float*>(sVt + kmaj(kRows, 4 * c + 2, tid)) = vv.z;
            *reinterpret_cast<float*>(sVt + kmaj(kRows, 4 * c + 3, tid)) = vv.w;
          }
        }
        fence_proxy_async_smem();
        __syncthreads();
        // S^T = K Q^T
        if (!run_mma(warp, bar, phase, p.wait_ns, &abort_flag, [&] {
#pragma unroll
              for (int kk = 0; kk < D / 8; ++kk)
                mma_ss_tf32(tmem, dK + kstep(kRows, kk), dQ + kstep(NP, kk), idS, kk > 0 ? 1u : 0u);
            })) {
          if (tid == 0) report_timeout(p.status, 3, &abort_flag);
          ok = false;
          break;
        }
        // u = score (log2 units); masked rows and columns read nothing
        const int mcols = min(NP, max(0, tok_t + j * tok_j - lim) * p.G);
        float u[NP];
        {
          uint32_t a[NP];
#pragma unroll
          for (int c = 0; c < NP / 16; ++c) tmem_ld16(lane_addr + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&a[16 * c]));
          tmem_ld_wait();
#pragma unroll
          for (int n = 0; n < NP; ++n)
            u[n] = valid && n >= mcols && n < p.ncols ? __uint_as_float(a[n]) * p.scale_log2 : -INFINITY;
        }
        // column maxima over the tile's rows; the running max of a column moves to them
#pragma unroll
        for (int n = 0; n < NP; ++n) {
          float v = u[n];
#pragma unroll
          for (int d = 16; d > 0; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
          if (lane == 0) sRed[warp][n] = v;
        }
        __syncthreads();
        if (tid < NP) {
          const float cm = fmaxf(fmaxf(sRed[0][tid], sRed[1][tid]), fmaxf(sRed[2][tid], sRed[3][tid]));
          const float mo = sM[tid], mn = fmaxf(mo, cm);
          sAlpha[tid] = mo == -INFINITY ? 0.f : ex2(mo - mn);
          sM[tid] = mn;
        }
        __syncthreads();
        bool moved = false;
        float pr[NP];
#pragma unroll
        for (int n = 0; n < NP; ++n) {
          const float a = sAlpha[n];
          moved |= a != 1.f;
          l[n] *= a;
          pr[n] = u[n] == -INFINITY ? 0.f : ex2(u[n] - sM[n]);
          l[n] += pr[n];
          *reinterpret_cast<float*>(sP + kmaj(NP, n, tid)) = pr[n];
        }
        if (j > 0 && __syncthreads_or(moved)) {
          // O^T holds the earlier tiles (their P.V completed): scale its columns
          uint32_t o[NP];
#pragma unroll
          for (int c = 0; c < NP / 16; ++c) tmem_ld16(lane_addr + NP + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&o[16 * c]));
          tmem_ld_wait();
#pragma unroll
          for (int n = 0; n < NP; ++n) o[n] = __float_as_uint(__uint_as_float(o[n]) * sAlpha[n]);
#pragma unroll
          for (int c = 0; c < NP / 16; ++c) tmem_st16(lane_addr + NP + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&o[16 * c]));
          tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // O^T (+)= V^T P^T
        if (!run_mma(warp, bar, phase, p.wait_ns, &abort_flag, [&] {
#pragma unroll
              for (int kk = 0; kk < kRows / 8; ++kk)
                mma_ss_tf32(tmem + NP, dVt + kstep(kRows, kk), dP + kstep(NP, kk), idO, (j > 0 || kk > 0) ? 1u : 0u);
            })) {
          if (tid == 0) report_timeout(p.status, 4, &abort_flag);
          ok = false;
          break;
        }
      }
      if (!ok) break;
      // ---- epilogue of the unit: column sums, O^T / sum, LSE
#pragma unroll
      for (int n = 0; n < NP; ++n) {
        float v = l[n];
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
        if (lane == 0) sRed[warp][n] = v;
      }
      __syncthreads();
      if (tid < NP) {
        const float tot = sRed[0][tid] + sRed[1][tid] + sRed[2][tid] + sRed[3][tid];
        sAlpha[tid] = tot > 0.f ? 1.f / tot : 0.f;
        if (tid < p.ncols) out_l[sCol[tid] + kh * p.G] = tot > 0.f ? (sM[tid] + lg2(tot)) * kLn2 : -INFINITY;
      }
      __syncthreads();
      {
        uint32_t o[NP];
#pragma unroll
        for (int c = 0; c < NP / 16; ++c) tmem_ld16(lane_addr + NP + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&o[16 * c]));
        tmem_ld_wait();
        if (tid < D) {
#pragma unroll
          for (int n = 0; n < NP; ++n)
            if (n < p.ncols) out_o[(long long)(sCol[n] + kh * p.G) * D + tid] = __uint_as_float(o[n]) * sAlpha[n];
        }
      }
      tc_fence_before();
      __syncthreads();  // sQ, sM, sAlpha and sRed are free for the next unit
      tc_fence_after();
    }
  }
  // Never free TMEM under a running product (a wait that gave up leaves one).
  if (warp == 0) {
    if (elect_one()) mma_commit(smem_u32(&bar_drain));
    __syncwarp();
    mbar_wait(smem_u32(&bar_drain), 0, 1000000000ull, &zero_flag);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

template <int D>
cudaError_t launch_prefill_d(const PrefillParams& p, cudaStream_t s) {
  constexpr int smem = 3 * kRows * D * 4 + 1024;
  cudaError_t e = cudaFuncSetAttribute(prefill_tf32_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  prefill_tf32_kernel<D><<<(unsigned)((long long)p.n_tiles * p.Hq), kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int D, int NP>
cudaError_t launch_decode_d(const DecodeParams& p, int grid, cudaStream_t s) {
  constexpr int smem = kRows * D * 4 + kRows * kRows * 4 + NP * D * 4 + NP * kRows * 4 + 1024;
  auto kern = decode_gqa_tf32_kernel<D, NP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tf32_supported(int D) { return D == 64 || D == 128; }

cudaError_t launch_prefill_tf32(const int32_t* dev_plan, const int32_t* host_plan, const cp_plan_header& h,
                                int rank, const void* q, const void* k, const void* v, int Hq, int Hkv, int D,
                                float sm_scale, void* o, float* lse, cudaStream_t s) {
  PrefillParams p;
  p.plan = dev_plan;
  p.off_seg = h.off_seg;
  if (rank < 0) {
    p.tile_list = h.off_tiles;
    p.n_tiles = h.n_tiles;
    p.row_sub = 0;
  } else {
    const int32_t* rto = host_plan + h.off_rtile;
    p.tile_list = h.off_rtile + h.C + 1 + 2 * rto[rank];
    p.n_tiles = rto[rank + 1] - rto[rank];
    p.row_sub = host_plan[h.off_rank + rank];
  }
  if (p.n_tiles == 0) return cudaSuccess;
  p.q = static_cast<const float*>(q);
  p.k = static_cast<const float*>(k);
  p.v = static_cast<const float*>(v);
  p.o = static_cast<float*>(o);
  p.lse = lse;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = Hq / Hkv;
  p.KV = h.KV;
  p.scale_log2 = sm_scale * kLog2e;
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevice;
  p.wait_ns = wait_limit_ns();
  return D == 128 ? launch_prefill_d<128>(p, s) : launch_prefill_d<64>(p, s);
}

bool gqa_tf32_supported(int Hq, int Hkv, int Dqk, int Dv, int s_q, bool paged) {
  return !paged && Dqk == Dv && (Dqk == 64 || Dqk == 128) && Hkv >= 1 && Hq % Hkv == 0 &&
         (Hq / Hkv) * s_q <= 64;
}

cudaError_t launch_decode_gqa_tf32(const int32_t* dev_plan, const cp_plan_header& h, const void* q,
                                   const ShardPtrs& k, const ShardPtrs& v, int Hq, int Hkv, int D, float sm_scale,
                                   float* o_part, float* lse_part, float* ws_o, float* ws_lse,
                                   const int32_t* pair_count, cudaStream_t s) {
  DecodeParams p;
  p.plan = dev_plan;
  p.B = h.R;
  p.off_pair = h.off_rank;
  p.off_worker = h.off_req;
  p.off_work = h.off_seg;
  p.q = static_cast<const float*>(q);
  p.k = k;
  p.v = v;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.s_q = plan_s_q(h);
  p.Hc = Hq * p.s_q;
  p.ncols = p.G * p.s_q;
  p.scale_log2 = sm_scale * kLog2e;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.ws_o = ws_o;
  p.ws_lse = ws_lse;
  p.pair_count = pair_count;
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevice;
  p.wait_ns = wait_limit_ns();
  const int grid = h.n_tiles;
  if (D == 64) {
    if (p.ncols <= 16) return launch_decode_d<64, 16>(p, grid, s);
    if (p.ncols <= 32) return launch_decode_d<64, 32>(p, grid, s);
    return launch_decode_d<64, 64>(p, grid, s);
  }
  if (p.ncols <= 16) return launch_decode_d<128, 16>(p, grid, s);
  if (p.ncols <= 32) return launch_decode_d<128, 32>(p, grid, s);
  return launch_decode_d<128, 64>(p, grid, s);
}

}  // namespace cpattn
