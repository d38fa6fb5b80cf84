// GQA split-KV decode over an FP8-E4M3 cache (head dim 128) on FP8 tensor-core
// products.
//
// The same computation as the bf16 GQA kernel ("How GPUs Share a Long
// Context During LLM Inference" §3.1-3.4): per work item (a row range of one
// (shard, request) pair) and kv head g, a partial O and the natural-log LSE of
// the G = Hq/Hkv query heads of g over the item's rows, merged later exactly
// (§3.3).  The cache holds E4M3 codes with one fp32 scale per token for both
// its K and V rows (k = code x scale, v = code x scale).
//
// The codes go from HBM to shared memory by TMA as stored and feed
// kind::f8f6f4 products directly, as in the FP8 MLA decode: the bf16 query and
// the softmax weights are carried as pairs hi + lo of E4M3 numbers (hi = x
// rounded to E4M3, lo = the remainder rounded to E4M3; 8 significant bits for
// |x| >= 2^-2, absolute error <= 2^-10 below):
//   query:   x = q 2^e_q, e_q per unit so that max |x| is in [128, 256)
//   weights: x = 2^(s - M_n) scale_row 2^gs, gs per unit so that
//            scale_row 2^gs < 32; the running max of a column moves when a
//            score passes it by more than 2^3, so x < 256
// The products, transposed so that M = 128 KV rows, with the unit's
// n = qi G + i query columns padded to NP (16 or 32):
//   S^T [128 rows x 2 NP] = K_codes_g [128 x 128] . [Q_hi | Q_lo]^T
//     score(row, n) = (S^T[row][n] + S^T[row][NP + n]) scale_row 2^-e_q
//   O^T [128 dims x NP]  += V_codes_g^T [128 x 128 rows] . (P_hi^T + P_lo^T)
// The hi and lo products of a K-step share A (a 128-dim x 32-row block of
// V_codes^T), which the second takes from the tensor core's A collector.
//
// Warp roles (352 threads): warps 0-7 softmax in two streams, warps 0-3 the
// tiles with even g and warps 4-7 those with odd g (thread = KV row of the
// tile = TMEM lane; in a unit's epilogue a dim row of O^T); warp 8 TMA (the K
// and V codes of a tile into one of six 32 KB slots); warp 9 QK^T issue;
// warp 10 P.V issue and TMEM owner.  Issuing a tcgen05.mma holds the issuing
// thread about as long as the product runs, so each product stream has its
// own issuing warp (one elected lane, the loop run warp-wide) and the tensor
// pipe interleaves them.  A softmax stream has its own S^T buffer, P buffer,
// O^T accumulator and running max, sum and weight exponent: loading a tile's
// scores from TMEM takes ~900 clk while products run, and one stream's loads
// overlap the other's exponentials.  The unit's epilogue merges the two
// streams' (O, max, sum) exactly, as the LSE merge would.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "internal.h"
#include "tc_ptx.cuh"

namespace cpattn {
namespace {
using namespace tc;

constexpr int kRows = 128;                  // KV rows per tile (MMA M)
constexpr int kD = 128;                     // head dim
constexpr int kCodeBytes = kRows * kD;      // E4M3 K or V tile of one kv head: 16 KB
constexpr int kSlotBytes = 2 * kCodeBytes;  // a slot: the tile's K and V codes
constexpr int kSlots = 6;
constexpr int kSoftmaxWarps = 8;  // two streams (even and odd tiles) of four TMEM lane quarters
constexpr int kSoftmax = 32 * kSoftmaxWarps;
constexpr int kWarpTma = kSoftmaxWarps, kWarpQk = kSoftmaxWarps + 1, kWarpPv = kSoftmaxWarps + 2;
constexpr int kThreads = 32 * (kSoftmaxWarps + 3);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 3.0f;  // the running max moves when a score passes it by > 2^3
constexpr int kWeightTop = 5;         // scale_row 2^gs < 2^5, so a weight 2^(s - M) scale_row 2^gs < 2^8
constexpr int kTmemCols = 256;

// Shared memory: the slots, the unit's query operand [Q_hi | Q_lo] (2 NP rows
// x 128 B, K-major, 128-byte swizzle), two P buffers [P_hi | P_lo] (each NP
// rows x 128 B, K-major: row n holds column n's weights of the tile's 128 KV
// rows).
template <int NP>
struct Geo {
  static constexpr int kQOff = kSlots * kSlotBytes;
  static constexpr int kQBytes = 2 * NP * 128;
  static constexpr int kPOff = kQOff + kQBytes;
  static constexpr int kPBytes = 2 * NP * 128;  // one buffer: hi then lo
  static constexpr int kSmem = kPOff + 2 * kPBytes + 1024;
};

struct Params {
  const int32_t* plan;
  int B, off_pair, off_worker, off_work;
  const __nv_bfloat16* q;  // [B][s_q][Hq][128]
  int Hq, Hkv, G;          // query heads, kv heads, query heads per kv head
  int s_q;                 // query rows per request
  int Hc;                  // output columns per request: s_q x Hq
  float scale_log2;        // sm_scale * log2(e)
  ScalePtrs sc;            // per-row scales of each shard
  float* o_part;
  float* lse_part;
  float* ws_o;
  float* ws_lse;
  const int32_t* pair_count;  // rows in use per pair (a selection buffer), or nullptr
  unsigned* status;
  unsigned long long wait_ns;
};

// Tensor maps of the shards' K and V codes ([rows, Hkv, 128] bytes, box 128
// bytes x 1 head x 128 rows, 128-byte swizzle).
struct CodeMaps {
  CUtensorMap k[CP_MAX_SHARDS];
  CUtensorMap v[CP_MAX_SHARDS];
};

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
__device__ __forceinline__ int ordered(float f) {
  const int b = __float_as_int(f);
  return b >= 0 ? b : b ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float unordered(int b) {
  return __int_as_float(b >= 0 ? b : b ^ 0x7FFFFFFF);
}
// 2^e for integer e in [-126, 127], exactly.
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }
// Byte offset of (row, byte) in a 128-byte-swizzled [rows][128 B] block.
__device__ __forceinline__ int sw128(int row, int byte) {
  return row * 128 + ((((byte >> 4) ^ (row & 7))) << 4) + (byte & 15);
}
// D[tmem] (+)= A . B with 8-bit operands, A read from shared memory into the
// tensor core's A collector buffer and kept for the next product (fill), or
// taken from that buffer, which the next product may not use again (lastuse).
__device__ __forceinline__ void mma_f8_fill_a(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4.collector::a::fill [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_f8_reuse_a(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4.collector::a::lastuse [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
// Two values -> E4M3 pairs (hi, lo) with hi + lo ~ (x0, x1); byte 0 holds x0's code.
__device__ __forceinline__ void split_e4m3x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  uint16_t a, b, h, l;
  uint32_t xh, back, rem;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(a) : "f"(x0));
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(b) : "f"(x1));
  asm("mov.b32 %0, {%1, %2};" : "=r"(xh) : "h"(a), "h"(b));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(h) : "r"(xh));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(back) : "h"(h));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(rem) : "r"(xh), "r"(back));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(l) : "r"(rem));
  hi = h;
  lo = l;
}
// Exponent that maps the largest |x| of a set into [2^(top-1), 2^top).
__device__ __forceinline__ int scale_exponent(float maxabs, int top, int fallback) {
  if (!(maxabs > 0.f)) return fallback;
  const int E = (__float_as_int(maxabs) >> 23) & 0xFF;
  const int e = E == 0 ? -126 : E - 126;
  return max(-120, min(120, top - e));
}
__device__ void report_timeout(unsigned* status, unsigned site, volatile int* abort) {
  *abort = 1;
  if (atomicCAS(status, 0u, 1u) == 0u) {
    status[1] = kKernDecodeGqaF8;
    status[2] = site;
    status[3] = blockIdx.x;
    __threadfence();
  }
}

// The fields of one work item that every role reads.
struct Item {
  int pair, r, b, part, row_begin, nrows, ntiles;
  long long row0;  // first shard row
  cp_pair_desc pd;
};
__device__ __forceinline__ Item read_item(const Params& p, int wi) {
  const cp_pair_desc* pairs = reinterpret_cast<const cp_pair_desc*>(p.plan + p.off_pair);
  const cp_work_desc* work = reinterpret_cast<const cp_work_desc*>(p.plan + p.off_work);
  const cp_work_desc wd = work[wi];
  Item it;
  it.pair = wd.pair;
  it.r = wd.pair / p.B;
  it.b = wd.pair % p.B;
  it.part = wd.part;
  it.pd = pairs[wd.pair];
  const int row_end = p.pair_count ? min(wd.row_end, max(wd.row_begin, __ldg(p.pair_count + wd.pair)))
                                   : wd.row_end;
  it.row_begin = wd.row_begin;
  it.nrows = row_end - wd.row_begin;
  it.ntiles = (it.nrows + kRows - 1) / kRows;
  it.row0 = (long long)it.pd.row_off + wd.row_begin;
  return it;
}
__device__ __forceinline__ float* out_rows(const Params& p, const Item& it) {
  return it.part < 0 ? p.o_part + (long long)it.pair * p.Hc * kD : p.ws_o + (long long)it.part * p.Hc * kD;
}
__device__ __forceinline__ float* out_lse(const Params& p, const Item& it) {
  return it.part < 0 ? p.lse_part + (long long)it.pair * p.Hc : p.ws_lse + (long long)it.part * p.Hc;
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(taddr));
}
// A unit (work item, kv head) covers the item's tiles; g counts tiles over all
// units of this CTA in the order every role walks them, so the parity of
// each barrier's wait follows from g (slot barriers complete once per use of
// their slot, S^T and P buffer barriers once per use of their buffer, bar_q
// once per unit).
template <int NP>
__global__ void __launch_bounds__(kThreads, 1)
    decode_gqa_f8_kernel(const __grid_constant__ CodeMaps maps, const Params p) {
  using Gm = Geo<NP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + Gm::kQOff;
  uint8_t* sP = smem + Gm::kPOff;
  // full[s]: slot s holds its tile's codes; empty[s]: the P.V of the slot's
  // tile has completed (and with it the QK^T before it), so the slot, the P
  // buffer of that tile and O^T's earlier columns are free.
  // s[b]: S^T buffer b holds its tile's scores; sfree[b]: the softmax loaded them.
  // p[b]: P buffer b holds its tile's weights.  q: the unit's query operand is written.
  __shared__ __align__(8) uint64_t bar_full[kSlots], bar_empty[kSlots], bar_s[2], bar_sfree[2], bar_p[2];
  __shared__ __align__(8) uint64_t bar_q, bar_drain_qk, bar_drain_pv;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ volatile int zero_flag;  // never set: drains ignore the abort flag
  __shared__ float sM[2][NP];       // each stream's running max per column (log2 units)
  __shared__ float sDelta[2][NP];   // its last move
  __shared__ int sRed[2][4][NP];    // each stream's cross-warp column maxima, then column sums
  __shared__ uint32_t sRed1[2][4];  // each stream's per-warp max of the token scales
  __shared__ uint32_t sQmax[kSoftmaxWarps];  // per-warp max of |q|
  __shared__ float sCoef[2][NP];    // epilogue: each stream's factor to the common max, / sum
  __shared__ int sGs[2];            // epilogue: each stream's weight exponent
  __shared__ int sCol[NP];       // output column of unit column n for kv head 0

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {  // buffer b serves the tiles of stream b
      mbar_init(smem_u32(&bar_s[b]), 1);
      mbar_init(smem_u32(&bar_sfree[b]), kSoftmax / 2);
      mbar_init(smem_u32(&bar_p[b]), kSoftmax / 2);
    }
    mbar_init(smem_u32(&bar_q), kSoftmax);
    mbar_init(smem_u32(&bar_drain_qk), 1);
    mbar_init(smem_u32(&bar_drain_pv), 1);
    abort_flag = 0;
    zero_flag = 0;
    mbar_init_fence();
  }
  if (threadIdx.x < NP) sCol[threadIdx.x] = (threadIdx.x / p.G) * p.Hq + threadIdx.x % p.G;
  // query operand rows past the unit's columns stay zero
  for (int i = threadIdx.x; i < Gm::kQBytes / 16; i += kThreads) reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == kWarpPv) tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // TMEM: S^T buffer b at columns [2 NP b, 2 NP b + 2 NP) (hi products, then
  // lo); stream b's O^T at [4 NP + NP b, 5 NP + NP b)
  const uint32_t tmem = tmem_slot;
  const uint32_t tmem_o = tmem + 4 * NP;
  const int w0 = p.plan[p.off_worker + blockIdx.x], w1 = p.plan[p.off_worker + blockIdx.x + 1];
  const int ncols = p.G * p.s_q;  // columns of a unit in use
  const uint32_t sbase = smem_u32(smem);

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA: codes into the slots
    bool ok = true;
    int g = 0;
    int last[kSlots];
#pragma unroll
    for (int s = 0; s < kSlots; ++s) last[s] = -1;
    for (int wi = w0; wi < w1 && ok; ++wi) {
      const Item it = read_item(p, wi);
      for (int kh = 0; kh < p.Hkv && it.ntiles > 0 && ok; ++kh) {
        for (int j = 0; j < it.ntiles; ++j, ++g) {
          const int s = g % kSlots, use = g / kSlots;
          // the slot's previous tile (g - kSlots) must have gone through its P.V
          if (use > 0 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_empty[s]), (use - 1) & 1,
                                                            p.wait_ns, &abort_flag))) {
            if (lane == 0) report_timeout(p.status, 1, &abort_flag);
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&bar_full[s]);
          if (elect_one()) {
            mbar_expect_tx(full, kSlotBytes);
            const int y = (int)(it.row0 + (long long)j * kRows);
            tma_load_3d(sbase + s * kSlotBytes, &maps.k[it.r], 0, kh, y, full);
            tma_load_3d(sbase + s * kSlotBytes + kCodeBytes, &maps.v[it.r], 0, kh, y, full);
          }
          __syncwarp();
          last[s] = g;
        }
      }
    }
    // Never leave with a copy in flight.
    for (int s = 0; s < kSlots; ++s)
      if (last[s] >= 0) mbar_wait(smem_u32(&bar_full[s]), (last[s] / kSlots) & 1, 1000000000ull, &zero_flag);
    __syncwarp();
  } else if (warp == kWarpQk) {
    // ------------------------------------------------------------ QK^T issue
    const uint32_t idQK = idesc_e4m3_f32(kRows, 2 * NP, 0, 0);
    // K codes and the query operand K-major, 128-byte swizzle; a K-step of 32
    // dims is 32 bytes of a row, 2 in the descriptor's start-address field
    const uint64_t dK = smem_desc(sbase, 16, 1024, 2);
    const uint64_t dQ = smem_desc(smem_u32(sQ), 16, 1024, 2);
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, p.wait_ns, &abort_flag));
    };
    bool ok = true;
    int g = 0, nu = 0;
    for (int wi = w0; wi < w1 && ok; ++wi) {
      const Item it = read_item(p, wi);
      for (int kh = 0; kh < p.Hkv && it.ntiles > 0 && ok; ++kh, ++nu) {
        // the unit's query operand is in place (written after every product of
        // the previous unit completed)
        if (!wait_all(smem_u32(&bar_q), nu & 1)) {
          if (lane == 0) report_timeout(p.status, 2, &abort_flag);
          ok = false;
          break;
        }
        for (int j = 0; j < it.ntiles; ++j, ++g) {
          const int s = g % kSlots, b = g & 1;
          // S^T buffer b is free once the softmax has loaded tile g - 2's scores
          if (g >= 2 && !wait_all(smem_u32(&bar_sfree[b]), ((g >> 1) & 1) ^ 1)) {
            if (lane == 0) report_timeout(p.status, 9, &abort_flag);
            ok = false;
            break;
          }
          if (!wait_all(smem_u32(&bar_full[s]), (g / kSlots) & 1)) {
            if (lane == 0) report_timeout(p.status, 3, &abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint64_t a = dK + (uint64_t)((s * kSlotBytes) >> 4);
#pragma unroll
            for (int ks = 0; ks < kD / 32; ++ks)
              mma_ss_f8(tmem + 2 * NP * b, a + 2 * ks, dQ + 2 * ks, idQK, ks > 0 ? 1u : 0u);
            mma_commit(smem_u32(&bar_s[b]));
          }
          __syncwarp();
        }
      }
    }
    // Never free TMEM under a running MMA.
    if (elect_one()) mma_commit(smem_u32(&bar_drain_qk));
    __syncwarp();
    mbar_wait(smem_u32(&bar_drain_qk), 0, 1000000000ull, &zero_flag);
  } else if (warp == kWarpPv) {
    // ------------------------------------------------------------ P.V issue, TMEM owner
    const uint32_t idPV = idesc_e4m3_f32(kRows, NP, 1, 0);
    // V^T: the V codes read MN-major (M = 128 dims of a 128-byte row; a K-step
    // of 32 rows is 4 KB); P_hi / P_lo K-major like the query operand
    const uint64_t dV = smem_desc(sbase + kCodeBytes, kCodeBytes, 1024, 2);
    const uint64_t dP = smem_desc(smem_u32(sP), 16, 1024, 2);
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, p.wait_ns, &abort_flag));
    };
    bool ok = true;
    int g = 0;
    for (int wi = w0; wi < w1 && ok; ++wi) {
      const Item it = read_item(p, wi);
      for (int kh = 0; kh < p.Hkv && it.ntiles > 0 && ok; ++kh) {
        for (int j = 0; j < it.ntiles; ++j, ++g) {
          const int s = g % kSlots, b = g & 1;
          if (!wait_all(smem_u32(&bar_p[b]), (g >> 1) & 1) ||
              !wait_all(smem_u32(&bar_full[s]), (g / kSlots) & 1)) {
            if (lane == 0) report_timeout(p.status, 4, &abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint64_t av = dV + (uint64_t)((s * kSlotBytes) >> 4);
            const uint64_t bh = dP + (uint64_t)((b * Gm::kPBytes) >> 4);
            const uint64_t bl = bh + (uint64_t)((NP * 128) >> 4);
#pragma unroll
            for (int kk = 0; kk < kRows / 32; ++kk) {
              const uint64_t a = av + (uint64_t)((kk * 4096) >> 4);
              // stream b's accumulator; its first tile of the unit (j < 2) starts it
              mma_f8_fill_a(tmem_o + NP * b, a, bh + 2 * kk, idPV, (j >= 2 || kk > 0) ? 1u : 0u);
              mma_f8_reuse_a(tmem_o + NP * b, a, bl + 2 * kk, idPV, 1u);
            }
            mma_commit(smem_u32(&bar_empty[s]));
          }
          __syncwarp();
        }
      }
    }
    if (elect_one()) mma_commit(smem_u32(&bar_drain_pv));
    __syncwarp();
    mbar_wait(smem_u32(&bar_drain_pv), 0, 1000000000ull, &zero_flag);
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    // Two streams: warps 0-3 take the unit's tiles with even g, warps 4-7 those
    // with odd g.  Each stream has its own S^T buffer, P buffer, O^T
    // accumulator and running max and sum, so one stream's score loads (slow
    // while products run) overlap the other's exponentials; a unit's epilogue
    // merges the two streams' (O, max, sum) exactly.
    const int st = warp >> 2;           // stream: tiles g with g % 2 == st
    const int quarter = warp & 3;       // TMEM lane quarter: tile rows [32 quarter, +32)
    const int t = quarter * 32 + lane;  // tile row = TMEM lane; in the epilogue a dim row of O^T
    const int tid = threadIdx.x;        // 0 .. kSoftmax - 1
    const int sid = tid & 127;          // thread within the stream
    const int bar_st = 1 + st;          // the stream's named barrier (128 threads)
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t o_addr = lane_addr + 4 * NP + NP * st;  // this stream's O^T
    auto pv_done = [&](int gg) {  // the P.V of tile gg has completed
      return __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_empty[gg % kSlots]), (gg / kSlots) & 1,
                                               p.wait_ns, &abort_flag));
    };
    bool ok = true;
    int g = 0, nu = 0;
    for (int wi = w0; wi < w1 && ok; ++wi) {
      const Item it = read_item(p, wi);
      if (it.ntiles == 0) {  // empty shard: O = 0, LSE = -inf
        float* out_o = out_rows(p, it);
        float* out_l = out_lse(p, it);
        for (int i = tid; i < p.Hc * kD; i += kSoftmax) out_o[i] = 0.f;
        for (int i = tid; i < p.Hc; i += kSoftmax) out_l[i] = -INFINITY;
        continue;
      }
      // token of tile row t of tile j: tok_t + j tok_j; a cache row is masked
      // for the columns of query rows below tok - lim
      const int tok_j = kRows * it.pd.tok_step;
      const int tok_t = it.pd.tok0 + (it.row_begin + t) * it.pd.tok_step;
      const int lim = it.pd.ctx_len - p.s_q;
      const float* srow = p.sc.p[it.r] + it.row0;  // the item's per-row scales
      for (int kh = 0; kh < p.Hkv && ok; ++kh, ++nu) {
        const int g0 = g;  // the unit's first tile
        // ---- the unit's [Q_hi | Q_lo]: x = q 2^eq with max |x| in [128, 256).
        // Every product of the previous unit has completed (its epilogue
        // waited for both streams' last P.V), so the operand can be overwritten.
        constexpr int kPieces = kD / 8;  // 16-byte pieces per query column
        constexpr int kPer = NP * kPieces / kSoftmax;
        uint4 qv[kPer];
        uint32_t qmax = 0;  // largest |q| as bf16 magnitude bits
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int i = tid + k * kSoftmax, n = i / kPieces, d0 = (i % kPieces) * 8;
          qv[k] = make_uint4(0, 0, 0, 0);
          if (n < ncols) {
            const int qi = n / p.G, hh = kh * p.G + n % p.G;
            qv[k] = __ldg(reinterpret_cast<const uint4*>(
                p.q + (((long long)it.b * p.s_q + qi) * p.Hq + hh) * kD + d0));
          }
          const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) qmax = max(qmax, max(w[e] & 0x7FFFu, (w[e] >> 16) & 0x7FFFu));
        }
        qmax = __reduce_max_sync(0xffffffffu, qmax);
        if (lane == 0) sQmax[warp] = qmax;
        if (sid < NP) sM[st][sid] = 0.f;  // each stream's running max restarts with the unit
        named_bar_sync(3, kSoftmax);
#pragma unroll
        for (int w = 0; w < kSoftmaxWarps; ++w) qmax = max(qmax, sQmax[w]);
        const int eq = scale_exponent(__uint_as_float(qmax << 16), 8, 0);
        const float qs = pow2i(eq);
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int i = tid + k * kSoftmax, n = i / kPieces, d0 = (i % kPieces) * 8;
          if (n < ncols) {
            const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
            uint32_t hs[4], ls[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              split_e4m3x2(__uint_as_float(w[e] << 16) * qs, __uint_as_float(w[e] & 0xFFFF0000u) * qs, hs[e],
                           ls[e]);
            *reinterpret_cast<uint2*>(sQ + sw128(n, d0)) = make_uint2(hs[0] | (hs[1] << 16), hs[2] | (hs[3] << 16));
            *reinterpret_cast<uint2*>(sQ + sw128(NP + n, d0)) =
                make_uint2(ls[0] | (ls[1] << 16), ls[2] | (ls[3] << 16));
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&bar_q));
        named_bar_sync(3, kSoftmax);  // sQmax read before its next write

        // ---- this stream's tiles of the unit
        const float cq = p.scale_log2 * pow2i(-eq);
        int gs = 0;  // weights carry scale_row 2^gs (set on the stream's first tile, only decreases)
        float l[NP];
#pragma unroll
        for (int n = 0; n < NP; ++n) l[n] = 0.f;
        const int j0 = (st ^ g0) & 1;  // the stream's first tile in the unit
        bool failed = false;
        for (int j = j0; j < it.ntiles; j += 2) {
          const int gg = g0 + j, b = st;
          const bool first = j < 2;
          const bool valid = j * kRows + t < it.nrows;
          const float rs = valid ? __ldg(srow + j * kRows + t) : 0.f;
          // several query rows (s_q > 1): row qi reads tokens up to L - s_q + qi,
          // so this cache row is masked for columns n = qi G + i with qi < tok - lim
          const int mcols = min(NP, max(0, tok_t + j * tok_j - lim) * p.G);
          // The stream's warps leave together: one that gave up meets the others at this vote.
          const bool got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_s[b]), (gg >> 1) & 1, p.wait_ns,
                                                             &abort_flag));
          if (bar_red_or(bar_st, 128, !got)) {
            if (!got) report_timeout(p.status, 5, &abort_flag);
            failed = true;
            break;
          }
          tc_fence_after();
          // u = score - running max (log2 units); masked rows and columns read nothing
          const float c = rs * cq;
          float u[NP];
          float over = -INFINITY;
#pragma unroll
          for (int h0 = 0; h0 < NP; h0 += 16) {  // 16 columns at a time keeps registers low
            uint32_t a[16], z[16];
            tmem_ld16(lane_addr + 2 * NP * b + h0, a);
            tmem_ld16(lane_addr + 2 * NP * b + NP + h0, z);
            tmem_ld_wait();
#pragma unroll
            for (int n = 0; n < 16; ++n) {
              const int col = h0 + n;
              u[col] = valid && col >= mcols && col < ncols
                           ? fmaf(__uint_as_float(a[n]) + __uint_as_float(z[n]), c, -sM[st][col])
                           : -INFINITY;
              over = fmaxf(over, u[col]);
            }
          }
          // the scores are in registers: the QK^T issuer may refill this S^T buffer
          tc_fence_before();
          mbar_arrive(smem_u32(&bar_sfree[b]));
          // Stream-wide vote: the stream's first tile, a score past its running max by
          // more than 2^3, or a token scale that would take a weight to 2^8 or more.
          const bool big = valid && rs * pow2i(gs) >= (float)(1 << kWeightTop);
          if (bar_red_or(bar_st, 128, first || over > kRescaleLog2 || big)) {
#pragma unroll
            for (int n = 0; n < NP; ++n) {
              const int m = __reduce_max_sync(0xffffffffu, ordered(u[n]));
              if (lane == 0) sRed[st][quarter][n] = m;
            }
            const uint32_t smx = __reduce_max_sync(0xffffffffu, __float_as_uint(rs));
            if (lane == 0) sRed1[st][quarter] = smx;
            named_bar_sync(bar_st, 128);
            const float smax = __uint_as_float(max(max(sRed1[st][0], sRed1[st][1]), max(sRed1[st][2], sRed1[st][3])));
            const int gs_new = first ? scale_exponent(smax, kWeightTop, 0)
                                     : min(gs, scale_exponent(smax, kWeightTop, gs));
            if (sid < NP) {
              const float cm = fmaxf(fmaxf(unordered(sRed[st][0][sid]), unordered(sRed[st][1][sid])),
                                     fmaxf(unordered(sRed[st][2][sid]), unordered(sRed[st][3][sid])));
              // the first tile sets the max; later it moves when it grew by more
              // than 2^3 (a column with no unmasked row in the stream's first tile
              // has none later: rows go up in token order; it keeps max 0, weight 0)
              const float delta = first ? (cm == -INFINITY ? 0.f : cm) : (cm > kRescaleLog2 ? cm : 0.f);
              sDelta[st][sid] = delta;
              sM[st][sid] += delta;
            }
            named_bar_sync(bar_st, 128);
            const float gf = pow2i(max(gs_new - gs, -126));
#pragma unroll
            for (int n = 0; n < NP; ++n) {
              const float dl = sDelta[st][n];
              u[n] -= dl;
              l[n] *= ex2(-dl);
            }
            if (!first) {
              // O^T holds the stream's earlier tiles: once its last P.V has landed, scale its columns
              const bool landed = pv_done(gg - 2);
              if (bar_red_or(bar_st, 128, !landed)) {
                if (!landed) report_timeout(p.status, 6, &abort_flag);
                failed = true;
                break;
              }
              tc_fence_after();
#pragma unroll
              for (int h0 = 0; h0 < NP; h0 += 16) {
                uint32_t o[16];
                tmem_ld16(o_addr + h0, o);
                tmem_ld_wait();
#pragma unroll
                for (int n = 0; n < 16; ++n)
                  o[n] = __float_as_uint(__uint_as_float(o[n]) * (ex2(-sDelta[st][h0 + n]) * gf));
                tmem_st16(o_addr + h0, o);
              }
              tmem_st_wait();
            }
            gs = gs_new;
            named_bar_sync(bar_st, 128);  // sRed, sRed1 and sDelta read before their next writes
          }
          // P row t: p = 2^u, weight x = p scale_row 2^gs as E4M3 hi + lo
          const float gr = rs * pow2i(gs);
          uint32_t hw[NP / 2], lw[NP / 2];
#pragma unroll
          for (int k = 0; k < NP / 2; ++k) {
            const float p0 = ex2(u[2 * k]), p1 = ex2(u[2 * k + 1]);
            l[2 * k] += p0;
            l[2 * k + 1] += p1;
            split_e4m3x2(p0 * gr, p1 * gr, hw[k], lw[k]);
          }
          // P buffer b was read by the P.V of the stream's previous tile
          if (!first) {
            const bool freed = pv_done(gg - 2);
            if (bar_red_or(bar_st, 128, !freed)) {
              if (!freed) report_timeout(p.status, 7, &abort_flag);
              failed = true;
              break;
            }
          }
          // K-major: row n of P_hi / P_lo holds column n's weights; this thread's KV row is byte t
          uint8_t* ph = sP + b * Gm::kPBytes;
#pragma unroll
          for (int k = 0; k < NP / 2; ++k) {
            ph[sw128(2 * k, t)] = (uint8_t)(hw[k] & 0xFF);
            ph[sw128(2 * k + 1, t)] = (uint8_t)(hw[k] >> 8);
            ph[NP * 128 + sw128(2 * k, t)] = (uint8_t)(lw[k] & 0xFF);
            ph[NP * 128 + sw128(2 * k + 1, t)] = (uint8_t)(lw[k] >> 8);
          }
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(smem_u32(&bar_p[b]));
        }
        g = g0 + it.ntiles;
        // ---- epilogue of the unit: both streams' column maxima and sums, the
        // two O^T accumulators scaled to the common max, / sum, LSE
#pragma unroll
        for (int n = 0; n < NP; ++n) {
          float v = l[n];
#pragma unroll
          for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
          if (lane == 0) sRed[st][quarter][n] = __float_as_int(v);
        }
        if (sid == 0) sGs[st] = gs;
        // both streams' last P.V have landed (the stream that gave up skips the wait)
        const bool aborted = __any_sync(0xffffffffu, abort_flag != 0);
        const bool landed = failed || aborted || ((it.ntiles < 2 || pv_done(g - 2)) && pv_done(g - 1));
        if (bar_red_or(3, kSoftmax, failed || !landed || aborted)) {
          if (!landed) report_timeout(p.status, 8, &abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        if (tid < NP) {
          const float l0 = __int_as_float(sRed[0][0][tid]) + __int_as_float(sRed[0][1][tid]) +
                           __int_as_float(sRed[0][2][tid]) + __int_as_float(sRed[0][3][tid]);
          const float l1 = __int_as_float(sRed[1][0][tid]) + __int_as_float(sRed[1][1][tid]) +
                           __int_as_float(sRed[1][2][tid]) + __int_as_float(sRed[1][3][tid]);
          // a stream with no weight in the column (or no tile in the unit) adds nothing
          const float m0 = l0 > 0.f ? sM[0][tid] : -INFINITY, m1 = l1 > 0.f ? sM[1][tid] : -INFINITY;
          const float m = fmaxf(m0, m1);
          const float c0 = l0 > 0.f ? ex2(m0 - m) : 0.f, c1 = l1 > 0.f ? ex2(m1 - m) : 0.f;
          const float tot = l0 * c0 + l1 * c1;
          const float inv = tot > 0.f ? 1.f / tot : 0.f;
          sCoef[0][tid] = c0 * inv * pow2i(-sGs[0]);
          sCoef[1][tid] = c1 * inv * pow2i(-sGs[1]);
          if (tid < ncols) out_lse(p, it)[sCol[tid] + kh * p.G] = tot > 0.f ? (m + lg2(tot)) * kLn2 : -INFINITY;
        }
        named_bar_sync(3, kSoftmax);
        {
          // warp (st, quarter): dim rows of the quarter, columns [st NP / 2, st NP / 2 + NP / 2)
          constexpr int NC = NP / 2;
          const int cb = st * NC;
          uint32_t o0[NC], o1[NC];
          if constexpr (NC == 8) {
            tmem_ld8(lane_addr + 4 * NP + cb, o0);
            tmem_ld8(lane_addr + 5 * NP + cb, o1);
          } else {
            tmem_ld16(lane_addr + 4 * NP + cb, o0);
            tmem_ld16(lane_addr + 5 * NP + cb, o1);
          }
          tmem_ld_wait();
          float* out_o = out_rows(p, it);
#pragma unroll
          for (int n = 0; n < NC; ++n) {
            const int col = cb + n;
            if (col < ncols) {
              // a stream without weight in the column may hold an earlier unit's values: select, not scale
              const float c0 = sCoef[0][col], c1 = sCoef[1][col];
              const float v = (c0 != 0.f ? __uint_as_float(o0[n]) * c0 : 0.f) +
                              (c1 != 0.f ? __uint_as_float(o1[n]) * c1 : 0.f);
              out_o[(long long)(sCol[col] + kh * p.G) * kD + t] = v;
            }
          }
        }
        tc_fence_before();
        // the softmax warps decide together whether to go on; shared state is
        // free for the next unit
        if (bar_red_or(3, kSoftmax, abort_flag != 0)) ok = false;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpPv) tmem_dealloc(tmem, kTmemCols);
}

template <int NP>
cudaError_t launch_np(const CodeMaps& maps, const Params& p, int grid, cudaStream_t s) {
  auto kern = decode_gqa_f8_kernel<NP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Geo<NP>::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, Geo<NP>::kSmem, s>>>(maps, p);
  return cudaGetLastError();
}

}  // namespace

bool gqa_f8_supported(int Hq, int Hkv, int Dqk, int Dv, int s_q, bool paged) {
  return !paged && Dqk == kD && Dv == kD && Hkv >= 1 && Hq % Hkv == 0 && (Hq / Hkv) * s_q <= 32;
}

cudaError_t launch_decode_gqa_f8(const int32_t* dev_plan, const cp_plan_header& h, const void* q,
                                 const ShardPtrs& k, const ShardPtrs& v, const ScalePtrs& sc,
                                 const long long* shard_rows, int Hq, int Hkv, float sm_scale, float* o_part,
                                 float* lse_part, float* ws_o, float* ws_lse, const int32_t* pair_count,
                                 unsigned long long wait_ns, cudaStream_t s) {
  Params p;
  p.plan = dev_plan;
  p.B = h.R;
  p.off_pair = h.off_rank;
  p.off_worker = h.off_req;
  p.off_work = h.off_seg;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.s_q = plan_s_q(h);
  p.Hc = Hq * p.s_q;
  p.scale_log2 = sm_scale * kLog2e;
  p.sc = sc;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.ws_o = ws_o;
  p.ws_lse = ws_lse;
  p.pair_count = pair_count;
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevice;
  p.wait_ns = wait_ns;
  CodeMaps maps;
  memset(&maps, 0, sizeof(maps));
  const uint64_t strides[2] = {(uint64_t)kD, (uint64_t)Hkv * kD};
  for (int r = 0; r < h.C; ++r) {
    if (shard_rows[r] == 0) continue;
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)Hkv, (uint64_t)shard_rows[r]};
    const uint32_t box[3] = {(uint32_t)kD, 1, (uint32_t)kRows};
    if (!encode_tensor_map_u8_3d(&maps.k[r], k.p[r], dims, strides, box) ||
        !encode_tensor_map_u8_3d(&maps.v[r], v.p[r], dims, strides, box))
      return cudaErrorInvalidValue;
  }
  return p.G * p.s_q <= 16 ? launch_np<16>(maps, p, h.n_tiles, s) : launch_np<32>(maps, p, h.n_tiles, s);
}

}  // namespace cpattn
