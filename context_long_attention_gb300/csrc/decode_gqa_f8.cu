// GQA split-KV decode over an FP8-E4M3 cache (head dim 128) on the tcgen05
// tensor cores.
//
// The same computation as the bf16 GQA kernel ("How GPUs Share a Long
// Context During LLM Inference" §3.1-3.4): per work item (a row range of one
// (shard, request) pair) and kv head g, a partial O and the natural-log LSE of
// the G = Hq/Hkv query heads of g over the item's rows, merged later exactly
// (§3.3).  The cache holds E4M3 codes with one fp32 scale per token for both
// its K and V rows (k = code x scale, v = code x scale).
//
// Every E4M3 value is exactly an f16 value, so the codes are expanded to f16
// in shared memory by six converter warps and the products run as kind::f16
// with f16 operands:
//   S^T [128 rows x NP]  = K_codes_g [128 x 128] . (Q_g 2^e)^T, scaled per row
//                           by scale_row 2^-e in the softmax,
//   O^T [128 dims x NP] += V_codes_g^T . (P scale_row)^T,
// the running sum counting the unscaled weights, so O = sum p v / sum p.
// The query of a unit (request, kv head) is scaled by a power of two 2^e that
// puts its largest magnitude in [2^13, 2^14), so its bf16 values are exact in
// f16.
//
// Warp roles (384 threads): warps 0-3 softmax (thread = KV row of the tile =
// TMEM lane; in the epilogue a dim row of O^T), warp 4 TMA (codes into two
// staging slots), warp 5 MMA issue (one elected lane, the loop run
// warp-wide), warps 6-11 expand the codes into two f16 stages and convert
// each unit's query; two S^T buffers in TMEM.
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
constexpr int kSlotBytes = 2 * kCodeBytes;  // a staging slot: K and V codes, 32 KB
constexpr int kChunkBytes = kRows * 128;    // 64 dims of an f16 tile: 16 KB
constexpr int kTileBytes = 2 * kChunkBytes; // f16 K or V tile: 32 KB
constexpr int kStageBytes = 2 * kTileBytes; // f16 K and V: 64 KB
constexpr int kSlots = 2, kStages = 2;
constexpr int kThreads = 384;
constexpr int kSoftmax = 128;
constexpr int kConvWarps = 6;
constexpr int kConv = kConvWarps * 32;  // converter threads (warps 6-11: three SM sub-partitions hold
                                        // three warps, the register cap of 168 a thread either way)
constexpr int kWarpTma = 4, kWarpMma = 5, kWarpConv0 = 6;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

template <int NP>
constexpr int smem_bytes() {
  return kSlots * kSlotBytes + kStages * kStageBytes + NP * 256 /* Q */ + NP * 256 /* P */ + 1024;
}

struct Params {
  const int32_t* plan;
  int B, off_pair, off_worker, off_work;
  int Hq, Hkv, G;    // query heads, kv heads, query heads per kv head
  int s_q;           // query rows per request
  int Hc;            // output columns per request: s_q x Hq
  float scale_log2;  // sm_scale * log2(e)
  ScalePtrs sc;      // per-row scales of each shard
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
__device__ __forceinline__ void report_timeout(unsigned* status, unsigned site, volatile int* abort) {
  *abort = 1;
  if (atomicCAS(status, 0u, 1u) == 0u) {
    status[1] = kKernDecodeGqaF8;
    status[2] = site;
    status[3] = blockIdx.x;
    __threadfence();
  }
}
// Two E4M3 codes of a word (bytes `lo` and `lo + 1`) to f16x2 holding the
// codes' values x 2^-8, exactly: an E4M3 code's sign, 4 exponent bits and 3
// mantissa bits, moved to the f16 sign, the low 4 exponent bits and the top 3
// mantissa bits, read as f16 with bias 15 instead of 7, give its value x 2^-8,
// subnormals included (both formats scale their subnormals the same way).
// Integer ALU work only: the 16-bit conversion instructions, issued at this
// rate, slow the tensor pipe.  Codes must be finite (0x7F, 0xFF are NaN).
template <int lo>
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_scaled(uint32_t word) {
  const uint32_t t = __byte_perm(word, 0u, lo == 0 ? 0x1404u : 0x3424u);  // codes into bytes 1 and 3
  return (t & 0x80008000u) | ((t >> 1) & 0x3F803F80u);
}
// Two E4M3 codes of a word (bytes `lo` and `lo + 1`) to f16x2 by the hardware
// conversion: the codes' values exactly.  Fewer instructions than the integer
// form, and the converter warps are issue-bound, so this is the one used.
template <int lo>
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_hw(uint32_t word) {
  uint32_t r;
  const uint32_t two = lo == 0 ? (word & 0xFFFFu) : (word >> 16);
  asm("{\n .reg .b16 c;\n cvt.u16.u32 c, %1;\n cvt.rn.f16x2.e4m3x2 %0, c;\n}" : "=r"(r) : "r"(two));
  return r;
}
constexpr float kCodeScale = 1.f;  // the f16 tiles hold the codes' values x 1 / kCodeScale

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

template <int NP>
__device__ __forceinline__ void tmem_ld_cols(uint32_t addr, uint32_t (&a)[NP]) {
  if constexpr (NP == 16) {
    tmem_ld16(addr, a);
  } else {
    tmem_ld32(addr, a);
  }
}
template <int NP>
__device__ __forceinline__ void tmem_st_cols(uint32_t addr, uint32_t (&a)[NP]) {
#pragma unroll
  for (int c = 0; c < NP / 16; ++c) tmem_st16(addr + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&a[16 * c]));
}

// A unit (work item, kv head) covers the item's tiles; g counts tiles over
// all units of this CTA in the order every role walks them; each barrier
// completes once per tile (per slot or stage use; bar_s[b] once per two
// tiles; bar_q and bar_qf once per unit), so the parity to wait for follows
// from g.
template <int NP>
__global__ void __launch_bounds__(kThreads, 1)
    decode_gqa_f8_kernel(const __grid_constant__ CodeMaps maps, const __grid_constant__ CUtensorMap qmap,
                         const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sSlot = smem;                            // [slot][K codes 16 KB | V codes 16 KB]
  uint8_t* sStage = smem + kSlots * kSlotBytes;     // [stage][K f16: 2 chunks | V f16: 2 chunks]
  uint8_t* sQ = sStage + kStages * kStageBytes;     // [2 chunks][NP rows x 128 B]: the unit's query
  uint8_t* sP = sQ + NP * 256;                      // [2 chunks of 64 rows][NP rows x 128 B]
  // code[s]: slot s holds its tile's codes; codefree[s]: the converters read them.
  // full[s]: f16 stage s holds its tile; empty[s]: the tile's products read it.
  // s[b]: S^T buffer b holds the scores; p: the four softmax warps wrote P;
  // pv: the tile's P.V has completed; q: the unit's bf16 query landed in sQ;
  // qf: the converters rewrote it as f16 (x 2^e), for the issuer; qe[u % 4]:
  // unit u's exponent is in sQe[u % 4], for the softmax, which may be two
  // units behind the converters (a unit's query load waits for the P.V of the
  // tile two before it, which waits for that tile's softmax), so one barrier
  // for it would let its phase run two ahead of the wait.
  __shared__ __align__(8) uint64_t bar_code[kSlots], bar_codefree[kSlots], bar_fullK[kStages], bar_fullV[kStages],
      bar_empty[kStages], bar_s[2], bar_p, bar_pv, bar_q, bar_qf, bar_qe[4], bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ volatile int zero_flag;
  __shared__ float sM[NP];      // running max per column (log2 units)
  __shared__ float sAlpha[NP];  // rescale of a moved max; in the epilogue 1 / column sum
  __shared__ float sDelta[NP];
  __shared__ int sRed[4][NP];   // cross-warp column maxima
  __shared__ float sL[4][NP];   // cross-warp column sums
  __shared__ int sCol[NP];      // output column of unit column n for kv head 0
  __shared__ uint32_t sQmax[kConvWarps];  // the converter warps' largest |q| (bf16 magnitude bits)
  __shared__ int sQe[4];        // unit u's query exponent e, at u % 4

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(smem_u32(&bar_code[s]), 1);
      mbar_init(smem_u32(&bar_codefree[s]), kConv);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bar_fullK[s]), kConv);
      mbar_init(smem_u32(&bar_fullV[s]), kConv);
      mbar_init(smem_u32(&bar_empty[s]), 1);
    }
    mbar_init(smem_u32(&bar_s[0]), 1);
    mbar_init(smem_u32(&bar_s[1]), 1);
    mbar_init(smem_u32(&bar_p), 4);
    mbar_init(smem_u32(&bar_pv), 1);
    mbar_init(smem_u32(&bar_q), 1);
    mbar_init(smem_u32(&bar_qf), kConv);
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bar_qe[i]), kConv);
    mbar_init(smem_u32(&bar_drain), 1);
    abort_flag = 0;
    zero_flag = 0;
    mbar_init_fence();
  }
  if (threadIdx.x < NP) sCol[threadIdx.x] = (threadIdx.x / p.G) * p.Hq + threadIdx.x % p.G;
  // rows of the query operand past the unit's G s_q columns stay zero
  for (int i = threadIdx.x; i < NP * 256 / 16; i += kThreads) reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == kWarpMma) tmem_alloc(smem_u32(&tmem_slot), 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // TMEM: S^T buffer b: cols [NP b, NP b + NP); O^T: [2 NP, 3 NP)
  const uint32_t tmem = tmem_slot;
  const int w0 = p.plan[p.off_worker + blockIdx.x], w1 = p.plan[p.off_worker + blockIdx.x + 1];
  const int ncols = p.G * p.s_q;  // columns of a unit in use

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA: codes into the slots
    bool ok = true;
    int g = 0;
    int last[kSlots] = {-1, -1};  // tile of each slot's last fill
    for (int wi = w0; wi < w1 && ok; ++wi) {
      const Item it = read_item(p, wi);
      for (int kh = 0; kh < p.Hkv && it.ntiles > 0 && ok; ++kh) {
        for (int j = 0; j < it.ntiles; ++j, ++g) {
          const int s = g % kSlots, use = g / kSlots;
          if (use > 0 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_codefree[s]), (use - 1) & 1,
                                                            p.wait_ns, &abort_flag))) {
            if (lane == 0) report_timeout(p.status, 1, &abort_flag);
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&bar_code[s]);
          if (elect_one()) {
            mbar_expect_tx(full, kSlotBytes);
            const int y = (int)(it.row0 + (long long)j * kRows);
            tma_load_3d(smem_u32(sSlot + s * kSlotBytes), &maps.k[it.r], 0, kh, y, full);
            tma_load_3d(smem_u32(sSlot + s * kSlotBytes + kCodeBytes), &maps.v[it.r], 0, kh, y, full);
          }
          __syncwarp();
          last[s] = g;
        }
      }
    }
    if (!ok) {
      // never leave with a copy in flight
      for (int s = 0; s < kSlots; ++s)
        if (last[s] >= 0) mbar_wait(smem_u32(&bar_code[s]), (last[s] / kSlots) & 1, 1000000000ull, &zero_flag);
      __syncwarp();
    }
  } else if (warp >= kWarpConv0) {
    // ------------------------------------------------------------ converters (warps 6-11):
    // each unit's query to f16 x 2^e, each tile's codes to f16
    const int ct = threadIdx.x - kWarpConv0 * 32;  // 0 .. kConv - 1
    bool ok = true;
    int g = 0, nu = 0;  // tiles and units so far
    int q_pending = -1; // parity of a query load that may still be in flight
    for (int wi = w0; wi < w1 && ok; ++wi) {
      const Item it = read_item(p, wi);
      for (int kh = 0; kh < p.Hkv && it.ntiles > 0 && ok; ++kh, ++nu) {
        for (int j = 0; j < it.ntiles; ++j, ++g) {
          const int s = g % kSlots, st = g % kStages;
          // f16 stage st is free once the P.V of tile g - 2 has completed; that
          // P.V was issued after the QK^T of tile g - 1, so sQ is free too (for
          // g = 1: the first QK^T's own barrier, whose first phase it is)
          bool got = true;
          if (g >= 2)
            got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_empty[st]), ((g - 2) / kStages) & 1,
                                                    p.wait_ns, &abort_flag));
          else if (g == 1 && j == 0)
            got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_s[0]), 0, p.wait_ns, &abort_flag));
          if (got && j == 0) {
            // ---- the unit's query: bf16 by TMA, then f16 x 2^e in place
            q_pending = nu & 1;
            if (ct == 0) {
              mbar_expect_tx(smem_u32(&bar_q), 2 * ncols * 128);
              for (int c = 0; c < 2; ++c)
                tma_load_4d(smem_u32(sQ + c * NP * 128), &qmap, c * 64, 0, kh, it.b * p.s_q, smem_u32(&bar_q));
            }
            got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_q), nu & 1, p.wait_ns, &abort_flag));
            if (got) {
              q_pending = -1;
              uint32_t mx = 0;  // largest |q| as bf16 magnitude bits
              for (int i = ct; i < 2 * ncols * 8; i += kConv) {
                const int c = i / (ncols * 8), n = (i / 8) % ncols, w = i % 8;
                const uint4 v = *reinterpret_cast<const uint4*>(sQ + c * NP * 128 + n * 128 + w * 16);
                const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) mx = max(mx, max(wd[e] & 0x7FFFu, (wd[e] >> 16) & 0x7FFFu));
              }
              mx = __reduce_max_sync(0xffffffffu, mx);
              if (lane == 0) sQmax[warp - kWarpConv0] = mx;
              named_bar_sync(2, kConv);
              for (int w2 = 0; w2 < kConvWarps; ++w2) mx = max(mx, sQmax[w2]);
              // 2^e puts the largest |q| in [2^13, 2^14); e kept where 2^e and 2^-e are normal
              const int ex = (int)((mx >> 7) & 0xFF) - 127;
              const int e = mx == 0 ? 0 : max(-126, min(126, 13 - ex));
              const float sc = __int_as_float((e + 127) << 23);
              for (int i = ct; i < 2 * ncols * 8; i += kConv) {
                const int c = i / (ncols * 8), n = (i / 8) % ncols, w = i % 8;
                uint4* ptr = reinterpret_cast<uint4*>(sQ + c * NP * 128 + n * 128 + w * 16);
                const uint4 v = *ptr;
                const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
                uint32_t o[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                  const __half2 h = __floats2half2_rn(__uint_as_float(wd[e2] << 16) * sc,
                                                      __uint_as_float(wd[e2] & 0xFFFF0000u) * sc);
                  o[e2] = *reinterpret_cast<const uint32_t*>(&h);
                }
                *ptr = make_uint4(o[0], o[1], o[2], o[3]);
              }
              if (ct == 0) sQe[nu & 3] = e;
              fence_proxy_async_smem();
              mbar_arrive(smem_u32(&bar_qf));
              mbar_arrive(smem_u32(&bar_qe[nu & 3]));
            }
          }
          got = got && __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_code[s]), (g / kSlots) & 1, p.wait_ns,
                                                         &abort_flag));
          if (!got) {
            if (lane == 0) report_timeout(p.status, 2, &abort_flag);
            ok = false;
            break;
          }
          // ---- codes of slot s -> f16 stage st: K, announced on its own so that
          // QK^T and the softmax overlap the conversion of V
          const uint8_t* src = sSlot + s * kSlotBytes;
          uint8_t* dst = sStage + st * kStageBytes;
#pragma unroll 1
          for (int tsr = 0; tsr < 2; ++tsr) {
#pragma unroll 4
            for (int i = ct; i < kRows * 8; i += kConv) {
              const int r = i >> 3, u = i & 7;  // row, 16-code unit
              const uint4 v =
                  *reinterpret_cast<const uint4*>(src + tsr * kCodeBytes + r * 128 + ((u ^ (r & 7)) << 4));
              const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
              uint32_t h[8];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                h[2 * e] = e4m3x2_to_f16x2_hw<0>(wd[e]);
                h[2 * e + 1] = e4m3x2_to_f16x2_hw<2>(wd[e]);
              }
              // dims 16u .. 16u + 15: chunk u / 4, 16-byte units 2 (u % 4) and 2 (u % 4) + 1
              uint8_t* rowp = dst + tsr * kTileBytes + (u >> 2) * kChunkBytes + r * 128;
              const int w0u = 2 * (u & 3);
              *reinterpret_cast<uint4*>(rowp + ((w0u ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
              *reinterpret_cast<uint4*>(rowp + (((w0u + 1) ^ (r & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
            }
            fence_proxy_async_smem();
            if (tsr == 0) mbar_arrive(smem_u32(&bar_fullK[st]));
          }
          mbar_arrive(smem_u32(&bar_codefree[s]));
          mbar_arrive(smem_u32(&bar_fullV[st]));
        }
      }
    }
    if (!ok && q_pending >= 0) {
      // never leave with the query copy in flight
      mbar_wait(smem_u32(&bar_q), q_pending, 1000000000ull, &zero_flag);
      __syncwarp();
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issue: per tile g,
    // S^T(g) first, then P.V of tile g - 1 once its P is written
    const uint32_t idS = idesc_f16_f32(kRows, NP, 0, 0);
    const uint32_t idPV = idesc_f16_f32(kRows, NP, 1, 0);
    const uint32_t st0 = smem_u32(sStage);
    // K tile K-major; V^T MN-major (its two 64-dim chunks kChunkBytes apart); Q and P K-major
    const uint64_t dK = smem_desc(st0, 16, 1024), dV = smem_desc(st0 + kTileBytes, kChunkBytes, 1024);
    const uint64_t dQ = smem_desc(smem_u32(sQ), 16, 1024), dP = smem_desc(smem_u32(sP), 16, 1024);
    bool ok = true;
    int g = 0, nu = 0;
    int prev_j = -1, prev_s = 0;  // tile index in its unit and stage of the tile whose P.V is pending
    auto pv = [&](int gp, int jp, int sp) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_p), gp & 1, p.wait_ns, &abort_flag))) return false;
      // every earlier phase of this stage's V barrier was waited for here
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_fullV[sp]), (gp / kStages) & 1, p.wait_ns,
                                             &abort_flag)))
        return false;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t v = dV + ((uint32_t)(sp * kStageBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kRows / 16; ++kk)
          mma_ss(tmem + 2 * NP, v + ((kk * 2048) >> 4), dP + (((kk >> 2) * NP * 128 + (kk & 3) * 32) >> 4), idPV,
                 (jp > 0 || kk > 0) ? 1u : 0u);
        mma_commit(smem_u32(&bar_empty[sp]));
        mma_commit(smem_u32(&bar_pv));
      }
      __syncwarp();
      return true;
    };
    for (int wi = w0; wi < w1 && ok; ++wi) {
      const Item it = read_item(p, wi);
      for (int kh = 0; kh < p.Hkv && it.ntiles > 0 && ok; ++kh, ++nu) {
        for (int j = 0; j < it.ntiles; ++j, ++g) {
          const int s = g % kStages;
          bool got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_fullK[s]), (g / kStages) & 1, p.wait_ns,
                                                       &abort_flag));
          if (got && j == 0)
            got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_qf), nu & 1, p.wait_ns, &abort_flag));
          if (!got) {
            if (lane == 0) report_timeout(p.status, 3, &abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          // S^T buffer g & 1 was last read by the softmax of tile g - 2, whose P
          // the P.V of tile g - 2 waited for
          if (elect_one()) {
            const uint64_t k = dK + ((uint32_t)(s * kStageBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
              const uint32_t qoff = (kk >> 2) * NP * 128 + (kk & 3) * 32;
              mma_ss(tmem + NP * (g & 1), k + (off >> 4), dQ + (qoff >> 4), idS, kk > 0);
            }
            mma_commit(smem_u32(&bar_s[g & 1]));
          }
          __syncwarp();
          if (prev_j >= 0 && !pv(g - 1, prev_j, prev_s)) {
            if (lane == 0) report_timeout(p.status, 4, &abort_flag);
            ok = false;
            break;
          }
          prev_j = j;
          prev_s = s;
        }
      }
    }
    if (ok && prev_j >= 0 && !pv(g - 1, prev_j, prev_s)) {
      if (lane == 0) report_timeout(p.status, 4, &abort_flag);
    }
    // never free TMEM under a running MMA
    if (elect_one()) mma_commit(smem_u32(&bar_drain));
    __syncwarp();
    mbar_wait(smem_u32(&bar_drain), 0, 1000000000ull, &zero_flag);
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax (warps 0-3)
    const int t = threadIdx.x;  // tile row = TMEM lane; in the epilogue a dim row of O^T
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    // P row n is K-major: KV row t sits in chunk t / 64, 16-byte unit (t % 64) / 8
    // (swizzled with n % 8), halfword t % 8
    uint8_t* prow = sP + (t >> 6) * NP * 128 + (t & 7) * 2;
    const int punit = (t & 63) >> 3;
    bool ok = true;
    int g = 0, nu = 0;
    for (int wi = w0; wi < w1 && ok; ++wi) {
      const Item it = read_item(p, wi);
      if (it.ntiles == 0) {  // empty shard: O = 0, LSE = -inf
        float* out_o = out_rows(p, it);
        float* out_l = out_lse(p, it);
        for (int i = t; i < p.Hc * kD; i += kSoftmax) out_o[i] = 0.f;
        for (int i = t; i < p.Hc; i += kSoftmax) out_l[i] = -INFINITY;
        continue;
      }
      // token of tile row t of tile j: tok_t + j * tok_j; a cache row is masked
      // for the columns of query rows below tok - lim
      const int tok_j = kRows * it.pd.tok_step;
      const int tok_t = it.pd.tok0 + (it.row_begin + t) * it.pd.tok_step;
      const int lim = it.pd.ctx_len - p.s_q;
      const float* srow = p.sc.p[it.r] + it.row0;  // the item's per-row scales
      for (int kh = 0; kh < p.Hkv && ok; ++kh, ++nu) {
        // the unit's query exponent: scores in log2 units are S x scale_row x 2^-e x scale_log2
        const bool qok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_qe[nu & 3]), (nu >> 2) & 1, p.wait_ns,
                                                           &abort_flag));
        if (bar_red_or(1, kSoftmax, !qok)) {
          if (!qok) report_timeout(p.status, 8, &abort_flag);
          ok = false;
          break;
        }
        const float cj = p.scale_log2 * kCodeScale * __int_as_float((127 - sQe[nu & 3]) << 23);
        // the running max restarts from the unit's first tile; every read of the
        // previous unit's maxima came before its epilogue's barriers
        if (t < NP) sM[t] = 0.f;
        named_bar_sync(1, kSoftmax);
        float l[NP];
#pragma unroll
        for (int n = 0; n < NP; ++n) l[n] = 0.f;
        for (int j = 0; j < it.ntiles; ++j, ++g) {
          const bool valid = j * kRows + t < it.nrows;
          const float rs = valid ? __ldg(srow + j * kRows + t) : 0.f;
          // several query rows (s_q > 1): row qi reads tokens up to L - s_q + qi,
          // so this cache row is masked for columns n = qi G + i with qi < tok - lim
          const int mcols = min(NP, max(0, tok_t + j * tok_j - lim) * p.G);
          const bool got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_s[g & 1]), (g >> 1) & 1, p.wait_ns,
                                                             &abort_flag));
          if (bar_red_or(1, kSoftmax, !got)) {
            if (!got) report_timeout(p.status, 5, &abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          // u = score - running max (log2 units); masked rows and columns read nothing
          float u[NP];
          float over = -INFINITY;
          {
            uint32_t a[NP];
            tmem_ld_cols<NP>(lane_addr + NP * (g & 1), a);
            tmem_ld_wait();
#pragma unroll
            for (int n = 0; n < NP; ++n) {
              u[n] = valid && n >= mcols ? fmaf(__uint_as_float(a[n]), cj * rs, -sM[n]) : -INFINITY;
              over = fmaxf(over, u[n]);
            }
          }
          // the previous tile's P.V has completed: P is free and O^T holds it
          const bool freed = g == 0 || __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_pv), (g - 1) & 1,
                                                                          p.wait_ns, &abort_flag));
          if (bar_red_or(1, kSoftmax, !freed)) {
            if (!freed) report_timeout(p.status, 7, &abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          // block-wide vote: does any score pass its running max by more than 2^8?
          if (bar_red_or(1, kSoftmax, j == 0 || over > kRescaleLog2)) {
#pragma unroll
            for (int n = 0; n < NP; ++n) {
              const int m = __reduce_max_sync(0xffffffffu, ordered(u[n]));
              if (lane == 0) sRed[warp][n] = m;
            }
            named_bar_sync(1, kSoftmax);
            if (t < NP) {
              const float cm = fmaxf(fmaxf(unordered(sRed[0][t]), unordered(sRed[1][t])),
                                     fmaxf(unordered(sRed[2][t]), unordered(sRed[3][t])));
              // the first tile sets the max; later the max moves when it grew by
              // more than 2^8, earlier sums and O^T shrinking by 2^-delta (a column
              // with no unmasked row in the unit's first tile has none at all:
              // rows go up in token order; it keeps max 0 and weight 0)
              const float delta = j == 0 ? (cm == -INFINITY ? 0.f : cm) : (cm > kRescaleLog2 ? cm : 0.f);
              sAlpha[t] = j == 0 ? 0.f : ex2(-delta);
              sDelta[t] = delta;
              sM[t] += delta;
            }
            named_bar_sync(1, kSoftmax);
#pragma unroll
            for (int n = 0; n < NP; ++n) {
              l[n] *= sAlpha[n];
              u[n] -= sDelta[n];
            }
            if (j > 0) {
              uint32_t o[NP];
              tmem_ld_cols<NP>(lane_addr + 2 * NP, o);
              tmem_ld_wait();
#pragma unroll
              for (int n = 0; n < NP; ++n) o[n] = __float_as_uint(__uint_as_float(o[n]) * sAlpha[n]);
              tmem_st_cols<NP>(lane_addr + 2 * NP, o);
              tmem_st_wait();
            }
          }
          // P[n][t] = 2^u x scale_row (f16): the value rows' scale; l counts 2^u
#pragma unroll
          for (int n = 0; n < NP; ++n) {
            const float pn = ex2(u[n]);
            l[n] += pn;
            *reinterpret_cast<__half*>(prow + n * 128 + ((punit ^ (n & 7)) << 4)) = __float2half_rn(pn * rs);
          }
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bar_p));
        }
        if (!ok) break;
        // ---- epilogue of the unit: column sums of l, O^T / l, LSE
        const bool landed =
            __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_pv), (g - 1) & 1, p.wait_ns, &abort_flag));
        if (bar_red_or(1, kSoftmax, !landed)) {
          if (!landed) report_timeout(p.status, 6, &abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int n = 0; n < NP; ++n) {
          float v = l[n];
#pragma unroll
          for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
          if (lane == 0) sL[warp][n] = v;
        }
        named_bar_sync(1, kSoftmax);
        // unit column n is output column (n / G) Hq + kh G + n % G
        float* out_o = out_rows(p, it);
        if (t < NP) {
          const float tot = sL[0][t] + sL[1][t] + sL[2][t] + sL[3][t];
          sAlpha[t] = tot > 0.f ? kCodeScale / tot : 0.f;
          if (t < ncols) out_lse(p, it)[sCol[t] + kh * p.G] = tot > 0.f ? (sM[t] + lg2(tot)) * kLn2 : -INFINITY;
        }
        named_bar_sync(1, kSoftmax);
        {
          uint32_t o[NP];
          tmem_ld_cols<NP>(lane_addr + 2 * NP, o);
          tmem_ld_wait();
#pragma unroll
          for (int n = 0; n < NP; ++n)
            if (n < ncols) out_o[(long long)(sCol[n] + kh * p.G) * kD + t] = __uint_as_float(o[n]) * sAlpha[n];
        }
        tc_fence_before();
        // the four softmax warps decide together whether to go on
        if (bar_red_or(1, kSoftmax, abort_flag != 0)) ok = false;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, 128);
}


template <int NP>
cudaError_t launch_np(const CodeMaps& maps, const CUtensorMap& qmap, const Params& p, int grid, cudaStream_t s) {
  auto kern = decode_gqa_f8_kernel<NP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<NP>());
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem_bytes<NP>(), s>>>(maps, qmap, p);
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
  // the bf16 queries [B s_q][Hkv][G][128]: one box per 64-dim chunk holds one
  // kv head's G heads of every query row of a request, rows n = qi G + i
  CUtensorMap qmap;
  {
    const uint64_t dims[4] = {(uint64_t)kD, (uint64_t)p.G, (uint64_t)Hkv, (uint64_t)h.R * p.s_q};
    const uint64_t qstrides[3] = {(uint64_t)kD * 2, (uint64_t)p.G * kD * 2, (uint64_t)Hq * kD * 2};
    const uint32_t box[4] = {64, (uint32_t)p.G, 1, (uint32_t)p.s_q};
    if (!encode_tensor_map_bf16(&qmap, q, 4, dims, qstrides, box)) return cudaErrorInvalidValue;
  }
  return p.G * p.s_q <= 16 ? launch_np<16>(maps, qmap, p, h.n_tiles, s) : launch_np<32>(maps, qmap, p, h.n_tiles, s);
}

}  // namespace cpattn
