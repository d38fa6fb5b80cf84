// GQA split-KV decode over a bf16 cache (head dim 64 or 128) on the tcgen05
// tensor cores.
//
// One decode step of every request against the rows a virtual shard stores
// ("How GPUs Share a Long Context During LLM Inference" §3.1-3.4): query head
// h reads kv head h / (Hq/Hkv) of each of the shard's rows of its request, and
// each work item (a row range of one (shard, request) pair, from the decode
// plan) yields a partial O and the natural-log LSE of every query head over
// those rows, merged later exactly (§3.3).
//
// A unit of work is (work item, kv head g).  The G = Hq/Hkv query heads of g,
// for each of the s_q query rows, form the unit's n = qi G + i columns
// (padded to NP = 16, 32 or 64), and the products are transposed so that the
// MMA M dimension is 128 KV rows:
//   S^T [128 rows x NP]  = K_g tile [128 x D dims] . Q_g^T            (K = D)
//   O^T [128 dims x NP] += V_g tile^T [128 dims x 128 rows] . P^T     (K = 128)
// (at D = 64 the upper 64 dims of V^T are a zero block).
// K_g and V_g tiles come by TMA (a 3-d map over [rows][Hkv][D], one box per
// 64-dim chunk); the request's query, all kv heads, by TMA into one operand
// per kv head (when those do not fit in 64 KB, as with many kv heads of one
// query head each, one kv head's operand, loaded at each unit); P goes
// through shared memory as a K-major operand.
//
// Warp roles (256 threads): warps 0-3 softmax (thread = KV row of the tile =
// TMEM lane; in the epilogue a dim row of O^T), warp 4 TMA, warp 5 MMA issue
// (one elected lane, the loop run warp-wide).  Two or four K/V stages; two S^T
// buffers in TMEM so the issuer runs the next tile's QK^T ahead of this
// tile's P.V.  The running max of a column moves only when a score passes it
// by more than 2^8 (one block-wide vote per tile), which keeps every
// exponential <= 2^8; any running max gives the exact result.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "internal.h"
#include "tc_ptx.cuh"

namespace cpattn {
namespace {
using namespace tc;

constexpr int kRows = 128;                      // KV rows per tile (MMA M)
constexpr int kChunkBytes = kRows * 128;        // 64 dims of a tile: 16 KB
constexpr int kMaxQCols = 256;                  // Hkv x NP, the query operands of all kv heads
constexpr int kThreads = 256;
constexpr int kSoftmax = 128;
constexpr int kWarpTma = 4, kWarpMma = 5;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

// Shared-memory geometry for head dim D (64 or 128): a row is D / 64 chunks of
// 64 dims (128 B, 128-byte swizzle); a stage holds the K and V tiles of one kv
// head (64 KB at D = 128, 32 KB at D = 64, which takes four stages).  At D = 64
// the P.V A operand V^T still spans M = 128: its second 64-dim chunk is a
// zero block.
template <int D>
struct Geo {
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  // at D = 128 a third 64 KB stage takes the room of the query operands of
  // all kv heads: the query slot holds one unit's operand, loaded per unit
  // (at 64 columns the three stages and the kernel's static arrays would pass
  // the 227 KB a block may hold: two stages there)
  template <int NP>
  __host__ __device__ static constexpr int stages() {
    return D == 64 ? 4 : (NP == 64 ? 2 : 3);
  }
  static constexpr bool kQPerUnit = D == 128;
  static constexpr int kQBytes = (kQPerUnit ? 64 : kMaxQCols) * 128 * kChunks;
  static constexpr int kZeroBytes = D == 64 ? kChunkBytes : 0;
  template <int NP>
  static constexpr int smem() {
    return stages<NP>() * kStageBytes + kQBytes + NP * 256 + kZeroBytes + 1024;
  }
};

struct Params {
  const int32_t* plan;
  int B, off_pair, off_worker, off_work;
  RowMap rm;         // paged cache: 64-row boxes of a pool, rows through the page table
  int Hq, Hkv, G;    // query heads, kv heads, query heads per kv head
  int s_q;           // query rows per request
  int Hc;            // output columns per request: s_q x Hq
  int q_per_unit;    // the operands of all kv heads do not fit: sQ holds one, loaded per unit
  float scale_log2;  // sm_scale * log2(e)
  float* o_part;
  float* lse_part;
  float* ws_o;
  float* ws_lse;
  const int32_t* pair_count;  // rows in use per pair (a selection buffer), or nullptr
  unsigned* status;
  unsigned long long wait_ns;
};

// Tensor maps of the shards' K and V caches ([rows, Hkv, D], box 64 dims x
// 1 head x 128 rows, 128-byte swizzle); a paged cache has one map of each pool
// with 64-row boxes.
struct KVMaps {
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
    status[1] = kKernDecodeGqaTc;
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

// Where an item's partial goes: its pair's row of the partials, or, for one
// part of a pair split between CTAs, a workspace row merged afterwards.
__device__ __forceinline__ float* out_rows(const Params& p, const Item& it, int D) {
  return it.part < 0 ? p.o_part + (long long)it.pair * p.Hc * D : p.ws_o + (long long)it.part * p.Hc * D;
}
__device__ __forceinline__ float* out_lse(const Params& p, const Item& it) {
  return it.part < 0 ? p.lse_part + (long long)it.pair * p.Hc : p.ws_lse + (long long)it.part * p.Hc;
}

// tcgen05.ld of NP fp32 columns of this warp's TMEM lanes.
template <int NP>
__device__ __forceinline__ void tmem_ld_cols(uint32_t addr, uint32_t (&a)[NP]) {
  if constexpr (NP == 16) {
    tmem_ld16(addr, a);
  } else if constexpr (NP == 32) {
    tmem_ld32(addr, a);
  } else {
    tmem_ld32(addr, *reinterpret_cast<uint32_t(*)[32]>(&a[0]));
    tmem_ld32(addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&a[32]));
  }
}
template <int NP>
__device__ __forceinline__ void tmem_st_cols(uint32_t addr, uint32_t (&a)[NP]) {
#pragma unroll
  for (int c = 0; c < NP / 16; ++c) tmem_st16(addr + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&a[16 * c]));
}

// A unit (work item, kv head) covers the item's tiles; g counts tiles over
// all units of this CTA in the order every role walks them, and each barrier
// completes once per tile (bar_s[b] once per two, bar_q once per query
// load), so the parity to wait for follows from g.
template <int NP, int D>
__global__ void __launch_bounds__(kThreads, 1)
    decode_gqa_tc_kernel(const __grid_constant__ KVMaps maps, const __grid_constant__ CUtensorMap qmap,
                         const Params p) {
  using Gm = Geo<D>;
  constexpr int kStages = Gm::template stages<NP>(), kStageBytes = Gm::kStageBytes, kTileBytes = Gm::kTileBytes;
  constexpr int kChunks = Gm::kChunks;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sStage = smem;                          // [stage][K: kChunks chunks | V: kChunks chunks]
  uint8_t* sQ = smem + kStages * kStageBytes;      // [Hkv][kChunks][NP rows x 128 B]
  uint8_t* sP = sQ + Gm::kQBytes;                  // [2 chunks of 64 rows][NP rows x 128 B]
  uint8_t* sZero = sP + NP * 256;                  // D = 64: the zero half of V^T
  // full[s]: stage s holds its tile; empty[s]: the tile's products have read it.
  // s[b]: S^T buffer b holds the scores; p: the four softmax warps wrote P;
  // pv: the tile's P.V has completed; q: sQ holds the request's query.
  __shared__ __align__(8) uint64_t bar_full[kStages], bar_empty[kStages], bar_s[2], bar_p, bar_pv, bar_q,
      bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ volatile int zero_flag;
  __shared__ float sM[NP];      // running max per column (log2 units)
  __shared__ float sAlpha[NP];  // rescale of a moved max; in the epilogue 1 / column sum
  __shared__ float sDelta[NP];
  __shared__ int sRed[4][NP];   // cross-warp column maxima
  __shared__ float sL[4][NP];   // cross-warp column sums
  __shared__ int sCol[NP];      // output column of unit column n for kv head 0

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_empty[s]), 1);
    }
    mbar_init(smem_u32(&bar_s[0]), 1);
    mbar_init(smem_u32(&bar_s[1]), 1);
    mbar_init(smem_u32(&bar_p), 4);
    mbar_init(smem_u32(&bar_pv), 1);
    mbar_init(smem_u32(&bar_q), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    abort_flag = 0;
    zero_flag = 0;
    mbar_init_fence();
  }
  if (threadIdx.x < NP) sCol[threadIdx.x] = (threadIdx.x / p.G) * p.Hq + threadIdx.x % p.G;
  // Rows of a kv head's query operand past its G s_q columns stay zero, and so
  // does the zero block.
  for (int i = threadIdx.x; i < Gm::kQBytes / 16; i += kThreads) reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0, 0, 0, 0);
  for (int i = threadIdx.x; i < Gm::kZeroBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(sZero)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == kWarpMma) tmem_alloc(smem_u32(&tmem_slot), 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // TMEM: S^T buffer b: cols [NP b, NP b + NP); O^T: [2 NP, 3 NP)
  const uint32_t tmem = tmem_slot;
  const int w0 = p.plan[p.off_worker + blockIdx.x], w1 = p.plan[p.off_worker + blockIdx.x + 1];
  const int ncols = p.G * p.s_q;  // columns of a unit in use

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA (the warp runs the
    // loop, one elected lane issues the copies)
    bool ok = true;
    int g = 0, q_b = -1, nq = 0;
    int last[kStages];  // tile of each stage's last fill
    for (int s = 0; s < kStages; ++s) last[s] = -1;
    for (int wi = w0; wi < w1 && ok; ++wi) {
      const Item it = read_item(p, wi);
      if (it.ntiles == 0) continue;
      const bool new_q = it.b != q_b;
      q_b = it.b;
      for (int kh = 0; kh < p.Hkv && ok; ++kh) {
        for (int j = 0; j < it.ntiles; ++j, ++g) {
          const int s = g % kStages, use = g / kStages;
          if (use > 0 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_empty[s]), (use - 1) & 1,
                                                            p.wait_ns, &abort_flag))) {
            if (lane == 0) report_timeout(p.status, 1, &abort_flag);
            ok = false;
            break;
          }
          if (j == 0 && (p.q_per_unit || (kh == 0 && new_q))) {
            // the previous tile's QK^T, the last read of sQ, has completed: for
            // g >= 2 the P.V of tile g - 2, issued after it, has (that phase of
            // its stage's barrier follows one this warp has already seen); for
            // g = 1 the first QK^T's own barrier, whose first phase it is
            const bool freed =
                g == 0 ||
                __all_sync(0xffffffffu,
                           g == 1 ? mbar_wait(smem_u32(&bar_s[0]), 0, p.wait_ns, &abort_flag)
                                  : mbar_wait(smem_u32(&bar_empty[(g - 2) % kStages]), ((g - 2) / kStages) & 1,
                                              p.wait_ns, &abort_flag));
            if (!freed) {
              if (lane == 0) report_timeout(p.status, 2, &abort_flag);
              ok = false;
              break;
            }
            if (elect_one()) {
              // every kv head's operand at its slot, or this unit's kv head at slot 0
              const int h0 = p.q_per_unit ? kh : 0, h1 = p.q_per_unit ? kh + 1 : p.Hkv;
              mbar_expect_tx(smem_u32(&bar_q), (h1 - h0) * kChunks * ncols * 128);
              for (int h2 = h0; h2 < h1; ++h2)
                for (int c = 0; c < kChunks; ++c)
                  tma_load_4d(smem_u32(sQ + ((h2 - h0) * kChunks + c) * NP * 128), &qmap, c * 64, 0, h2,
                              it.b * p.s_q, smem_u32(&bar_q));
            }
            __syncwarp();
            ++nq;
          }
          const uint32_t full = smem_u32(&bar_full[s]);
          uint8_t* st = sStage + s * kStageBytes;
          if (elect_one()) {
            mbar_expect_tx(full, kStageBytes);
            if (!p.rm.table) {
              const int y = (int)(it.row0 + (long long)j * kRows);
              for (int c = 0; c < kChunks; ++c) {
                tma_load_3d(smem_u32(st + c * kChunkBytes), &maps.k[it.r], c * 64, kh, y, full);
                tma_load_3d(smem_u32(st + kTileBytes + c * kChunkBytes), &maps.v[it.r], c * 64, kh, y, full);
              }
            } else {
              // the pool rows of the tile's two 64-row halves (each inside one page); past
              // the pair's rows the coordinate is past the pool and the copy reads zeros
              for (int hh = 0; hh < 2; ++hh) {
                const int i0 = it.row_begin + j * kRows + 64 * hh;
                const int y = (int)(i0 < it.pd.rows ? map_row(p.rm, it.pair, 0, i0) : p.rm.pool_rows);
                for (int c = 0; c < kChunks; ++c) {
                  tma_load_3d(smem_u32(st + c * kChunkBytes + hh * 64 * 128), &maps.k[0], c * 64, kh, y, full);
                  tma_load_3d(smem_u32(st + kTileBytes + c * kChunkBytes + hh * 64 * 128), &maps.v[0], c * 64,
                              kh, y, full);
                }
              }
            }
          }
          __syncwarp();
          last[s] = g;
        }
      }
    }
    if (!ok) {
      // never leave with a copy in flight: each stage's last fill and the last query load
      for (int s = 0; s < kStages; ++s)
        if (last[s] >= 0)
          mbar_wait(smem_u32(&bar_full[s]), (last[s] / kStages) & 1, 1000000000ull, &zero_flag);
      if (nq > 0) mbar_wait(smem_u32(&bar_q), (nq - 1) & 1, 1000000000ull, &zero_flag);
      __syncwarp();
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issue: per tile g,
    // S^T(g) first, then P.V of tile g - 1 once its P is written
    const uint32_t idS = idesc_bf16_f32(kRows, NP, 0, 0);
    const uint32_t idPV = idesc_bf16_f32(kRows, NP, 1, 0);
    const uint32_t st0 = smem_u32(sStage), zero = smem_u32(sZero);
    // K tile K-major; V^T MN-major (its two 64-dim chunks along M kChunkBytes
    // apart, or the V chunk and the zero block at D = 64); Q_g and P K-major
    // (64-element chunks NP x 128 B apart)
    const uint64_t dK = smem_desc(st0, 16, 1024);
    const uint64_t dQ = smem_desc(smem_u32(sQ), 16, 1024), dP = smem_desc(smem_u32(sP), 16, 1024);
    bool ok = true;
    int g = 0, q_b = -1, nq = 0;
    int prev_j = -1, prev_s = 0;  // tile index in its unit and stage of the tile whose P.V is pending
    // O^T += V^T P^T for tile gp (the unit's first tile overwrites O^T)
    auto pv = [&](int gp, int jp, int sp) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_p), gp & 1, p.wait_ns, &abort_flag))) return false;
      tc_fence_after();
      if (elect_one()) {
        const uint32_t vaddr = st0 + sp * kStageBytes + kTileBytes;
        const uint64_t v = smem_desc(vaddr, D == 128 ? kChunkBytes : zero - vaddr, 1024);
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
      if (it.ntiles == 0) continue;
      const bool new_q = it.b != q_b;
      q_b = it.b;
      for (int kh = 0; kh < p.Hkv && ok; ++kh) {
        for (int j = 0; j < it.ntiles; ++j, ++g) {
          const int s = g % kStages, use = g / kStages;
          bool got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_full[s]), use & 1, p.wait_ns, &abort_flag));
          if (got && j == 0 && (p.q_per_unit || (kh == 0 && new_q))) {
            got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_q), nq & 1, p.wait_ns, &abort_flag));
            ++nq;
          }
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
            const uint64_t qd = dQ + ((uint32_t)((p.q_per_unit ? 0 : kh) * kChunks * NP * 128) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
              const uint32_t qoff = (kk >> 2) * NP * 128 + (kk & 3) * 32;
              mma_ss(tmem + NP * (g & 1), k + (off >> 4), qd + (qoff >> 4), idS, kk > 0);
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
    const float cj = p.scale_log2;  // scores in log2 units
    // P row n is K-major: KV row t sits in chunk t / 64, 16-byte unit (t % 64) / 8
    // (swizzled with n % 8), halfword t % 8
    uint8_t* prow = sP + (t >> 6) * NP * 128 + (t & 7) * 2;
    const int punit = (t & 63) >> 3;
    bool ok = true;
    int g = 0;
    for (int wi = w0; wi < w1 && ok; ++wi) {
      const Item it = read_item(p, wi);
      if (it.ntiles == 0) {  // empty shard: O = 0, LSE = -inf
        float* out_o = out_rows(p, it, D);
        float* out_l = out_lse(p, it);
        for (int i = t; i < p.Hc * D; i += kSoftmax) out_o[i] = 0.f;
        for (int i = t; i < p.Hc; i += kSoftmax) out_l[i] = -INFINITY;
        continue;
      }
      // token of tile row t of tile j: tok_t + j * tok_j; a cache row is masked
      // for the columns of query rows below tok - lim
      const int tok_j = kRows * it.pd.tok_step;
      const int tok_t = it.pd.tok0 + (it.row_begin + t) * it.pd.tok_step;
      const int lim = it.pd.ctx_len - p.s_q;
      for (int kh = 0; kh < p.Hkv && ok; ++kh) {
        // the running max restarts from the unit's first tile; every read of the
        // previous unit's maxima came before its epilogue's barriers
        if (t < NP) sM[t] = 0.f;
        named_bar_sync(1, kSoftmax);
        float l[NP];
#pragma unroll
        for (int n = 0; n < NP; ++n) l[n] = 0.f;
        for (int j = 0; j < it.ntiles; ++j, ++g) {
          const bool valid = j * kRows + t < it.nrows;
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
              u[n] = valid && n >= mcols ? fmaf(__uint_as_float(a[n]), cj, -sM[n]) : -INFINITY;
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
          // P[n][t] = 2^u (bf16)
#pragma unroll
          for (int n = 0; n < NP; ++n) {
            const float pn = ex2(u[n]);
            l[n] += pn;
            *reinterpret_cast<__nv_bfloat16*>(prow + n * 128 + ((punit ^ (n & 7)) << 4)) = __float2bfloat16_rn(pn);
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
        float* out_o = out_rows(p, it, D);
        if (t < NP) {
          const float tot = sL[0][t] + sL[1][t] + sL[2][t] + sL[3][t];
          sAlpha[t] = tot > 0.f ? 1.f / tot : 0.f;
          if (t < ncols) out_lse(p, it)[sCol[t] + kh * p.G] = tot > 0.f ? (sM[t] + lg2(tot)) * kLn2 : -INFINITY;
        }
        named_bar_sync(1, kSoftmax);
        {
          uint32_t o[NP];
          tmem_ld_cols<NP>(lane_addr + 2 * NP, o);
          tmem_ld_wait();
#pragma unroll
          for (int n = 0; n < NP; ++n)
            if (n < ncols && t < D) out_o[(long long)(sCol[n] + kh * p.G) * D + t] = __uint_as_float(o[n]) * sAlpha[n];
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
  if (warp == kWarpMma) tmem_dealloc(tmem, 256);
}

template <int NP, int D>
cudaError_t launch_np(const KVMaps& maps, const CUtensorMap& qmap, const Params& p, int grid, cudaStream_t s) {
  auto kern = decode_gqa_tc_kernel<NP, D>;
  constexpr int smem = Geo<D>::template smem<NP>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, s>>>(maps, qmap, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const KVMaps& maps, const CUtensorMap& qmap, const Params& p, int np, int grid,
                     cudaStream_t s) {
  switch (np) {
    case 16:
      return launch_np<16, D>(maps, qmap, p, grid, s);
    case 32:
      return launch_np<32, D>(maps, qmap, p, grid, s);
    default:
      return launch_np<64, D>(maps, qmap, p, grid, s);
  }
}

// Columns of a unit padded to the MMA N: 16, 32 or 64.
int padded_cols(int ncols) { return ncols <= 16 ? 16 : ncols <= 32 ? 32 : 64; }

}  // namespace

bool gqa_tc_supported(cp_dtype kv_dtype, int Hq, int Hkv, int Dqk, int Dv, int s_q) {
  if (kv_dtype != CP_BF16 || (Dqk != 64 && Dqk != 128) || Dv != Dqk || Hkv < 1 || Hq % Hkv) return false;
  const int ncols = (Hq / Hkv) * s_q;
  return ncols <= 64;
}

cudaError_t launch_decode_gqa_tc(const int32_t* dev_plan, const cp_plan_header& h, const void* q,
                                 const ShardPtrs& k, const ShardPtrs& v, const long long* shard_rows,
                                 const RowMap& rm, int Hq, int Hkv, int D, float sm_scale, float* o_part,
                                 float* lse_part, float* ws_o, float* ws_lse, const int32_t* pair_count,
                                 unsigned long long wait_ns, cudaStream_t s) {
  Params p;
  p.plan = dev_plan;
  p.B = h.R;
  p.off_pair = h.off_rank;
  p.off_worker = h.off_req;
  p.off_work = h.off_seg;
  p.rm = rm;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.s_q = plan_s_q(h);
  p.Hc = Hq * p.s_q;
  p.q_per_unit = (D == 128 || Hkv * padded_cols(p.G * p.s_q) > kMaxQCols) ? 1 : 0;
  p.scale_log2 = sm_scale * kLog2e;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.ws_o = ws_o;
  p.ws_lse = ws_lse;
  p.pair_count = pair_count;
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevice;
  p.wait_ns = wait_ns;
  KVMaps maps;
  memset(&maps, 0, sizeof(maps));
  // a kv head's slice of a row is 2 D bytes: at D = 64 a 128-byte slice, whose
  // neighbours (the other kv heads) are read in later units, so L2 fetches stay 128 bytes
  const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)Hkv * D * 2};
  if (rm.table) {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)Hkv, (uint64_t)rm.pool_rows};
    const uint32_t box[3] = {64, 1, 64};
    if (!encode_tensor_map_bf16(&maps.k[0], k.p[0], 3, dims, strides, box, D == 128) ||
        !encode_tensor_map_bf16(&maps.v[0], v.p[0], 3, dims, strides, box, D == 128))
      return cudaErrorInvalidValue;
  } else {
    for (int r = 0; r < h.C; ++r) {
      if (shard_rows[r] == 0) continue;
      const uint64_t dims[3] = {(uint64_t)D, (uint64_t)Hkv, (uint64_t)shard_rows[r]};
      const uint32_t box[3] = {64, 1, (uint32_t)kRows};
      if (!encode_tensor_map_bf16(&maps.k[r], k.p[r], 3, dims, strides, box, D == 128) ||
          !encode_tensor_map_bf16(&maps.v[r], v.p[r], 3, dims, strides, box, D == 128))
        return cudaErrorInvalidValue;
    }
  }
  // the queries [B s_q][Hkv][G][D]: one box per (kv head, 64-dim chunk) holds
  // the kv head's G heads of every query row of a request, rows n = qi G + i
  CUtensorMap qmap;
  {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)p.G, (uint64_t)Hkv, (uint64_t)h.R * p.s_q};
    const uint64_t qstrides[3] = {(uint64_t)D * 2, (uint64_t)p.G * D * 2, (uint64_t)Hq * D * 2};
    const uint32_t box[4] = {64, (uint32_t)p.G, 1, (uint32_t)p.s_q};
    if (!encode_tensor_map_bf16(&qmap, q, 4, dims, qstrides, box)) return cudaErrorInvalidValue;
  }
  const int np = padded_cols(p.G * p.s_q);
  return D == 64 ? launch_d<64>(maps, qmap, p, np, h.n_tiles, s) : launch_d<128>(maps, qmap, p, np, h.n_tiles, s);
}

}  // namespace cpattn
