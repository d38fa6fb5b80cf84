// MLA split-KV decode over an FP8-E4M3 cache, on FP8 tensor-core products.
//
// The work is that of the bf16 MLA decode: one decode query per request (64
// heads x 576 dims) against the rows one virtual shard stores ("How GPUs Share
// a Long Context During LLM Inference" §3.1-3.4); keys are the whole 576-dim
// latent entry and values its first 512 dims (vLLM blog "GLM-5.3 Part 2",
// footnote 1); each work item (a row range of one (shard, request) pair of
// the decode plan) yields a partial O and the natural-log LSE over its rows,
// merged later exactly (§3.3).  A cache entry is 576 E4M3 codes and one fp32
// scale per token (value = code x scale).
//
// The codes go from HBM to shared memory by TMA as stored and feed
// kind::f8f6f4 products directly: nothing is expanded to 16 bits.  The bf16
// query and the softmax weights are not E4M3 numbers, so each is carried as
// a pair hi + lo of E4M3 numbers (hi = x rounded to E4M3, lo = x - hi rounded
// to E4M3), which keeps 8 significant bits (relative error <= 2^-8) for
// |x| >= 2^-2 and an absolute error <= 2^-10 below that:
//   query:   x = q 2^e_q, with e_q per request so that max |x| is in [128, 256)
//   weights: x = 2^(s - M_h) scale_row 2^g, with M_h the running max of head h
//            and g per run of work items so that scale_row 2^g < 32; the running max
//            moves when a score passes it by more than 2^3, so x < 256
// The products (transposed so that M = 128 KV rows):
//   S^T [128 rows x 128] = K_codes [128 x 576] . [Q_hi | Q_lo]^T   (N = 128)
//     score(row, h) = (S^T[row][h] + S^T[row][64 + h]) scale_row 2^-e_q
//   O^T [512 x 64]      += V_codes^T [512 x 128] . (P_hi^T + P_lo^T) (K = 2 x 128)
// V_codes^T is the tile's first four 128-dim chunks read as an MN-major
// operand; P_hi^T goes over the tile's rope chunk once S^T is computed.
//
// Roles (352 threads): warps 0-7 softmax (thread = KV row of the tile = TMEM
// lane, warps w and w + 4 taking heads 0-31 and 32-63 of the same rows; in
// the epilogue, a dim row of O^T); warp 8 TMA producer; warp 9 P.V issuer and
// TMEM owner; warp 10 QK^T issuer.  Issuing a tcgen05.mma holds the issuing
// thread about as long as the product runs, so a single issuer serialises the
// two streams behind its own waits: with one per stream the tensor pipe runs
// the next tile's QK^T groups, which arrive chunk by chunk, while this tile's
// P.V waits for its weights.  Two tile stages in shared memory, each refilled
// chunk by chunk as P.V's M-blocks release it, and two S^T buffers in TMEM
// (each released by the softmax once it has loaded the scores) let the next
// tile's QK^T run while this tile's softmax works.
// TMEM: S^T buffer b at columns [128 b, 128 b + 128); O^T M-block mb at
// [256 + 64 mb, 320 + 64 mb).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstring>

#include "internal.h"
#include "tc_ptx.cuh"

namespace cpattn {
namespace {
using namespace tc;

constexpr int kRows = 128;   // KV rows per tile (MMA M)
constexpr int kHeads = 64;   // query heads (zero-padded)
constexpr int kDqk = 576, kDv = 512;
constexpr int kChunkBytes = kRows * 128;           // dims [128c, 128c + 128) of 128 rows: 16 KB
constexpr int kRopeOff = 4 * kChunkBytes;          // dims [512, 576): 128 rows x 64 B
constexpr int kStageBytes = kRopeOff + kRows * 64; // 73,728 B
constexpr int kQOff = 2 * kStageBytes;             // [Q_hi | Q_lo]: 128 operand rows x 576 B
constexpr int kPloOff = kQOff + kStageBytes;       // P_lo^T: 128 rows x 64 heads
constexpr int kSmem = kPloOff + kRows * 64 + 1024;
constexpr int kSoftmaxWarps = 8;  // a row's 64 heads in two groups of 32
constexpr int kSoftmax = 32 * kSoftmaxWarps;
constexpr int kHpw = kHeads / (kSoftmaxWarps / 4);  // heads per softmax warp
static_assert(kHpw % 16 == 0, "a softmax warp takes whole 16-head TMEM loads");
constexpr int kWarpTma = kSoftmaxWarps, kWarpPv = kSoftmaxWarps + 1, kWarpQk = kSoftmaxWarps + 2;
constexpr int kThreads = 32 * (kSoftmaxWarps + 3);
constexpr int kPrefetchAhead = 1;  // tiles between the L2 prefetch and the shared-memory copy
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 3.0f;  // the running max moves when a score passes it by > 2^3
constexpr int kWeightTop = 5;         // scale_row 2^g < 2^5, so a weight 2^(s - M) scale_row 2^g < 2^8

struct Params {
  const int32_t* plan;
  int B, off_pair, off_worker, off_work;
  const __nv_bfloat16* q;
  ShardPtrs k;  // code arrays (for the L2 prefetch; the tiles come through the tensor maps)
  ScalePtrs sc;
  RowMap rm;    // paged cache: 64-row boxes of a pool, rows through the page table
  int H;        // columns = s_q query rows x Hrow heads (<= 64)
  int Hrow, s_q;
  float scale_log2;  // sm_scale * log2(e)
  float* o_part;
  float* lse_part;
  float* ws_o;
  float* ws_lse;
  const int32_t* pair_count;  // rows in use per pair (a selection buffer), or nullptr
  // Merged output: run_out is the plan's run table (nullptr: one partial per
  // work item).  A worker's consecutive items of one request accumulate as
  // one run; a run holding its whole request writes the result to o_fin /
  // lse_fin, any other run a part to ws_o / ws_lse at its slot.
  const int32_t* run_out;
  void* o_fin;     // [B][H][512], bf16 (o_fin_bf16) or fp32
  int o_fin_bf16;
  float* lse_fin;  // [B][H]
  unsigned* status;
  unsigned long long wait_ns;
};

// Tensor maps of the shards' code arrays ([rows, 576] bytes): dims [0, 512)
// in 128-byte boxes with a 128-byte swizzle, dims [512, 576) with a 64-byte
// one; 128 rows a box, or for a paged cache one pool map with 64-row boxes.
struct CodeMaps {
  CUtensorMap body[CP_MAX_SHARDS];
  CUtensorMap rope[CP_MAX_SHARDS];
};

// D[tmem] (+)= A . B with 8-bit operands, A read from shared memory into the
// tensor core's A collector buffer and kept there for the next product
// (fill), or taken from that buffer, which the next product may not use
// again (lastuse).  Consecutive products with the same A read it once.
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

// Byte offset of (row, byte) in a 128-byte-swizzled [rows][128 B] block and
// in a 64-byte-swizzled [rows][64 B] block (the TMA and MMA layouts).
__device__ __forceinline__ int sw128(int row, int byte) {
  return row * 128 + ((((byte >> 4) ^ (row & 7))) << 4) + (byte & 15);
}
__device__ __forceinline__ int sw64(int row, int byte) {
  return row * 64 + ((((byte >> 4) ^ ((row >> 1) & 3))) << 4) + (byte & 15);
}

// Two values -> E4M3 pairs (hi, lo) with hi + lo ~ (x0, x1); byte 0 holds x0's code.
// The fp32 -> f16 step uses single conversions (the paired form slows the
// tensor-core products of the CTA); the E4M3 steps work on f16x2.
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

// Exponent e with |x| < 2^e for the largest |x| of a set (x > 0 normal);
// the scaling exponent that maps it into [2^(top-1), 2^top) is top - e.
__device__ __forceinline__ int scale_exponent(float maxabs, int top, int fallback) {
  if (!(maxabs > 0.f)) return fallback;
  const int E = (__float_as_int(maxabs) >> 23) & 0xFF;
  const int e = E == 0 ? -126 : E - 126;
  return max(-120, min(120, top - e));
}

__device__ void report_timeout(unsigned* status, unsigned site, volatile int* abort) {
  *abort = 1;
  if (atomicCAS(status, 0u, 1u) == 0u) {
    status[1] = kKernDecodeMlaFp8;
    status[2] = site;
    status[3] = blockIdx.x;
    __threadfence();
  }
}

// One work item of this CTA as every role sees it.
struct Item {
  int r, b, nrows, ntiles;
  int pair, row_begin, pair_rows;  // the pair, the item's first row in it, the pair's rows
  int tok0, tok_step, ctx_len;     // token of the pair's row i = tok0 + i tok_step; L
  long long row0;  // first shard row (contiguous caches)
  void* out_o;     // where the item's run writes O: fp32, or bf16 when out_bf16
  float* out_l;
  bool out_bf16;
  bool run_end;    // the item ends its run (always, without the run table)
  bool skip;       // an empty pair's item in a merged decode: nothing to do
};
template <bool kRuns>
__device__ __forceinline__ Item read_item(const Params& p, int wi) {
  const cp_work_desc wd = reinterpret_cast<const cp_work_desc*>(p.plan + p.off_work)[wi];
  const cp_pair_desc pd = reinterpret_cast<const cp_pair_desc*>(p.plan + p.off_pair)[wd.pair];
  Item it;
  it.r = wd.pair / p.B;
  it.b = wd.pair % p.B;
  const int row_end = p.pair_count ? min(wd.row_end, max(wd.row_begin, __ldg(p.pair_count + wd.pair)))
                                    : wd.row_end;
  it.nrows = row_end - wd.row_begin;
  it.ntiles = (it.nrows + kRows - 1) / kRows;
  it.row0 = (long long)pd.row_off + wd.row_begin;
  it.pair = wd.pair;
  it.row_begin = wd.row_begin;
  it.pair_rows = pd.rows;
  it.tok0 = pd.tok0;
  it.tok_step = pd.tok_step;
  it.ctx_len = pd.ctx_len;
  it.out_bf16 = false;
  it.run_end = true;
  it.skip = false;
  if (!kRuns) {
    it.out_o = wd.part < 0 ? p.o_part + (long long)wd.pair * p.H * kDv
                           : p.ws_o + (long long)wd.part * p.H * kDv;
    it.out_l = wd.part < 0 ? p.lse_part + (long long)wd.pair * p.H
                           : p.ws_lse + (long long)wd.part * p.H;
    return it;
  }
  const int ro = p.run_out[wi];
  it.skip = ro == -3;
  it.run_end = ro >= 0 || ro == -2;
  if (ro >= 0) {  // a part
    it.out_o = p.ws_o + (long long)ro * p.H * kDv;
    it.out_l = p.ws_lse + (long long)ro * p.H;
  } else {  // the request's result (read only when ro == -2)
    it.out_bf16 = p.o_fin_bf16 != 0;
    it.out_o = static_cast<uint8_t*>(p.o_fin) + (long long)it.b * p.H * kDv * (it.out_bf16 ? 2 : 4);
    it.out_l = p.lse_fin + (long long)it.b * p.H;
  }
  return it;
}

// kRuns: the launch has a run table (a merged decode); the split decode's
// instance folds the run branches away.
template <bool kRuns>
__global__ void __launch_bounds__(kThreads, 1)
    decode_mla_fp8_kernel(const __grid_constant__ CodeMaps maps, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // bar_full[s][q]: chunk group q of stage s (q < 4: dims [128q, 128q + 128);
  //   q = 4: the rope dims) holds its tile.
  // bar_done[s][mb]: P.V M-block mb of the tile in stage s has completed
  //   (and every product issued before it), so chunk mb of the stage may be
  //   refilled; mb = 3 also frees the rope chunk (it holds P_hi^T) and the
  //   P_lo^T buffer.
  // bar_s[b]: S^T buffer b holds its tile's products.  bar_p: this tile's
  // P^T is written.  bar_q: the work item's query is in shared memory.
  __shared__ __align__(8) uint64_t bar_full[2][5], bar_done[2][4], bar_s[2], bar_sfree[2];
  __shared__ __align__(8) uint64_t bar_p, bar_q, bar_drain, bar_drain_qk;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ volatile int zero_flag;  // never set: drains ignore the abort flag
  __shared__ __align__(16) float sM[kHeads];  // running max per head (log2 units)
  __shared__ float sDelta[kHeads];            // its last move; in the epilogue 1 / column sum
  __shared__ int sRed[4][kHeads];             // per row-quarter column maxima, then column sums
  __shared__ uint32_t sRed1[kSoftmaxWarps];   // per-warp max of |q| or of the token scales
  __shared__ uint32_t sInit[kHeads / 32];     // bit h: head h has had an unmasked row in the current run
  __shared__ int sMoved;                      // a vote moved some running max
  // (static shared memory has 2 KB beside the 225 KB of operands: keep these small)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      for (int q = 0; q < 5; ++q) mbar_init(smem_u32(&bar_full[s][q]), 1);
      for (int mb = 0; mb < 4; ++mb) mbar_init(smem_u32(&bar_done[s][mb]), 1);
      mbar_init(smem_u32(&bar_s[s]), 1);
      mbar_init(smem_u32(&bar_sfree[s]), kSoftmax);
    }
    mbar_init(smem_u32(&bar_p), kSoftmax);
    mbar_init(smem_u32(&bar_q), kSoftmax);
    mbar_init(smem_u32(&bar_drain), 1);
    mbar_init(smem_u32(&bar_drain_qk), 1);
    abort_flag = 0;
    zero_flag = 0;
    mbar_init_fence();
  }
  if (warp == kWarpPv) tmem_alloc(smem_u32(&tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t sbase = smem_u32(smem);
  const int w0 = p.plan[p.off_worker + blockIdx.x], w1 = p.plan[p.off_worker + blockIdx.x + 1];

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    // Warp-wide like the issuer: one elected lane issues the copies.
    {
      int last_g[2] = {-1, -1}, last_n[2] = {0, 0};  // last tile per stage, groups issued for it
      bool ok = true;
      int g = 0;
      for (int wi = w0; wi < w1 && ok; ++wi) {
        const Item it = read_item<kRuns>(p, wi);
        const uint8_t* codes = static_cast<const uint8_t*>(p.k.p[it.r]);
        // Cache row of the item's row i; past the pair's rows, a row past the
        // pool, where the copy reads zeros.
        auto cache_row = [&](int i) -> long long {
          const int ip = it.row_begin + i;
          if (!p.rm.table) return it.row0 + i;
          return ip < it.pair_rows ? map_row(p.rm, it.pair, 0, ip) : p.rm.pool_rows;
        };
        auto prefetch = [&](int jt) {  // tile jt of the item into L2, 64 contiguous rows at a time
          for (int hh = 0; hh < 2; ++hh) {
            const int i = jt * kRows + 64 * hh;
            const int rows = min(64, it.nrows - i);
            const long long row = rows > 0 ? cache_row(i) : 0;
            if (rows > 0 && elect_one()) prefetch_l2_bulk(codes + row * kDqk, (uint32_t)rows * kDqk);
            __syncwarp();
          }
        };
        for (int jt = 0; jt < kPrefetchAhead && jt < it.ntiles; ++jt) prefetch(jt);
        for (int j = 0; j < it.ntiles && ok; ++j, ++g) {
          const int s = g & 1;
          const uint32_t stage = sbase + s * kStageBytes;
          const int y = (int)(it.row0 + (long long)j * kRows);
          if (j + kPrefetchAhead < it.ntiles) prefetch(j + kPrefetchAhead);
          // paged: the pool rows of the tile's two 64-row halves, looked up once
          const long long yh[2] = {p.rm.table ? cache_row(j * kRows) : 0,
                                   p.rm.table ? cache_row(j * kRows + 64) : 0};
          for (int q = 0; q < 5 && ok; ++q) {
            // chunk q < 4 of the stage is free once P.V M-block q of its previous
            // tile (g - 2) has completed; the rope chunk once the whole P.V has
            if (g >= 2 && q < 4 &&
                !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_done[s][q]), ((g >> 1) & 1) ^ 1,
                                                   p.wait_ns, &abort_flag))) {
              if (lane == 0) report_timeout(p.status, 1, &abort_flag);
              ok = false;
              break;
            }
            const uint32_t full = smem_u32(&bar_full[s][q]);
            const uint32_t dst = stage + (q < 4 ? q * kChunkBytes : kRopeOff);
            const int x = 128 * q, row_bytes = q < 4 ? 128 : 64;
            const CUtensorMap* map = q < 4 ? &maps.body[it.r] : &maps.rope[it.r];
            if (elect_one()) {
              mbar_expect_tx(full, kRows * row_bytes);
              if (!p.rm.table) {
                tma_load_2d(dst, map, x, y, full);
              } else {  // two 64-row halves, each inside one page
                for (int hh = 0; hh < 2; ++hh)
                  tma_load_2d(dst + hh * 64 * row_bytes, &(q < 4 ? maps.body : maps.rope)[0], x,
                              (int)yh[hh], full);
              }
            }
            __syncwarp();
            last_g[s] = g;
            last_n[s] = q + 1;
          }
        }
      }
      // Never leave with a copy in flight.
      for (int s = 0; s < 2; ++s)
        for (int q = 0; q < last_n[s]; ++q)
          mbar_wait(smem_u32(&bar_full[s][q]), (last_g[s] >> 1) & 1, 1000000000ull, &zero_flag);
    }
  } else if (warp == kWarpQk) {
    // ------------------------------------------------------------ QK^T issuer
    // Issuing a tcgen05.mma holds the issuing thread for about as long as the
    // product runs, so one thread cannot run ahead of the tensor pipe: QK^T and
    // P.V each have an issuing warp, and the pipe interleaves the two streams
    // (the next tile's QK^T groups, which arrive chunk by chunk, fill the pipe
    // while this tile's P.V waits for its weights).  The whole warp runs the
    // loop so that descriptors and loop state stay warp-uniform; one elected
    // lane issues and commits.
    {
      const uint32_t idQK = idesc_e4m3_f32(kRows, 2 * kHeads, 0, 0);
      // Descriptors are built once; an MMA adds its byte offset / 16 to the
      // start-address field (shared addresses stay below 2^18, so it never carries).
      const uint32_t st0 = sbase, st1 = sbase + kStageBytes;
      const uint64_t dK[2] = {smem_desc(st0, 16, 1024, 2), smem_desc(st1, 16, 1024, 2)};
      const uint64_t dKr[2] = {smem_desc(st0 + kRopeOff, 16, 512, 4),
                               smem_desc(st1 + kRopeOff, 16, 512, 4)};
      const uint64_t dQ = smem_desc(sbase + kQOff, 16, 1024, 2);
      const uint64_t dQr = smem_desc(sbase + kQOff + kRopeOff, 16, 512, 4);
      auto wait_all = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, p.wait_ns, &abort_flag));
      };
      bool ok = true;
      int g = 0, nq = 0;  // tiles and query loads so far
      int q_b = -1;       // request whose query the operand holds
      for (int wi = w0; wi < w1 && ok; ++wi) {
        const Item it = read_item<kRuns>(p, wi);
        if (it.ntiles == 0) continue;
        // a new request's query is in place (written after every earlier product completed)
        if (it.b != q_b) {
          if (!wait_all(smem_u32(&bar_q), nq & 1)) {
            if (lane == 0) report_timeout(p.status, 2, &abort_flag);
            break;
          }
          ++nq;
          q_b = it.b;
        }
        for (int j = 0; j < it.ntiles && ok; ++j, ++g) {
          const int s = g & 1;
          const uint32_t d = tmem + 128 * s;
          // S^T buffer s is free once the softmax has loaded tile g - 2's scores
          if (g >= 2 && !wait_all(smem_u32(&bar_sfree[s]), ((g >> 1) & 1) ^ 1)) {
            if (lane == 0) report_timeout(p.status, 9, &abort_flag);
            ok = false;
            break;
          }
          // S^T(g) = K_codes . [Q_hi | Q_lo]^T, chunk group by chunk group as the codes land
          for (int q = 0; q < 5; ++q) {
            if (!wait_all(smem_u32(&bar_full[s][q]), (g >> 1) & 1)) {
              if (lane == 0) report_timeout(p.status, 3, &abort_flag);
              ok = false;
              break;
            }
            tc_fence_after();
            if (q < 4) {
              const uint64_t a = (s ? dK[1] : dK[0]) + (uint64_t)((q * kChunkBytes) >> 4);
              const uint64_t b = dQ + (uint64_t)((q * kChunkBytes) >> 4);
              if (elect_one()) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                  mma_ss_f8(d, a + 2 * ks, b + 2 * ks, idQK, (q | ks) != 0 ? 1u : 0u);
              }
            } else {
              const uint64_t a = s ? dKr[1] : dKr[0];
              if (elect_one()) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) mma_ss_f8(d, a + 2 * ks, dQr + 2 * ks, idQK, 1u);
                mma_commit(smem_u32(&bar_s[s]));
              }
            }
            __syncwarp();
          }
        }
      }
      // Never free TMEM under a running MMA.
      if (elect_one()) mma_commit(smem_u32(&bar_drain_qk));
      __syncwarp();
      mbar_wait(smem_u32(&bar_drain_qk), 0, 1000000000ull, &zero_flag);
    }
  } else if (warp == kWarpPv) {
    // ------------------------------------------------------------ P.V issuer and TMEM owner
    // O^T[M-block mb] (+)= V_codes^T . (P_hi^T + P_lo^T): the hi and lo
    // products of a K-step read the same A (a 128-dim x 32-row block of
    // V_codes^T), which the second one takes from the tensor core's A
    // collector buffer instead of shared memory.  Each block's commit releases
    // its chunk of the stage (block 3's also the rope chunk and P_lo^T's buffer).
    {
      const uint32_t idPV = idesc_e4m3_f32(kRows, kHeads, 1, 1);
      const uint32_t st0 = sbase, st1 = sbase + kStageBytes;
      const uint64_t dPhi[2] = {smem_desc(st0 + kRopeOff, 16, 512, 4),  // P_hi^T over the rope chunk
                                smem_desc(st1 + kRopeOff, 16, 512, 4)};
      const uint64_t dV[2] = {smem_desc(st0, kChunkBytes, 1024, 2),
                              smem_desc(st1, kChunkBytes, 1024, 2)};
      const uint64_t dPlo = smem_desc(sbase + kPloOff, 16, 512, 4);
      bool ok = true;
      int g = 0;
      int run_tiles = 0;  // tiles of the current run issued so far (O^T accumulates after the first)
      for (int wi = w0; wi < w1 && ok; ++wi) {
        const Item it = read_item<kRuns>(p, wi);
        for (int j = 0; j < it.ntiles && ok; ++j, ++g) {
          const int s = g & 1;
          const bool acc = run_tiles > 0;
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_p), g & 1, p.wait_ns, &abort_flag))) {
            if (lane == 0) report_timeout(p.status, 4, &abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int mb = 0; mb < 4; ++mb) {
            const uint64_t av = (s ? dV[1] : dV[0]) + (uint64_t)((mb * kChunkBytes) >> 4);
            const uint64_t bh = s ? dPhi[1] : dPhi[0];
            const uint32_t d = tmem + 256 + 64 * mb;
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < kRows / 32; ++kk) {
                const uint64_t a = av + (uint64_t)((kk * 4096) >> 4);
                mma_f8_fill_a(d, a, bh + (uint64_t)((kk * 2048) >> 4), idPV, (kk > 0 || acc) ? 1u : 0u);
                mma_f8_reuse_a(d, a, dPlo + (uint64_t)((kk * 2048) >> 4), idPV, 1u);
              }
              mma_commit(smem_u32(&bar_done[s][mb]));
            }
            __syncwarp();
          }
          ++run_tiles;
        }
        if (it.run_end) run_tiles = 0;
      }
      if (elect_one()) mma_commit(smem_u32(&bar_drain));
      __syncwarp();
      mbar_wait(smem_u32(&bar_drain), 0, 1000000000ull, &zero_flag);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int quarter = warp & 3;          // TMEM lane quarter: tile rows [32 quarter, +32)
    const int hb = (warp >> 2) * kHpw;     // this warp's heads [hb, hb + kHpw)
    const int t = quarter * 32 + lane;     // tile row = TMEM lane; in the epilogue a dim row
    const int tid = threadIdx.x;           // 0 .. kSoftmax - 1
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    uint8_t* sQ = smem + kQOff;
    uint8_t* sPlo = smem + kPloOff;
    bool ok = true;
    int g = 0;
    int q_b = -1, eq = 0;  // request whose query the operand holds, its scale exponent
    // the run's state: tiles so far, the weights' scale exponent (set on the
    // run's first tile, only decreases), this row's sums per head
    int run_tiles = 0, gs = 0;
    float l[kHpw];
    for (int wi = w0; wi < w1 && ok; ++wi) {
      const Item it = read_item<kRuns>(p, wi);
      if (it.skip) continue;
      // the run's result or part: O in fp32, or bf16 for a bf16 result
      void* const out_o = it.out_o;
      const bool out_bf16 = it.out_bf16;
      auto put_o = [out_o, out_bf16](long long i, float v) {
        if (out_bf16) static_cast<__nv_bfloat16*>(out_o)[i] = __float2bfloat16_rn(v);
        else static_cast<float*>(out_o)[i] = v;
      };
      if (it.ntiles > 0) {
        // ---- [Q_hi | Q_lo] of request b: x = q 2^eq with max |x| in [128, 256).
        // Every product of the previous item has completed (its epilogue waited
        // for the last P.V), so the operand can be overwritten; an item of the
        // same request as the previous one keeps it.
        const bool new_q = it.b != q_b;
        if (new_q) {
          q_b = it.b;
          const uint4* qsrc = reinterpret_cast<const uint4*>(p.q + (long long)it.b * p.H * kDqk);
          constexpr int kPieces = kDqk / 8;                   // 16-byte pieces per head
          constexpr int kPer = kHeads * kPieces / kSoftmax;   // pieces per thread
          static_assert(kHeads * kPieces % kSoftmax == 0, "query pieces split evenly");
          constexpr int kBatch = kPer % 6 == 0 ? 6 : 3;  // pieces in flight at once per thread
          static_assert(kPer % kBatch == 0, "whole batches of pieces");
          // a batch of this thread's pieces (heads past H are zero)
          auto load_batch = [&](int k0, uint4* qv) {
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
              const int i = tid + (k0 + k) * kSoftmax;
              qv[k] = i < p.H * kPieces ? __ldg(qsrc + i) : make_uint4(0, 0, 0, 0);
            }
          };
          uint32_t qmax = 0;  // largest |q| as bf16 magnitude bits
#pragma unroll 1
          for (int k0 = 0; k0 < kPer; k0 += kBatch) {
            uint4 qv[kBatch];
            load_batch(k0, qv);
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
              const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) qmax = max(qmax, max(w[e] & 0x7FFFu, (w[e] >> 16) & 0x7FFFu));
            }
          }
          qmax = __reduce_max_sync(0xffffffffu, qmax);
          if (lane == 0) sRed1[warp] = qmax;
          named_bar_sync(1, kSoftmax);
#pragma unroll
          for (int w = 0; w < kSoftmaxWarps; ++w) qmax = max(qmax, sRed1[w]);
          eq = scale_exponent(__uint_as_float(qmax << 16), 8, 0);
          const float qs = pow2i(eq);
#pragma unroll 1
          for (int k0 = 0; k0 < kPer; k0 += kBatch) {
            uint4 qv[kBatch];
            load_batch(k0, qv);
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
              const int i = tid + (k0 + k) * kSoftmax;
              const int h = i / kPieces, d0 = (i % kPieces) * 8;
              const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
              uint32_t hs[4], ls[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                split_e4m3x2(__uint_as_float(w[e] << 16) * qs, __uint_as_float(w[e] & 0xFFFF0000u) * qs,
                             hs[e], ls[e]);
              const uint2 hw = make_uint2(hs[0] | (hs[1] << 16), hs[2] | (hs[3] << 16));
              const uint2 lw = make_uint2(ls[0] | (ls[1] << 16), ls[2] | (ls[3] << 16));
              int oh, ol;
              if (d0 < 4 * 128) {
                const int base = (d0 >> 7) * kChunkBytes;
                oh = base + sw128(h, d0 & 127);
                ol = base + sw128(kHeads + h, d0 & 127);
              } else {
                oh = kRopeOff + sw64(h, d0 - 512);
                ol = kRopeOff + sw64(kHeads + h, d0 - 512);
              }
              *reinterpret_cast<uint2*>(sQ + oh) = hw;
              *reinterpret_cast<uint2*>(sQ + ol) = lw;
            }
          }
        }
        if (run_tiles == 0) {  // a new run: maxima set from its first tile
          if (tid < kHeads) sM[tid] = 0.f;
          if (tid < kHeads / 32) sInit[tid] = 0u;
          gs = 0;
#pragma unroll
          for (int h = 0; h < kHpw; ++h) l[h] = 0.f;
        }
        if (new_q) {
          fence_proxy_async_smem();
          mbar_arrive(smem_u32(&bar_q));  // the issuer's first QK^T orders the reset too
        } else {
          named_bar_sync(1, kSoftmax);    // the reset before any reader
        }

        const float* srow = p.sc.p[it.r] + it.row0;
        const float cq = p.scale_log2 * pow2i(-eq);
        for (int j = 0; j < it.ntiles; ++j, ++g) {
          const int row = j * kRows + t;
          const bool valid = row < it.nrows;
          // Several query rows (s_q > 1): query row qi reads tokens up to
          // L - s_q + qi, so this cache row is masked for columns [0, mcols).
          const int tok = it.tok0 + (it.row_begin + row) * it.tok_step;
          const int mcols = min(kHeads, max(0, tok - (it.ctx_len - p.s_q)) * p.Hrow);
          const float scale =
              !valid ? 0.f
                     : p.rm.table ? __ldg(p.sc.p[0] + map_row(p.rm, it.pair, 0, it.row_begin + row))
                                  : __ldg(srow + row);
          const int b = g & 1;
          // The softmax warps leave together: one that gave up meets the others at this vote.
          const bool got = __all_sync(
              0xffffffffu, mbar_wait(smem_u32(&bar_s[b]), (g >> 1) & 1, p.wait_ns, &abort_flag));
          if (bar_red_or(1, kSoftmax, !got)) {
            if (!got) report_timeout(p.status, 5, &abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          // u = score - running max (log2 units); rows past the item read nothing
          const float c = scale * cq;
          float u[kHpw];
          float over = -INFINITY;
          {  // one wait for all of the row's scores (the loads are slow while P.V runs)
            static_assert(kHpw == 32, "the score load takes 32 heads");
            uint32_t a[32], z[32];
            tmem_ld32(lane_addr + 128 * b + hb, a);
            tmem_ld32(lane_addr + 128 * b + kHeads + hb, z);
            tmem_ld_wait();
#pragma unroll
            for (int h4 = 0; h4 < 8; ++h4) {
              const float4 m4 = *reinterpret_cast<const float4*>(&sM[hb + 4 * h4]);
              const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int h = 4 * h4 + e;
                u[h] = valid && hb + h >= mcols ? fmaf(__uint_as_float(a[h]) + __uint_as_float(z[h]), c, -mm[e])
                             : -INFINITY;
                over = fmaxf(over, u[h]);
              }
            }
          }
          // the scores are in registers: the QK^T issuer may refill this S^T buffer
          tc_fence_before();
          mbar_arrive(smem_u32(&bar_sfree[b]));
          // Block-wide vote: the item's first tile, a score past its running max by
          // more than 2^3, or a token scale that would take a weight to 2^8 or more.
          const bool big = valid && scale * pow2i(gs) >= (float)(1 << kWeightTop);
          // A run's first tile sets the maxima.  A later item's first tile votes
          // only with several query rows, when heads masked so far may meet
          // their first rows (with one row every head is set on the run's
          // first tile).
          const bool first = j == 0 && (run_tiles == 0 || p.s_q > 1);
          if (bar_red_or(1, kSoftmax, first || over > kRescaleLog2 || big)) {
            if (tid == 0) sMoved = 0;
#pragma unroll
            for (int h = 0; h < kHpw; ++h) {
              const int m = __reduce_max_sync(0xffffffffu, ordered(u[h]));
              if (lane == 0) sRed[quarter][hb + h] = m;
            }
            const uint32_t smx = __reduce_max_sync(0xffffffffu, __float_as_uint(scale));
            if (lane == 0) sRed1[warp] = smx;
            named_bar_sync(1, kSoftmax);
            uint32_t smb = 0;
#pragma unroll
            for (int w = 0; w < kSoftmaxWarps; ++w) smb = max(smb, sRed1[w]);
            const float smax = __uint_as_float(smb);
            const int gs_new = run_tiles == 0 ? scale_exponent(smax, kWeightTop, 0)
                                              : min(gs, scale_exponent(smax, kWeightTop, gs));
            if (tid < kHeads) {
              const float cm = fmaxf(fmaxf(unordered(sRed[0][tid]), unordered(sRed[1][tid])),
                                     fmaxf(unordered(sRed[2][tid]), unordered(sRed[3][tid])));
              // A column takes its max from its first unmasked rows; until then it
              // keeps max 0 and weight 0.  Within an item rows go up in token
              // order, so a column masked in an item's first tile stays masked in
              // the item; a later item of the run (another shard) may unmask it,
              // and its first tile always votes.
              float delta;
              if (!((sInit[tid >> 5] >> (tid & 31)) & 1u)) {
                delta = cm == -INFINITY ? 0.f : cm;
                if (cm != -INFINITY) atomicOr(&sInit[tid >> 5], 1u << (tid & 31));
              } else {
                delta = cm > kRescaleLog2 ? cm : 0.f;
              }
              sDelta[tid] = delta;
            if (delta != 0.f) sMoved = 1;
              sM[tid] += delta;
            }
            named_bar_sync(1, kSoftmax);
            const float gf = pow2i(max(gs_new - gs, -126));
#pragma unroll
            for (int h = 0; h < kHpw; ++h) {
              const float dl = sDelta[hb + h];
              u[h] -= dl;
              l[h] *= ex2(-dl);
            }
            if (run_tiles > 0 && (sMoved || gs_new != gs)) {
              // O^T holds the run's earlier tiles: once the last P.V has landed, scale its columns
              const bool landed = __all_sync(
                  0xffffffffu, mbar_wait(smem_u32(&bar_done[(g - 1) & 1][3]), ((g - 1) >> 1) & 1, p.wait_ns,
                                         &abort_flag));
              if (bar_red_or(1, kSoftmax, !landed)) {
                if (!landed) report_timeout(p.status, 6, &abort_flag);
                ok = false;
                break;
              }
              tc_fence_after();
              // column h of O^T becomes O^T 2^-delta_h 2^(gs_new - gs)
#pragma unroll 1
              for (int c = 0; c < (kHpw / 16) * (kDv / 128); ++c) {
                const int mb = c / (kHpw / 16), h0 = 16 * (c % (kHpw / 16));
                uint32_t a[16];
                tmem_ld16(lane_addr + 256 + 64 * mb + hb + h0, a);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  a[e] = __float_as_uint(__uint_as_float(a[e]) * (ex2(-sDelta[hb + h0 + e]) * gf));
                tmem_st16(lane_addr + 256 + 64 * mb + hb + h0, a);
              }
              tmem_st_wait();
            }
            gs = gs_new;
          }
          // P^T row t, heads [hb, hb + kHpw): p = 2^u, weight x = p scale_row 2^gs as E4M3 hi + lo
          const float gr = scale * pow2i(gs);
          uint32_t hw[kHpw / 4], lw[kHpw / 4];
#pragma unroll
          for (int k = 0; k < kHpw / 4; ++k) {
            float pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              pk[e] = ex2(u[4 * k + e]);
              l[4 * k + e] += pk[e];
            }
            uint32_t h0, l0, h1, l1;
            split_e4m3x2(pk[0] * gr, pk[1] * gr, h0, l0);
            split_e4m3x2(pk[2] * gr, pk[3] * gr, h1, l1);
            hw[k] = h0 | (h1 << 16);
            lw[k] = l0 | (l1 << 16);
          }
          // P_lo^T has one buffer: the previous tile's P.V must have read it
          if (g > 0) {
            const bool freed = __all_sync(
                0xffffffffu, mbar_wait(smem_u32(&bar_done[(g - 1) & 1][3]), ((g - 1) >> 1) & 1, p.wait_ns,
                                       &abort_flag));
            if (bar_red_or(1, kSoftmax, !freed)) {
              if (!freed) report_timeout(p.status, 7, &abort_flag);
              ok = false;
              break;
            }
          }
          // MN-major operands [128 rows][64 heads], 64-byte swizzle; P_hi^T over the
          // rope chunk of this tile's stage (QK^T(g) has read it)
          uint8_t* phi = smem + b * kStageBytes + kRopeOff;
#pragma unroll
          for (int k = 0; k < kHpw / 16; ++k) {
            *reinterpret_cast<uint4*>(phi + sw64(t, hb + 16 * k)) =
                make_uint4(hw[4 * k], hw[4 * k + 1], hw[4 * k + 2], hw[4 * k + 3]);
            *reinterpret_cast<uint4*>(sPlo + sw64(t, hb + 16 * k)) =
                make_uint4(lw[4 * k], lw[4 * k + 1], lw[4 * k + 2], lw[4 * k + 3]);
          }
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(smem_u32(&bar_p));
          ++run_tiles;
        }
        if (!ok) break;
      }
      if (!it.run_end) continue;
      if (run_tiles == 0) {  // no rows in the run (an empty shard): O = 0, LSE = -inf
        for (int i = tid; i < p.H * kDv; i += kSoftmax) put_o(i, 0.f);
        for (int i = tid; i < p.H; i += kSoftmax) it.out_l[i] = -INFINITY;
        continue;
      }
      run_tiles = 0;
      // ---- epilogue: column sums of l, O^T 2^-gs / l, LSE
      const bool landed = __all_sync(
          0xffffffffu, mbar_wait(smem_u32(&bar_done[(g - 1) & 1][3]), ((g - 1) >> 1) & 1, p.wait_ns, &abort_flag));
      if (bar_red_or(1, kSoftmax, !landed)) {
        if (!landed) report_timeout(p.status, 8, &abort_flag);
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < kHpw; ++h) {
        float v = l[h];
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
        if (lane == 0) sRed[quarter][hb + h] = __float_as_int(v);
      }
      named_bar_sync(1, kSoftmax);
      if (tid < kHeads) {
        const float tot = __int_as_float(sRed[0][tid]) + __int_as_float(sRed[1][tid]) +
                          __int_as_float(sRed[2][tid]) + __int_as_float(sRed[3][tid]);
        sDelta[tid] = tot > 0.f ? 1.f / tot : 0.f;
        if (tid < p.H) it.out_l[tid] = tot > 0.f ? (sM[tid] + lg2(tot)) * kLn2 : -INFINITY;
      }
      named_bar_sync(1, kSoftmax);
      const float og = pow2i(-gs);
#pragma unroll 1
      for (int c = 0; c < (kHpw / 16) * (kDv / 128); ++c) {
        const int mb = c / (kHpw / 16), h0 = 16 * (c % (kHpw / 16));
        uint32_t a[16];
        tmem_ld16(lane_addr + 256 + 64 * mb + hb + h0, a);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const int hh = hb + h0 + h;
          if (hh < p.H) put_o((long long)hh * kDv + 128 * mb + t, __uint_as_float(a[h]) * og * sDelta[hh]);
        }
      }
      tc_fence_before();
      named_bar_sync(1, kSoftmax);  // shared state is free for the next item
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpPv) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_decode_mla_fp8(const int32_t* dev_plan, const cp_plan_header& h, const void* q,
                                  const ShardPtrs& k, const ScalePtrs& sc,
                                  const long long* shard_rows, const RowMap& rm, int H, float sm_scale,
                                  float* o_part, float* lse_part, float* ws_o, float* ws_lse,
                                  const int32_t* pair_count, unsigned long long wait_ns,
                                  cudaStream_t s, const MergedOut* mo) {
  Params p;
  p.pair_count = pair_count;
  p.run_out = mo ? mo->run_out : nullptr;
  p.o_fin = mo ? mo->o : nullptr;
  p.o_fin_bf16 = mo && mo->o_bf16 ? 1 : 0;
  p.lse_fin = mo ? mo->lse : nullptr;
  p.plan = dev_plan;
  p.B = h.R;
  p.off_pair = h.off_rank;
  p.off_worker = h.off_req;
  p.off_work = h.off_seg;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = k;
  p.sc = sc;
  p.rm = rm;
  p.s_q = plan_s_q(h);
  p.Hrow = H;
  p.H = H * p.s_q;
  p.scale_log2 = sm_scale * kLog2e;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.ws_o = ws_o;
  p.ws_lse = ws_lse;
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevice;
  p.wait_ns = wait_ns;
  CodeMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (rm.table) {
    const uint64_t rows = (uint64_t)rm.pool_rows;
    if (!encode_tensor_map_u8_2d(&maps.body[0], k.p[0], kDqk, rows, kDqk, 128, 64, true) ||
        !encode_tensor_map_u8_2d(&maps.rope[0], k.p[0], kDqk, rows, kDqk, 64, 64, false))
      return cudaErrorInvalidValue;
  } else {
    for (int r = 0; r < h.C; ++r) {
      if (shard_rows[r] == 0) continue;
      const uint64_t rows = (uint64_t)shard_rows[r];
      if (!encode_tensor_map_u8_2d(&maps.body[r], k.p[r], kDqk, rows, kDqk, 128, kRows, true) ||
          !encode_tensor_map_u8_2d(&maps.rope[r], k.p[r], kDqk, rows, kDqk, 64, kRows, false))
        return cudaErrorInvalidValue;
    }
  }
  auto kern = p.run_out ? decode_mla_fp8_kernel<true> : decode_mla_fp8_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  kern<<<h.n_tiles, kThreads, kSmem, s>>>(maps, p);
  return cudaGetLastError();
}

}  // namespace cpattn
