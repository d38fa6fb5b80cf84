// MLA split-KV decode over a bf16 cache on the tcgen05 tensor cores.
//
// One decode query per request (64 heads x 576 dims) against the rows a
// virtual shard stores ("How GPUs Share a Long Context During LLM Inference"
// §3.1-3.4): every head reads the same 576-dim latent entry of each token
// (§1.3); keys are the whole entry and values its first 512 dims (vLLM blog
// "GLM-5.3 Part 2", footnote 1).  Each work item (a row range of one
// (shard, request) pair, from the decode plan) yields a partial O and the
// natural-log LSE over its rows, merged later exactly (§3.3).  (An FP8 cache
// takes the FP8 tensor-core kernel instead.)
//
// The products are transposed so that the MMA M dimension is 128 KV rows:
//   S^T [128 rows x 64 heads]  = K_tile [128 x 576] . Q^T          (K = 576)
//   O^T [512 dims x 64 heads] += V_tile^T [512 x 128] . P^T        (K = 128)
// V_tile^T is the same shared-memory tile as K_tile read as an MN-major
// operand (V is the first 512 latent dims), so one bf16 tile serves both
// products.  P^T (bf16) goes over the tile's last 64-dim chunk, which only
// the first product reads.
//
// Warp roles (256 threads): warps 0-3 softmax, thread = KV row of the tile
// (TMEM lane) and, in the epilogue, dim row of O^T; warp 0 also owns TMEM
// and issues the MMAs (one elected lane, the loop run warp-wide); warp 4
// refills the tile by TMA chunk group by chunk group as the previous tile's
// P.V releases it.
// Softmax down the KV axis needs per-head maxima over the 128 rows of a tile.
// The running maximum M_h used in the exponentials only moves when some score
// exceeds it by more than 2^8 (checked per tile with one block-wide vote);
// then a column max is reduced with redux.sync and O^T and the per-thread
// partial sums are rescaled.  Any M_h gives the exact result; this one keeps
// every exponential <= 2^8.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>

#include "internal.h"
#include "tc_ptx.cuh"

namespace cpattn {
namespace {
using namespace tc;

constexpr int kRows = 128;      // KV rows per tile (MMA M)
constexpr int kHeads = 64;      // MMA N (query heads, zero-padded)
constexpr int kDqk = 576, kDv = 512;
constexpr int kChunks = kDqk / 64;          // 9 chunks of 64 dims (128 B bf16 rows)
constexpr int kChunkBytes = kRows * 128;    // one chunk of the tile: 16 KB
constexpr int kTileBytes = kChunks * kChunkBytes;  // 147,456 B
constexpr int kQChunkBytes = kHeads * 128;  // one chunk of Q: 8 KB
constexpr int kQBytes = kChunks * kQChunkBytes;    // 73,728 B
constexpr int kSmem = kTileBytes + kQBytes + 1024;
constexpr int kThreads = 256;  // 8 warps: 2 per SM sub-partition, up to 255 registers
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

struct Params {
  const int32_t* plan;
  int B, off_pair, off_worker, off_work;
  ShardPtrs k;
  RowMap rm;  // paged cache: 64-row boxes of a pool, rows through the page table
  int H;             // columns = s_q query rows x Hrow heads (<= 64)
  int Hrow, s_q;
  float scale_log2;  // sm_scale * log2(e)
  float* o_part;
  float* lse_part;
  float* ws_o;
  float* ws_lse;
  const int32_t* pair_count;  // rows in use per pair (a selection buffer), or nullptr
  // Merged output (as in the FP8 MLA decode): run_out is the plan's run table,
  // nullptr for one partial per work item.
  const int32_t* run_out;
  void* o_fin;     // [B][H][512], bf16 (o_fin_bf16) or fp32
  int o_fin_bf16;
  float* lse_fin;  // [B][H]
  unsigned* status;
  unsigned long long wait_ns;
};

// Tensor maps of the shards' bf16 caches ([rows, 576], box 64 dims x 128 rows,
// 128-byte swizzle); a paged cache has one map of the pool with 64-row boxes.
struct ShardMaps {
  CUtensorMap m[CP_MAX_SHARDS];
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
    status[1] = kKernDecodeMlaTc;
    status[2] = site;
    status[3] = blockIdx.x;
    __threadfence();
  }
}

// Chunk groups of a tile: q = 0..3 hold dims [128q, 128q + 128) (chunks 2q,
// 2q+1, also the M-block q of V^T); q = 4 holds the rope dims [512, 576),
// overwritten by P^T once S^T is computed.
__device__ __forceinline__ int group_chunks(int q) { return q < 4 ? 2 : 1; }

// The fields of one work item that every role reads.
struct Item {
  int pair, r, b, part, row_begin, nrows, ntiles;
  long long row0;  // first shard row
  cp_pair_desc pd;
};

__device__ __forceinline__ Item read_item(const Params& p, const cp_pair_desc* pairs,
                                          const cp_work_desc* work, int wi) {
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
__device__ __forceinline__ float* out_rows(const Params& p, const Item& it) {
  return it.part < 0 ? p.o_part + (long long)it.pair * p.H * kDv : p.ws_o + (long long)it.part * p.H * kDv;
}
__device__ __forceinline__ float* out_lse(const Params& p, const Item& it) {
  return it.part < 0 ? p.lse_part + (long long)it.pair * p.H : p.ws_lse + (long long)it.part * p.H;
}

// Where a run ending at item it writes: the item's partial (no run table),
// a part slot, or the request's result (bf16 or fp32).
struct RunOut {
  float* f;
  __nv_bfloat16* b;  // non-null: a bf16 result
  float* l;
  __device__ __forceinline__ void put(long long i, float v) const {
    if (b) b[i] = __float2bfloat16_rn(v);
    else f[i] = v;
  }
};
template <bool kRuns>
__device__ __forceinline__ RunOut run_out_of(const Params& p, const Item& it, int ro) {
  RunOut o;
  o.b = nullptr;
  if (!kRuns) {
    o.f = out_rows(p, it);
    o.l = out_lse(p, it);
  } else if (ro >= 0) {
    o.f = p.ws_o + (long long)ro * p.H * kDv;
    o.l = p.ws_lse + (long long)ro * p.H;
  } else {
    o.f = static_cast<float*>(p.o_fin) + (long long)it.b * p.H * kDv;
    if (p.o_fin_bf16) o.b = static_cast<__nv_bfloat16*>(p.o_fin) + (long long)it.b * p.H * kDv;
    o.l = p.lse_fin + (long long)it.b * p.H;
  }
  return o;
}

// Warp roles run their loops over all work items of the CTA without meeting
// at item boundaries: the TMA warp fills the next item's first tile as soon
// as the previous tile's P.V releases the buffer, and loads a new request's
// query (one TMA box per 64-dim chunk; heads past H read as zeros) once the
// previous QK^T has completed.  Every barrier completes once per tile (bar_q
// once per query load), so the parity to wait for is that of the tile's index
// g over all items of this CTA.
// kRuns: the launch has a run table (a merged decode).  The split decode's
// instance folds every run branch away, so the per-item path keeps its
// registers.
template <bool kRuns>
__global__ void __launch_bounds__(kThreads, 1)
    decode_mla_tc_kernel(const __grid_constant__ ShardMaps maps, const __grid_constant__ CUtensorMap qmap,
                         const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sTile = smem;                  // [9 chunks][128 rows x 128 B]
  uint8_t* sQ = smem + kTileBytes;        // [9 chunks][64 heads x 128 B]
  uint8_t* sP = sTile + 8 * kChunkBytes;  // P^T over the last chunk: [128 rows][64 heads]
  // fill[q]: chunk group q of the tile holds the current tile.
  // mb[q]: the P.V product of M-block q (dims of group q) has completed; mb[3]
  //        also means the whole P.V (and every read of P^T) has completed.
  // q: sQ holds the query of the item's request.
  __shared__ __align__(8) uint64_t bar_fill[5], bar_mb[4], bar_s, bar_q, bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ volatile int zero_flag;
  __shared__ float sM[kHeads];     // running max per head (log2 units)
  __shared__ float sAlpha[kHeads];
  __shared__ float sDelta[kHeads];
  __shared__ int sRed[4][kHeads];  // cross-warp column maxima
  __shared__ float sL[4][kHeads];  // cross-warp column sums
  __shared__ uint32_t sInit[kHeads / 32];  // bit h: head h has had an unmasked row in the current run
  __shared__ int sMoved;                   // a vote moved some running max

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int q = 0; q < 5; ++q) mbar_init(smem_u32(&bar_fill[q]), 1);
    for (int q = 0; q < 4; ++q) mbar_init(smem_u32(&bar_mb[q]), 1);
    mbar_init(smem_u32(&bar_s), 1);
    mbar_init(smem_u32(&bar_q), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    abort_flag = 0;
    zero_flag = 0;
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // TMEM: S^T cols [0,64); O^T block mb: [64 + 64 mb, 128 + 64 mb)
  const uint32_t tmem = tmem_slot;

  const cp_pair_desc* pairs = reinterpret_cast<const cp_pair_desc*>(p.plan + p.off_pair);
  const cp_work_desc* work = reinterpret_cast<const cp_work_desc*>(p.plan + p.off_work);
  const int w0 = p.plan[p.off_worker + blockIdx.x], w1 = p.plan[p.off_worker + blockIdx.x + 1];
  bool ok = true;

  if (warp == 4) {
    // ------------------------------------------------------------ tile fill (TMA; the
    // warp runs the loop, one elected lane issues the copies)
    int g = 0;             // tiles of this CTA so far
    int q_b = -1, nq = 0;  // request whose query was loaded last, query loads issued
    int last_fill[5] = {-1, -1, -1, -1, -1};  // tile of each group's last issued fill
    for (int wi = w0; wi < w1 && ok; ++wi) {
      const Item it = read_item(p, pairs, work, wi);
      if (it.ntiles == 0) continue;
      const bool new_q = it.b != q_b;
      q_b = it.b;
      for (int j = 0; j < it.ntiles && ok; ++j, ++g) {
        // paged: the pool rows of the tile's two 64-row halves (each inside one page);
        // past the pair's rows the coordinate is past the pool and the copy reads zeros
        long long yh[2] = {0, 0};
        if (p.rm.table) {
          for (int hh = 0; hh < 2; ++hh) {
            const int i0 = it.row_begin + j * kRows + 64 * hh;
            yh[hh] = i0 < it.pd.rows ? map_row(p.rm, it.pair, 0, i0) : p.rm.pool_rows;
          }
        }
#pragma unroll
        for (int q = 0; q < 5; ++q) {
          // group q is free once the previous tile's P.V M-block q (or, for the
          // rope group that holds P^T, the whole P.V) has read it
          if (g > 0 &&
              !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_mb[q < 4 ? q : 3]), (g - 1) & 1,
                                                 p.wait_ns, &abort_flag))) {
            if (lane == 0) report_timeout(p.status, 1, &abort_flag);
            ok = false;
            break;
          }
          if (j == 0 && q == 0 && new_q) {
            // P.V block 0 of the previous tile follows its QK^T, the last read of sQ
            if (elect_one()) {
              mbar_expect_tx(smem_u32(&bar_q), kQBytes);
              for (int c = 0; c < kChunks; ++c)
                tma_load_3d(smem_u32(sQ + c * kQChunkBytes), &qmap, c * 64, 0, it.b, smem_u32(&bar_q));
            }
            __syncwarp();
            ++nq;
          }
          const uint32_t full = smem_u32(&bar_fill[q]);
          if (elect_one()) {
            mbar_expect_tx(full, group_chunks(q) * kChunkBytes);
            for (int cc = 0; cc < group_chunks(q); ++cc) {
              const int c = 2 * q + cc;
              if (!p.rm.table) {
                tma_load_2d(smem_u32(sTile + c * kChunkBytes), &maps.m[it.r], c * 64,
                            (int)(it.row0 + (long long)j * kRows), full);
              } else {
                for (int hh = 0; hh < 2; ++hh)
                  tma_load_2d(smem_u32(sTile + c * kChunkBytes + hh * 64 * 128), &maps.m[0],
                              c * 64, (int)yh[hh], full);
              }
            }
          }
          __syncwarp();
          last_fill[q] = g;
        }
      }
    }
    if (!ok) {
      // never leave with a copy in flight: each group's last fill and the last query load
      for (int q = 0; q < 5; ++q)
        if (last_fill[q] >= 0)
          mbar_wait(smem_u32(&bar_fill[q]), last_fill[q] & 1, 1000000000ull, &zero_flag);
      if (nq > 0) mbar_wait(smem_u32(&bar_q), (nq - 1) & 1, 1000000000ull, &zero_flag);
      __syncwarp();
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax (warps 0-3)
    const int t = threadIdx.x;  // tile row = TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t idS = idesc_bf16_f32(kRows, kHeads, 0, 0);
    const uint32_t idPV = idesc_bf16_f32(kRows, kHeads, 1, 1);
    const uint32_t tile = smem_u32(sTile), qb = smem_u32(sQ), pb = smem_u32(sP);
    // Warp 0 issues the products warp-wide (one elected lane); descriptors are
    // built once and an MMA adds its byte offset / 16 to the address field.
    const uint64_t dK = smem_desc(tile, 16, 1024), dQ = smem_desc(qb, 16, 1024);
    const uint64_t dV = smem_desc(tile, kChunkBytes, 1024), dP = smem_desc(pb, 16, 1024);
    int g0 = 0;
    int q_b = -1, nq = 0;  // request whose query sQ holds, query loads so far
    // the run (a worker's consecutive items of one request, or one item
    // without the run table): its tiles so far; this row's sums per head live
    // in registers within an item and in TMEM columns [320, 384) between the
    // items of a run (kept in registers across items they spilled)
    int run_tiles = 0;
    const uint32_t l_addr = lane_addr + 320;
    auto l_save = [&](const float (&l)[kHeads]) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t a[32];
#pragma unroll
        for (int h = 0; h < 32; ++h) a[h] = __float_as_uint(l[32 * h2 + h]);
        tmem_st32(l_addr + 32 * h2, a);
      }
      tmem_st_wait();
    };
    auto l_load = [&](float (&l)[kHeads]) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t a[32];
        tmem_ld32(l_addr + 32 * h2, a);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < 32; ++h) l[32 * h2 + h] = __uint_as_float(a[h]);
      }
    };
    for (int wi = w0; wi < w1 && ok; ++wi) {
      const Item it = read_item(p, pairs, work, wi);
      float l[kHeads];
      // where the item's run writes: the per-item partial, a part slot, or the result
      const int ro = kRuns ? p.run_out[wi] : -2;
      if (!kRuns) run_tiles = 0;
      if (ro == -3) continue;  // an empty pair's item of a merged decode
      const bool run_end = !kRuns || ro != -1;
      if (it.ntiles == 0) {
        if (!run_end) continue;
        if (run_tiles == 0) {  // no rows in the run (an empty shard): O = 0, LSE = -inf
          const RunOut out = run_out_of<kRuns>(p, it, ro);
          for (int i = t; i < p.H * kDv; i += 128) out.put(i, 0.f);
          for (int i = t; i < p.H; i += 128) out.l[i] = -INFINITY;
          continue;
        }
      }
      if (it.ntiles > 0) {
        // a new request: warp 0 waits for its query before the first QK^T
        bool q_ok = true;
        if (it.b != q_b) {
          if (warp == 0)
            q_ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_q), nq & 1, p.wait_ns, &abort_flag));
          ++nq;
        }
        q_b = it.b;
        // a run's running max starts from its first tile's maxima; every read of
        // the previous run's maxima came before its epilogue's barrier
        if (run_tiles == 0) {
          if (t < kHeads) sM[t] = 0.f;
          if (t < kHeads / 32) sInit[t] = 0u;
#pragma unroll
          for (int h = 0; h < kHeads; ++h) l[h] = 0.f;
        } else {
          l_load(l);  // the run's sums so far
        }
        named_bar_sync(1, 128);
        // token of tile row t of tile j: tok_t + j * tok_j; a cache row is masked
        // for the columns of query rows below tok - lim
        const int tok_j = kRows * it.pd.tok_step;
        const int tok_t = it.pd.tok0 + (it.row_begin + t) * it.pd.tok_step;
        const int lim = it.pd.ctx_len - p.s_q;
        const int nrows = it.nrows, ntiles = it.ntiles;
        for (int j = 0; j < ntiles; ++j) {
          const int g = g0 + j;
          bool issued = q_ok;
          q_ok = true;
          if (warp == 0) {  // S^T = K_tile Q^T, chunk group by chunk group as they fill
            for (int q = 0; q < 5 && issued; ++q) {
              issued = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_fill[q]), g & 1, p.wait_ns,
                                                         &abort_flag));
              if (!issued) break;
              tc_fence_after();
              if (elect_one()) {
                for (int ks = 0; ks < 4 * group_chunks(q); ++ks) {
                  const int kk = 8 * q + ks;
                  const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                  const uint32_t qoff = (kk >> 2) * kQChunkBytes + (kk & 3) * 32;
                  mma_ss(tmem, dK + (off >> 4), dQ + (qoff >> 4), idS, kk > 0);
                }
              }
              __syncwarp();
            }
            if (issued && elect_one()) mma_commit(smem_u32(&bar_s));
            __syncwarp();
          }
          const bool valid = j * kRows + t < nrows;
          // Several query rows (s_q > 1): row qi of the request reads tokens up
          // to L - s_q + qi, so this cache row is masked for the columns of the
          // query rows qi < tok - (L - s_q), columns [0, mcols).
          const int tok = tok_t + j * tok_j;
          const int mcols = min(kHeads, max(0, tok - lim) * p.Hrow);
          const float cj = p.scale_log2;  // scores in log2 units
          // The four softmax warps leave together: a warp that gave up still
          // meets the others at the named barrier of this vote.
          const bool got = __all_sync(
              0xffffffffu, issued && mbar_wait(smem_u32(&bar_s), g & 1, p.wait_ns, &abort_flag));
          if (bar_red_or(1, 128, !got)) {
            if (!got) report_timeout(p.status, 6, &abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          // u = score - running max (log2 units); invalid rows read nothing
          float u[kHeads];
          float over = -INFINITY;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t a[32];
            tmem_ld32(lane_addr + 32 * half, a);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 32; ++h) {
              const int hh = 32 * half + h;
              u[hh] = valid && hh >= mcols ? fmaf(__uint_as_float(a[h]), cj, -sM[hh]) : -INFINITY;
              over = fmaxf(over, u[hh]);
            }
          }
          // Block-wide vote: does any score pass its running max by more than 2^8?
          // A run's first tile sets the maxima; a later item's first tile votes
          // only with several query rows (heads masked so far may meet their first rows).
          const bool first = j == 0 && (run_tiles == 0 || p.s_q > 1);
          if (bar_red_or(1, 128, first || over > kRescaleLog2)) {
            if (t == 0) sMoved = 0;
            // column maxima of this tile (relative to the old running max)
#pragma unroll
            for (int h = 0; h < kHeads; ++h) {
              const int m = __reduce_max_sync(0xffffffffu, ordered(u[h]));
              if (lane == 0) sRed[warp][h] = m;
            }
            named_bar_sync(1, 128);
            if (t < kHeads) {
              const float cm = fmaxf(fmaxf(unordered(sRed[0][t]), unordered(sRed[1][t])),
                                     fmaxf(unordered(sRed[2][t]), unordered(sRed[3][t])));
              // move the running max to a column's first unmasked maxima, or when it
              // grew by more than 2^8; earlier sums and O^T shrink by 2^-delta.  A
              // column masked so far keeps max 0 and weight 0: within an item rows
              // go up in token order, and a later item of the run (another shard)
              // that unmasks it votes on its first tile.
              float delta;
              if (!((sInit[t >> 5] >> (t & 31)) & 1u)) {
                delta = cm == -INFINITY ? 0.f : cm;
                if (cm != -INFINITY) atomicOr(&sInit[t >> 5], 1u << (t & 31));
              } else {
                delta = cm > kRescaleLog2 ? cm : 0.f;
              }
              if (delta != 0.f) sMoved = 1;
              sAlpha[t] = run_tiles == 0 ? 0.f : ex2(-delta);
              sDelta[t] = delta;
              sM[t] += delta;
            }
            named_bar_sync(1, 128);
#pragma unroll
            for (int h = 0; h < kHeads; ++h) {
              l[h] *= sAlpha[h];
              u[h] -= sDelta[h];
            }
            if (run_tiles > 0 && sMoved) {  // O^T holds the run's earlier tiles (their P.V completed before this S)
              // 16 columns at a time: u and l stay in registers meanwhile
#pragma unroll 1
              for (int c = 0; c < 4 * kHeads / 16; ++c) {
                uint32_t a[16];
                tmem_ld16(lane_addr + 64 + 16 * c, a);
                tmem_ld_wait();
                const float* al = sAlpha + ((16 * c) & (kHeads - 1));
#pragma unroll
                for (int h = 0; h < 16; ++h) a[h] = __float_as_uint(__uint_as_float(a[h]) * al[h]);
                tmem_st16(lane_addr + 64 + 16 * c, a);
              }
              tmem_st_wait();
            }
          }
          // P^T row t: p = 2^u.
          // MN-major B operand: row t = 64 heads x 2 B = one 128-byte swizzled row.
          uint8_t* prow = sP + t * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int h = 8 * c + 2 * e;
              const float p0 = ex2(u[h]), p1 = ex2(u[h + 1]);
              l[h] += p0;
              l[h + 1] += p1;
              pk[e] = pack_bf16x2(p0, p1);
            }
            *reinterpret_cast<uint4*>(prow + ((c ^ (t & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
          fence_proxy_async_smem();
          tc_fence_before();
          named_bar_sync(1, 128);  // every row of P^T is written
          if (warp == 0) {         // O^T += V_tile^T P^T, one M-block (128 dims) at a time
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
              for (int mb = 0; mb < kDv / 128; ++mb) {
#pragma unroll
                for (int kk = 0; kk < kRows / 16; ++kk)
                  mma_ss(tmem + 64 + 64 * mb, dV + ((2 * mb * kChunkBytes + kk * 2048) >> 4),
                         dP + ((kk * 2048) >> 4), idPV, (run_tiles > 0 || kk > 0) ? 1u : 0u);
                mma_commit(smem_u32(&bar_mb[mb]));
              }
            }
            __syncwarp();
          }
          ++run_tiles;
        }
      }
      if (!run_end && run_tiles > 0) l_save(l);  // the run goes on to the next item
      // ---- epilogue at a run's end: column sums of l, O^T / l, LSE
      if (run_end && run_tiles > 0) {
      if (it.ntiles == 0) l_load(l);  // an item with no rows ends the run
      run_tiles = 0;
      const bool landed =
          ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_mb[3]), (g0 + it.ntiles - 1) & 1,
                                                  p.wait_ns, &abort_flag));
      if (bar_red_or(1, 128, !landed)) {
        if (ok && !landed) report_timeout(p.status, 7, &abort_flag);
        ok = false;
      }
      if (ok) {
        tc_fence_after();
        const RunOut out = run_out_of<kRuns>(p, it, ro);
        float* const out_l = out.l;
#pragma unroll
        for (int h = 0; h < kHeads; ++h) {
          float v = l[h];
#pragma unroll
          for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
          if (lane == 0) sL[warp][h] = v;
        }
        named_bar_sync(1, 128);
        // one reciprocal per head (sAlpha is free until the next item's first
        // tile): a division per element made the epilogue cost more than a tile
        if (t < kHeads) {
          const float tot = sL[0][t] + sL[1][t] + sL[2][t] + sL[3][t];
          sAlpha[t] = tot > 0.f ? 1.f / tot : 0.f;
          if (t < p.H) out_l[t] = tot > 0.f ? (sM[t] + lg2(tot)) * kLn2 : -INFINITY;
        }
        named_bar_sync(1, 128);
#pragma unroll 1
        for (int mb = 0; mb < kDv / 128; ++mb) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t a[32];
            tmem_ld32(lane_addr + 64 + 64 * mb + 32 * half, a);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 32; ++h) {
              const int hh = 32 * half + h;
              if (hh < p.H) out.put((long long)hh * kDv + 128 * mb + t, __uint_as_float(a[h]) * sAlpha[hh]);
            }
          }
        }
      }
      }

      g0 += it.ntiles;
      // the four softmax warps decide together whether to go on
      if (bar_red_or(1, 128, !ok || abort_flag != 0)) ok = false;
    }
  }
  // Never free TMEM under a running MMA.
  if (warp == 0) {
    if (elect_one()) mma_commit(smem_u32(&bar_drain));
    __syncwarp();
    mbar_wait(smem_u32(&bar_drain), 0, 1000000000ull, &zero_flag);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_decode_mla_tc(const int32_t* dev_plan, const cp_plan_header& h,
                                 const void* q, const ShardPtrs& k,
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
  p.k = k;
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
  ShardMaps local;
  memset(&local, 0, sizeof(local));
  if (rm.table) {
    const uint64_t dims[2] = {(uint64_t)kDqk, (uint64_t)rm.pool_rows};
    const uint64_t strides[1] = {(uint64_t)kDqk * 2};
    const uint32_t box[2] = {64, 64};
    if (!encode_tensor_map_bf16(&local.m[0], k.p[0], 2, dims, strides, box))
      return cudaErrorInvalidValue;
  } else {
    for (int r = 0; r < h.C; ++r) {
      if (shard_rows[r] == 0) continue;
      const uint64_t dims[2] = {(uint64_t)kDqk, (uint64_t)shard_rows[r]};
      const uint64_t strides[1] = {(uint64_t)kDqk * 2};
      const uint32_t box[2] = {64, (uint32_t)kRows};
      if (!encode_tensor_map_bf16(&local.m[r], k.p[r], 2, dims, strides, box))
        return cudaErrorInvalidValue;
    }
  }
  // the queries [B][H][576]: one box per 64-dim chunk of a request's 64 columns
  // (columns past H fall outside the map and read as zeros)
  CUtensorMap qmap;
  {
    const uint64_t dims[3] = {(uint64_t)kDqk, (uint64_t)p.H, (uint64_t)h.R};
    const uint64_t strides[2] = {(uint64_t)kDqk * 2, (uint64_t)p.H * kDqk * 2};
    const uint32_t box[3] = {64, (uint32_t)kHeads, 1};
    if (!encode_tensor_map_bf16(&qmap, q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  auto kern = p.run_out ? decode_mla_tc_kernel<true> : decode_mla_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  kern<<<h.n_tiles, kThreads, kSmem, s>>>(local, qmap, p);
  return cudaGetLastError();
}

}  // namespace cpattn
