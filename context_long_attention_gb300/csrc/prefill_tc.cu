// Causal GQA prefill on the tcgen05 tensor cores (bf16 in, fp32 accumulate).
//
// What it computes is the attention of "How GPUs Share a Long Context During
// LLM Inference" §1.1 for every query a virtual shard owns (§2.3 zigzag
// blocks, §2.4 interleave runs): each query at position p reads the keys at
// positions 0..p of its request, and the kernel emits O and the natural-log
// LSE of the scaled scores (§3.3).
//
// One CTA = one plan tile (up to 256 consecutive queries of one segment) x
// one query head, as two 128-row M tiles that share every K/V tile:
//   warps 0-15  softmax: warp w takes rows [32 (w % 4), +32) of M tile
//               (w / 4) % 2, columns [64 h, 64 h + 64) of S and dims
//               [D/2 h, D/2 h + D/2) of O with h = w / 8 (four softmax warps
//               per SM sub-partition hide each other's latency)
//   warp 16     TMA producer: K_j, V_j tiles [128 keys x D] into a slot ring,
//               V_(j-1) and K_j as one unit under one barrier
//   warp 17     MMA issuer (one elected lane; the warp runs the loop) and
//               TMEM owner.  Each of its mbarrier waits leaves the tensor
//               pipe idle (the pipe takes few products ahead), so a step has
//               two: the two tiles' P
//   warp 18     relay: one more arrival on each tile's P barrier per step,
//               once the step's K/V unit has landed, so the wait for P
//               covers the unit; the slots are freed by a softmax thread
// TMEM (512 columns): tile t holds S_t = Q_t K_j^T in columns [256t, 256t+128)
// and its output accumulator O_t in [256t+128, 256t+128+D).  Each half of a
// row writes its P (bf16 pairs) over the first 32 of its own 64 S columns,
// and O_t += P_t V_j reads P from TMEM there.  The MMA thread alternates the
// two M tiles so that one tile's softmax overlaps the other tile's matrix
// products.  The running max used in the exponentials only moves when a
// row's max grows by more than 2^8 (the two halves of the row exchange their
// maxima then, and O is rescaled); P is first computed with the max as it
// stands and recomputed only then.  The result is exact either way because
// O = sum_t exp(s_t - m) v_t / sum_t exp(s_t - m) holds for any m.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "internal.h"
#include "tc_ptx.cuh"

namespace cpattn {
namespace {
using namespace tc;

constexpr int BM = 128;        // query rows per M tile
constexpr int BN = 128;        // keys per K/V tile
constexpr int kSoftmaxWarps = 16;                 // two per row quarter of each M tile
constexpr int kThreads = 32 * (kSoftmaxWarps + 3);  // + TMA warp + MMA warp + relay warp
constexpr int kWarpTma = kSoftmaxWarps;
constexpr int kWarpMma = kSoftmaxWarps + 1;
constexpr int kWarpRelay = kSoftmaxWarps + 2;
// Registers are capped as for five warps per SM sub-partition (warps 16-18
// share sub-partitions 0-2 with four softmax warps each).
constexpr int kLaunchBoundThreads = 640;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;  // move the running max when it grows by > 2^8
constexpr float kSpecSum = 64.f * 256.f;  // a half row's P sum that may hide a P above 2^8

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;                   // 128-byte column chunks per row
  static constexpr int kQBytes = BM * D * 2;               // one Q tile
  static constexpr int kSlotBytes = BN * D * 2;            // one K or V tile
  static constexpr int kSlots = D == 128 ? 5 : 10;         // ring of K/V tiles (5 x 32 KB fits beside Q)
  static constexpr int kSmem = 2 * kQBytes + kSlots * kSlotBytes + 1024;
};

struct Params {
  const int32_t* plan;
  int off_seg;
  int tile_list;  // word offset of this launch's cp_tile_desc list
  int n_tiles;
  int row_sub;    // subtracted from rank-major rows (per-rank output)
  const __nv_bfloat16* q;
  __nv_bfloat16* o;
  float* lse;
  int Hq, group;
  float sm_scale, scale_log2;
  unsigned* status;
  unsigned long long wait_ns;
  int stall_test;  // test hook: the MMA thread waits on a barrier nobody arrives at
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed pairs of fp32 (one instruction for two lanes of work).
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
  asm("{\n .reg .b64 a, b, c, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n"
      " mov.b64 c, {%6, %7};\n fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n"
      " add.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, d;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ void report_timeout(unsigned* status, unsigned site, volatile int* abort) {
  *abort = 1;
  if (atomicCAS(status, 0u, 1u) == 0u) {
    status[1] = kKernPrefillTc;
    status[2] = site;
    status[3] = blockIdx.x;
    __threadfence();
  }
}

template <int D>
__global__ void __launch_bounds__(kLaunchBoundThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                    // two Q tiles
  uint8_t* sKV = smem + 2 * C::kQBytes;  // K/V slot ring
  // Loads go out in units that one wait covers: unit 0 = K_0, unit k = {V_(k-1), K_k},
  // unit nK = V_(nK-1); unit k completes bar_unit[k % kUnitBars].  A barrier
  // comes round again for unit k + kSlots, whose slots last held K/V tiles
  // k + 2 or later, freed only once S_(k+2) has completed; that needs
  // P_(k+1), which the relay warp completes after it has waited for unit k
  // (it takes the units in order; the MMA thread waits for unit 0), so no
  // phase completes before the one waited for.
  constexpr int kUnitBars = C::kSlots;
  // Slots are freed once per step: release j frees V_(j-1) and K_j (release
  // 0: K_0), on bar_rel[j % kSlots].  The last product the MMA thread issues
  // before tile rt's S_j is that of step j - 1, so one softmax thread of tile
  // rt (the tile that runs every step) arrives there when it sees S_j
  // complete: the issuing thread spends no commit on it.  The TMA warp waits
  // for release r of load u - kSlots (r about u / 2 - kSlots / 2) before it
  // loads u, while release r + kSlots needs S_(r+kSlots) and so a unit it has
  // not loaded yet: no release barrier completes twice unobserved.
  __shared__ __align__(8) uint64_t bar_unit[kUnitBars], bar_rel[C::kSlots];
  __shared__ __align__(8) uint64_t bar_q[2], bar_s[2], bar_p[2], bar_o[2], bar_never, bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ volatile int zero_flag;  // never set: drains ignore the abort flag

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTAs go kv head by kv head (each head's tiles longest first, the q heads
  // of its group side by side): the CTAs in flight then read one kv head's
  // K/V, which the L2 holds, instead of all of them
  const int per_g = p.n_tiles * p.group;
  const int gi = blockIdx.x / per_g, rem = blockIdx.x - gi * per_g;
  const int tile_i = rem / p.group, h = gi * p.group + rem % p.group;
  const cp_tile_desc td = reinterpret_cast<const cp_tile_desc*>(p.plan + p.tile_list)[tile_i];
  const cp_seg_desc sg = reinterpret_cast<const cp_seg_desc*>(p.plan + p.off_seg)[td.seg];
  const int g = h / p.group;

  // Rows and K/V tile counts of the two M tiles (scalars: no local-memory arrays).
  const int rows0 = min(BM, max(0, sg.count - td.q_off));
  const int rows1 = min(BM, max(0, sg.count - td.q_off - BM));
  const int nkv0 = rows0 > 0 ? (sg.first_pos + (td.q_off + rows0 - 1) * sg.stride + BN) / BN : 0;
  const int nkv1 = rows1 > 0 ? (sg.first_pos + (td.q_off + BM + rows1 - 1) * sg.stride + BN) / BN : 0;
  const int nK = max(nkv0, nkv1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kSlots; ++s) mbar_init(smem_u32(&bar_rel[s]), 1);
    for (int s = 0; s < kUnitBars; ++s) mbar_init(smem_u32(&bar_unit[s]), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bar_q[t]), 2 * BM);
      mbar_init(smem_u32(&bar_s[t]), 1);
      mbar_init(smem_u32(&bar_p[t]), 2 * BM + 1);  // + the relay warp
      mbar_init(smem_u32(&bar_o[t]), 1);
    }
    mbar_init(smem_u32(&bar_never), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    abort_flag = 0;
    zero_flag = 0;
    mbar_init_fence();
  }
  if (warp == kWarpMma) tmem_alloc(smem_u32(&tmem_slot), 512);
  if (warp == kWarpTma && lane == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp < kSoftmaxWarps) {
    // ------------------------------------------------------------ softmax
    // Warps w and w + 8 take the same 32 rows (TMEM lanes) of M tile t,
    // columns [64 half, 64 half + 64) of each S row and dims [D/2 half,
    // D/2 half + D/2) of each O row.  They exchange row maxima and sums
    // through column 63 of each half's S columns, which P never covers and
    // which S no longer needs once a tile's values are in registers.
    const int quarter = warp & 3;
    const int t = (warp >> 2) & 1;
    const int half = warp >> 3;
    const int i = quarter * 32 + lane;  // row within the M tile = TMEM lane
    const int pbar = 2 + t * 4 + quarter;  // named barrier of the two warps of these rows
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t colS = t * 256 + 64 * half, colO = t * 256 + 128 + (D / 2) * half;
    const int rows_t = t ? rows1 : rows0;
    const bool valid = i < rows_t;
    // the thread that frees K/V slots (bar_rel): tile 1 runs every step when it has rows
    const bool releaser = t == (rows1 > 0 ? 1 : 0) && quarter == 0 && half == 0;
    // value of the other half of this row
    auto exchange = [&](float v) -> float {
      tmem_st1(lane_addr + t * 256 + 64 * half + 63, __float_as_uint(v));
      tmem_st_wait();
      tc_fence_before();
      named_bar_sync(pbar, 64);
      tc_fence_after();
      const uint32_t o = tmem_ld1(lane_addr + t * 256 + 64 * (half ^ 1) + 63);
      tmem_ld_wait();
      return __uint_as_float(o);
    };
    // Q row -> shared memory in the 128-byte-swizzled K-major layout (half of its pieces).
    {
      const long long f = (long long)sg.first_f + (long long)(td.q_off + t * BM + i) * sg.stride;
      const uint4* src = reinterpret_cast<const uint4*>(p.q + (f * p.Hq + h) * D);
      uint8_t* dst = sQ + t * C::kQBytes + i * 128;
#pragma unroll
      for (int c = half * (D / 16); c < (half + 1) * (D / 16); ++c) {
        uint4 val = make_uint4(0, 0, 0, 0);
        if (valid) val = __ldg(src + c);
        const int a = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4*>(dst + a * (BM * 128) + ((cc ^ (i & 7)) << 4)) = val;
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bar_q[t]));
    }
    const int n_t = t ? nkv1 : nkv0;
    if (n_t > 0) {
      const int my_row = valid ? i : rows_t - 1;
      const int pos = sg.first_pos + (td.q_off + t * BM + my_row) * sg.stride;
      const float sl2 = p.scale_log2;
      const float thr = kRescaleLog2 / sl2;  // threshold in raw score units
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      // this half of the S row to registers, masked past the row's position
      // (P overwrites only these columns, so the two halves never touch each
      // other's S)
      auto load_s = [&](int j, uint32_t (&sr)[64]) {
        const int kbase = j * BN + 64 * half;
        tmem_ld32(lane_addr + colS, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(lane_addr + colS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_ld_wait();
        if (kbase + 63 > pos) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (kbase + e > pos) sr[e] = __float_as_uint(-INFINITY);
        }
      };
      // P = 2^(s c - m c) as bf16 pairs; returns this half's sum of P
      auto exps = [&](const uint32_t (&sr)[64], uint32_t (&pk)[32]) -> float {
        const float neg = -m_used * sl2;
        float s0sum = 0.f, s1sum = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float s0 = __uint_as_float(sr[2 * e]), s1 = __uint_as_float(sr[2 * e + 1]);
          float u0, u1;
          fma2(u0, u1, s0, s1, sl2, sl2, neg, neg);
          const float p0 = ex2(u0), p1 = ex2(u1);
          add2(s0sum, s1sum, s0sum, s1sum, p0, p1);
          pk[e] = pack_bf16x2(p0, p1);
        }
        return s0sum + s1sum;
      };
      for (int j = 0; j < n_t && ok; ++j) {
        const bool got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_s[t]), j & 1, p.wait_ns,
                                                           &abort_flag));
        if (got && releaser && lane == 0) mbar_arrive(smem_u32(&bar_rel[j % C::kSlots]));
        tc_fence_after();
        uint32_t sr[64], pk[32];
        float part = 0.f;
        bool slow = j == 0;
        if (j > 0) {
          // P with the running max as it stands, before anything is known of
          // this tile's maxima: a half whose P sums past 64 x 2^8 holds a P
          // above 2^8, its max passed the running max by more than 2^8 (NaN
          // counts as that too), and the row takes the exact path below.  Else
          // every P of the row is at most 2^14 and the running max stays.  (S
          // of a warp that gave up is read but never used.)
          load_s(j, sr);
          part = exps(sr, pk);
          slow = bar_red_or(pbar, 64, !got || !(part <= kSpecSum));
        }
        if (slow) {
          // Both warps of these rows leave together: one that gave up meets
          // the other at this vote.
          if (bar_red_or(pbar, 64, !got)) {
            if (!got) report_timeout(p.status, 1, &abort_flag);
            ok = false;
            break;
          }
          load_s(j, sr);
          float mx = -INFINITY;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            mx = fmax3(mx, __uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]));
          // The running max is the first tile's row max, and moves when a row's
          // max grows by more than 2^8: the halves exchange maxima so both move
          // it together.
          const float mrow = fmaxf(mx, exchange(mx));
          if (j == 0) {
            m_used = mrow;
          } else {
            // Each row (lane) moves its own max; the wait and the pair's barrier
            // below are taken by every lane of both warps (a lane whose max
            // stays scales by 1), since the vote to be here was the pair's.
            const bool need = mrow > m_used + thr;
            const float alpha = need ? ex2((m_used - mrow) * sl2) : 1.f;
            if (need) {
              l *= alpha;
              m_used = mrow;
            }
            // rescale this half of O_t once its previous P V product has landed
            const bool landed = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_o[t]), (j - 1) & 1,
                                                                  p.wait_ns, &abort_flag));
            if (bar_red_or(pbar, 64, !landed)) {
              if (!landed) report_timeout(p.status, 2, &abort_flag);
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r[16];
              tmem_ld16(lane_addr + colO + c * 16, r);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
              tmem_st16(lane_addr + colO + c * 16, r);
            }
          }
          part = exps(sr, pk);
        }
        l += part;
        // P over this half's first 32 columns of S, one store
        tmem_st32(lane_addr + colS, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_p[t]));
      }
      // epilogue: O / l and LSE (l summed over the two halves)
      const bool landed =
          ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_o[t]), (n_t - 1) & 1, p.wait_ns,
                                                  &abort_flag));
      if (!bar_red_or(pbar, 64, !landed)) {
        tc_fence_after();
        const float lt = l + exchange(l);
        const float inv = 1.f / lt;
        const long long out_row =
            (long long)sg.local_start + td.q_off + t * BM + i - p.row_sub;
        __nv_bfloat16* dst = p.o + (out_row * p.Hq + h) * D + (D / 2) * half;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t r[32];
          tmem_ld32(lane_addr + colO + c * 32, r);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(r[8 * v4 + 0]) * inv, __uint_as_float(r[8 * v4 + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(r[8 * v4 + 2]) * inv, __uint_as_float(r[8 * v4 + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(r[8 * v4 + 4]) * inv, __uint_as_float(r[8 * v4 + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(r[8 * v4 + 6]) * inv, __uint_as_float(r[8 * v4 + 7]) * inv);
              reinterpret_cast<uint4*>(dst + c * 32)[v4] = w;
            }
          }
        }
        if (valid && half == 0) p.lse[out_row * p.Hq + h] = m_used * p.sm_scale + logf(lt);
      } else if (ok) {
        report_timeout(p.status, 3, &abort_flag);
      }
    }
  } else if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    // The warp runs the loop; one elected lane issues the copies.
    {
      int last_unit = -1;
      bool ok = true;
      for (int k = 0; k <= nK && nK > 0 && ok; ++k) {
        // load u = 2j (K_j) or 2j + 1 (V_j) goes to slot u % kSlots
        const int u0 = k == 0 ? 0 : 2 * k - 1, u1 = k == nK ? 2 * k - 1 : 2 * k;
        for (int u = u0; u <= u1 && ok; ++u) {
          if (u < C::kSlots) continue;  // the slot's first load
          const int r = (u - C::kSlots + 1) >> 1;  // the release of load u - kSlots
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_rel[r % C::kSlots]), (r / C::kSlots) & 1,
                                                 p.wait_ns, &abort_flag))) {
            if (lane == 0) report_timeout(p.status, 4, &abort_flag);
            ok = false;
          }
        }
        if (!ok) break;
        const uint32_t full = smem_u32(&bar_unit[k % kUnitBars]);
        if (elect_one()) {
          mbar_expect_tx(full, (u1 - u0 + 1) * C::kSlotBytes);
          for (int u = u0; u <= u1; ++u) {
            const uint32_t dst = smem_u32(sKV + (u % C::kSlots) * C::kSlotBytes);
            const CUtensorMap* map = (u & 1) ? &vmap : &kmap;
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(dst + c * (BN * 128), map, c * 64, g, sg.kv_base + (u >> 1) * BN, full);
          }
        }
        __syncwarp();
        last_unit = k;
      }
      // Never leave with a copy in flight: wait for the last unit of every barrier.
      for (int k = max(0, last_unit - kUnitBars + 1); k <= last_unit; ++k)
        mbar_wait(smem_u32(&bar_unit[k % kUnitBars]), (k / kUnitBars) & 1, 1000000000ull, &zero_flag);
      __syncwarp();
    }
  } else if (warp == kWarpRelay) {
    // ------------------------------------------------------------ relay
    // P_j of tile t completes only once V_j and K_(j+1) have landed: this warp
    // adds one arrival per step to bar_p[t] after their unit is in and the
    // barrier's previous phase (step j - 1) is over, so the MMA thread's wait
    // for P_j covers the unit.  (A wait costs the issuing thread ~140 clk even
    // on a completed phase, and the tensor pipe runs dry meanwhile.)  Phase j
    // cannot complete before this arrival, so the wait for phase j - 1 never
    // sees two phases pass.
    bool ok = true;
    for (int j = 0; j < nK && ok; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_unit[(j + 1) % kUnitBars]),
                                             ((j + 1) / kUnitBars) & 1, p.wait_ns, &abort_flag));
      for (int t = 0; t < 2 && ok; ++t) {
        if (j >= (t ? nkv1 : nkv0)) continue;
        if (j > 0)
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_p[t]), (j - 1) & 1, p.wait_ns, &abort_flag));
        if (ok && lane == 0) mbar_arrive(smem_u32(&bar_p[t]));
        __syncwarp();
      }
      if (!ok && lane == 0) report_timeout(p.status, 17, &abort_flag);
    }
  } else {
    // ------------------------------------------------------------ MMA issuer
    // The warp runs the loop so that descriptors stay warp-uniform; one elected
    // lane (the same one every time, which also commits) issues the products.
    {
      constexpr unsigned kAll = 0xffffffffu;
      const uint32_t idS = idesc_bf16_f32(BM, BN, 0, 0);
      const uint32_t idPV = idesc_bf16_f32(BM, D, 0, 1);
      auto fail = [&](unsigned site) {
        if (lane == 0) report_timeout(p.status, site, &abort_flag);
      };
      auto wait_all = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(kAll, mbar_wait(bar, parity, p.wait_ns, &abort_flag));
      };
      auto wait_unit = [&](int k) -> bool {
        return wait_all(smem_u32(&bar_unit[k % kUnitBars]), (k / kUnitBars) & 1);
      };
      auto commit = [&](uint64_t* bar) {
        if (elect_one()) mma_commit(smem_u32(bar));
        __syncwarp();
      };
      // Descriptors are built once; an MMA adds its byte offset / 16 to the
      // start-address field (shared addresses stay below 2^18, so it never
      // carries).  The issuing thread shares its SM sub-partition with four
      // softmax warps: few instructions per MMA keep the tensor pipe fed.
      const uint64_t dQ0 = smem_desc(smem_u32(sQ), 16, 1024);
      const uint64_t dK0 = smem_desc(smem_u32(sKV), 16, 1024);
      const uint64_t dV0 = smem_desc(smem_u32(sKV), BN * 128, 1024);
      auto issue_s = [&](int t, int u) {
        const uint64_t a0 = dQ0 + (uint64_t)((t * C::kQBytes) >> 4);
        const uint64_t b0 = dK0 + (uint64_t)(((u % C::kSlots) * C::kSlotBytes) >> 4);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4;
            mma_ss(tmem + t * 256, a0 + off, b0 + off, idS, kk > 0);
          }
          mma_commit(smem_u32(&bar_s[t]));
        }
        __syncwarp();
      };
      auto issue_pv = [&](int t, int u, bool acc) {
        const uint64_t v0 = dV0 + (uint64_t)(((u % C::kSlots) * C::kSlotBytes) >> 4);
        const uint32_t pa = tmem + t * 256, d = tmem + t * 256 + 128;
        // P of keys [64 h, 64 h + 64) sits over the first 32 of S's columns [64 h, 64 h + 64)
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(d, pa + (kk >> 2) * 64 + (kk & 3) * 8, v0 + (uint64_t)((kk * 16 * 128) >> 4),
                   idPV, (acc || kk > 0) ? 1u : 0u);
          mma_commit(smem_u32(&bar_o[t]));
        }
        __syncwarp();
      };
      bool ok = true;
      if (p.stall_test && !wait_all(smem_u32(&bar_never), 0)) {
        fail(10);
        ok = false;
      }
      for (int t = 0; t < 2 && ok; ++t)
        if ((t ? nkv1 : nkv0) > 0 && !wait_all(smem_u32(&bar_q[t]), 0)) {
          fail(11);
          ok = false;
        }
      if (ok && nK > 0) {
        if (!wait_unit(0)) {
          fail(12);
          ok = false;
        } else {
          tc_fence_after();
          if (nkv0 > 0) issue_s(0, 0);
          if (nkv1 > 0) issue_s(1, 0);
        }
      }
      for (int j = 0; j < nK && ok; ++j) {
        const int uV = 2 * j + 1, uK = 2 * j + 2;
        // V_j and K_(j+1) are in place once a tile's P_j has completed (the
        // relay warp's arrival)
        for (int t = 0; t < 2 && ok; ++t) {
          const int nt = t ? nkv1 : nkv0;
          if (j >= nt) continue;
          if (!wait_all(smem_u32(&bar_p[t]), j & 1)) {
            fail(14 + t);
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(t, uV, j > 0);
          if (j + 1 < nt) issue_s(t, uK);
        }
        if (!ok) break;
      }
      // Never free TMEM under a running MMA: wait for everything issued.
      commit(&bar_drain);
      mbar_wait(smem_u32(&bar_drain), 0, 1000000000ull, &zero_flag);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, 512);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// [rows, H, D] bf16 viewed as 3-D (D, H, rows); box (64, 1, 128), 128-byte swizzle.
bool make_kv_map(CUtensorMap* m, const void* base, int rows, int H, int D) {
  const uint64_t dims[3] = {(uint64_t)D, (uint64_t)H, (uint64_t)rows};
  const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)H * D * 2};
  const uint32_t box[3] = {64, 1, (uint32_t)BN};
  return encode_tensor_map_bf16(m, base, 3, dims, strides, box);
}

template <int D>
cudaError_t launch_d(const CUtensorMap& km, const CUtensorMap& vm, const Params& p,
                     cudaStream_t s) {
  const int smem = Cfg<D>::kSmem;
  cudaError_t e =
      cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)p.n_tiles * p.Hq;
  prefill_tc_kernel<D><<<(unsigned)blocks, kThreads, smem, s>>>(km, vm, p);
  return cudaGetLastError();
}

}  // namespace

bool encode_tensor_map_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                            const uint64_t* strides, const uint32_t* box, bool promote_256) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rank < 2 || rank > 4) return false;
  cuuint64_t d[4], st[3];
  cuuint32_t b[4], es[4] = {1, 1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) st[i] = strides[i];
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, st, b, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             promote_256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tensor_map_u8_3d(CUtensorMap* m, const void* base, const uint64_t* dims, const uint64_t* strides,
                             const uint32_t* box) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]}, st[2] = {strides[0], strides[1]};
  const cuuint32_t b[3] = {box[0], box[1], box[2]}, es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), d, st, b, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tensor_map_u8_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                             uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows,
                             bool swizzle_128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t d[2] = {cols, rows}, st[1] = {row_bytes};
  const cuuint32_t b[2] = {box_cols, box_rows}, es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), d, st, b, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle_128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Limit of every bounded device wait: CPATTN_WAIT_LIMIT_MS (default 4000 ms),
// read once per process.
unsigned long long wait_limit_ns() {
  static unsigned long long v = [] {
    const char* s = getenv("CPATTN_WAIT_LIMIT_MS");
    const long long ms = s ? atoll(s) : 4000;
    return (unsigned long long)(ms > 0 ? ms : 4000) * 1000000ull;
  }();
  return v;
}

cudaError_t launch_prefill_tc(const int32_t* dev_plan, const int32_t* host_plan,
                              const cp_plan_header& h, int rank, const void* q, const void* k,
                              const void* v, int Hq, int Hkv, int D, float sm_scale, void* o,
                              float* lse, bool stall_test, cudaStream_t s) {
  Params p;
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
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.Hq = Hq;
  p.group = Hq / Hkv;
  p.sm_scale = sm_scale;
  p.scale_log2 = sm_scale * kLog2e;
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevice;
  p.wait_ns = stall_test ? 50000000ull : wait_limit_ns();
  p.stall_test = stall_test ? 1 : 0;
  CUtensorMap km, vm;
  if (!make_kv_map(&km, k, h.KV, Hkv, D) || !make_kv_map(&vm, v, h.KV, Hkv, D))
    return cudaErrorInvalidValue;
  return D == 128 ? launch_d<128>(km, vm, p, s) : launch_d<64>(km, vm, p, s);
}

}  // namespace cpattn
