// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cpattn.h"

namespace cpattn {

constexpr int kHeaderWords = (int)(sizeof(cp_plan_header) / 4);
constexpr int kSegWords = (int)(sizeof(cp_seg_desc) / 4);
constexpr int kPairWords = (int)(sizeof(cp_pair_desc) / 4);
constexpr int kWorkWords = (int)(sizeof(cp_work_desc) / 4);
constexpr int kPrefillTileRows = 256;  // queries per prefill tile (two 128-row MMA tiles)
constexpr int kDecodeTileRows = 128;   // KV rows per decode scheduling tile (MMA M)
constexpr long long kDecodeItemCost = 2;  // a work item's fixed work, in tiles, for the schedule

// Query rows per request of a decode plan (plans without the field have one).
inline int plan_s_q(const cp_plan_header& h) { return h.s_q > 0 ? h.s_q : 1; }

// Device status word layout (written by kernels, read by cp_device_error_check).
//   [0] non-zero once any bounded wait gave up
//   [1] kernel id   [2] wait site   [3] block index
enum KernelId : unsigned {
  kKernPrefillTc = 1,
  kKernDecodeMlaTc = 2,
  kKernDecodeMlaFp8 = 3,
  kKernDecodeGqaTc = 4,
  kKernDecodeGqaF8 = 5,
  kKernTf32 = 6
};

struct ShardPtrs {
  const void* p[CP_MAX_SHARDS];
};
struct ScalePtrs {
  const float* p[CP_MAX_SHARDS];
};
using ScorePtrs = ScalePtrs;  // per-shard fp32 arrays of token scores
struct MutShardPtrs {
  void* p[CP_MAX_SHARDS];
};
struct MutScalePtrs {
  float* p[CP_MAX_SHARDS];
};

// Where the rows of a (shard r, request b) decode pair live.  Contiguous:
// rows [row_off, row_off + rows) of shard r's own buffer.  Paged: row i is
// row i % page_size of page table[pair][i / page_size] of one pool shared by
// all shards (every shard pointer is then the pool).  page_size is a multiple
// of 64, so a 64-row half of a 128-row decode tile never crosses a page.
struct RowMap {
  const int32_t* table;  // device [C * B][max_pages] page ids, or nullptr
  int max_pages;
  int page_size;
  long long pool_rows;   // num_pages * page_size (paged)
};
#ifdef __CUDACC__
__device__ __forceinline__ long long map_row(const RowMap& m, int pair, long long row_off, int i) {
  if (!m.table) return row_off + i;
  const int page = __ldg(m.table + (long long)pair * m.max_pages + i / m.page_size);
  return (long long)page * m.page_size + i % m.page_size;
}
#endif

// Returns the device address of this device's status words (set up once per device).
unsigned* device_status_ptr();

// Records a message for cp_last_error() on this thread and returns `st`.
cp_status report_error(cp_status st, const char* fmt, ...);

// ---- plan / pack / merge kernels (plan_kernels.cu)
cudaError_t launch_plan_maps(const int32_t* dev_plan, int n_seg, int off_seg, int off_idx,
                             int off_qpos, int off_qreq, cudaStream_t s);
cudaError_t launch_kv_pack(const int32_t* dev_plan, const cp_plan_header& h, int elem_bytes,
                           const void* kv, const float* kv_scale, int row_elems,
                           const MutShardPtrs& dst, const MutScalePtrs& dst_scale, bool has_scale,
                           const RowMap& rm, cudaStream_t s);
// Paged caches: zero the rows past each pair's last row on its last page (they
// enter the decode products with zero weight, and must hold finite values).
cudaError_t launch_page_tail_zero(const int32_t* dev_plan, const cp_plan_header& h,
                                  size_t row_bytes, void* pool, float* scale_pool,
                                  const RowMap& rm, cudaStream_t s);
cudaError_t launch_lse_merge(int P, int N, int H, int Dv, const float* o_part,
                             const float* lse_part, void* o, bool o_bf16, float* lse,
                             cudaStream_t s);
cudaError_t launch_lse_fold(int N, int H, int Dv, float* o, float* lse, const float* o_add,
                            const float* lse_add, cudaStream_t s);
// The merged decode's requests whose result comes from parts (the plan's
// merge list, n_list entries {request, first slot, parts}).
cudaError_t launch_merge_runs(const int32_t* dev_plan, const cp_plan_header& h, int n_list, int H, int Dv,
                              const float* ws_o, const float* ws_lse, void* o, bool o_bf16, float* lse,
                              cudaStream_t s);
cudaError_t launch_decode_fixup(const int32_t* dev_plan, const cp_plan_header& h, int H, int Dv,
                                const float* ws_o, const float* ws_lse, float* o_part,
                                float* lse_part, cudaStream_t s);

// ---- tensor-core prefill (prefill_tc.cu)
cudaError_t launch_prefill_tc(const int32_t* dev_plan, const int32_t* host_plan,
                              const cp_plan_header& h, int rank, const void* q, const void* k,
                              const void* v, int Hq, int Hkv, int D, float sm_scale, void* o,
                              float* lse, bool stall_test, cudaStream_t s);

// bf16 tensor map with a 128-byte swizzle (rank 2 to 4; strides in bytes for
// dims 1..rank-1).  False if the driver entry point is missing or rejects it.
// promote_256: L2 fetches widened to 256 bytes (the box rows are 256 bytes or
// neighbouring boxes are read together); else 128 bytes (a box row is a
// 128-byte slice whose neighbours are read much later).
bool encode_tensor_map_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                            const uint64_t* strides, const uint32_t* box, bool promote_256 = true);

// [rows, cols] byte tensor (row stride row_bytes), box [box_rows, box_cols],
// 128-byte swizzle if swizzle_128 else 64-byte.
// 3-d byte tensor (strides in bytes for dims 1..2), 128-byte swizzle, L2
// fetches of 128 bytes (a box row is one kv head's 128-byte slice of a row).
bool encode_tensor_map_u8_3d(CUtensorMap* m, const void* base, const uint64_t* dims, const uint64_t* strides,
                             const uint32_t* box);
bool encode_tensor_map_u8_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                             uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows,
                             bool swizzle_128);

// The merged-output decode's destinations: the plan's run table (device),
// the requests' results O [B][H][Dv] (bf16 or fp32) and LSE [B][H]; parts go
// to the workspace slots ws_o / ws_lse.
struct MergedOut {
  const int32_t* run_out;
  void* o;
  bool o_bf16;
  float* lse;
};

// ---- MLA decode over an FP8 cache on FP8 tensor-core products (decode_mla_fp8.cu)
// With mo, a worker's consecutive items of one request accumulate as one run
// (per-item partials otherwise).
cudaError_t launch_decode_mla_fp8(const int32_t* dev_plan, const cp_plan_header& h, const void* q,
                                  const ShardPtrs& k, const ScalePtrs& sc,
                                  const long long* shard_rows, const RowMap& rm, int H, float sm_scale,
                                  float* o_part, float* lse_part, float* ws_o, float* ws_lse,
                                  const int32_t* pair_count, unsigned long long wait_ns,
                                  cudaStream_t s, const MergedOut* mo = nullptr);

// ---- tensor-core MLA decode over a bf16 cache (decode_mla_tc.cu)
cudaError_t launch_decode_mla_tc(const int32_t* dev_plan, const cp_plan_header& h,
                                 const void* q, const ShardPtrs& k,
                                 const long long* shard_rows, const RowMap& rm, int H, float sm_scale,
                                 float* o_part, float* lse_part, float* ws_o, float* ws_lse,
                                 const int32_t* pair_count, unsigned long long wait_ns,
                                 cudaStream_t s, const MergedOut* mo = nullptr);
unsigned long long wait_limit_ns();

// ---- CUDA-core attention (simt_attn.cu)
cudaError_t launch_prefill_simt(const int32_t* dev_plan, const cp_plan_header& h, int rank,
                                int row_begin, int n_rows, bool bf16, const void* q,
                                const void* k, const void* v, int Hq, int Hkv, int D,
                                float sm_scale, void* o, float* lse, cudaStream_t s);
// The tensor-core GQA decode takes a bf16 cache with head dim 64 or 128 and at most
// 64 query columns per kv head (G s_q).
bool gqa_tc_supported(cp_dtype kv_dtype, int Hq, int Hkv, int Dqk, int Dv, int s_q);
cudaError_t launch_decode_gqa_tc(const int32_t* dev_plan, const cp_plan_header& h, const void* q,
                                 const ShardPtrs& k, const ShardPtrs& v, const long long* shard_rows,
                                 const RowMap& rm, int Hq, int Hkv, int D, float sm_scale, float* o_part,
                                 float* lse_part, float* ws_o, float* ws_lse, const int32_t* pair_count,
                                 unsigned long long wait_ns, cudaStream_t s);
// The tensor-core GQA decode over an E4M3 cache (codes expanded to f16 in
// shared memory): head dim 128, at most 32 query columns per kv head, per-shard
// buffers (not a paged pool).
bool gqa_f8_supported(int Hq, int Hkv, int Dqk, int Dv, int s_q, bool paged);
cudaError_t launch_decode_gqa_f8(const int32_t* dev_plan, const cp_plan_header& h, const void* q,
                                 const ShardPtrs& k, const ShardPtrs& v, const ScalePtrs& sc,
                                 const long long* shard_rows, int Hq, int Hkv, float sm_scale, float* o_part,
                                 float* lse_part, float* ws_o, float* ws_lse, const int32_t* pair_count,
                                 unsigned long long wait_ns, cudaStream_t s);
// ---- fp32 inputs on the tensor cores, kind::tf32 (tf32_attn.cu): the prefill
// at head dim 64 or 128; the GQA decode over per-shard fp32 buffers at head
// dim 64 or 128 with at most 64 query columns per kv head (G s_q).
bool prefill_tf32_supported(int D);
cudaError_t launch_prefill_tf32(const int32_t* dev_plan, const int32_t* host_plan, const cp_plan_header& h,
                                int rank, const void* q, const void* k, const void* v, int Hq, int Hkv, int D,
                                float sm_scale, void* o, float* lse, cudaStream_t s);
bool gqa_tf32_supported(int Hq, int Hkv, int Dqk, int Dv, int s_q, bool paged);
cudaError_t launch_decode_gqa_tf32(const int32_t* dev_plan, const cp_plan_header& h, const void* q,
                                   const ShardPtrs& k, const ShardPtrs& v, int Hq, int Hkv, int D, float sm_scale,
                                   float* o_part, float* lse_part, float* ws_o, float* ws_lse,
                                   const int32_t* pair_count, cudaStream_t s);
cudaError_t launch_decode_simt(const int32_t* dev_plan, const cp_plan_header& h,
                               cp_dtype kv_dtype, const void* q, const ShardPtrs& k,
                               const ShardPtrs& v, const ScalePtrs& sc, const RowMap& rm, int Hq,
                               int Hkv, int Dqk,
                               int Dv, float sm_scale, float* o_part, float* lse_part,
                               float* ws_o, float* ws_lse, const int32_t* pair_count,
                               cudaStream_t s);

// ---- sparse decode: exact sharded top-k and the owners' gather (sparse_kernels.cu)
// Decode kernels given a pair_count (device, one per (shard, request) pair)
// read only the first pair_count[pair] rows of each pair.
// range [C * B]: each pair's score range for the merge (hi << 32 | lo, ordered scores).
cudaError_t launch_topk_local(const int32_t* dev_plan, const cp_plan_header& h, const ScorePtrs& scores,
                              int k, int max_pair_rows, uint64_t* cand_keys, int32_t* cand_n, uint64_t* range,
                              cudaStream_t s);
cudaError_t launch_topk_merge(const int32_t* dev_plan, const cp_plan_header& h, int k, const uint64_t* cand_keys,
                              const int32_t* cand_n, const uint64_t* range, uint64_t* thresh, int32_t* sel_ids,
                              int32_t* sel_count, cudaStream_t s);
cudaError_t launch_sparse_gather(const int32_t* dev_plan, const cp_plan_header& h, int k,
                                 const uint64_t* cand_keys, const int32_t* cand_n,
                                 const uint64_t* thresh, const ShardPtrs& src,
                                 const ScalePtrs& src_scale, int row_bytes, const MutShardPtrs& dst,
                                 const MutScalePtrs& dst_scale, bool has_scale, int32_t* pair_count,
                                 cudaStream_t s);

}  // namespace cpattn
