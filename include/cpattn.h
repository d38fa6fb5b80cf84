/*
 * cpattn.h — context-parallel attention on one GPU (sm_103a), C ABI.
 *
 * The library computes the data-parallel hot path of context parallelism for
 * long-context LLM inference, with C *virtual* shards executed as
 * independent partitions on one GPU:
 *
 *   cp_shard_plan      prompt-token shard maps (zigzag, interleave)
 *   cp_decode_plan     decode KV-cache token shards + split-KV schedule
 *   cp_prefill_attn    causal GQA prefill per shard, emitting (O, LSE)
 *   cp_kv_shard_pack   gather a token-ordered cache into token shards
 *   cp_decode_attn     one decode query per request against each shard,
 *                      emitting per-shard partial (O, LSE)
 *   cp_lse_merge       exact log-sum-exp combine of partial results
 *
 * Sources (page title, section):
 *   [CTX] "How GPUs Share a Long Context During LLM Inference"
 *   [SGL] SGLang documentation, "Prefill context parallelism"
 *   [V4]  "DeepSeek-V4 Attention Inference Systems", §5
 *   [GLM] vLLM blog "GLM-5.3 Part 2: PCP, DCP and Hybrid HiSparse on 16 H200"
 *   [DCP] vLLM blog on Decode Context Parallelism, §4.1 and §5.3
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Ownership: the caller allocates every host and device buffer; the
 *   library never allocates memory and never synchronises the device, except
 *   cp_device_error_check(), which reads a device status word.
 * - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy
 *   default stream).  All device work is enqueued on it, in order.
 * - Errors: every entry point validates its arguments on the host and returns
 *   a cp_status before launching anything; on error nothing is enqueued and
 *   cp_last_error() returns a message for the calling thread.
 * - LSE is the natural logarithm of the sum of exponentiated (scaled)
 *   scores ([CTX] §3.3).  An empty key set has O = 0 and LSE = -inf.
 * - Tensors are dense, row-major, with the innermost dimension last.
 *   Device pointers must be 16-byte aligned.
 * - Kernels never wait without a bound: an mbarrier wait that runs past its
 *   iteration limit sets a device status word and the kernel returns;
 *   cp_device_error_check() then reports CP_ERR_DEVICE_TIMEOUT.
 */
#ifndef CPATTN_H
#define CPATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CPATTN_VERSION 1
#define CP_PLAN_MAGIC 0x4c504350 /* 'CPPL' */
#define CP_MAX_SHARDS 64         /* C limit: per-shard pointers travel as kernel arguments */

typedef enum {
  CP_OK = 0,
  CP_ERR_INVALID_ARG = -1,    /* a null pointer, a bad size, a misaligned pointer */
  CP_ERR_UNSUPPORTED = -2,    /* a valid combination this build does not implement */
  CP_ERR_CUDA = -3,           /* a CUDA runtime/driver call failed (message has details) */
  CP_ERR_DEVICE_TIMEOUT = -4, /* a kernel gave up a bounded wait (see cp_device_error_check) */
  CP_ERR_WORKSPACE = -5       /* the workspace passed is too small */
} cp_status;

typedef enum { CP_ZIGZAG = 0, CP_INTERLEAVE = 1 } cp_strategy;
typedef enum { CP_BF16 = 0, CP_FP32 = 1, CP_FP8_E4M3 = 2 } cp_dtype;
typedef enum { CP_DECODE_GQA = 0, CP_DECODE_MLA = 1 } cp_decode_mode;
/* Which decode shard holds token p of a request of L cached tokens. */
typedef enum {
  CP_DCP_ROUND_ROBIN = 0, /* shard p mod C, row p / C ([CTX] §3.1; [V4] §5) */
  CP_DCP_CONTIGUOUS = 1,  /* C consecutive chunks, the first L mod C one token longer ([DCP] §4) */
  CP_DCP_SELECTED = 2     /* selection buffers of a sparse decode (cp_sparse_plan only) */
} cp_dcp_layout;

/* ---------------------------------------------------------------------------
 * Plan layout.  A plan is an array of int32 words: a cp_plan_header, then
 * tables at the word offsets the header gives.  The host part (header and
 * tables) is written by the host into `host_plan` and copied, in stream
 * order, to the front of `dev_plan`; per-token arrays exist only in
 * `dev_plan` and are written there by a device kernel.
 * ------------------------------------------------------------------------- */
typedef struct {
  int32_t magic;      /* CP_PLAN_MAGIC */
  int32_t kind;       /* 0 zigzag prefill, 1 interleave prefill, 2 decode */
  int32_t C;          /* number of virtual shards (ranks) */
  int32_t R;          /* number of requests */
  int32_t T;          /* prefill: total new tokens; decode: total cached tokens */
  int32_t KV;         /* prefill: total K/V rows = sum(prefix + new); decode: 0 */
  int32_t n_seg;      /* prefill: number of segments; decode: number of work items */
  int32_t n_tiles;    /* prefill: number of 256-query tiles; decode: number of workers */
  int32_t off_rank;   /* prefill: int32 rank_off[C+1]; decode: cp_pair_desc[C*R] */
  int32_t off_req;    /* prefill: cp_req_desc[R]; decode: int32 worker_off[n_workers+1] */
  int32_t off_seg;    /* prefill: cp_seg_desc[n_seg]; decode: cp_work_desc[n_seg] */
  int32_t off_tiles;  /* prefill: cp_tile_desc[n_tiles], all ranks, longest first */
  int32_t off_rtile;  /* prefill: int32 rank_tile_off[C+1] + cp_tile_desc[n_tiles] by rank */
  int32_t off_idx;    /* prefill, device only: int32 idx[T]  (flattened new-token index) */
  int32_t off_qpos;   /* prefill, device only: int32 qpos[T] (position incl. prefix) */
  int32_t off_qreq;   /* prefill, device only: int32 qreq[T] (request of the query) */
  int32_t host_words; /* words in the host part */
  int32_t dev_words;  /* words in the device plan */
  int32_t n_parts;    /* decode: partial slots in the workspace (split pairs) */
  int32_t tile_rows;  /* decode: KV rows per scheduling tile (work boundaries) */
  int32_t n_split;    /* decode: pairs covered by more than one work item */
  int32_t layout;     /* decode: cp_dcp_layout of the token shards */
  int32_t s_q;        /* decode: query rows per request (1, or more for MTP) */
  int32_t off_run;    /* decode: the merged-output run table (cp_decode_attn_merged) */
} cp_plan_header;
/* Decode plans reuse the table offsets: off_tiles -> int32 [R][2]
 * {ctx_len, first token of the request in the token-ordered cache};
 * off_rtile -> int32 split_pairs[n_split]. */

/* One request of a prefill batch. */
typedef struct {
  int32_t new_len;    /* newly extended tokens (queries) */
  int32_t prefix_len; /* cached prefix read by every query of the request */
  int32_t q_base;     /* flattened index of the request's first new token */
  int32_t kv_base;    /* first K/V row of the request (prefix, then new tokens) */
} cp_req_desc;

/* A run of one rank's queries inside one request: a zigzag block, or the
 * C-strided interleave run.  Segments are ordered by (rank, local_start). */
typedef struct {
  int32_t rank;        /* owning virtual shard */
  int32_t req;         /* request index */
  int32_t block;       /* zigzag: block 0..2C-1; interleave: -1 */
  int32_t which;       /* zigzag: 0 early block, 1 late block; interleave: 0 */
  int32_t local_start; /* first row of the segment in the rank-major output */
  int32_t count;       /* queries in the segment (q_len) */
  int32_t first_f;     /* flattened new-token index of its first query */
  int32_t stride;      /* flattened-index step between its queries: 1 or C */
  int32_t q_start;     /* offset of its first query within the request's new tokens */
  int32_t first_pos;   /* position of its first query, prefix included */
  int32_t kv_len;      /* keys read by its last query (zigzag: prefix + block end);
                          0 for an empty interleave run */
  int32_t kv_base;     /* first K/V row of the request */
} cp_seg_desc;

/* A tile of up to 256 consecutive queries of one segment. */
typedef struct {
  int32_t seg;   /* segment index */
  int32_t q_off; /* offset of the tile's first query within the segment */
} cp_tile_desc;

/* Decode: one (shard r, request b) pair; pair index = r * R + b. */
typedef struct {
  int32_t rows;       /* tokens of request b stored on shard r (round robin: ceil((L_b - r) / C)) */
  int32_t row_off;    /* first row of request b in shard r's cache */
  int32_t ctx_len;    /* L_b, the request's cached tokens */
  int32_t n_parts;    /* work items that cover this pair (>1: merged from the workspace) */
  int32_t first_part; /* first workspace slot of this pair when n_parts > 1, else -1 */
  int32_t tok0;       /* token (position in the request) of the pair's row 0 */
  int32_t tok_step;   /* token distance between consecutive rows: C or 1 */
  int32_t reserved;
} cp_pair_desc;

/* Decode: a contiguous row range of one pair, processed by one worker. */
typedef struct {
  int32_t pair;      /* pair index */
  int32_t row_begin; /* first row within the pair */
  int32_t row_end;   /* one past the last row within the pair */
  int32_t part;      /* workspace slot, or -1 when the item covers the whole pair */
} cp_work_desc;

/* ---------------------------------------------------------------------------
 * Library state
 * ------------------------------------------------------------------------- */

/* Message of the last failed call on this thread ("" if none). */
const char* cp_last_error(void);

/* CPATTN_VERSION of the loaded library. */
int cp_version(void);

/* Reads (and clears) the device status word that bounded waits set.  Blocks
 * until `stream` has drained.  CP_OK, or CP_ERR_DEVICE_TIMEOUT with the
 * failing kernel and wait site in cp_last_error(). */
cp_status cp_device_error_check(void* stream);

/* ---------------------------------------------------------------------------
 * cp_shard_plan — prompt-token shard maps.
 *
 * Zigzag ([CTX] §2.3 "Zigzag"; [SGL] "Zigzag strategy"): each request's
 * new_len[j] new tokens are cut into 2C contiguous blocks; block sizes are
 * floor(n/2C), plus one for the first n mod 2C blocks (early blocks receive
 * the remainder); rank r takes blocks r and 2C-1-r; the split restarts for
 * every request.  A block's queries read the cached prefix and every new
 * token up to themselves, so its kv length is prefix_len[j] + block end.
 *
 * Interleave ([CTX] §2.4 "Interleave"; [SGL] "Interleave strategy"): the new
 * tokens of all requests are flattened (f = 0..T-1, no reset at request
 * boundaries) and rank r owns f = r, r+C, r+2C, ...; a query keeps its
 * position in its request, prefix included, and reads keys 0..position.
 *
 * Local order: rank-major.  Rank r's queries occupy rows
 * [rank_off[r], rank_off[r+1]) of every per-rank output; within a rank,
 * zigzag orders request by request, early block then late block, and
 * interleave orders by ascending f.
 *
 * cp_plan_size: host and device plan sizes in bytes for this batch.
 * cp_shard_plan: writes the host part into host_plan (host_bytes), copies it
 *   to dev_plan (dev_bytes, device memory) on `stream` and launches the
 *   kernel that fills idx/qpos/qreq.  If host_plan is pinned memory the copy
 *   is asynchronous: keep host_plan unchanged until the stream passes it.
 * Arguments: strategy; C in [1, CP_MAX_SHARDS]; R >= 1 requests;
 *   new_len[R] >= 0, prefix_len[R] >= 0 (host arrays); totals < 2^31.
 * ------------------------------------------------------------------------- */
cp_status cp_plan_size(cp_strategy strategy, int C, int R, const int32_t* new_len,
                       const int32_t* prefix_len, size_t* host_bytes, size_t* dev_bytes);
cp_status cp_shard_plan(cp_strategy strategy, int C, int R, const int32_t* new_len,
                        const int32_t* prefix_len, void* host_plan, size_t host_bytes,
                        void* dev_plan, size_t dev_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * cp_prefill_attn — causal GQA prefill for every query a rank owns.
 *
 * For each owned query at position p of request j and each q head h, with
 * kv head g = h / (Hq / Hkv) (consecutive grouping):
 *   s_t = sm_scale * <q_h, k_{t,g}> for t = 0..p  (keys up to and including
 *   itself, [CTX] §1.1; the prefix and the request's new tokens);
 *   LSE = ln sum_t exp(s_t);  O = sum_t exp(s_t - LSE) v_{t,g}.
 * With virtual shards the KV all-gather of [CTX] §2.1 is the identity: every
 * rank reads the same global K/V buffers.
 *
 * q   [T, Hq, D]    flattened new-token order, dtype `dtype`
 * k,v [KV, Hkv, D]  per request: prefix rows then new-token rows
 * o   [rows, Hq, D] same dtype as q; rows = T (rank = -1, rank-major order)
 *                   or rank r's count (rank = r, its local order)
 * lse [rows, Hq]    fp32
 * dtype: CP_BF16 (tensor cores, bf16 products; D in {64, 128}) or CP_FP32
 *   (D <= 128, D % 32 == 0): at D = 64 or 128 on the tensor cores as tf32
 *   products (fp32 values read with a 10-bit mantissa, fp32 accumulation),
 *   at D = 32 or 96 on the CUDA cores.  Hq % Hkv == 0.  host_plan and
 *   dev_plan come from cp_shard_plan (the host part is read for the launch
 *   shape).
 * ------------------------------------------------------------------------- */
cp_status cp_prefill_attn(const void* host_plan, const void* dev_plan, int rank, cp_dtype dtype,
                          const void* q, const void* k, const void* v, int Hq, int Hkv, int D,
                          float sm_scale, void* o, float* lse, void* stream);

/* ---------------------------------------------------------------------------
 * cp_decode_plan — decode KV-cache token shards and split-KV schedule.
 *
 * Token p of request b lives on shard p mod C at row p / C ([CTX] §3.1
 * "Storing each token once": gpu = slot % C, row = slot // C; [V4] §5
 * owner(j) = j mod P).  Shard r holds rows_{r,b} = ceil((L_b - r)/C) rows of
 * request b, requests back to back (row_off).  The work of all (r, b) pairs,
 * walked request by request, is cut into contiguous row ranges over
 * `n_workers` CTAs (0 = the SM count of the current device), balanced in
 * 128-row tiles plus a fixed two-tile cost per work item; a pair split over
 * several workers gets workspace slots that cp_decode_attn merges exactly.
 *
 * Arguments: C in [1, CP_MAX_SHARDS]; B >= 1; ctx_len[B] >= 0 host array.
 * ------------------------------------------------------------------------- */
cp_status cp_decode_plan_size(int C, int B, const int32_t* ctx_len, int n_workers,
                              size_t* host_bytes, size_t* dev_bytes);
cp_status cp_decode_plan(int C, int B, const int32_t* ctx_len, int n_workers, void* host_plan,
                         size_t host_bytes, void* dev_plan, size_t dev_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * cp_decode_plan_ex — cp_decode_plan with a choice of shard layout and
 * several query rows per request.
 *
 * layout CP_DCP_ROUND_ROBIN is cp_decode_plan's map.  CP_DCP_CONTIGUOUS
 *   gives shard r one chunk of consecutive tokens (the example of [DCP] §4:
 *   four GPUs holding tokens 0-50K, 50K-100K, ... of one request): with
 *   L = C q + m, shards r < m hold
 *   q + 1 tokens and the others q, in token order, so token p of shard r sits
 *   at row p - (r q + min(r, m)).  The merged result is the same for both
 *   layouts (the exact combine does not depend on the partition).
 * s_q >= 1 query rows per request ([V4] §2.2: MTP or speculative decode
 *   raises the query rows per request above one).  Query row i of request b
 *   stands at position L_b - s_q + i and reads the cached tokens 0 ..
 *   L_b - s_q + i (the s_q new tokens are already in the cache, the last
 *   one read by the last row only); every request then needs L_b >= s_q.
 *   cp_decode_attn takes q [B, s_q, H, Dqk] and writes o_part
 *   [C, B, s_q, H, Dv], lse_part [C, B, s_q, H]; the MLA kernels treat the
 *   s_q H query rows as their columns (s_q H <= 64) and read each cache row
 *   once for all of them.
 * Shard sizes per pair, the split-KV schedule and the pack map follow the
 *   layout; cp_kv_shard_pack(_paged) and the paged entry points accept
 *   these plans unchanged.
 * Errors: CP_ERR_INVALID_ARG for a layout outside the enum, s_q < 1 or
 *   s_q > 64, or a request with L_b < s_q when s_q > 1.
 * ------------------------------------------------------------------------- */
cp_status cp_decode_plan_ex_size(int C, int B, const int32_t* ctx_len, cp_dcp_layout layout, int s_q,
                                 int n_workers, size_t* host_bytes, size_t* dev_bytes);
cp_status cp_decode_plan_ex(int C, int B, const int32_t* ctx_len, cp_dcp_layout layout, int s_q,
                            int n_workers, void* host_plan, size_t host_bytes, void* dev_plan,
                            size_t dev_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * cp_kv_shard_pack — copy a token-ordered cache into its token shards
 * (the decode side's store of [CTX] §5 case C: each decode GPU keeps only the
 * tokens it owns).
 *
 * kv        [sum_b L_b, row_elems] device, requests back to back, dtype `dtype`
 * kv_scale  [sum_b L_b] fp32 per-token scales, or NULL (copied when non-NULL)
 * shard_kv  host array of C device pointers; shard r: [sum_b rows_{r,b}, row_elems]
 * shard_scale host array of C device pointers (fp32 [sum_b rows_{r,b}]) or NULL
 * Row bytes (row_elems * element size) must be a multiple of 16.
 * ------------------------------------------------------------------------- */
cp_status cp_kv_shard_pack(const void* host_plan, const void* dev_plan, cp_dtype dtype,
                           const void* kv, const float* kv_scale, int row_elems,
                           void* const* shard_kv, float* const* shard_scale, void* stream);

/* ---------------------------------------------------------------------------
 * cp_decode_attn — one decode query per request against every shard.
 *
 * For shard r and request b, the same attention as cp_prefill_attn restricted
 * to the tokens stored on shard r ([CTX] §3.2, §3.4 step 3), giving a partial
 * (O_r, LSE_r); merging the C partials with cp_lse_merge gives the
 * attention over the whole cache ([CTX] §3.3; [V4] §5).
 *
 * With a plan of s_q > 1 query rows (cp_decode_plan_ex) q is [B, s_q, H, Dqk]
 * and the outputs [C, B, s_q, H, ...]: below, read B as B s_q rows.
 *
 * mode CP_DECODE_MLA: one latent KV head shared by all H <= 64 query heads
 *   (s_q H <= 64)
 *   ([CTX] §1.3; [DCP] §5.3), on the tensor cores.  Dqk = 576, Dv = 512,
 *   Hkv = 1: keys are the whole
 *   576-dim entry, values its first 512 dims ([GLM] footnote 1).
 *   q [B, H, 576] bf16; shard_k[r] [rows_r, 576] as kv_dtype CP_BF16, or
 *   CP_FP8_E4M3 codes with shard_scale[r] [rows_r] fp32 (value = code *
 *   scale); shard_v must be NULL.  FP8 codes must be finite (0x7F and 0xFF
 *   are NaN in E4M3 and propagate), scales finite and >= 0.  The FP8 path
 *   multiplies the codes on the tensor cores as they are stored; the bf16
 *   query and the softmax weights enter those products as pairs of E4M3
 *   numbers whose sum keeps 8 significant bits (see the kernel's notes).
 * mode CP_DECODE_GQA: q [B, Hq, D] and shard_k[r], shard_v[r]
 *   [rows_r, Hkv, D], all of kv_dtype CP_BF16 or CP_FP32 (shard_scale NULL),
 *   or shard_k/shard_v E4M3 codes (CP_FP8_E4M3, q bf16) with
 *   shard_scale[r] [rows_r] fp32, one scale per token for both its K and V
 *   rows (k = code x scale, v = code x scale); Dqk = Dv = D, D % 32 == 0,
 *   D <= 256.  Which kernel runs (the results agree within the bf16
 *   tolerance either way; Hq = Hkv, plain multi-head attention, included):
 *   - FP8 cache, D = 128, at most 32 query columns per kv head
 *     ((Hq/Hkv) s_q), per-shard buffers: tensor cores, FP8 products on the
 *     codes as stored (query and weights as E4M3 hi + lo pairs);
 *   - bf16 cache, D = 64 or 128, at most 64 query columns per kv head, per
 *     shard or paged: tensor cores, bf16 products;
 *   - fp32 cache, D = 64 or 128, at most 64 query columns per kv head,
 *     per-shard buffers: tensor cores, tf32 products;
 *   - every other shape (other head dims, more query columns per kv head, a
 *     paged FP8 or fp32 pool): CUDA cores.
 * o_part [C, B, H, Dv] fp32 and lse_part [C, B, H] fp32 (normalised partial
 *   outputs; an empty shard gives O = 0, LSE = -inf).
 * ws: workspace of cp_decode_workspace_size() bytes (NULL if that is 0).
 * ------------------------------------------------------------------------- */
cp_status cp_decode_workspace_size(const void* host_plan, int H, int Dv, size_t* bytes);
cp_status cp_decode_attn(const void* host_plan, const void* dev_plan, cp_decode_mode mode,
                         cp_dtype kv_dtype, const void* q, const void* const* shard_k,
                         const void* const* shard_v, const float* const* shard_scale, int Hq,
                         int Hkv, int Dqk, int Dv, float sm_scale, float* o_part, float* lse_part,
                         void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * cp_decode_attn_merged — cp_decode_attn followed by cp_lse_merge over the C
 * partials, in one call: o [B, H, Dv] (o_dtype CP_BF16 or CP_FP32) and
 * lse [B, H] fp32 (natural log), the attention over each request's whole
 * cache ([CTX] §3.3; [V4] §5).  Arguments as for cp_decode_attn.
 *
 * With an MLA cache (FP8 or bf16, per-shard buffers) the partials never
 * leave the GPU's tensor memory where they need not: the plan's run table (the header's
 * off_run, built with every decode plan) groups each worker's consecutive
 * work items of one request into a run, and the run accumulates all of them
 * (the shards' partial softmax combines exactly across them, as in the
 * merge).  A run holding all of its request's rows writes the result; the
 * runs of a request cut by a worker boundary write fp32 parts, which a merge
 * combines.  Short requests, whose C shards fit in one worker, then cost no
 * partial at all.  GQA caches run cp_decode_attn into the workspace and
 * merge there.
 *
 * Run table at off_run (int32): n_parts, n_list, then run_out[n_work] (per
 * work item: -1 the run goes on to the worker's next item, -2 the last item
 * of a run holding its whole request, k >= 0 the last item of a run that is
 * one of its request's parts, written to part slot k, -3 an empty pair's
 * item), then n_list entries {request, first part slot, parts} (a request's
 * parts are consecutive slots; a request with no rows is listed with none
 * and gets O = 0, LSE = -inf).
 * ws: cp_decode_merged_workspace_size() bytes (NULL if 0).  Errors as for
 * cp_decode_attn; CP_ERR_INVALID_ARG also for a selection plan.
 * ------------------------------------------------------------------------- */
cp_status cp_decode_merged_workspace_size(const void* host_plan, cp_decode_mode mode, cp_dtype kv_dtype,
                                          int H, int Dv, size_t* bytes);
cp_status cp_decode_attn_merged(const void* host_plan, const void* dev_plan, cp_decode_mode mode,
                                cp_dtype kv_dtype, const void* q, const void* const* shard_k,
                                const void* const* shard_v, const float* const* shard_scale, int Hq,
                                int Hkv, int Dqk, int Dv, float sm_scale, void* o, cp_dtype o_dtype,
                                float* lse, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Sparse decode with an exact sharded top-k ("DeepSeek-V4 Attention
 * Inference Systems" §5.2; [CTX] §4.1, the index split with the cache).
 *
 * Each shard holds the relevance scores of the tokens it stores (the output
 * of its local index scan; the scoring function belongs to the model and is
 * an input here) and the steps run as the pages list them:
 *   cp_sparse_topk    every (shard, request) pair keeps its k best tokens,
 *                     then the at most C k candidates of a request give the
 *                     exact global top-k (the union of the local top-k lists
 *                     contains it, so nothing is approximated);
 *   cp_sparse_gather  every owner packs the cache rows of the selected tokens
 *                     it stores into its selection buffer (route to owners);
 *   cp_sparse_decode_attn  every owner attends to its selected rows; the
 *                     partials merge exactly with cp_lse_merge.
 * Order: higher score first; equal scores by lower token index (the pages
 * ask only for deterministic ties).  Scores must not be NaN.
 *
 * cp_sparse_topk: host_plan/dev_plan = the cache's decode plan (any layout,
 *   one query row); shard_scores[r] fp32 [rows_r] device, shard r's scores in
 *   the plan's row order; k in [1, 4096].  Writes sel_ids [B][k] int32 (the
 *   selected token indices of request b in increasing order, -1 past the
 *   count) and sel_count [B] = min(k, L_b).  ws: cp_sparse_workspace_size()
 *   bytes, 16-byte aligned; it keeps the candidates for cp_sparse_gather.
 * cp_sparse_gather: after cp_sparse_topk with the same plan, k and ws.
 *   shard_kv[r] [rows_r, row_elems] (and shard_scale[r] fp32 [rows_r] or
 *   NULL) as packed by cp_kv_shard_pack; sel_kv[r] [B kp, row_elems] (and
 *   sel_scale[r] [B kp]), kp = CP_SPARSE_SLOT_ROWS(k), receive the selected
 *   rows of request b at rows b kp .. b kp + pair_count[r B + b] - 1, in
 *   token order, and zeros up to the next multiple of 128 rows (the decode
 *   reads whole 128-row tiles; a row past the count enters with weight 0 and
 *   must hold finite values); pair_count [C B] int32 device.  Call once per
 *   array (K and V for GQA).
 * cp_sparse_plan: the decode plan over those selection buffers (room for kp
 *   rows per pair; the rows in use are pair_count's, read on the device).
 * cp_sparse_decode_attn: cp_decode_attn over the selection buffers with
 *   that plan and pair_count; same shapes and outputs (o_part [C, B, H, Dv],
 *   lse_part [C, B, H]); ws: cp_decode_workspace_size(sparse plan).
 * Errors: CP_ERR_INVALID_ARG for k outside [1, 4096], a selection plan given
 *   to top-k or a cache plan to the sparse attention, NULL or misaligned
 *   pointers; CP_ERR_UNSUPPORTED for a plan with s_q > 1; CP_ERR_WORKSPACE.
 * ------------------------------------------------------------------------- */
#define CP_SPARSE_SLOT_ROWS(k) ((((k) + 127) / 128) * 128)
cp_status cp_sparse_workspace_size(const void* host_plan, int k, size_t* bytes);
cp_status cp_sparse_topk(const void* host_plan, const void* dev_plan, const float* const* shard_scores,
                         int k, int32_t* sel_ids, int32_t* sel_count, void* ws, size_t ws_bytes,
                         void* stream);
cp_status cp_sparse_gather(const void* host_plan, const void* dev_plan, int k, const void* ws,
                           size_t ws_bytes, cp_dtype dtype, const void* const* shard_kv,
                           const float* const* shard_scale, int row_elems, void* const* sel_kv,
                           float* const* sel_scale, int32_t* pair_count, void* stream);
cp_status cp_sparse_plan_size(int C, int B, int k, int n_workers, size_t* host_bytes,
                              size_t* dev_bytes);
cp_status cp_sparse_plan(int C, int B, int k, int n_workers, void* host_plan, size_t host_bytes,
                         void* dev_plan, size_t dev_bytes, void* stream);
cp_status cp_sparse_decode_attn(const void* host_plan, const void* dev_plan, const int32_t* pair_count,
                                cp_decode_mode mode, cp_dtype kv_dtype, const void* q,
                                const void* const* sel_k, const void* const* sel_v,
                                const float* const* sel_scale, int Hq, int Hkv, int Dqk, int Dv,
                                float sm_scale, float* o_part, float* lse_part, void* ws,
                                size_t ws_bytes, void* stream);
/* cp_sparse_decode_attn_merged: cp_sparse_decode_attn and cp_lse_merge of
 * its partials in one call, as cp_decode_attn_merged: o [B, H, Dv] (o_dtype
 * CP_BF16 or CP_FP32), lse [B, H]; ws: cp_decode_merged_workspace_size(the
 * sparse plan) bytes.  Over MLA selections the owners' items of one request
 * combine in tensor memory. */
cp_status cp_sparse_decode_attn_merged(const void* host_plan, const void* dev_plan, const int32_t* pair_count,
                                       cp_decode_mode mode, cp_dtype kv_dtype, const void* q,
                                       const void* const* sel_k, const void* const* sel_v,
                                       const float* const* sel_scale, int Hq, int Hkv, int Dqk, int Dv,
                                       float sm_scale, void* o, cp_dtype o_dtype, float* lse, void* ws,
                                       size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Paged token-sharded decode cache ("How GPUs Share a Long Context During LLM
 * Inference" §3.1: a slot maps to (GPU, row); serving caches keep those rows
 * in fixed-size pages, "DeepSeek-V4 Attention Inference Systems" §9.2).
 *
 * The rows of pair (shard r, request b) = pair index r * R + b of a decode
 * plan are the shard's rows of that request in order (row i = token
 * p = i * C + r).  Row i lives at row i % page_size of page
 * page_table[pair][i / page_size] of one pool shared by all shards:
 *   pool row = page_id * page_size + i % page_size,
 *   pool: [num_pages * page_size, row] with row = 576 (MLA) or Hkv x D (GQA).
 * page_table: int32 [C * R][max_pages], a host copy (validated: page ids in
 *   [0, num_pages), ceil(rows / page_size) <= max_pages) and a device copy
 *   (read by the kernels; must hold the same ids).  page_size is a multiple
 *   of 64.  Entries past a pair's pages are ignored.
 * Rows past a pair's last row on its last page enter the decode products
 * with zero weight and must hold finite values; cp_kv_shard_pack_paged
 * zeroes them.
 * ------------------------------------------------------------------------- */

/* cp_kv_shard_pack_paged — cp_kv_shard_pack into a paged pool: token p of
 * request b goes to shard p mod C, row p / C, at the pool row its page table
 * gives; then the tail rows of every pair's last page are zeroed.  No page
 * may be used by two pairs.  pool / scale_pool (FP8: one fp32 scale per pool
 * row, or NULL with kv_scale NULL) are caller-owned device buffers. */
cp_status cp_kv_shard_pack_paged(const void* host_plan, const void* dev_plan, cp_dtype dtype,
                                 const void* kv, const float* kv_scale, int row_elems, void* pool,
                                 float* scale_pool, const int32_t* host_page_table,
                                 const int32_t* dev_page_table, int max_pages, int page_size,
                                 int num_pages, void* stream);

/* cp_decode_attn_paged — cp_decode_attn over a paged pool: the same partials
 * (O_r, LSE_r), with shard_k / shard_v / shard_scale replaced by k_pool,
 * v_pool (GQA; NULL for MLA) and scale_pool (FP8; NULL otherwise). */
cp_status cp_decode_attn_paged(const void* host_plan, const void* dev_plan, cp_decode_mode mode,
                               cp_dtype kv_dtype, const void* q, const void* k_pool,
                               const void* v_pool, const float* scale_pool,
                               const int32_t* host_page_table, const int32_t* dev_page_table,
                               int max_pages, int page_size, int num_pages, int Hq, int Hkv,
                               int Dqk, int Dv, float sm_scale, float* o_part, float* lse_part,
                               void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * cp_lse_merge — exact combine of P partial results ([CTX] §3.3; [V4] §5).
 *
 * Per (n, h): g = max_p LSE_p; w_p = exp(LSE_p - g) (0 for LSE_p = -inf);
 * O = sum_p w_p O_p / sum_p w_p; LSE = g + ln sum_p w_p.  If every part is
 * empty, O = 0 and LSE = -inf.
 * o_part [P, N, H, Dv] fp32; lse_part [P, N, H] fp32;
 * o [N, H, Dv] of o_dtype CP_BF16 or CP_FP32; lse [N, H] fp32 or NULL.
 * P in [1, CP_MAX_SHARDS]; Dv % 4 == 0.
 * ------------------------------------------------------------------------- */
cp_status cp_lse_merge(int P, int N, int H, int Dv, const float* o_part, const float* lse_part,
                       void* o, cp_dtype o_dtype, float* lse, void* stream);

/* ---------------------------------------------------------------------------
 * cp_lse_fold — exact combine of one partial into another, in place:
 * (O, LSE) <- combine((O, LSE), (O_add, LSE_add)) with the weights of
 * cp_lse_merge ([V4] §5).  The designated-rank rule of [V4] §5.3: a window
 * (or sink) cache that every shard holds a copy of is attended once, as its
 * own partial, and folded into exactly one shard's partial, so its
 * probability mass is counted once when the shards are merged.
 * o, o_add [N, H, Dv] fp32; lse, lse_add [N, H] fp32 (may alias nothing else).
 * ------------------------------------------------------------------------- */
cp_status cp_lse_fold(int N, int H, int Dv, float* o, float* lse, const float* o_add,
                      const float* lse_add, void* stream);

/* ---------------------------------------------------------------------------
 * cp_decode_attn_noalloc — cp_decode_attn for callers that cannot allocate.
 *
 * The pages have no counterpart: this is an interface convenience.  Some
 * callers cannot allocate device memory where they call the decode: serving
 * loops held to a fixed memory budget, and plugins reached through a C
 * interface that gives them no allocator.  This entry point takes the same arguments as
 * cp_decode_attn minus the workspace, and keeps the split-KV partial results
 * in a library-owned static device array of CP_NOALLOC_SCRATCH_BYTES.
 *
 * - Memory: the array is part of the loaded library; every GPU that loads it
 *   holds the array until the process exits.  Nothing is allocated per call.
 * - Limit: a plan that needs more scratch than the array
 *   (cp_decode_workspace_size > CP_NOALLOC_SCRATCH_BYTES) is rejected with
 *   CP_ERR_WORKSPACE and a message; nothing is launched.
 * - Sharing: all calls use the same array and it keeps the last call's
 *   contents; nothing in it needs to start at zero (each slot is fully written
 *   before it is read within one call).  Calls that overlap on the GPU race
 *   on the array: serialise them on one stream.
 * - Device: the array used is the current device's; q must live on the
 *   current device, else CP_ERR_INVALID_ARG.
 * - Set-up: every call on a stream that is not capturing looks up the array's
 *   device address (cudaGetSymbolAddress, the current device) and caches it
 *   per device, so a context torn down and re-created (cudaDeviceReset) never
 *   leaves a stale address; a call on a capturing stream uses that cache, so
 *   the first call on a device must come before any stream capture begins
 *   (else CP_ERR_CUDA).
 * ------------------------------------------------------------------------- */
#define CP_NOALLOC_SCRATCH_BYTES (16u << 20) /* 16 MiB per device */
/* The array's size in bytes (CP_NOALLOC_SCRATCH_BYTES of the built library). */
size_t cp_noalloc_scratch_bytes(void);
cp_status cp_decode_attn_noalloc(const void* host_plan, const void* dev_plan, cp_decode_mode mode,
                                 cp_dtype kv_dtype, const void* q, const void* const* shard_k,
                                 const void* const* shard_v, const float* const* shard_scale,
                                 int Hq, int Hkv, int Dqk, int Dv, float sm_scale, float* o_part,
                                 float* lse_part, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CPATTN_H */
