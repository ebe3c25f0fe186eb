/*
 * pkvd.h -- paged-KV split-KV decode attention on GB300 (sm_103a): C ABI.
 *
 * The new query token(s) of each request are scored against that request's
 * paged KV cache. The work is cut into splits along the sequence; each split
 * runs an online softmax over its tokens and leaves a normalised P.V partial
 * with its log-sum-exp, and a second kernel merges the splits of every
 * (request, query token, head). With one query token per request the
 * operation is
 *
 *     out[b,h,:] = sum_t softmax_t(scale * q[b,h,:] . K[row(b,t,kv),:]) * V[row(b,t,kv),:Dv]
 *     lse[b,h]   = ln sum_t exp(scale * q[b,h,:] . K[row(b,t,kv),:])
 *
 * over t = 0 .. L_b - 1, with kv = h / (heads / kv_heads) and row(b,t,kv) =
 * (page_table[b][t/ps] * kv_heads + kv) * ps + t % ps. With q_len > 1 query
 * tokens per request (draft tokens verified in one step), the request's last
 * q_len positions are its queries, already written to the cache: query token
 * j (0-based) sits at position L_b - q_len + j and its sums run over
 * t = 0 .. L_b - q_len + j only (causal among the new tokens). Sources for
 * the pieces:
 *   - the split policy, the split-major grid and the head-dim-tiled merge:
 *     aiter pull 4758, "[Gluon][MLA] Deeper async-copy pipeline in the bh16
 *     stage-1 decode loop", Motivation and Technical Details 1-3;
 *   - several keys per warp and xor-fold warp sums for the scores:
 *     TensorFold pull 1932, "What this changes";
 *   - the bank-conflict-free shared-memory pitch for K/V tiles:
 *     ROCm/rocm-libraries pull 10102 (attention_dense LDS group padding),
 *     Motivation and Technical Details.
 *
 * Two families:
 *   GQA  head_dim D in {128, 256}, head_dim_v == D, heads / kv_heads from 1
 *        to 16 (the FMA variant: 1, 2, 4 or 8); K and V in separate pools.
 *   MLA  head_dim 576 (512 no-rope + 64 rope), head_dim_v 512, kv_heads 1,
 *        heads a multiple of 16; V is the first 512 elements of the same
 *        576-wide row (pass v_pages == k_pages, both row pitches equal).
 *
 * Layouts (row-major, contiguous unless a pitch says otherwise):
 *   q          [batch, q_len, heads, head_dim]            bf16 or fp16
 *   k_pages    [num_pool_pages, kv_heads, page_size, k_row_pitch]
 *   v_pages    [num_pool_pages, kv_heads, page_size, v_row_pitch]
 *   page_table [batch, max_pages_per_seq]                  int32 page ids
 *   out        [batch, q_len, heads, head_dim_v]           fp32
 *   lse        [batch, q_len, heads]                       fp32, natural log
 * Every device pointer must be 16-byte aligned, and each row pitch times the
 * element size a multiple of 16 bytes.
 *
 * Ownership. The caller owns every tensor above. A plan owns its device work
 * list and its partial workspace, allocated when the plan is made and freed
 * by decode_plan_destroy. A plan holds a copy of seq_lens and is valid only
 * for those lengths (and for the shapes it was made with): re-plan when they
 * change.
 *
 * Errors. Every call returns a pkvd_status (0 = success) and never aborts.
 * decode_run is asynchronous: it reports argument and launch errors only.
 * Faults the kernels detect themselves (with checks on: a page id outside
 * the pool, or members of a shared-prefix group whose prefix pages differ;
 * always: a pipeline wait that ran out) are recorded in a device status word
 * and come back from decode_last_device_status.
 *
 * Streams. decode_run enqueues work on the given stream and neither
 * allocates nor synchronises, so it can be captured in a CUDA graph.
 */
#ifndef PKVD_H_
#define PKVD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkvd_plan pkvd_plan;          /* opaque; immutable once made */
typedef struct CUstream_st *pkvd_stream_t;   /* a cudaStream_t; NULL = legacy default stream */
typedef struct CUevent_st *pkvd_event_t;     /* a cudaEvent_t */

typedef enum pkvd_status {
  PKVD_OK = 0,
  PKVD_EINVAL = -1,         /* bad argument: null pointer, size, alignment  */
  PKVD_EUNSUPPORTED = -2,   /* valid but unsupported shape or dtype         */
  PKVD_ECUDA = -3,          /* a CUDA runtime call failed                   */
  PKVD_ENOMEM = -4,         /* host or device allocation failed             */
  PKVD_EDEVICE_CHECK = -5,  /* a kernel's page-id check failed (checks on)  */
  PKVD_ETIMEOUT = -6        /* a kernel's bounded pipeline wait ran out     */
} pkvd_status;

typedef enum pkvd_dtype { PKVD_BF16 = 0, PKVD_FP16 = 1 } pkvd_dtype;

typedef enum pkvd_family { PKVD_FAMILY_GQA = 0, PKVD_FAMILY_MLA = 1 } pkvd_family;

/* Stage-1 kernel variants. AUTO picks per shape. */
typedef enum pkvd_variant {
  PKVD_VARIANT_AUTO = 0,
  PKVD_VARIANT_GQA_FMA = 1,   /* fp32 FMA scores and P.V, four keys per warp pass  */
  PKVD_VARIANT_GQA_MMA = 2,   /* mma.sync m16n8k16: keys as M, the head group as N */
  PKVD_VARIANT_MLA_MMA = 3,   /* mma.sync, a block of 16 heads per work item       */
  PKVD_VARIANT_MLA_TC = 4     /* tcgen05 with tensor-memory accumulators, a block
                                 of 64 (query token, head) rows per work item,
                                 the last block of a request zero-padded when
                                 q_len * heads is not a multiple of 64; P is
                                 rounded to one 16-bit value, so it is taken
                                 (AUTO) and accepted (forced) only when every
                                 non-empty request has >= 1024 tokens; else
                                 PKVD_EUNSUPPORTED                              */
} pkvd_variant;

/* Order of stage-1 work items in the grid. Both orders compute the same
 * items with the same reduction order, so results are bit-identical. */
typedef enum pkvd_grid_order {
  PKVD_ORDER_AUTO = 0,          /* split-major when batch > 1              */
  PKVD_ORDER_SPLIT_MAJOR = 1,   /* item id = split-major over (s, b, unit) */
  PKVD_ORDER_REQUEST_MAJOR = 2  /* item id = request-major over (b, unit, s) */
} pkvd_grid_order;

/* Full plan description. Zero in an optional field means "default". */
typedef struct pkvd_plan_desc {
  int32_t batch;              /* requests, >= 1                                   */
  int32_t heads;              /* query heads per request                          */
  int32_t kv_heads;           /* KV heads (MLA: 1)                                 */
  int32_t head_dim;           /* D: 128, 256 (GQA) or 576 (MLA)                   */
  int32_t head_dim_v;         /* Dv: 0 = D for GQA, 512 for MLA                   */
  int32_t page_size;          /* tokens per page, >= 1                            */
  int32_t dtype;              /* pkvd_dtype of q, K and V                         */
  int32_t splits;             /* 0 = planner; > 0 = this many splits per request
                                 (fewer when a request has fewer tokens)         */
  int32_t grid_order;         /* pkvd_grid_order                                  */
  int32_t stage2_tiles;       /* 0 = planner; else 1, 2, 4 or 8 slices of Dv      */
  int32_t variant;            /* pkvd_variant                                     */
  int32_t checks;             /* 1 = kernels bounds-check page ids (needs
                                 num_pool_pages) and report via the status word  */
  int32_t num_sms;            /* 0 = query the device                             */
  int32_t ctas_per_sm;        /* 0 = query the occupancy of the chosen kernel     */
  int32_t min_chunk;          /* 0 = default: smallest split, in tokens           */
  int32_t q_len;              /* query tokens per request, 0 = 1; at most 8. Every
                                 non-empty request needs L_b >= q_len. GQA: the
                                 mma variant with q_len * heads / kv_heads <= 16
                                 (the FMA variant takes q_len 1 only); MLA: both
                                 variants; no shared-prefix plans                 */
  int64_t max_pages_per_seq;  /* page_table row stride; 0 = max ceil(L_b / ps)    */
  int64_t num_pool_pages;     /* pages in the pools; 0 = unknown (no checks)      */
  int64_t k_row_pitch;        /* elements between K rows; 0 = D (MLA: 576)        */
  int64_t v_row_pitch;        /* elements between V rows; 0 = Dv (MLA: 576)       */
  float scale;                /* 0 = 1 / sqrt(D)                                  */
  int32_t reserved2;          /* must be 0                                        */
} pkvd_plan_desc;

/* What the planner decided (decode_plan_query / decode_plan_compute). */
typedef struct pkvd_plan_info {
  int32_t family;             /* pkvd_family                                      */
  int32_t variant;            /* resolved pkvd_variant                            */
  int32_t grid_order;         /* resolved pkvd_grid_order                         */
  int32_t stage2_tiles;       /* resolved slices of Dv in the merge               */
  int32_t stage2_threads;     /* threads per merge block                          */
  int32_t num_sms;            /* SMs the plan fills                               */
  int32_t ctas_per_sm;        /* resident stage-1 blocks per SM                   */
  int32_t heads_per_unit;     /* (query token, head) rows one stage-1 item covers */
  int32_t units_per_request;  /* stage-1 items per (request, split)               */
  int32_t num_items;          /* stage-1 grid size                                */
  int32_t num_partial_rows;   /* sum over requests of their split counts          */
  int32_t max_splits;         /* largest split count of any request               */
  int64_t chunk;              /* tokens per split when uniform, else 0            */
  int64_t workspace_bytes;    /* device bytes the plan owns                       */
  int32_t block_tokens;       /* tokens per pipeline stage of the stage-1 kernel  */
  int32_t pipeline_stages;    /* shared-memory stages of the stage-1 kernel       */
  int32_t stage1_smem_bytes;  /* dynamic shared memory of a stage-1 block         */
  int32_t stage1_threads;     /* threads of a stage-1 block                       */
  int32_t kv_tiles;           /* 1: K/V pages move as whole 16-row TMA tiles
                                 (page size a multiple of 16, splits on 16-token
                                 boundaries); 0: one bulk copy per row            */
  int32_t num_prefix_items;   /* shared-prefix plans: grouped prefix items, run
                                 before the num_items per-request items; else 0  */
} pkvd_plan_info;

/* One stage-1 work item as the planner lays it out (decode_plan_compute). */
typedef struct pkvd_work_item {
  int32_t request;            /* b                                                */
  int32_t unit;               /* GQA: KV head; MLA: head block                    */
  int32_t split;              /* s, 0-based within the request                    */
  int32_t partial_row;        /* row of this split in the partial workspace      */
  int32_t tok_begin;          /* first logical token                              */
  int32_t tok_end;            /* one past the last logical token                 */
  int32_t grouped;            /* 1: a shared-prefix item: `request` is the first
                                 of `unit` consecutive requests whose heads fill
                                 the 64 query rows, `split` their prefix split,
                                 partial_row unused (each member's row is its
                                 first partial row + split); else 0              */
  int32_t query_pos;          /* L_b - q_len: query token j of the request sees the
                                 tokens t <= query_pos + j                       */
} pkvd_work_item;

/* GQA shorthand of decode_plan_ex (head_dim_v = head_dim, bf16, all other
 * fields default); head_dim 576 selects the MLA family (Dv 512, pitches 576).
 * seq_lens: host array of `batch` lengths, copied. splits: 0 = planner.
 * Defined by: aiter pull 4758, Motivation (the split count per request, about
 * 256 / batch on that part, trades loop length against parallelism). */
int decode_plan(pkvd_plan **out, int batch, int heads, int kv_heads, int head_dim,
                int page_size, const int32_t *seq_lens, int splits);

/* Make a plan on the current CUDA device: checks the shape, runs the split
 * planner, allocates and fills the device work list and the partial
 * workspace. *out receives the plan (NULL on error). PKVD_EINVAL for a bad
 * field, PKVD_EUNSUPPORTED for a shape no kernel takes, PKVD_ENOMEM /
 * PKVD_ECUDA if the device allocation or upload failed. The fields and
 * seq_lens are checked before the kernel variant, so a request shorter than
 * q_len gives PKVD_EINVAL even for a shape no variant takes.
 * Defined by: aiter pull 4758, Motivation (split count) and Technical
 * Details 2 (split-major grid order) and 3 (head-dim-tiled merge gated on
 * idle SMs); ROCm/rocm-libraries pull 10102, Motivation (a launch must be
 * keyed by every shape field: a plan is valid only for its own). */
int decode_plan_ex(pkvd_plan **out, const pkvd_plan_desc *desc, const int32_t *seq_lens);

/* Shared-prefix plan (MLA only, heads in {16, 32, 64}). prefix_group[b] >= 0
 * puts request b in a group; the members of a group must be consecutive
 * requests with equal prefix_len[b] (1 <= prefix_len[b] <= seq_lens[b]) and
 * page_table rows whose first ceil(prefix_len / page_size) entries name the
 * same pages (the caller's promise: the shared tokens are read through the
 * first member's row; with desc->checks on, the kernels compare every
 * member's prefix entries with the first member's and report a difference
 * as PKVD_EDEVICE_CHECK). prefix_group[b] < 0: no sharing. A group's
 * shared tokens are read once per 64/heads members, with the members' query
 * heads batched as the N side of the tensor-core products (64 rows); each
 * request's private tokens run as usual (their variant is chosen on the
 * private lengths), and the merge combines both kinds of partials. Groups
 * whose prefix is shorter than 1024 tokens are not batched (their members
 * read the prefix as private tokens): the batched items run on the
 * tensor-memory kernel, whose one-part P needs long items. Results equal
 * the plain plan's within the usual tolerance. desc->splits applies to the
 * private tokens only.
 * Defined by: aiter pull 4758, Technical Details 2 (the split-major grid
 * hopes for L2 reuse when requests share a prefix; this call makes the
 * reuse explicit) and Test Plan (68,000-token contexts whose first 63,240
 * tokens are shared by groups of 8). */
int decode_plan_prefix(pkvd_plan **out, const pkvd_plan_desc *desc, const int32_t *seq_lens,
                       const int32_t *prefix_group, const int32_t *prefix_len);

/* Host-only planning of a shared-prefix plan (no CUDA call): the grouped
 * prefix items come first in `items`, then the per-request items; capacity
 * must cover info->num_prefix_items + info->num_items. desc->num_sms and
 * desc->ctas_per_sm (of the per-request kernel) must be set.
 * Defined by: as decode_plan_prefix. */
int decode_plan_prefix_compute(const pkvd_plan_desc *desc, const int32_t *seq_lens,
                               const int32_t *prefix_group, const int32_t *prefix_len,
                               pkvd_plan_info *info, pkvd_work_item *items, int64_t capacity);

/* ------------------------------------------------------------------------
 * Context-parallel decode: one request's tokens spread over `world` GPUs
 * (ranks), each holding the whole paged cache and page table. Rank r of
 * world takes of request b the contiguous token range [begin, begin + len)
 * with ceil(ceil(L_b / world) / page_size) pages per rank from the start
 * (ranges start on page boundaries; trailing ranks may be empty). Each rank
 * runs an ordinary decode over its range (decode_plan_cp + decode_run) and
 * gets a normalised output and its log-sum-exp per (request, head); the
 * ranks exchange those rows (an all-gather, the caller's collective) and
 * decode_merge_ranks combines them into the whole-context result. One query
 * token per request (q_len 0 or 1); no shared-prefix plans.
 * Defined by: aiter pull 4758, Technical Details 3 (the split partials'
 * log-sum-exp merge: here the ranks' ranges are the splits).
 *
 * decode_cp_ranges: the token range of every request on rank `rank` (host,
 * no CUDA call); begin and len are host arrays of `batch` entries. PKVD_EINVAL
 * for world outside 1 .. 1024, rank outside 0 .. world - 1 or a negative
 * length. */
int decode_cp_ranges(int world, int rank, int batch, int page_size, const int32_t *seq_lens,
                     int32_t *begin, int32_t *len);

/* A plan of rank `rank`'s token ranges (on the current device): seq_lens are
 * the whole requests' lengths, and decode_run of this plan takes the whole
 * page table and writes the range's normalised out and lse (an empty range:
 * out 0, lse -inf). The variant is chosen on the range lengths. Errors as
 * decode_plan_ex, and PKVD_EINVAL for a bad world or rank, PKVD_EUNSUPPORTED
 * for q_len > 1. */
int decode_plan_cp(pkvd_plan **out, const pkvd_plan_desc *desc, const int32_t *seq_lens,
                   int world, int rank);

/* Host-only planning of decode_plan_cp (no CUDA call; desc->num_sms and
 * desc->ctas_per_sm must be set), items in grid order with absolute token
 * positions. Capacity as decode_plan_compute. */
int decode_plan_cp_compute(const pkvd_plan_desc *desc, const int32_t *seq_lens, int world,
                           int rank, pkvd_plan_info *info, pkvd_work_item *items,
                           int64_t capacity);

/* Merge n_ranks ranks' rows: o_parts [n_ranks, rows, dv] fp32 and lse_parts
 * [n_ranks, rows] fp32 natural log (device, o 16-byte aligned) into out
 * [rows, dv] and lse [rows]; rows = batch * heads. Ranks are summed in rank
 * order, so the bits do not depend on which rank merges. dv a multiple of 4
 * up to 512 (PKVD_EUNSUPPORTED otherwise); PKVD_EINVAL for bad sizes or
 * pointers, PKVD_ECUDA if the launch failed. Asynchronous on `stream`,
 * allocates nothing. */
int decode_merge_ranks(int n_ranks, int64_t rows, int dv, const float *o_parts,
                       const float *lse_parts, float *out, float *lse, pkvd_stream_t stream);

/* Launch stage 1 and the merge on `stream`. q, k_pages, v_pages, page_table,
 * out and lse are device pointers laid out as above. Asynchronous; returns
 * PKVD_EINVAL for a null or misaligned pointer or a plan made on another
 * device, PKVD_ECUDA if a launch failed.
 * Defined by: aiter pull 4758, Motivation (stage 1 writes one normalised
 * partial and its log-sum-exp per split; stage 2 merges them) and Technical
 * Details 1 (two KV blocks in flight in the stage-1 loop) and 3 (the merge
 * recomputes its scalar statistics per Dv tile); TensorFold pull 1932, "What
 * this changes" (one score per key for each query head of a KV group). */
int decode_run(const pkvd_plan *plan, const void *q, const void *k_pages,
               const void *v_pages, const int32_t *page_table, float *out, float *lse,
               pkvd_stream_t stream);

/* decode_run that also records caller-made events on `stream`: ev_begin
 * before stage 1, ev_mid between stage 1 and the merge, ev_end after the
 * merge (any may be NULL). Recording ev_mid keeps the merge from overlapping
 * stage 1's tail; otherwise identical to decode_run. For timing each stage.
 * Defined by: aiter pull 4758, Test Plan (device time from events around
 * the op) and Technical Details 3 (stage-2's own share is measured). */
int decode_run_timed(const pkvd_plan *plan, const void *q, const void *k_pages,
                     const void *v_pages, const int32_t *page_table, float *out,
                     float *lse, pkvd_stream_t stream, pkvd_event_t ev_begin,
                     pkvd_event_t ev_mid, pkvd_event_t ev_end);

/* Free a plan and its device memory (NULL is a no-op). Synchronises the
 * plan's device so no run still reads the freed memory. PKVD_ECUDA if the
 * synchronisation or the free failed (the plan is freed on the host anyway).
 * Defined by: the plan / run split of decode_plan_ex (ROCm/rocm-libraries
 * pull 10102, Motivation). */
int decode_plan_destroy(pkvd_plan *plan);

/* Device bytes the plan owns (work list, split table, partials, status); 0
 * for NULL. Defined by: aiter pull 4758, Motivation (the per-split partials
 * and their log-sum-exps that stage 1 leaves for the merge). */
size_t decode_workspace_bytes(const pkvd_plan *plan);

/* Copy the planner's decisions into *info (PKVD_EINVAL for NULL).
 * Defined by: aiter pull 4758, Motivation and Technical Details 2-3 (split
 * count, grid order and merge tiling are the planner's decisions). */
int decode_plan_query(const pkvd_plan *plan, pkvd_plan_info *info);

/* Synchronise `stream`, then read and clear the plan's device status word:
 * PKVD_OK, PKVD_EDEVICE_CHECK or PKVD_ETIMEOUT (PKVD_ECUDA if the
 * synchronisation or the read failed).
 * Defined by: TensorFold pull 1932, "What this changes" and "Tests run" (a
 * key or block the kernel skips must be caught, not pass silently): here
 * every pipeline wait is bounded and reports, and page ids can be checked. */
int decode_last_device_status(const pkvd_plan *plan, pkvd_stream_t stream);

/* ------------------------------------------------------------------------
 * Dense causal prefill attention, head_dim 64 (a second workload: the whole
 * prompt at once instead of one decode step). Every token t of request b
 * attends to that request's tokens 0 .. t:
 *
 *     out[b,t,h,:] = sum_{u<=t} softmax_u(scale * q[b,t,h,:] . k[b,kv,u,:]) * v[b,kv,u,:]
 *     lse[b,t,h]   = ln sum_{u<=t} exp(scale * q[b,t,h,:] . k[b,kv,u,:])
 *
 * with kv = h / (heads / kv_heads). It is the multi-token decode above with
 * q_len = seq_len on an unpaged cache (one page of seq_len tokens per
 * request). The rocm-libraries pull 10102 page is about this kernel's
 * shared-memory pitch at D = 64; here the tiles use the 128-byte TMA swizzle,
 * which a 64-element row fills exactly (no pad needed).
 *
 * Layouts (contiguous, 16-byte aligned):
 *   q    [batch, seq_len, heads, 64]       bf16 or fp16
 *   k, v [batch, kv_heads, seq_len, 64]    same type
 *   out  [batch, seq_len, heads, 64]       fp32
 *   lse  [batch, seq_len, heads]           fp32, natural log
 *   status  one caller-owned device int32: a pipeline wait that ran out ORs
 *           in a nonzero bit (the caller zeroes it and reads it after a sync)
 */
typedef struct pkvd_prefill_desc {
  int32_t batch;              /* requests, >= 1                                   */
  int32_t heads;              /* query heads                                       */
  int32_t kv_heads;           /* KV heads; heads % kv_heads == 0                   */
  int32_t seq_len;            /* tokens per request, >= 1                          */
  int32_t dtype;              /* pkvd_dtype                                        */
  float scale;                /* 0 = 1 / 8 (= 1 / sqrt(64))                        */
  int32_t reserved[2];        /* must be 0                                         */
} pkvd_prefill_desc;

/* Launch the prefill on `stream` (asynchronous, allocates nothing). Returns
 * PKVD_EINVAL for a bad argument or pointer alignment, PKVD_EUNSUPPORTED for
 * heads % kv_heads != 0 or a grid too large, PKVD_ECUDA if a tensor map or
 * the launch failed. */
int prefill_d64_run(const pkvd_prefill_desc *desc, const void *q, const void *k, const void *v,
                    float *out, float *lse, int32_t *status, pkvd_stream_t stream);

/* Self-test of the kernels' bounded pipeline waits. Launches one block on
 * `stream` that waits, through the same bounded barrier wait the stage-1
 * kernels use, on a shared-memory barrier that nothing completes, with a
 * limit of limit_us microseconds (1 .. 10,000,000). The wait runs out; the
 * block writes status[0] = PKVD_ETIMEOUT (PKVD_OK would mean the barrier
 * completed, PKVD_ECUDA that the wait gave up before its limit) and
 * status[1] = the microseconds it waited, then exits: nothing hangs or
 * faults, and the context stays usable. status: caller-owned device array
 * of two int32. Asynchronous; returns PKVD_EINVAL for a bad argument,
 * PKVD_ECUDA if the launch failed. */
int decode_selftest_wait_timeout(int32_t *status, int64_t limit_us, pkvd_stream_t stream);

/* The split planner alone, on the host, with no CUDA call: desc->num_sms and
 * desc->ctas_per_sm must be set (> 0). Fills *info and, when `items` is not
 * NULL, up to `capacity` work items in grid order. Returns PKVD_OK, or
 * PKVD_EINVAL when capacity is smaller than info->num_items (info is still
 * filled).
 * Defined by: aiter pull 4758, Motivation (split count) and Technical
 * Details 2 (split-major order); ROCm/rocm-libraries pull 10102, Technical
 * Details (the structure is checked on the host, without a GPU). */
int decode_plan_compute(const pkvd_plan_desc *desc, const int32_t *seq_lens,
                        pkvd_plan_info *info, pkvd_work_item *items, int64_t capacity);

/* A decode op that allocates no device memory. The paper has no counterpart
 * to this call. It is for callers that cannot call cudaMalloc: a host
 * application that owns all device memory through its own pool, or code that
 * runs where allocating is forbidden or would stall the stream. It plans on
 * the host like decode_plan_ex (same desc and seq_lens rules) and launches
 * the same kernels, but keeps all scratch (status word, split table, work
 * list, split partials) in one static 16 MiB device array that the library
 * holds on every device that loads it until the process exits.
 *   - The scratch a call needs must fit 16 MiB (about rows * heads * (Dv + 1)
 *     * 4 bytes for the partials); larger problems return PKVD_ENOMEM and
 *     queue nothing.
 *   - All calls share the array: calls on one stream run in order, calls that
 *     overlap on the GPU (other streams, unsynchronised threads) race.
 *   - The first call on a device looks up the array's address with that
 *     device current.
 *   - The call copies its work list from host memory it frees on return, so
 *     on a stream that is being captured it returns PKVD_EUNSUPPORTED and
 *     queues nothing.
 *   - Device-side page-id checks (desc->checks) and wait timeouts are
 *     recorded in the array's status word, which each call clears first;
 *     decode_run_static_status reports the last call's.
 * q, k_pages, v_pages, page_table, out and lse are as for decode_run;
 * desc and seq_lens are host pointers, read during the call only. */
int decode_run_static(const pkvd_plan_desc *desc, const int32_t *seq_lens, const void *q,
                      const void *k_pages, const void *v_pages, const int32_t *page_table,
                      float *out, float *lse, pkvd_stream_t stream);

/* Status of the last decode_run_static call on the current device, also
 * allocation-free (the paper has no counterpart to this call either):
 * synchronises `stream`, then reads and clears the static array's status
 * word. PKVD_OK, PKVD_EDEVICE_CHECK (a page id outside the pool, with
 * checks on) or PKVD_ETIMEOUT (a pipeline wait ran out). */
int decode_run_static_status(pkvd_stream_t stream);

/* Static description of a status code (never NULL). Defined by: the
 * error conventions above. */
const char *decode_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* PKVD_H_ */
