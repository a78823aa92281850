/*
 * cpattn.h -- C ABI of libcpattn: attention over a context-parallel ("striped")
 * paged KV pool on one GB300 GPU (sm_103a).
 *
 * The method (mstar PR #1124 "Context / Sequence Parallel 1/5", description):
 * a paged KV pool shared by P partners stripes the token slots of every page
 * over the partners -- the slot at offset s of a logical page belongs to
 * partner s % P, where it is physical slot s / P of the same page id.  Page ids
 * stay logical, so one page table serves every partner.  Each partner attends
 * its own slots and returns a partial output with its log-sum-exp; the
 * partials are merged exactly.  A step that is not one token a row attends the
 * pool for the context only and attends its new tokens apart (own-token
 * attention) from the K/V the layer passes; the own-token partial is merged
 * with the context partials (vLLM "[Core] Add explicit layer parallel plans",
 * flash_attn.py, FlashAttentionImpl._forward_with_dcp: context partial,
 * own-token partial with cu_seqlens_k = cu_seqlens_q, merge_attn_states).
 * Here all P partners live on one GPU, so the cross-partner exchange of the
 * pages is replaced by lse_merge reading the P partials from device memory.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is DEVICE memory owned by the caller, except the
 *   cpattn_pool_desc pointer, which is HOST memory read during the call.  The
 *   library allocates nothing, never synchronises, and launches only on the
 *   given stream (0 = legacy default).  It keeps no state between calls,
 *   except cp_paged_attn_partial_noalloc: that entry point owns a fixed
 *   device array inside the library and caches its address per device (see
 *   its own block below).
 * - Return value: CPATTN_OK (0) or a negative CPATTN_ERR_* code.  Argument
 *   checks happen on the host before any launch; a failed check launches
 *   nothing.  CPATTN_ERR_CUDA means a launch failed (cudaGetLastError);
 *   kernels already queued may have run.  The library never aborts or prints.
 * - Device-side checks: table entries that would address memory outside the
 *   pool (a page id >= num_pages, a position past the row's page table) are
 *   skipped, and, when dev_status is not NULL, the first such event stores a
 *   nonzero CPATTN_DEV_* code in *dev_status (the caller reads it after the
 *   stream synchronises; the library never clears it).
 * - Device pointers must be 16-byte aligned (CPATTN_ERR_MISALIGNED), and every
 *   row of head_dim values must be a multiple of 16 bytes.
 * - Element types: CPATTN_DTYPE_BF16 (bfloat16 values) or CPATTN_DTYPE_FP32.
 *   A bf16 layer may keep its pool in CPATTN_DTYPE_FP8_E4M3 (kv_dtype of the
 *   descriptor): the vLLM page "[Core] Add explicit layer parallel plans"
 *   passes per-tensor k_descale / v_descale to the attention call of an FP8
 *   cache.  A stored code is the OCP FP8 E4M3 value nearest to x / descale
 *   (IEEE float32 quotient, round to nearest even, magnitudes past 448
 *   saturated to 448); a read key or value is code value * descale.  Queries,
 *   new K/V and outputs stay bf16; the pool bytes halve.
 *   Partial outputs and log-sum-exps are always fp32.  Log-sum-exps use the
 *   natural logarithm; an empty key set gives output 0 and LSE -inf.
 *
 * Pool layout (HND per partner)
 * -----------------------------
 *   pool_k: [P][num_pages][num_kv_heads][page_size / P][head_dim]
 *   pool_v: [P][num_pages][num_kv_heads][page_size / P][head_dim_v]
 * Logical position pos of a row whose page table is pages[] lives in page id
 * pages[pos / page_size] at offset off = pos % page_size, i.e. partner
 * off % P, physical slot off / P.  P must divide page_size.
 * With an interleave size I > 1 (the vLLM page "[Core] Add explicit layer
 * parallel plans", FlashAttentionMetadataBuilder: cp_kv_cache_interleave_size)
 * runs of I consecutive offsets stay together: partner (off / I) % P,
 * physical slot (off / (I * P)) * I + off % I, and I * P must divide
 * page_size.  I = 1 is the plain striping.  MLA pools keep one
 * latent row per token (num_kv_heads = 1, head_dim = 576) and no pool_v: the
 * value is the first head_dim_v values of the latent row (pool_v == NULL).
 */
#ifndef CPATTN_H_
#define CPATTN_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CPATTN_VERSION 3

/* exported symbols (the library is built with hidden visibility otherwise) */
#if defined(__GNUC__)
#define CPATTN_API __attribute__((visibility("default")))
#else
#define CPATTN_API
#endif

/* status codes */
#define CPATTN_OK 0
#define CPATTN_ERR_INVALID_ARG (-1)               /* null pointer, bad count or size */
#define CPATTN_ERR_P_NOT_DIVIDING_PAGE_SIZE (-2)  /* P < 1, interleave < 0 or page_size % (P * I) != 0 */
#define CPATTN_ERR_UNSUPPORTED_SHAPE (-3)         /* head dims / group size not compiled */
#define CPATTN_ERR_MISALIGNED (-4)                /* a device pointer not 16-byte aligned */
#define CPATTN_ERR_WORKSPACE_TOO_SMALL (-5)       /* workspace_bytes below the requirement */
#define CPATTN_ERR_CUDA (-6)                      /* a launch failed */

/* device-side status codes (written to *dev_status) */
#define CPATTN_DEV_OK 0
#define CPATTN_DEV_PAGE_OUT_OF_RANGE 1   /* page id outside [0, num_pages) */
#define CPATTN_DEV_POS_PAST_TABLE 2      /* position beyond the row's page table */
#define CPATTN_DEV_BAD_INDPTR 3          /* qo_indptr not within [0, num_tokens] */
#define CPATTN_DEV_TC_TIMEOUT 4          /* a tensor-core completion wait ran out; that CTA's output is not written */

/* element types */
#define CPATTN_DTYPE_BF16 0
#define CPATTN_DTYPE_FP32 1
#define CPATTN_DTYPE_FP8_E4M3 2 /* pools only (kv_dtype), with a bf16 layer */

typedef struct cpattn_pool_desc {
  int32_t P;            /* partners (stripes); divides page_size */
  int32_t page_size;    /* logical page size in tokens */
  int32_t num_pages;    /* page ids per partner pool (same ids for every partner) */
  int32_t num_kv_heads; /* GQA KV heads; 1 for MLA */
  int32_t head_dim;     /* key width (MLA: latent + rope, 576) */
  int32_t head_dim_v;   /* value width (== head_dim for GQA; MLA: 512) */
  int32_t dtype;        /* CPATTN_DTYPE_* of pool, q and new K/V */
  int32_t interleave;   /* interleave size I (0 or 1: plain striping); I * P divides page_size */
  int32_t kv_dtype;     /* element type of pool_k / pool_v: 0 or dtype (the same), or
                           CPATTN_DTYPE_FP8_E4M3 with dtype CPATTN_DTYPE_BF16 */
  float k_descale;      /* FP8 pools: key = code value * k_descale (finite, > 0) */
  float v_descale;      /* FP8 pools: value = code value * v_descale (finite, > 0) */
} cpattn_pool_desc;

/* Library version (CPATTN_VERSION) -- lets a binding check it loaded the right .so. */
CPATTN_API int cpattn_version(void);

/* Static, NUL-terminated text for a status code. */
CPATTN_API const char* cpattn_status_string(int status);

/* Bytes of one pool tensor: pool_k (which_v = 0) or pool_v (which_v = 1).
 * Returns 0 for an invalid descriptor. */
CPATTN_API size_t cpattn_pool_bytes(const cpattn_pool_desc* desc, int which_v);

/*
 * cp_kv_write -- write a step's new K/V into the striped pool.
 *
 * Follows the write path of mstar PR #1124 "Context / Sequence Parallel 1/5"
 * (description: a token is written by its owner; review thread: every
 * write-addressing path maps through the placement, none takes the offset at
 * the logical page size).  Token t belongs to row b with
 * qo_indptr[b] <= t < qo_indptr[b+1]; its logical position is positions[t].
 * Its K row k_new[t] ([num_kv_heads][head_dim]) is copied bit for bit to
 * pool_k[off % P][page][h][off / P][:] with page = kv_page_indices[
 * kv_page_indptr[b] + positions[t] / page_size], off = positions[t] % page_size
 * (V likewise into pool_v).  Tokens with positions[t] < 0 and tokens at or past
 * qo_indptr[num_rows] are padding and are not written (and never read).
 *
 *   k_new, v_new     [num_tokens][num_kv_heads][head_dim | head_dim_v];
 *                    v_new and pool_v are NULL for MLA (latent rows only)
 *   positions        [num_tokens] int32
 *   qo_indptr        [num_rows + 1] int32, non-decreasing
 *   kv_page_indptr   [num_rows + 1] int32; kv_page_indices [kv_page_indptr[num_rows]]
 *   dev_status       optional device int32 (see conventions)
 * Deterministic: the result does not depend on launch order (distinct tokens
 * own distinct slots when positions are distinct within a row).
 */
CPATTN_API int cp_kv_write(const cpattn_pool_desc* desc, void* pool_k, void* pool_v,
                const void* k_new, const void* v_new, const int32_t* positions,
                const int32_t* qo_indptr, int32_t num_rows, int32_t num_tokens,
                const int32_t* kv_page_indptr, const int32_t* kv_page_indices,
                int32_t* dev_status, cudaStream_t stream);

/*
 * cp_paged_attn_partial -- every partner's partial attention over the pool.
 *
 * Follows mstar PR #1124 "Context / Sequence Parallel 1/5" (description: each
 * partner attends its own slots and returns the partial with its
 * log-sum-exp) and the context partial of vLLM "[Core] Add explicit layer
 * parallel plans", FlashAttentionImpl._forward_with_dcp.  For partner p,
 * query token t of row b and query head h (KV head h / (num_q_heads /
 * num_kv_heads)), with S_p = { j < kv_len[b] : j % P == p }:
 *   o_part[p][t][h][:] = sum_{j in S_p} softmax_j(scale * q[t][h] . K_j) V_j
 *   lse_part[p][t][h]  = ln sum_{j in S_p} exp(scale * q[t][h] . K_j)
 * (empty S_p: 0 and -inf).  Every query token of a row sees the same kv_len[b]
 * keys: a decode row passes its full length (its own key already written), a
 * multi-token row of a non-decode step passes its context length.  Tokens of
 * rows >= num_rows' span end (t >= qo_indptr[num_rows]) get 0 / -inf.
 *
 *   q          [num_tokens][num_q_heads][head_dim]
 *   qo_indptr  [num_rows + 1]; NULL means one token a row (num_tokens == num_rows)
 *   kv_len     [num_rows] int32
 *   max_kv_len host upper bound of kv_len[] (sizes the grid and workspace;
 *              larger kv_len entries are clamped to it and flagged)
 *   o_part     [P][num_tokens][num_q_heads][head_dim_v] fp32
 *   lse_part   [P][num_tokens][num_q_heads] fp32
 *   workspace  device scratch of cp_paged_attn_workspace_bytes(...) bytes, or
 *              more; its contents need no initialisation and are clobbered.
 * Supported: GQA with head_dim in {64, 128}, group size in {1, 2, 4, 8, 16};
 * MLA (num_kv_heads 1, head_dim 576, head_dim_v 512, bf16, 128 query heads).
 * Other shapes, and multi-token rows over a bf16 pool of 2^31 or more K rows
 * (P * num_pages * num_kv_heads * page_size / P), return
 * CPATTN_ERR_UNSUPPORTED_SHAPE before any launch.
 */
CPATTN_API int cp_paged_attn_partial(const cpattn_pool_desc* desc, const void* pool_k,
                          const void* pool_v, const void* q, int32_t num_q_heads,
                          int32_t num_rows, int32_t num_tokens, const int32_t* qo_indptr,
                          const int32_t* kv_len, int32_t max_kv_len,
                          const int32_t* kv_page_indptr, const int32_t* kv_page_indices,
                          float scale, float* o_part, float* lse_part, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream);

/* Workspace bytes cp_paged_attn_partial needs for these sizes (0 on bad args). */
CPATTN_API size_t cp_paged_attn_workspace_bytes(const cpattn_pool_desc* desc, int32_t num_q_heads,
                                     int32_t num_tokens, int32_t max_kv_len);

/* LSE layouts of cp_paged_attn_partial_ex's lse_part */
#define CPATTN_LSE_TOKEN_MAJOR 0 /* [P][num_tokens][num_q_heads] (as cp_paged_attn_partial) */
#define CPATTN_LSE_HEAD_MAJOR 1  /* [P][num_q_heads][num_tokens] */

/*
 * cp_paged_attn_partial_ex -- cp_paged_attn_partial with a choice of LSE
 * layout and of the rows' dispatch order.  In the vLLM page "[Core] Add
 * explicit layer parallel plans" (_forward_with_dcp) the context attention
 * returns its LSE head-major ("[H, B]") while the DCP combine takes it
 * token-major ("[B, H]"); a TP-mode caller gathers the query heads of all
 * partners (query_across_dcp), has each partner attend all of them, and
 * combines per head.  lse_layout selects CPATTN_LSE_TOKEN_MAJOR or
 * CPATTN_LSE_HEAD_MAJOR (anything else: CPATTN_ERR_INVALID_ARG).  row_order
 * is as for cp_paged_attn_fused (a device permutation of the rows, used when
 * qo_indptr is NULL; longest rows first shortens the last wave; NULL: row
 * order).  Every other argument is as for cp_paged_attn_partial, and the
 * values written are the same.
 */
CPATTN_API int cp_paged_attn_partial_ex(const cpattn_pool_desc* desc, const void* pool_k,
                                        const void* pool_v, const void* q, int32_t num_q_heads,
                                        int32_t num_rows, int32_t num_tokens, const int32_t* qo_indptr,
                                        const int32_t* kv_len, int32_t max_kv_len,
                                        const int32_t* kv_page_indptr, const int32_t* kv_page_indices,
                                        float scale, float* o_part, float* lse_part, int32_t lse_layout,
                                        const int32_t* row_order, void* workspace, size_t workspace_bytes,
                                        int32_t* dev_status, cudaStream_t stream);

/*
 * cp_paged_attn_fused -- the partials of all P partners and their exact merge
 * in one call: the final attention output of every query token.
 *
 * The method computes one partial (output, LSE) per partner over its stripe
 * and combines them exactly (mstar PR #1124 "Context / Sequence Parallel
 * 1/5", description: each partner returns its partial with its log-sum-exp,
 * merged on the device; vLLM "[Core] Add explicit layer parallel plans",
 * _forward_with_dcp: merge_attn_states of the context and query partials).
 * Here the merge is fused into the partial kernels.  GQA heads: every chunk
 * of every partner leaves its partial in the workspace and the last CTA of
 * each (token, KV head) merges them.  MLA over pages of 64 slots: one tile
 * holds a logical page of every partner, so the online softmax merges the
 * partners as it goes and the kernel writes final rows; a token whose pages
 * are split between two CTA pairs leaves normalised pieces in the workspace,
 * merged by a second kernel on the same stream.  The exact merge is
 * associative, so the result is the one cp_paged_attn_partial followed by
 * lse_merge gives (up to rounding order), without the [P, T, Hq, Dv] partial
 * tensor round trip.  Pages give the captured buckets of a step (fixed
 * shapes, replayed as a graph); this call makes no host synchronisation and
 * no allocation, so it can be captured.
 *
 * Arguments as cp_paged_attn_partial, except:
 *   row_order   optional device [num_rows] permutation of the rows: the order
 *               in which CTAs take rows when each row is one token (qo_indptr
 *               NULL).  Longest rows first shortens the last wave; the
 *               caller's host-side plan knows the lengths.  NULL: row order.
 *               Entries outside [0, num_rows) are skipped and reported
 *               (CPATTN_DEV_BAD_INDPTR); a non-permutation gives wrong rows.
 *               Ignored when qo_indptr is given.
 *   extra_o, extra_lse  optional precomputed partial merged in too
 *               ([num_tokens][num_q_heads][head_dim_v] fp32 and
 *               [num_tokens][num_q_heads] fp32, e.g. own_token_attn's); both
 *               NULL or both set
 *   out_dtype   CPATTN_DTYPE_BF16 (round to nearest even) or CPATTN_DTYPE_FP32
 *   out         [num_tokens][num_q_heads][head_dim_v] of out_dtype
 *   lse_out     [num_tokens][num_q_heads] fp32 natural-log LSE, or NULL
 *   workspace   cp_paged_attn_fused_workspace_bytes(...) bytes or more.
 * Tokens of no row, of padding rows (kv_len 0) and empty stripes merge to
 * output 0 and LSE -inf unless the extra partial covers them.  max_kv_len may
 * be a capacity (a captured bucket's largest length): shorter rows only leave
 * idle CTAs.
 */
CPATTN_API int cp_paged_attn_fused(const cpattn_pool_desc* desc, const void* pool_k,
                                   const void* pool_v, const void* q, int32_t num_q_heads,
                                   int32_t num_rows, int32_t num_tokens, const int32_t* qo_indptr,
                                   const int32_t* kv_len, int32_t max_kv_len,
                                   const int32_t* kv_page_indptr, const int32_t* kv_page_indices,
                                   const int32_t* row_order, float scale, const float* extra_o,
                                   const float* extra_lse,
                                   int32_t out_dtype, void* out, float* lse_out, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream);

/* Workspace bytes cp_paged_attn_fused needs for these sizes (0 on bad args). */
CPATTN_API size_t cp_paged_attn_fused_workspace_bytes(const cpattn_pool_desc* desc, int32_t num_q_heads,
                                                      int32_t num_tokens, int32_t max_kv_len);

/*
 * cp_paged_attn_partial_noalloc -- cp_paged_attn_partial for callers that
 * cannot allocate device memory.  The pages have no counterpart: this is a
 * convenience of this library.
 *
 * Some callers cannot call cudaMalloc: a plugin that is handed raw input and
 * output pointers but no allocator, a runtime whose memory pool owns the whole
 * GPU, or a step that must not allocate once it has started.  This call takes
 * the same inputs and outputs as cp_paged_attn_partial but no workspace: the
 * split-KV scratch is a fixed 16 MiB __device__ array inside libcpattn (every
 * GPU that loads the library holds it until the process exits; see
 * cp_paged_attn_noalloc_scratch_bytes).
 *   - Returns CPATTN_ERR_WORKSPACE_TOO_SMALL, launching nothing, when
 *     cp_paged_attn_workspace_bytes(desc, num_q_heads, num_tokens, max_kv_len)
 *     exceeds that size.
 *   - Allocates nothing; all calls share the one array, which keeps the last
 *     call's contents.  The split tickets, the only part that must start at
 *     zero, are cleared on `stream` whenever the call splits a stripe (the
 *     only time they are read).  Calls whose kernels can overlap on the GPU
 *     (other streams, other host threads) race on the array: order them on
 *     one stream.
 *   - The first call on each device looks up the array's device address with
 *     that device current and caches it; make that first call before any
 *     stream capture begins.  The cached address belongs to the device's
 *     primary context: after cudaDeviceReset (or any teardown of that
 *     context) it is stale, and this entry point must not be called again in
 *     the same process.
 * Results equal those of cp_paged_attn_partial with a caller workspace.
 */
CPATTN_API int cp_paged_attn_partial_noalloc(const cpattn_pool_desc* desc, const void* pool_k,
                                             const void* pool_v, const void* q, int32_t num_q_heads,
                                             int32_t num_rows, int32_t num_tokens,
                                             const int32_t* qo_indptr, const int32_t* kv_len,
                                             int32_t max_kv_len, const int32_t* kv_page_indptr,
                                             const int32_t* kv_page_indices, float scale,
                                             float* o_part, float* lse_part, int32_t* dev_status,
                                             cudaStream_t stream);

/* Size in bytes of the library-owned scratch behind cp_paged_attn_partial_noalloc. */
CPATTN_API size_t cp_paged_attn_noalloc_scratch_bytes(void);

/*
 * own_token_attn -- causal attention of a step's new tokens over the K/V the
 * layer passes (mstar PR #1124 "Context / Sequence Parallel 1/5",
 * description: a step that is not one token a row attends its own tokens
 * apart; vLLM "[Core] Add explicit layer parallel plans", _forward_with_dcp:
 * flash_attn_varlen_func with cu_seqlens_k = cu_seqlens_q, causal).
 * For real row b < num_real_rows and its i-th token t = qo_indptr[b] + i:
 *   o_own[t][h] = sum_{j <= i} softmax_j(scale * q[t][h] . k_new[qo_indptr[b]+j]) v_new[...]
 *   lse_own[t][h] = ln of the same sum of exponentials.
 * Padding rows (b >= num_real_rows) and tokens at or past
 * qo_indptr[num_real_rows] get 0 / -inf, and their keys and values are never
 * read (review thread of the same PR: padding rows' keys must not reach real
 * rows in a captured bucket).
 *
 *   q      [num_tokens][num_q_heads][head_dim]
 *   k_new  [num_tokens][num_kv_heads][head_dim]; v_new [..][head_dim_v]
 *          (v_new NULL: the value is the first head_dim_v values of k_new)
 *   qo_indptr [num_rows_bucket + 1]
 *   max_q_len the most new tokens of any row (sizes the launch; an
 *          underestimate only costs time)
 *   o_own  [num_tokens][num_q_heads][head_dim_v] fp32, lse_own [num_tokens][num_q_heads]
 * Supported: head_dim == head_dim_v in {64, 128}; group size in {1, 2, 4, 8,
 * 16} (bf16, tensor cores) or {1, 2, 4, 8} (fp32).  MLA: num_kv_heads 1,
 * head_dim 576, head_dim_v 512, bf16, v_new NULL (the value is the first 512
 * values of each latent key row), any num_q_heads.
 */
CPATTN_API int own_token_attn(const void* q, const void* k_new, const void* v_new, int32_t num_q_heads,
                   int32_t num_kv_heads, int32_t head_dim, int32_t head_dim_v, int32_t dtype,
                   const int32_t* qo_indptr, int32_t num_rows_bucket, int32_t num_real_rows,
                   int32_t num_tokens, int32_t max_q_len, float scale, float* o_own,
                   float* lse_own, cudaStream_t stream);

/*
 * lse_merge -- exact merge of N partials over disjoint key sets (mstar PR #1124
 * "Context / Sequence Parallel 1/5", description: partials merged exactly;
 * vLLM "[Core] Add explicit layer parallel plans", merge_attn_states).
 * Per token t and head h, with M = max_i lse_i:
 *   M == -inf : out = 0, lse_out = -inf (padding merges to zero)
 *   otherwise : w_i = exp(lse_i - M), lse_out = M + ln sum w_i,
 *               out = sum_i w_i o_i / sum_i w_i  (rounded to out_dtype, RNE)
 *   o_parts    partial i at o_parts + i * stride_o, laid out [num_tokens][num_heads][head_dim_v]
 *   lse_parts  partial i at lse_parts + i * stride_lse, laid out [num_tokens][num_heads]
 *   out        [num_tokens][num_heads][head_dim_v] of out_dtype; lse_out may be NULL
 * stride_o and stride_lse are in elements; head_dim_v must be a multiple of 4.
 */
CPATTN_API int lse_merge(int32_t num_partials, const float* o_parts, const float* lse_parts,
              int64_t stride_o, int64_t stride_lse, int32_t num_tokens, int32_t num_heads,
              int32_t head_dim_v, int32_t out_dtype, void* out, float* lse_out,
              cudaStream_t stream);

/* One partial as a strided view: the output row of (token t, head h) is the
 * head_dim_v fp32 values at o + t * o_stride_token + h * o_stride_head; its
 * natural-log LSE is lse[t * lse_stride_token + h * lse_stride_head].  Strides
 * count elements; o and its strides must keep rows 16-byte aligned. */
typedef struct cpattn_partial_view {
  const float* o;
  const float* lse;
  int64_t o_stride_token, o_stride_head;
  int64_t lse_stride_token, lse_stride_head;
} cpattn_partial_view;

#define CPATTN_MAX_MERGE_VIEWS 16

/*
 * lse_merge_views -- lse_merge over partials of any layout.
 *
 * Same exact merge as lse_merge (mstar PR #1124 "Context / Sequence Parallel
 * 1/5", description; vLLM _forward_with_dcp, merge_attn_states), but each of
 * the num_views (1 .. CPATTN_MAX_MERGE_VIEWS) partials is a strided view (a
 * HOST array of cpattn_partial_view read during the call; the pointers in it
 * are device memory), and the output row of (t, h) goes to out + t *
 * out_stride_token + h * out_stride_head (elements of out_dtype), its LSE to
 * lse_out[t * lse_out_stride_token + h * lse_out_stride_head] (lse_out may be
 * NULL).  With it a TP-mode caller combines the partners' partials of one
 * rank's head slice from head-major LSEs, writes the rank's slice of the
 * output, and merges the context result with the own-token partial without
 * copies.  Views may not overlap the output.  Errors: bad counts or dims
 * (CPATTN_ERR_INVALID_ARG), rows not 16-byte aligned (CPATTN_ERR_MISALIGNED).
 */
CPATTN_API int lse_merge_views(int32_t num_views, const cpattn_partial_view* views, int32_t num_tokens,
                               int32_t num_heads, int32_t head_dim_v, int32_t out_dtype, void* out,
                               int64_t out_stride_token, int64_t out_stride_head, float* lse_out,
                               int64_t lse_out_stride_token, int64_t lse_out_stride_head,
                               cudaStream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* CPATTN_H_ */
