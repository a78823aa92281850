// Host-side launchers of the libcpattn kernels (internal; the C ABI is in cpattn.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace cpattn {

// Raise a kernel's dynamic shared-memory limit once per device (and again
// only if a launch needs more), so that launches recorded into a CUDA graph
// make no attribute call.  One `cache` per kernel instantiation.
template <typename Kernel>
inline cudaError_t ensure_smem(Kernel kern, size_t bytes, std::atomic<int> (&cache)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::atomic<int>& c = cache[dev & 63];
  if (c.load(std::memory_order_acquire) >= static_cast<int>(bytes)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) c.store(static_cast<int>(bytes), std::memory_order_release);
  return e;
}

struct WriteArgs {
  void* pool_k;
  void* pool_v;
  const void* k_new;
  const void* v_new;
  const int32_t* positions;
  const int32_t* qo_indptr;
  const int32_t* page_indptr;
  const int32_t* page_indices;
  int32_t* dev_status;
  int P, interleave, page_size, num_pages, num_kv_heads, num_rows, num_tokens;
  int row_bytes_k, row_bytes_v;  // bytes of one head's K / V row in the pool
  int src_row_bytes_k, src_row_bytes_v;  // ... in k_new / v_new
  int quant_fp8;                 // pool holds E4M3 codes of x / descale
  float k_descale, v_descale;
};
cudaError_t launch_kv_write(const WriteArgs& a, cudaStream_t s);

struct MergeArgs {
  int num_partials;
  const float* o_parts;
  const float* lse_parts;
  int64_t stride_o, stride_lse;
  int num_tokens, num_heads, head_dim_v;
  int out_bf16;
  void* out;
  float* lse_out;
};
cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t s);

// lse_merge_views: partials given as strided views (any token / head layout).
constexpr int kMaxMergeViews = 16;
struct MergeView {
  const float* o;
  const float* lse;
  int64_t o_st, o_sh, lse_st, lse_sh;
};
struct MergeViewArgs {
  int n;
  MergeView v[kMaxMergeViews];
  int num_tokens, num_heads, head_dim_v;
  int out_bf16;
  void* out;
  int64_t out_st, out_sh;
  float* lse_out;
  int64_t lse_out_st, lse_out_sh;
};
cudaError_t launch_lse_merge_views(const MergeViewArgs& a, cudaStream_t s);

// Shared by every partial-attention kernel.
struct PartialArgs {
  const void* pool_k;
  const void* pool_v;  // == pool_k for MLA (value = prefix of the latent row)
  const void* q;
  float* o_part;
  float* lse_part;
  int64_t lse_sp, lse_st, lse_sh;  // lse_part element of (partner, token, query head): strides
  const int32_t* qo_indptr;  // may be null: one token a row
  const int32_t* kv_len;
  const int32_t* page_indptr;
  const int32_t* page_indices;
  int32_t* dev_status;
  // workspace (split-KV partials)
  float* ws_o;
  float* ws_lse;
  int32_t* ws_cnt;   // [T * P * Hkv] chunk tickets
  int32_t* ws_pair;  // [T * Hkv] partner tickets (fused calls)
  int P, interleave, page_size, ps_l, num_pages, num_kv_heads, num_q_heads, head_dim, head_dim_v;
  int ps_shift;  // log2(ps_l) when ps_l is a power of two, else -1
  int num_rows, num_tokens, max_kv_len;
  int seg;         // tokens per staged segment (divides ps_l)
  int chunk;       // stripe tokens per CTA (multiple of seg)
  int max_chunks;  // chunks per (token, partner, kv head), = grid.x
  float scale;
  int kv_fp8;                 // pool holds E4M3 codes: key = code * k_descale, value = code * v_descale
  float k_descale, v_descale;
  // fused calls: o_part / lse_part point into the workspace, and the last
  // partner to finish a (token, KV head) writes the merged output
  int fused;
  const float* extra_o;    // [T][Hq][Dv] fp32 partial merged in too, or null
  const float* extra_lse;  // [T][Hq]
  void* out;               // [T][Hq][Dv], bf16 when out_bf16 else fp32
  int out_bf16;
  float* lse_out;          // [T][Hq] or null
  // dispatch order of the grid's row axis (a permutation, e.g. longest rows
  // first so the last wave holds the short ones), or null: natural order.
  // Used where the grid's z axis walks rows (one token a row); ignored by
  // the multi-token kernel.
  const int32_t* row_order;
};

// Geometry of a partial launch (shared by workspace sizing and the launch).
struct PartialPlan {
  int seg, chunk, max_chunks;
  size_t ws_o_floats, ws_lse_floats, ws_cnt_ints;
  size_t ws_part_floats, ws_part_lse_floats, ws_pair_ints;  // fused calls: partner partials, pair tickets
  size_t bytes() const;
};
// Returns false if the shape is unsupported.
bool plan_partial(int mla, int fused, int P, int interleave, int page_size, int num_kv_heads, int num_q_heads, int head_dim,
                  int num_tokens, int max_kv_len, int dtype_bytes, PartialPlan* plan);

// status: 0 ok, CPATTN_ERR_UNSUPPORTED_SHAPE, or the cudaError via *err
int launch_gqa_partial(const PartialArgs& a, int dtype_bf16, cudaStream_t s, cudaError_t* err);
int launch_gqa_partial_mma(const PartialArgs& a, cudaStream_t s, cudaError_t* err);
int launch_gqa_partial_ext(const PartialArgs& a, cudaStream_t s, cudaError_t* err);
int launch_gqa_partial_ext_ws(const PartialArgs& a, cudaStream_t s, cudaError_t* err);  // bf16 and E4M3 pools
int launch_mla_partial(const PartialArgs& a, cudaStream_t s, cudaError_t* err);
// MLA kernel: workspace slots for the pieces of cut stripes (0: no stripe can be
// cut); `grouped`: fused calls whose tiles are logical pages (cut tokens)
int mla_ws_slots(int P, int interleave, int num_tokens, int max_kv_len, int grouped);
constexpr int kMlaGroupMaxTokens = 511;  // grouped MLA plans keep two tables of this many tokens

struct OwnArgs {
  const void* q;
  const void* k_new;
  const void* v_new;
  float* o_own;
  float* lse_own;
  const int32_t* qo_indptr;
  int num_q_heads, num_kv_heads, head_dim, num_rows_bucket, num_real_rows, num_tokens, max_q_len;
  float scale;
};
int launch_own_token(const OwnArgs& a, int dtype_bf16, cudaStream_t s, cudaError_t* err);
int launch_own_token_mma(const OwnArgs& a, cudaStream_t s, cudaError_t* err);  // bf16, tensor cores
int launch_gqa_partial_mmat(const PartialArgs& a, cudaStream_t s, cudaError_t* err);  // decode rows, groups <= 8

}  // namespace cpattn
