// C ABI of libcpattn (declared in include/cpattn.h): argument checks on the
// host, then the kernel launches.  Nothing here allocates, synchronises or
// keeps state between calls.
#include <cstdint>

#include "cpattn.h"
#include "launch.h"

using namespace cpattn;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int dtype_bytes(int dtype) {
  if (dtype == CPATTN_DTYPE_BF16) return 2;
  if (dtype == CPATTN_DTYPE_FP32) return 4;
  return 0;
}

// Interleave size: 0 in the descriptor means 1 (plain striping).
int interleave_of(const cpattn_pool_desc* d) { return d->interleave > 1 ? d->interleave : 1; }

// Pool element type: kv_dtype 0 means the layer's dtype.
int kv_dtype_of(const cpattn_pool_desc* d) { return d->kv_dtype == 0 ? d->dtype : d->kv_dtype; }

int kv_bytes(const cpattn_pool_desc* d) {
  const int kt = kv_dtype_of(d);
  return kt == CPATTN_DTYPE_FP8_E4M3 ? 1 : dtype_bytes(kt);
}

bool is_fp8(const cpattn_pool_desc* d) { return kv_dtype_of(d) == CPATTN_DTYPE_FP8_E4M3; }

// Common descriptor checks.
int check_desc(const cpattn_pool_desc* d) {
  if (d == nullptr) return CPATTN_ERR_INVALID_ARG;
  if (d->P < 1 || d->page_size < 1 || d->interleave < 0 || d->page_size % (d->P * interleave_of(d)) != 0)
    return CPATTN_ERR_P_NOT_DIVIDING_PAGE_SIZE;
  if (d->num_pages < 1 || d->num_kv_heads < 1 || d->head_dim < 1 || d->head_dim_v < 1)
    return CPATTN_ERR_INVALID_ARG;
  const int eb = dtype_bytes(d->dtype);
  if (eb == 0) return CPATTN_ERR_INVALID_ARG;
  const int kt = kv_dtype_of(d);
  if (kt != d->dtype && kt != CPATTN_DTYPE_FP8_E4M3) return CPATTN_ERR_INVALID_ARG;
  if (kt == CPATTN_DTYPE_FP8_E4M3) {
    if (d->dtype != CPATTN_DTYPE_BF16) return CPATTN_ERR_UNSUPPORTED_SHAPE;
    const float ks = d->k_descale, vs = d->v_descale;
    if (!(ks > 0.f && ks <= 3.0e38f) || !(vs > 0.f && vs <= 3.0e38f)) return CPATTN_ERR_INVALID_ARG;
  }
  const int kb = kv_bytes(d);
  if ((d->head_dim * eb) % 16 != 0 || (d->head_dim_v * eb) % 16 != 0) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  if ((d->head_dim * kb) % 16 != 0 || (d->head_dim_v * kb) % 16 != 0) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  if (d->head_dim_v > d->head_dim) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  return CPATTN_OK;
}

bool is_mla(const cpattn_pool_desc* d) { return d->head_dim_v != d->head_dim; }

}  // namespace

namespace {

// Output side of a partial launch: per-partner partials (o_part / lse_part)
// or, fused, the merged output.
struct FusedOut {
  int fused = 0;
  const float* extra_o = nullptr;
  const float* extra_lse = nullptr;
  void* out = nullptr;
  int out_bf16 = 0;
  float* lse_out = nullptr;
  const int32_t* row_order = nullptr;
};

size_t partial_workspace(const cpattn_pool_desc* desc, int fused, int32_t num_q_heads, int32_t num_tokens,
                         int32_t max_kv_len) {
  if (check_desc(desc) != CPATTN_OK || num_q_heads < 1 || num_tokens < 0 || max_kv_len < 0) return 0;
  if (num_q_heads % desc->num_kv_heads != 0) return 0;
  PartialPlan plan;
  if (!plan_partial(is_mla(desc), fused, desc->P, interleave_of(desc), desc->page_size, desc->num_kv_heads,
                    num_q_heads, desc->head_dim, num_tokens, max_kv_len, dtype_bytes(desc->dtype), &plan))
    return 0;
  return plan.bytes();
}

int run_partial(const cpattn_pool_desc* desc, const void* pool_k, const void* pool_v, const void* q,
                int32_t num_q_heads, int32_t num_rows, int32_t num_tokens, const int32_t* qo_indptr,
                const int32_t* kv_len, int32_t max_kv_len, const int32_t* kv_page_indptr,
                const int32_t* kv_page_indices, float scale, float* o_part, float* lse_part, int lse_layout,
                const FusedOut& f, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                cudaStream_t stream) {
  int st = check_desc(desc);
  if (st != CPATTN_OK) return st;
  if (num_q_heads < 1 || num_rows < 0 || num_tokens < 0 || max_kv_len < 0) return CPATTN_ERR_INVALID_ARG;
  if (num_q_heads % desc->num_kv_heads != 0) return CPATTN_ERR_INVALID_ARG;
  if (qo_indptr == nullptr && num_tokens != num_rows) return CPATTN_ERR_INVALID_ARG;
  if (num_tokens == 0) return CPATTN_OK;
  const bool mla = is_mla(desc);
  if (pool_k == nullptr || q == nullptr || num_rows < 1 || kv_len == nullptr || kv_page_indptr == nullptr ||
      kv_page_indices == nullptr)
    return CPATTN_ERR_INVALID_ARG;
  if (!f.fused && (o_part == nullptr || lse_part == nullptr)) return CPATTN_ERR_INVALID_ARG;
  if (lse_layout != CPATTN_LSE_TOKEN_MAJOR && lse_layout != CPATTN_LSE_HEAD_MAJOR) return CPATTN_ERR_INVALID_ARG;
  if (!mla && pool_v == nullptr) return CPATTN_ERR_INVALID_ARG;
  if (mla && pool_v != nullptr && pool_v != pool_k) return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(pool_k) || !aligned16(pool_v) || !aligned16(q) || !aligned16(o_part) || !aligned16(workspace))
    return CPATTN_ERR_MISALIGNED;
  if (mla && desc->dtype != CPATTN_DTYPE_BF16) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  // E4M3 pools: GQA (the MLA kernel reads bf16 latent rows only)
  if (is_fp8(desc) && mla) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  // multi-token rows over a bf16 pool: the kernel's copy warps pass pool row
  // indices as 32-bit values (checked here, before the one-token rows' launch)
  if (!mla && qo_indptr != nullptr && !is_fp8(desc) &&
      static_cast<int64_t>(desc->num_pages) * desc->num_kv_heads * desc->page_size >= (int64_t{1} << 31))
    return CPATTN_ERR_UNSUPPORTED_SHAPE;

  PartialPlan plan;
  if (!plan_partial(mla, f.fused, desc->P, interleave_of(desc), desc->page_size, desc->num_kv_heads, num_q_heads,
                    desc->head_dim, num_tokens, max_kv_len, dtype_bytes(desc->dtype), &plan))
    return CPATTN_ERR_UNSUPPORTED_SHAPE;
  const size_t need = plan.bytes();
  if (workspace == nullptr || workspace_bytes < need) return CPATTN_ERR_WORKSPACE_TOO_SMALL;

  // workspace: chunk partials, chunk LSEs, partner partials, partner LSEs
  // (fused), then the two ticket arrays side by side (one memset)
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  PartialArgs a;
  size_t off = 0;
  a.ws_o = reinterpret_cast<float*>(ws + off);
  off += al(plan.ws_o_floats * 4);
  a.ws_lse = reinterpret_cast<float*>(ws + off);
  off += al(plan.ws_lse_floats * 4);
  float* ws_part = reinterpret_cast<float*>(ws + off);
  off += al(plan.ws_part_floats * 4);
  float* ws_part_lse = reinterpret_cast<float*>(ws + off);
  off += al(plan.ws_part_lse_floats * 4);
  a.ws_cnt = reinterpret_cast<int32_t*>(ws + off);
  const size_t cnt_bytes = al(plan.ws_cnt_ints * 4);
  a.ws_pair = reinterpret_cast<int32_t*>(ws + off + cnt_bytes);
  const size_t ticket_bytes = cnt_bytes + plan.ws_pair_ints * 4;
  if (f.fused) {
    o_part = ws_part;
    lse_part = ws_part_lse;
  }
  a.pool_k = pool_k;
  a.pool_v = mla ? pool_k : pool_v;
  a.q = q;
  a.o_part = o_part;
  a.lse_part = lse_part;
  // LSE of (partner, token, head): [P][T][Hq], or [P][Hq][T] (FlashAttention's [H, B] per partner);
  // the partner partials of fused calls are internal and token-major
  const int64_t TH = static_cast<int64_t>(num_tokens) * num_q_heads;
  const bool head_major = !f.fused && lse_layout == CPATTN_LSE_HEAD_MAJOR;
  a.lse_sp = TH;
  a.lse_st = head_major ? 1 : num_q_heads;
  a.lse_sh = head_major ? num_tokens : 1;
  a.qo_indptr = qo_indptr;
  a.kv_len = kv_len;
  a.page_indptr = kv_page_indptr;
  a.page_indices = kv_page_indices;
  a.dev_status = dev_status;
  a.P = desc->P;
  a.interleave = interleave_of(desc);
  a.page_size = desc->page_size;
  a.ps_l = desc->page_size / desc->P;
  a.ps_shift = -1;
  for (int sh = 0; sh < 31; ++sh)
    if ((1 << sh) == a.ps_l) a.ps_shift = sh;
  a.num_pages = desc->num_pages;
  a.num_kv_heads = desc->num_kv_heads;
  a.num_q_heads = num_q_heads;
  a.head_dim = desc->head_dim;
  a.head_dim_v = desc->head_dim_v;
  a.num_rows = num_rows;
  a.num_tokens = num_tokens;
  a.max_kv_len = max_kv_len;
  a.seg = plan.seg;
  a.chunk = plan.chunk;
  a.max_chunks = plan.max_chunks;
  a.scale = scale;
  a.kv_fp8 = is_fp8(desc);
  a.k_descale = desc->k_descale;
  a.v_descale = desc->v_descale;
  a.fused = f.fused;
  a.extra_o = f.extra_o;
  a.extra_lse = f.extra_lse;
  a.out = f.out;
  a.out_bf16 = f.out_bf16;
  a.lse_out = f.lse_out;
  a.row_order = f.row_order;

  // tickets start from zero (each call's last arrivals also reset them)
  if (plan.max_chunks > 1 || f.fused) {
    if (cudaMemsetAsync(a.ws_cnt, 0, ticket_bytes, stream) != cudaSuccess) return CPATTN_ERR_CUDA;
  }
  cudaError_t err = cudaSuccess;
  if (mla) return launch_mla_partial(a, stream, &err);
  return launch_gqa_partial(a, desc->dtype == CPATTN_DTYPE_BF16, stream, &err);
}

}  // namespace

extern "C" {

int cpattn_version(void) { return CPATTN_VERSION; }

const char* cpattn_status_string(int status) {
  switch (status) {
    case CPATTN_OK: return "ok";
    case CPATTN_ERR_INVALID_ARG: return "invalid argument";
    case CPATTN_ERR_P_NOT_DIVIDING_PAGE_SIZE: return "P and interleave must be >= 1 and P * interleave divide page_size";
    case CPATTN_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (head dims / group size)";
    case CPATTN_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case CPATTN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case CPATTN_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}

size_t cpattn_pool_bytes(const cpattn_pool_desc* d, int which_v) {
  if (check_desc(d) != CPATTN_OK) return 0;
  const size_t rows = static_cast<size_t>(d->P) * d->num_pages * d->num_kv_heads * (d->page_size / d->P);
  return rows * (which_v ? d->head_dim_v : d->head_dim) * kv_bytes(d);
}

int cp_kv_write(const cpattn_pool_desc* desc, void* pool_k, void* pool_v, const void* k_new, const void* v_new,
                const int32_t* positions, const int32_t* qo_indptr, int32_t num_rows, int32_t num_tokens,
                const int32_t* kv_page_indptr, const int32_t* kv_page_indices, int32_t* dev_status,
                cudaStream_t stream) {
  int st = check_desc(desc);
  if (st != CPATTN_OK) return st;
  if (num_rows < 0 || num_tokens < 0) return CPATTN_ERR_INVALID_ARG;
  if (num_tokens == 0) return CPATTN_OK;
  const bool mla = is_mla(desc);
  if (pool_k == nullptr || k_new == nullptr || positions == nullptr || qo_indptr == nullptr ||
      kv_page_indptr == nullptr || kv_page_indices == nullptr || num_rows < 1)
    return CPATTN_ERR_INVALID_ARG;
  if (!mla && (pool_v == nullptr || v_new == nullptr)) return CPATTN_ERR_INVALID_ARG;
  if (mla && (pool_v != nullptr || v_new != nullptr)) return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(pool_k) || !aligned16(pool_v) || !aligned16(k_new) || !aligned16(v_new))
    return CPATTN_ERR_MISALIGNED;
  const int eb = dtype_bytes(desc->dtype);
  WriteArgs a;
  a.pool_k = pool_k;
  a.pool_v = pool_v;
  a.k_new = k_new;
  a.v_new = v_new;
  a.positions = positions;
  a.qo_indptr = qo_indptr;
  a.page_indptr = kv_page_indptr;
  a.page_indices = kv_page_indices;
  a.dev_status = dev_status;
  a.P = desc->P;
  a.interleave = interleave_of(desc);
  a.page_size = desc->page_size;
  a.num_pages = desc->num_pages;
  a.num_kv_heads = desc->num_kv_heads;
  a.num_rows = num_rows;
  a.num_tokens = num_tokens;
  const int kb = kv_bytes(desc);
  a.row_bytes_k = desc->head_dim * kb;
  a.row_bytes_v = mla ? 0 : desc->head_dim_v * kb;
  a.src_row_bytes_k = desc->head_dim * eb;
  a.src_row_bytes_v = mla ? 0 : desc->head_dim_v * eb;
  a.quant_fp8 = is_fp8(desc);
  a.k_descale = desc->k_descale;
  a.v_descale = desc->v_descale;
  return launch_kv_write(a, stream) == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

size_t cp_paged_attn_workspace_bytes(const cpattn_pool_desc* desc, int32_t num_q_heads, int32_t num_tokens,
                                     int32_t max_kv_len) {
  return partial_workspace(desc, 0, num_q_heads, num_tokens, max_kv_len);
}

size_t cp_paged_attn_fused_workspace_bytes(const cpattn_pool_desc* desc, int32_t num_q_heads, int32_t num_tokens,
                                           int32_t max_kv_len) {
  return partial_workspace(desc, 1, num_q_heads, num_tokens, max_kv_len);
}

int cp_paged_attn_partial(const cpattn_pool_desc* desc, const void* pool_k, const void* pool_v, const void* q,
                          int32_t num_q_heads, int32_t num_rows, int32_t num_tokens, const int32_t* qo_indptr,
                          const int32_t* kv_len, int32_t max_kv_len, const int32_t* kv_page_indptr,
                          const int32_t* kv_page_indices, float scale, float* o_part, float* lse_part,
                          void* workspace, size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream) {
  FusedOut none;
  return run_partial(desc, pool_k, pool_v, q, num_q_heads, num_rows, num_tokens, qo_indptr, kv_len, max_kv_len,
                     kv_page_indptr, kv_page_indices, scale, o_part, lse_part, CPATTN_LSE_TOKEN_MAJOR, none,
                     workspace, workspace_bytes, dev_status, stream);
}

int cp_paged_attn_partial_ex(const cpattn_pool_desc* desc, const void* pool_k, const void* pool_v, const void* q,
                             int32_t num_q_heads, int32_t num_rows, int32_t num_tokens, const int32_t* qo_indptr,
                             const int32_t* kv_len, int32_t max_kv_len, const int32_t* kv_page_indptr,
                             const int32_t* kv_page_indices, float scale, float* o_part, float* lse_part,
                             int32_t lse_layout, const int32_t* row_order, void* workspace, size_t workspace_bytes,
                             int32_t* dev_status, cudaStream_t stream) {
  FusedOut none;
  none.row_order = qo_indptr == nullptr ? row_order : nullptr;
  return run_partial(desc, pool_k, pool_v, q, num_q_heads, num_rows, num_tokens, qo_indptr, kv_len, max_kv_len,
                     kv_page_indptr, kv_page_indices, scale, o_part, lse_part, lse_layout, none, workspace,
                     workspace_bytes, dev_status, stream);
}

int cp_paged_attn_fused(const cpattn_pool_desc* desc, const void* pool_k, const void* pool_v, const void* q,
                        int32_t num_q_heads, int32_t num_rows, int32_t num_tokens, const int32_t* qo_indptr,
                        const int32_t* kv_len, int32_t max_kv_len, const int32_t* kv_page_indptr,
                        const int32_t* kv_page_indices, const int32_t* row_order, float scale,
                        const float* extra_o, const float* extra_lse,
                        int32_t out_dtype, void* out, float* lse_out, void* workspace, size_t workspace_bytes,
                        int32_t* dev_status, cudaStream_t stream) {
  const int st = check_desc(desc);
  if (st != CPATTN_OK) return st;
  if (out_dtype != CPATTN_DTYPE_BF16 && out_dtype != CPATTN_DTYPE_FP32) return CPATTN_ERR_INVALID_ARG;
  if ((extra_o == nullptr) != (extra_lse == nullptr)) return CPATTN_ERR_INVALID_ARG;
  if (num_tokens > 0 && out == nullptr) return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(extra_o)) return CPATTN_ERR_MISALIGNED;
  if (out_dtype == CPATTN_DTYPE_BF16 && (desc->head_dim_v % 8) != 0) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  FusedOut f;
  f.fused = 1;
  f.extra_o = extra_o;
  f.extra_lse = extra_lse;
  f.out = out;
  f.out_bf16 = out_dtype == CPATTN_DTYPE_BF16;
  f.lse_out = lse_out;
  f.row_order = qo_indptr == nullptr ? row_order : nullptr;
  return run_partial(desc, pool_k, pool_v, q, num_q_heads, num_rows, num_tokens, qo_indptr, kv_len, max_kv_len,
                     kv_page_indptr, kv_page_indices, scale, nullptr, nullptr, CPATTN_LSE_TOKEN_MAJOR, f, workspace,
                     workspace_bytes, dev_status, stream);
}

int own_token_attn(const void* q, const void* k_new, const void* v_new, int32_t num_q_heads, int32_t num_kv_heads,
                   int32_t head_dim, int32_t head_dim_v, int32_t dtype, const int32_t* qo_indptr,
                   int32_t num_rows_bucket, int32_t num_real_rows, int32_t num_tokens, int32_t max_q_len,
                   float scale, float* o_own, float* lse_own, cudaStream_t stream) {
  const int eb = dtype_bytes(dtype);
  if (eb == 0 || num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0 || num_tokens < 0 ||
      num_rows_bucket < 1 || num_real_rows < 0 || num_real_rows > num_rows_bucket || max_q_len < 0)
    return CPATTN_ERR_INVALID_ARG;
  // MLA: one latent head, keys of 576 values whose first 512 are the value (v_new NULL)
  const bool mla = num_kv_heads == 1 && head_dim == 576 && head_dim_v == 512;
  if (mla ? (dtype != CPATTN_DTYPE_BF16 || v_new != nullptr) : head_dim != head_dim_v)
    return CPATTN_ERR_UNSUPPORTED_SHAPE;
  if (num_tokens == 0) return CPATTN_OK;
  if (q == nullptr || k_new == nullptr || qo_indptr == nullptr || o_own == nullptr || lse_own == nullptr)
    return CPATTN_ERR_INVALID_ARG;
  if (v_new == nullptr) v_new = k_new;  // value = prefix of the key row
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(o_own)) return CPATTN_ERR_MISALIGNED;
  OwnArgs a;
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.o_own = o_own;
  a.lse_own = lse_own;
  a.qo_indptr = qo_indptr;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.num_rows_bucket = num_rows_bucket;
  a.num_real_rows = num_real_rows;
  a.num_tokens = num_tokens;
  a.max_q_len = max_q_len;
  a.scale = scale;
  cudaError_t err = cudaSuccess;
  return launch_own_token(a, dtype == CPATTN_DTYPE_BF16, stream, &err);
}

int lse_merge(int32_t num_partials, const float* o_parts, const float* lse_parts, int64_t stride_o,
              int64_t stride_lse, int32_t num_tokens, int32_t num_heads, int32_t head_dim_v, int32_t out_dtype,
              void* out, float* lse_out, cudaStream_t stream) {
  if (num_partials < 1 || num_tokens < 0 || num_heads < 1 || head_dim_v < 4 || head_dim_v % 4 != 0)
    return CPATTN_ERR_INVALID_ARG;
  if (out_dtype != CPATTN_DTYPE_BF16 && out_dtype != CPATTN_DTYPE_FP32) return CPATTN_ERR_INVALID_ARG;
  if (num_tokens == 0) return CPATTN_OK;
  if (o_parts == nullptr || lse_parts == nullptr || out == nullptr) return CPATTN_ERR_INVALID_ARG;
  const int64_t per_o = static_cast<int64_t>(num_tokens) * num_heads * head_dim_v;
  const int64_t per_l = static_cast<int64_t>(num_tokens) * num_heads;
  if (num_partials > 1 && (stride_o < per_o || stride_lse < per_l)) return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(out) || (stride_o % 4) != 0) return CPATTN_ERR_MISALIGNED;
  if (out_dtype == CPATTN_DTYPE_BF16 && (head_dim_v % 8) != 0) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  MergeArgs a;
  a.num_partials = num_partials;
  a.o_parts = o_parts;
  a.lse_parts = lse_parts;
  a.stride_o = stride_o;
  a.stride_lse = stride_lse;
  a.num_tokens = num_tokens;
  a.num_heads = num_heads;
  a.head_dim_v = head_dim_v;
  a.out_bf16 = out_dtype == CPATTN_DTYPE_BF16;
  a.out = out;
  a.lse_out = lse_out;
  return launch_lse_merge(a, stream) == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

int lse_merge_views(int32_t num_views, const cpattn_partial_view* views, int32_t num_tokens, int32_t num_heads,
                    int32_t head_dim_v, int32_t out_dtype, void* out, int64_t out_stride_token,
                    int64_t out_stride_head, float* lse_out, int64_t lse_out_stride_token,
                    int64_t lse_out_stride_head, cudaStream_t stream) {
  if (num_views < 1 || num_views > CPATTN_MAX_MERGE_VIEWS || views == nullptr || num_tokens < 0 || num_heads < 1 ||
      head_dim_v < 4 || head_dim_v % 4 != 0)
    return CPATTN_ERR_INVALID_ARG;
  if (out_dtype != CPATTN_DTYPE_BF16 && out_dtype != CPATTN_DTYPE_FP32) return CPATTN_ERR_INVALID_ARG;
  if (num_tokens == 0) return CPATTN_OK;
  if (out == nullptr) return CPATTN_ERR_INVALID_ARG;
  // 16-byte row starts: every row pointer and row stride a multiple of 4 elements
  if (!aligned16(out) || out_stride_token % 4 != 0 || out_stride_head % 4 != 0) return CPATTN_ERR_MISALIGNED;
  MergeViewArgs a;
  a.n = num_views;
  for (int i = 0; i < num_views; ++i) {
    const cpattn_partial_view& v = views[i];
    if (v.o == nullptr || v.lse == nullptr) return CPATTN_ERR_INVALID_ARG;
    if (!aligned16(v.o) || v.o_stride_token % 4 != 0 || v.o_stride_head % 4 != 0) return CPATTN_ERR_MISALIGNED;
    a.v[i].o = v.o;
    a.v[i].lse = v.lse;
    a.v[i].o_st = v.o_stride_token;
    a.v[i].o_sh = v.o_stride_head;
    a.v[i].lse_st = v.lse_stride_token;
    a.v[i].lse_sh = v.lse_stride_head;
  }
  a.num_tokens = num_tokens;
  a.num_heads = num_heads;
  a.head_dim_v = head_dim_v;
  a.out_bf16 = out_dtype == CPATTN_DTYPE_BF16;
  a.out = out;
  a.out_st = out_stride_token;
  a.out_sh = out_stride_head;
  a.lse_out = lse_out;
  a.lse_out_st = lse_out_stride_token;
  a.lse_out_sh = lse_out_stride_head;
  return launch_lse_merge_views(a, stream) == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

}  // extern "C"
