// cp_kv_write: copy a step's new K/V rows into the P-way striped paged pool.
//
// Placement (mstar PR #1124 "Context / Sequence Parallel 1/5", description):
// offset off of a logical page belongs to partner off % P at physical slot
// off / P of the same page id.  With an interleave size I (vLLM's
// cp_kv_cache_interleave_size), runs of I offsets go together: partner
// (off / I) % P, physical slot (off / (I * P)) * I + off % I.  The review thread of that PR shows the failure
// this kernel must avoid: taking the slot at the logical page size, which makes
// every partner write every token at offsets up to page_size - 1.
//
// One thread moves one 16-byte chunk of one (token, KV head) row; the chunks of
// a row are adjacent threads, so both the read of k_new and the write into the
// pool are coalesced 16-byte accesses.
#include "common.cuh"
#include "launch.h"

namespace cpattn {

// E4M3 code of a float32 value, rounded once to the nearest E4M3 value (ties
// to the even code), magnitudes of 448 and more (and infinities) saturated to
// 448, NaN to 0x7F.  Written from the format: normal codes are the float32
// exponent rebiased from 127 to 7 and the mantissa rounded to 3 bits;
// below 2^-6 the codes are the multiples m * 2^-9 (m = 0..8).
__device__ __forceinline__ uint32_t e4m3_rn_satfinite(float x) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t sign = (u >> 24) & 0x80u;
  const float ax = fabsf(x);
  if (ax != ax) return 0x7Fu;
  if (ax >= 448.f) return sign | 0x7Eu;
  if (ax < 0.015625f) return sign | static_cast<uint32_t>(__float2int_rn(ax * 512.f));  // exact scaling
  const uint32_t bits = u & 0x7fffffffu;
  const uint32_t r = (bits + 0x7ffffu + ((bits >> 20) & 1u)) >> 20;  // exponent | 3 mantissa bits, to nearest even
  return sign | (r - ((127u - 7u) << 3));
}

// E4M3 codes of 16 bf16 values (byte offset src_off of src, chunk c) divided
// by the descale: IEEE float32 quotient, then e4m3_rn_satfinite.
__device__ __forceinline__ void store_fp8_chunk(const void* src, int64_t src_off, void* dst, int64_t dst_off, int c,
                                                float descale) {
  const uint4* s = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(src) + src_off) + 2 * c;
  const uint4 w0 = __ldg(s), w1 = __ldg(s + 1);
  const uint32_t in[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t pair = in[2 * i + j];
      const float lo = __fdiv_rn(bf16_lo(pair), descale);
      const float hi = __fdiv_rn(bf16_hi(pair), descale);
      const uint32_t b0 = e4m3_rn_satfinite(lo);
      const uint32_t b1 = e4m3_rn_satfinite(hi);
      word |= (b0 | (b1 << 8)) << (16 * j);
    }
    out[i] = word;
  }
  *(reinterpret_cast<uint4*>(static_cast<uint8_t*>(dst) + dst_off) + c) = make_uint4(out[0], out[1], out[2], out[3]);
}

__global__ void __launch_bounds__(256) kv_write_kernel(const WriteArgs a, int chunks_per_row) {
  pdl_trigger();
  pdl_wait();
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t per_token = static_cast<int64_t>(a.num_kv_heads) * chunks_per_row;
  const int64_t total = per_token * a.num_tokens;
  if (gid >= total) return;
  const int t = static_cast<int>(gid / per_token);
  const int rem = static_cast<int>(gid - static_cast<int64_t>(t) * per_token);
  const int h = rem / chunks_per_row;
  const int c = rem - h * chunks_per_row;

  const int end = __ldg(a.qo_indptr + a.num_rows);
  if (t >= end) return;  // padding token past the last row
  const int pos = __ldg(a.positions + t);
  if (pos < 0) return;  // padding token
  const int b = find_row(a.qo_indptr, a.num_rows, t);

  const int page_idx = pos / a.page_size;
  const int pbeg = __ldg(a.page_indptr + b);
  const int pend = __ldg(a.page_indptr + b + 1);
  if (page_idx >= pend - pbeg) {
    if (c == 0 && h == 0) report(a.dev_status, CPATTN_DEV_POS_PAST_TABLE);
    return;
  }
  const int page = __ldg(a.page_indices + pbeg + page_idx);
  if (page < 0 || page >= a.num_pages) {
    if (c == 0 && h == 0) report(a.dev_status, CPATTN_DEV_PAGE_OUT_OF_RANGE);
    return;
  }
  const int off = pos - page_idx * a.page_size;
  const int run = off / a.interleave;
  const int partner = run % a.P;
  const int slot = (run / a.P) * a.interleave + (off - run * a.interleave);
  const int ps_l = a.page_size / a.P;
  // row index inside the pool tensor [P][num_pages][H][ps_l]
  const int64_t prow =
      ((static_cast<int64_t>(partner) * a.num_pages + page) * a.num_kv_heads + h) * ps_l + slot;
  const int64_t srow = static_cast<int64_t>(t) * a.num_kv_heads + h;

  if (a.quant_fp8) {
    // 16 codes of the pool row from 16 bf16 values of the new row
    if (c * 16 < a.row_bytes_k) store_fp8_chunk(a.k_new, srow * a.src_row_bytes_k, a.pool_k, prow * a.row_bytes_k, c,
                                               a.k_descale);
    if (a.pool_v != nullptr && c * 16 < a.row_bytes_v)
      store_fp8_chunk(a.v_new, srow * a.src_row_bytes_v, a.pool_v, prow * a.row_bytes_v, c, a.v_descale);
    return;
  }
  if (c * 16 < a.row_bytes_k) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.k_new) +
                                                      srow * a.row_bytes_k) + c;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.pool_k) + prow * a.row_bytes_k) + c;
    *dst = __ldg(src);
  }
  if (a.pool_v != nullptr && c * 16 < a.row_bytes_v) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.v_new) +
                                                      srow * a.row_bytes_v) + c;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.pool_v) + prow * a.row_bytes_v) + c;
    *dst = __ldg(src);
  }
}

cudaError_t launch_kv_write(const WriteArgs& a, cudaStream_t s) {
  const int rb = a.row_bytes_k > a.row_bytes_v ? a.row_bytes_k : a.row_bytes_v;
  const int chunks = rb / 16;
  const int64_t total = static_cast<int64_t>(a.num_tokens) * a.num_kv_heads * chunks;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  return launch_pdl(kv_write_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, s, a, chunks);
}

}  // namespace cpattn
