// cp_paged_attn_partial, MLA path on CUDA cores (128 query heads over one
// latent KV head; QK over 576 latent+rope values, PV over the first 512).
//
// MLA's one latent head is striped like a GQA head (mstar PR #1124 "Context /
// Sequence Parallel 1/5", description: MLA's one latent head included; MLA
// copy_slots indexes the token axis).  CTA (chunk c, partner p, value block
// vb, query token t): thread h owns query head h, scores a segment of <= 16
// latent rows at a time against its query (held transposed in shared memory
// so a warp's 32 heads read 32 consecutive words), and accumulates 128 of the
// 512 value dims.  Rows come in through a two-stage cp.async ring.
#include "common.cuh"
#include "launch.h"
#include "split_combine.cuh"

namespace cpattn {

constexpr int kMlaHeads = 128;
constexpr int kMlaDqk = 576;
constexpr int kMlaDv = 512;
constexpr int kMlaVB = 128;                  // value dims per CTA
constexpr int kMlaVBlocks = kMlaDv / kMlaVB;  // 4
constexpr int kMlaSeg = 16;
constexpr int kMlaRowB = kMlaDqk * 2;         // 1152 bytes
constexpr size_t kMlaSmemQ = static_cast<size_t>(kMlaDqk / 2) * kMlaHeads * 4;  // bf16 pairs, transposed
constexpr size_t kMlaSmemK = static_cast<size_t>(kMlaSeg) * kMlaRowB;
constexpr size_t kMlaSmem = kMlaSmemQ + 2 * kMlaSmemK;

__global__ void __launch_bounds__(kMlaHeads) mla_partial_fma_kernel(const PartialArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* qT = reinterpret_cast<uint32_t*>(smem);  // [288][128] bf16x2 words
  uint8_t* kbuf = smem + kMlaSmemQ;                  // [2][16][576] bf16

  const int c = blockIdx.x;
  const int p = blockIdx.y / kMlaVBlocks;
  const int vb = blockIdx.y - p * kMlaVBlocks;
  const int t = blockIdx.z;
  const int h = threadIdx.x;
  const int P = a.P;

  int b = -1;
  if (a.qo_indptr != nullptr) {
    if (t < __ldg(a.qo_indptr + a.num_rows)) b = find_row(a.qo_indptr, a.num_rows, t);
  } else if (t < a.num_rows) {
    b = t;
  }
  int n_p = 0;
  if (b >= 0) {
    int L = __ldg(a.kv_len + b);
    if (L > a.max_kv_len) {
      if (c == 0 && h == 0) report(a.dev_status, CPATTN_DEV_POS_PAST_TABLE);
      L = a.max_kv_len;
    }
    n_p = (L > p) ? (L - p + P - 1) / P : 0;
  }
  const int nchunks = n_p > 0 ? (n_p + a.chunk - 1) / a.chunk : 1;
  if (c >= nchunks) return;
  const int k_begin = c * a.chunk;
  const int k_end = min(n_p, k_begin + a.chunk);
  const int nseg = k_end > k_begin ? (k_end - k_begin + a.seg - 1) / a.seg : 0;

  const int32_t* pages = nullptr;
  int npages = 0;
  if (b >= 0) {
    const int pb = __ldg(a.page_indptr + b);
    pages = a.page_indices + pb;
    npages = __ldg(a.page_indptr + b + 1) - pb;
  }
  auto page_of = [&](int k0, bool rep) -> int {
    const int j = k0 / a.ps_l;
    if (j >= npages) {
      if (rep) report(a.dev_status, CPATTN_DEV_POS_PAST_TABLE);
      return -1;
    }
    const int pg = __ldg(pages + j);
    if (pg < 0 || pg >= a.num_pages) {
      if (rep) report(a.dev_status, CPATTN_DEV_PAGE_OUT_OF_RANGE);
      return -1;
    }
    return pg;
  };
  auto issue = [&](int i) {
    if (i < nseg) {
      const int k0 = k_begin + i * a.seg;
      const int n = min(a.seg, k_end - k0);
      const int pg = page_of(k0, h == 0);
      if (pg >= 0) {
        const int64_t row = (static_cast<int64_t>(p) * a.num_pages + pg) * a.ps_l + (k0 % a.ps_l);
        const uint8_t* g = static_cast<const uint8_t*>(a.pool_k) + row * kMlaRowB;
        uint8_t* s = kbuf + (i & 1) * kMlaSmemK;
        const int pieces = n * (kMlaRowB / 16);
        for (int x = h; x < pieces; x += kMlaHeads) cp_async16(s + x * 16, g + x * 16);
      }
    }
    cp_async_commit();
  };
  issue(0);

  // query of head h, transposed: qT[d/2][h] = (q[d], q[d+1])
  if (b >= 0) {
    const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.q) +
                                                       (static_cast<int64_t>(t) * a.num_q_heads + h) * kMlaRowB);
    for (int x = 0; x < kMlaRowB / 16; ++x) {
      const uint4 u = __ldg(qrow + x);
      qT[(x * 4 + 0) * kMlaHeads + h] = u.x;
      qT[(x * 4 + 1) * kMlaHeads + h] = u.y;
      qT[(x * 4 + 2) * kMlaHeads + h] = u.z;
      qT[(x * 4 + 3) * kMlaHeads + h] = u.w;
    }
  }
  const float qs = a.scale * kLog2e;

  float m = -INFINITY, l = 0.f;
  float o[kMlaVB];
#pragma unroll
  for (int e = 0; e < kMlaVB; ++e) o[e] = 0.f;

  for (int i = 0; i < nseg; ++i) {
    issue(i + 1);
    cp_async_wait<1>();
    __syncthreads();
    const int k0 = k_begin + i * a.seg;
    const int n = page_of(k0, false) >= 0 ? min(a.seg, k_end - k0) : 0;
    const uint8_t* ks = kbuf + (i & 1) * kMlaSmemK;

    float s[kMlaSeg];
#pragma unroll
    for (int j = 0; j < kMlaSeg; ++j) s[j] = 0.f;
    for (int d8 = 0; d8 < kMlaDqk / 8; ++d8) {
      float qv[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t w = qT[(d8 * 4 + e) * kMlaHeads + h];
        qv[2 * e] = bf16_lo(w);
        qv[2 * e + 1] = bf16_hi(w);
      }
#pragma unroll
      for (int j = 0; j < kMlaSeg; ++j) {
        const uint4 u = *reinterpret_cast<const uint4*>(ks + j * kMlaRowB + d8 * 16);
        float kf[8];
        Chunk16<__nv_bfloat16>::widen(u, kf);
#pragma unroll
        for (int e = 0; e < 8; ++e) s[j] = fmaf(qv[e], kf[e], s[j]);
      }
    }
    float mt = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMlaSeg; ++j) {
      s[j] = (j < n) ? s[j] * qs : -INFINITY;
      mt = fmaxf(mt, s[j]);
    }
    if (n > 0) {
      const float mn = fmaxf(m, mt);
      const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - mn);
      l *= alpha;
#pragma unroll
      for (int e = 0; e < kMlaVB; ++e) o[e] *= alpha;
      m = mn;
#pragma unroll
      for (int j = 0; j < kMlaSeg; ++j) {
        s[j] = (j < n) ? exp2f(s[j] - m) : 0.f;
        l += s[j];
      }
      for (int j = 0; j < n; ++j) {  // only written rows: unwritten (NaN) slots never mix in
        const uint8_t* vrow = ks + j * kMlaRowB + vb * kMlaVB * 2;
#pragma unroll
        for (int d8 = 0; d8 < kMlaVB / 8; ++d8) {
          const uint4 u = *reinterpret_cast<const uint4*>(vrow + d8 * 16);
          float vf[8];
          Chunk16<__nv_bfloat16>::widen(u, vf);
#pragma unroll
          for (int e = 0; e < 8; ++e) o[d8 * 8 + e] = fmaf(s[j], vf[e], o[d8 * 8 + e]);
        }
      }
    }
    __syncthreads();  // stage i & 1 is refilled by the next step's issue
  }
  cp_async_wait<0>();

  const bool empty = (l == 0.f);
  const float inv = empty ? 0.f : 1.f / l;
  const float lse = empty ? -INFINITY : (m + log2f(l)) * kLn2;
  const int64_t orow = (static_cast<int64_t>(p) * a.num_tokens + t) * a.num_q_heads + h;
  const int64_t slot = static_cast<int64_t>(t) * P + p;
  if (nchunks == 1) {
    float4* dst = reinterpret_cast<float4*>(a.o_part + orow * kMlaDv + vb * kMlaVB);
#pragma unroll
    for (int e = 0; e < kMlaVB / 4; ++e)
      dst[e] = make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv, o[4 * e + 3] * inv);
    if (vb == 0) a.lse_part[orow] = lse;
    return;
  }
  const int64_t wrow = (slot * a.max_chunks + c) * kMlaHeads + h;
  float4* dst = reinterpret_cast<float4*>(a.ws_o + wrow * kMlaDv + vb * kMlaVB);
#pragma unroll
  for (int e = 0; e < kMlaVB / 4; ++e)
    dst[e] = make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv, o[4 * e + 3] * inv);
  if (vb == 0) a.ws_lse[wrow] = lse;
  if (!take_ticket(a.ws_cnt + slot, nchunks * kMlaVBlocks)) return;
  const int64_t orow0 = (static_cast<int64_t>(p) * a.num_tokens + t) * a.num_q_heads;
  merge_chunks(a, slot, nchunks, kMlaHeads, kMlaDv, a.o_part + orow0 * kMlaDv, a.lse_part + orow0);
  if (threadIdx.x == 0) a.ws_cnt[slot] = 0;
}

int launch_mla_partial(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  if (a.num_q_heads != kMlaHeads || a.head_dim != kMlaDqk || a.head_dim_v != kMlaDv || a.num_kv_heads != 1 ||
      a.seg > kMlaSeg)
    return CPATTN_ERR_UNSUPPORTED_SHAPE;
  *err = cudaFuncSetAttribute(mla_partial_fma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kMlaSmem));
  if (*err != cudaSuccess) return CPATTN_ERR_CUDA;
  dim3 grid(a.max_chunks, a.P * kMlaVBlocks, a.num_tokens);
  mla_partial_fma_kernel<<<grid, kMlaHeads, kMlaSmem, s>>>(a);
  *err = cudaGetLastError();
  return *err == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

}  // namespace cpattn
