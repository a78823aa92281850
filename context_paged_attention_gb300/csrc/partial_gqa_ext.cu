// cp_paged_attn_partial, GQA rows with several query tokens (bf16 pools,
// tensor cores).
//
// A non-decode step attends the pool for its context only and every new token
// of a row sees the same context (mstar PR #1124 "Context / Sequence Parallel
// 1/5", description: context-only plans; vLLM "[Core] Add explicit layer
// parallel plans", _forward_with_dcp: the context partial over the paged
// cache).  So the queries of a row's new tokens form a dense tile against the
// partner's stripe of that context: this kernel reads each stripe key once per
// block of 64 / G tokens instead of once per token.
//
// CTA = (chunk, partner p, KV head h, token block j of 64 / G consecutive
// tokens).  It handles the rows of two or more tokens that intersect the block
// (rows of one token are left to the decode kernel).  The 64 query rows
// (token, head) are split over 4 warps of 16 rows; all warps consume the same
// 16-key stages, copied by all threads with 16-byte cp.async into an
// XOR-swizzled ring (the stripe addressing and the tile math are those of
// partial_gqa_mma.cu).  A chunk split of a stripe is merged by the last CTA to
// arrive, per token.
#include "gqa_core.cuh"
#include "launch.h"
#include "mma_sync.cuh"
#include "split_combine.cuh"

namespace cpattn {

constexpr int kExtWarps = 4;
constexpr int kExtStages = 4;
constexpr int kExtKeys = 16;

template <int D, int G>
__global__ void __launch_bounds__(kExtWarps * 32, 2) gqa_partial_ext_kernel(const PartialArgs a) {
  constexpr int NW = kExtWarps;
  constexpr int NST = kExtStages;
  constexpr int KT = kExtKeys;
  constexpr int ROWB = D * 2;
  constexpr int CH = ROWB / 16;
  constexpr int STAGE_B = KT * ROWB;
  constexpr int KSTEPS = D / 16;
  constexpr int NT = D / 8;
  constexpr int QB = NW * 16 / G;  // tokens per block
  static_assert(G >= 1 && G <= 16 && NT % 4 == 0, "shape");
  extern __shared__ __align__(128) uint8_t smem[];
  int* spg = reinterpret_cast<int*>(smem + static_cast<size_t>(NST) * STAGE_B * 2);

  const int c = blockIdx.x;
  const int p = blockIdx.y / a.num_kv_heads;
  const int h = blockIdx.y - p * a.num_kv_heads;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int quad = lane >> 2;
  const int qi = lane & 3;
  const int mrow = lane & 7;
  const int mi = lane >> 3;
  const int P = a.P;
  const uint8_t* poolk = static_cast<const uint8_t*>(a.pool_k);
  const uint8_t* poolv = static_cast<const uint8_t*>(a.pool_v);
  const float sl = a.scale * kLog2e;

  const int t_lo = blockIdx.z * QB;
  const int t_real = __ldg(a.qo_indptr + a.num_rows);
  const int t_hi = min(t_lo + QB, t_real);
  if (c == 0) {
    // padding tokens past the last row: this (partner, KV head)'s 0 / -inf
    for (int tok = max(t_lo, t_real); tok < min(t_lo + QB, a.num_tokens); ++tok) {
      const int64_t orow0 = (static_cast<int64_t>(p) * a.num_tokens + tok) * a.num_q_heads + h * G;
      for (int x = tid; x < G * D; x += blockDim.x) a.o_part[orow0 * D + x] = 0.f;
      if (tid < G) a.lse_part[orow0 + tid] = -INFINITY;
    }
  }
  if (t_lo >= t_hi) return;

  for (int b = find_row(a.qo_indptr, a.num_rows, t_lo); b < a.num_rows; ++b) {
    const int r0 = __ldg(a.qo_indptr + b);
    if (r0 >= t_hi) break;
    const int r1 = __ldg(a.qo_indptr + b + 1);
    if (r1 - r0 < 2) continue;  // one-token rows: the decode kernel's
    const int s0 = max(r0, t_lo), s1 = min(r1, t_hi);
    if (s1 <= s0) continue;

    int L = __ldg(a.kv_len + b);
    if (L > a.max_kv_len) {
      if (c == 0 && tid == 0) report(a.dev_status, CPATTN_DEV_POS_PAST_TABLE);
      L = a.max_kv_len;
    }
    const int n_p = (L > p) ? (L - p + P - 1) / P : 0;
    const int nchunks = n_p > 0 ? (n_p + a.chunk - 1) / a.chunk : 1;
    if (c >= nchunks) continue;
    const int k_begin = c * a.chunk;
    const int k_end = min(n_p, k_begin + a.chunk);
    const int nstage = k_end > k_begin ? (k_end - k_begin + KT - 1) / KT : 0;

    // rows of this warp: r = 16 * warp + quad (+ 8): token s0 + r / G, head h * G + r % G
    const int ra = warp * 16 + quad, rb = ra + 8;
    const int ta = s0 + ra / G, tb = s0 + rb / G;
    const bool oka = ta < s1, okb = tb < s1;
    uint32_t qa[KSTEPS][4];
    {
      const uint32_t* qwa = reinterpret_cast<const uint32_t*>(
          static_cast<const uint8_t*>(a.q) + (static_cast<int64_t>(oka ? ta : s0) * a.num_q_heads + h * G + ra % G) * ROWB);
      const uint32_t* qwb = reinterpret_cast<const uint32_t*>(
          static_cast<const uint8_t*>(a.q) + (static_cast<int64_t>(okb ? tb : s0) * a.num_q_heads + h * G + rb % G) * ROWB);
#pragma unroll
      for (int s = 0; s < KSTEPS; ++s) {
        const int w0 = s * 8 + qi;
        qa[s][0] = oka ? __ldg(qwa + w0) : 0u;
        qa[s][1] = okb ? __ldg(qwb + w0) : 0u;
        qa[s][2] = oka ? __ldg(qwa + w0 + 4) : 0u;
        qa[s][3] = okb ? __ldg(qwb + w0 + 4) : 0u;
      }
    }

    // page ids of the chunk
    const int j0 = k_begin / a.ps_l;
    if (nstage > 0) {
      const int j1 = (k_end - 1) / a.ps_l;
      const int pb = __ldg(a.page_indptr + b);
      const int npages = __ldg(a.page_indptr + b + 1) - pb;
      for (int x = tid; x <= j1 - j0; x += blockDim.x) {
        const int j = j0 + x;
        int pg = -1;
        if (j >= npages) {
          report(a.dev_status, CPATTN_DEV_POS_PAST_TABLE);
        } else {
          pg = __ldg(a.page_indices + pb + j);
          if (pg < 0 || pg >= a.num_pages) {
            report(a.dev_status, CPATTN_DEV_PAGE_OUT_OF_RANGE);
            pg = -1;
          }
        }
        spg[x] = pg;
      }
    }
    __syncthreads();
    const int64_t head_row0 = static_cast<int64_t>(p) * a.num_pages * a.num_kv_heads + h;
    auto row_of = [&](int k) -> int64_t {
      if (k >= k_end) return -1;
      const int j = k / a.ps_l;
      const int pg = spg[j - j0];
      if (pg < 0) return -1;
      return (head_row0 + static_cast<int64_t>(pg) * a.num_kv_heads) * a.ps_l + (k - j * a.ps_l);
    };
    // all threads copy a stage: 16 keys x CH chunks x (K, V)
    auto issue = [&](int i) {
      if (i < nstage) {
        const int k0 = k_begin + i * KT;
        uint8_t* sk = smem + (i % NST) * STAGE_B * 2;
        uint8_t* sv = sk + STAGE_B;
        for (int x = tid; x < KT * CH; x += blockDim.x) {
          const int key = x / CH;
          const int ch = x - key * CH;
          const int64_t row = row_of(k0 + key);
          const int soff = (key * CH + (ch ^ (key & 7))) * 16;
          if (row >= 0) {
            cp_async16(sk + soff, poolk + row * ROWB + ch * 16);
            cp_async16(sv + soff, poolv + row * ROWB + ch * 16);
          } else {
            *reinterpret_cast<uint4*>(sv + soff) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      cp_async_commit();
    };

    float o[NT][4];
#pragma unroll
    for (int u = 0; u < NT; ++u) o[u][0] = o[u][1] = o[u][2] = o[u][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

#pragma unroll
    for (int i = 0; i < NST - 1; ++i) issue(i);
    for (int i = 0; i < nstage; ++i) {
      cp_async_wait<NST - 2>();
      __syncthreads();  // stage i complete for all threads; stage i - 1 no longer read
      issue(i + NST - 1);
      const uint32_t sk = smem_u32(smem + (i % NST) * STAGE_B * 2);
      const uint32_t sv = sk + STAGE_B;
      uint32_t vm;
      {
        const int k = k_begin + i * KT + (lane & (KT - 1));
        vm = __ballot_sync(0xffffffffu, row_of(k) >= 0) & 0xffffu;
      }
      float s[2][4], s_alt[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[j][e] = s_alt[j][e] = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < KSTEPS; s2 += 2) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int key = j * 8 + mrow;
          const int ch = s2 * 2 + mi;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(sk + (key * CH + (ch ^ (key & 7))) * 16, b0, b1, b2, b3);
          mma_bf16(s[j], qa[s2], b0, b1);
          mma_bf16(s_alt[j], qa[s2 + 1], b2, b3);
        }
      }
      float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool ok = (vm >> (j * 8 + 2 * qi + e)) & 1u;
          s[j][e] = ok ? (s[j][e] + s_alt[j][e]) * sl : -INFINITY;
          s[j][e + 2] = ok ? (s[j][e + 2] + s_alt[j][e + 2]) * sl : -INFINITY;
          bm0 = fmaxf(bm0, s[j][e]);
          bm1 = fmaxf(bm1, s[j][e + 2]);
        }
      }
      bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 1));
      bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 2));
      bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 1));
      bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 2));
      const bool up0 = bm0 > m0 + 8.f;
      const bool up1 = bm1 > m1 + 8.f;
      if (__any_sync(0xffffffffu, up0 || up1)) {
        const float a0 = up0 ? exp2f(m0 - bm0) : 1.f;
        const float a1 = up1 ? exp2f(m1 - bm1) : 1.f;
        if (up0) m0 = bm0;
        if (up1) m1 = bm1;
        l0 *= a0;
        l1 *= a1;
#pragma unroll
        for (int u = 0; u < NT; ++u) {
          o[u][0] *= a0;
          o[u][1] *= a0;
          o[u][2] *= a1;
          o[u][3] *= a1;
        }
      }
      uint32_t pa[4], pl[4];
      {
        const float p00 = exp2f(s[0][0] - m0), p01 = exp2f(s[0][1] - m0);
        const float p02 = exp2f(s[0][2] - m1), p03 = exp2f(s[0][3] - m1);
        const float p10 = exp2f(s[1][0] - m0), p11 = exp2f(s[1][1] - m0);
        const float p12 = exp2f(s[1][2] - m1), p13 = exp2f(s[1][3] - m1);
        l0 += (p00 + p01) + (p10 + p11);
        l1 += (p02 + p03) + (p12 + p13);
        split_bf16(p00, p01, pa[0], pl[0]);
        split_bf16(p02, p03, pa[1], pl[1]);
        split_bf16(p10, p11, pa[2], pl[2]);
        split_bf16(p12, p13, pa[3], pl[3]);
      }
      {
        const int key = (mi & 1) * 8 + mrow;
#pragma unroll
        for (int u = 0; u < NT; u += 4) {
          uint32_t bv[2][4];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int ch = u + 2 * hh + (mi >> 1);
            ldsm_x4_t(sv + (key * CH + (ch ^ (key & 7))) * 16, bv[hh][0], bv[hh][1], bv[hh][2], bv[hh][3]);
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            mma_bf16(o[u + 2 * hh], pa, bv[hh][0], bv[hh][1]);
            mma_bf16(o[u + 2 * hh + 1], pa, bv[hh][2], bv[hh][3]);
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            mma_bf16(o[u + 2 * hh], pl, bv[hh][0], bv[hh][1]);
            mma_bf16(o[u + 2 * hh + 1], pl, bv[hh][2], bv[hh][3]);
          }
        }
      }
    }
    cp_async_wait<0>();
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    // ---- rows of this warp: normalised output and LSE, to o_part or the workspace
    const bool single = (nchunks == 1);
    auto emit = [&](int tok, int g, float m, float l, int half) {
      const bool empty = (l == 0.f);
      const float inv = empty ? 0.f : 1.f / l;
      const float lse = empty ? -INFINITY : (m + log2f(l)) * kLn2;
      float* dst;
      float* ldst;
      if (single) {
        const int64_t orow = (static_cast<int64_t>(p) * a.num_tokens + tok) * a.num_q_heads + h * G + g;
        dst = a.o_part + orow * D;
        ldst = a.lse_part + orow;
      } else {
        const int64_t slot = (static_cast<int64_t>(tok) * P + p) * a.num_kv_heads + h;
        const int64_t wrow = (slot * a.max_chunks + c) * G + g;
        dst = a.ws_o + wrow * D;
        ldst = a.ws_lse + wrow;
      }
#pragma unroll
      for (int u = 0; u < NT; ++u)
        *reinterpret_cast<float2*>(dst + u * 8 + 2 * qi) = make_float2(o[u][2 * half] * inv, o[u][2 * half + 1] * inv);
      if (qi == 0) *ldst = lse;
    };
    if (oka) emit(ta, ra % G, m0, l0, 0);
    if (okb) emit(tb, rb % G, m1, l1, 1);

    if (!single) {
      // the segment's first token keys the ticket; the last CTA merges every token of it
      const int64_t slot0 = (static_cast<int64_t>(s0) * P + p) * a.num_kv_heads + h;
      if (take_ticket(a.ws_cnt + slot0, nchunks)) {
        for (int tok = s0; tok < s1; ++tok) {
          const int64_t slot = (static_cast<int64_t>(tok) * P + p) * a.num_kv_heads + h;
          const int64_t orow0 = (static_cast<int64_t>(p) * a.num_tokens + tok) * a.num_q_heads + h * G;
          merge_chunks(a, slot, nchunks, G, D, a.o_part + orow0 * D, a.lse_part + orow0);
        }
        if (tid == 0) a.ws_cnt[slot0] = 0;
      }
    }
    __syncthreads();  // the ring and the page table are reused by the next row of the block
  }
}

template <int D, int G>
static int launch_ext_t(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  constexpr int QB = kExtWarps * 16 / G;
  const size_t smem = static_cast<size_t>(kExtStages) * kExtKeys * D * 2 * 2 +
                      (static_cast<size_t>(a.chunk) / a.ps_l + 2) * sizeof(int);
  auto kern = gqa_partial_ext_kernel<D, G>;
  *err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (*err != cudaSuccess) return CPATTN_ERR_CUDA;
  dim3 grid(a.max_chunks, a.P * a.num_kv_heads, (a.num_tokens + QB - 1) / QB);
  kern<<<grid, kExtWarps * 32, smem, s>>>(a);
  *err = cudaGetLastError();
  return *err == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

template <int D>
static int ext_dispatch_g(const PartialArgs& a, int G, cudaStream_t s, cudaError_t* err) {
  switch (G) {
    case 1: return launch_ext_t<D, 1>(a, s, err);
    case 2: return launch_ext_t<D, 2>(a, s, err);
    case 4: return launch_ext_t<D, 4>(a, s, err);
    case 8: return launch_ext_t<D, 8>(a, s, err);
    case 16: return launch_ext_t<D, 16>(a, s, err);
    default: return CPATTN_ERR_UNSUPPORTED_SHAPE;
  }
}

int launch_gqa_partial_ext(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  const int G = a.num_q_heads / a.num_kv_heads;
  if (a.head_dim == 128) return ext_dispatch_g<128>(a, G, s, err);
  if (a.head_dim == 64) return ext_dispatch_g<64>(a, G, s, err);
  return CPATTN_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace cpattn
