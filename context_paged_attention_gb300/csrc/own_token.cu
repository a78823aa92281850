// own_token_attn: causal attention of a step's new tokens over the K/V the
// layer passes (mstar PR #1124 "Context / Sequence Parallel 1/5", description:
// a step that is not one token a row attends its own tokens apart; vLLM
// "[Core] Add explicit layer parallel plans", _forward_with_dcp: the own-token
// flash_attn_varlen_func call with cu_seqlens_k = cu_seqlens_q, causal).
//
// CTA (token t, KV head h): 4 warps split the keys qo_indptr[b] .. t of t's
// row and read them straight from global memory with 16-byte loads (each key
// is read by the few query tokens after it, so L1/L2 serve the reuse).  Only
// rows below num_real_rows are touched: a padding row's keys are never
// loaded, whatever they hold (review thread of the same PR: NaN in padding
// rows' keys must not reach real rows of a captured bucket).
#include "gqa_core.cuh"
#include "launch.h"

namespace cpattn {

constexpr int kOwnWarps = 4;

template <typename T, int D, int G>
__global__ void __launch_bounds__(kOwnWarps * 32) own_token_kernel(const OwnArgs a) {
  using C = GqaCfg<T, D, G>;
  constexpr int NW = kOwnWarps;
  __shared__ float sm[(NW * G * D + 2 * NW * G)];

  const int t = blockIdx.x;
  const int h = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int real_end = __ldg(a.qo_indptr + a.num_real_rows);
  int start = 0;
  const bool real = t < real_end;
  if (real) start = __ldg(a.qo_indptr + find_row(a.qo_indptr, a.num_real_rows, t));

  GqaLaneState<T, D, G> st;
  st.init(lane);
  st.load_q(static_cast<const uint8_t*>(a.q) + (static_cast<int64_t>(t) * a.num_q_heads + h * G) * C::ROWB, real,
            a.scale * kLog2e);

  if (real) {
    const int64_t stride = static_cast<int64_t>(a.num_kv_heads) * C::ROWB;
    const uint8_t* kb = static_cast<const uint8_t*>(a.k_new) + static_cast<int64_t>(h) * C::ROWB;
    const uint8_t* vb = static_cast<const uint8_t*>(a.v_new) + static_cast<int64_t>(h) * C::ROWB;
    for (int base = start + warp * C::TPW; base <= t; base += NW * C::TPW) {
      const int j = base + st.grp;
      const bool valid = j <= t;
      const int jj = valid ? j : t;
      st.template step<true>(kb + jj * stride, vb + jj * stride, valid);
    }
  }
  st.merge_groups();
  st.store(sm, NW, warp);
  __syncthreads();
  const int64_t orow0 = static_cast<int64_t>(t) * a.num_q_heads + h * G;
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int g = idx / D;
    const int d = idx - g * D;
    float out, lse;
    merge_stored<D, G>(sm, NW, g, d, out, lse);
    a.o_own[(orow0 + g) * D + d] = out;
    if (d == 0) a.lse_own[orow0 + g] = lse;
  }
}

template <typename T, int D, int G>
static int launch_own_t(const OwnArgs& a, cudaStream_t s, cudaError_t* err) {
  dim3 grid(a.num_tokens, a.num_kv_heads);
  own_token_kernel<T, D, G><<<grid, kOwnWarps * 32, 0, s>>>(a);
  *err = cudaGetLastError();
  return *err == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

template <typename T, int D>
static int own_dispatch_g(const OwnArgs& a, int G, cudaStream_t s, cudaError_t* err) {
  switch (G) {
    case 1: return launch_own_t<T, D, 1>(a, s, err);
    case 2: return launch_own_t<T, D, 2>(a, s, err);
    case 4: return launch_own_t<T, D, 4>(a, s, err);
    case 8: return launch_own_t<T, D, 8>(a, s, err);
    default: return CPATTN_ERR_UNSUPPORTED_SHAPE;
  }
}

// MLA (one latent KV head, keys of 576 values, values = their first 512):
// warp w of CTA (token t, head block y) takes query head 8 y + w.  Lane l
// holds bf16 pairs l + 32 i of the query and of each key (i < 9; the value
// pairs are those with i < 8), so every key is read once a warp, coalesced,
// and its value needs no second load.  Same row and padding rules as above.
constexpr int kOwnMlaHeads = 8;
__global__ void __launch_bounds__(kOwnMlaHeads * 32) own_token_mla_kernel(const OwnArgs a) {
  constexpr int kPairs = 576 / 2, kPL = kPairs / 32, kVPL = 512 / 2 / 32;  // 9 pairs a lane, 8 of them values
  const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * kOwnMlaHeads + warp;
  if (h >= a.num_q_heads) return;
  const int real_end = __ldg(a.qo_indptr + a.num_real_rows);
  const bool real = t < real_end;
  const int start = real ? __ldg(a.qo_indptr + find_row(a.qo_indptr, a.num_real_rows, t)) : 0;
  const float sl = a.scale * kLog2e;
  const uint32_t* qrow =
      reinterpret_cast<const uint32_t*>(a.q) + (static_cast<int64_t>(t) * a.num_q_heads + h) * kPairs;
  float qv[2 * kPL];
#pragma unroll
  for (int i = 0; i < kPL; ++i) {
    const float2 f = real ? __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(qrow + lane + 32 * i))
                          : make_float2(0.f, 0.f);
    qv[2 * i] = f.x * sl;
    qv[2 * i + 1] = f.y * sl;
  }
  float m = -INFINITY, l = 0.f, o[2 * kVPL];
#pragma unroll
  for (int i = 0; i < 2 * kVPL; ++i) o[i] = 0.f;
  if (real) {
    for (int j = start; j <= t; ++j) {
      const uint32_t* krow = reinterpret_cast<const uint32_t*>(a.k_new) + static_cast<int64_t>(j) * kPairs;
      float kv[2 * kPL];
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < kPL; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(krow + lane + 32 * i));
        kv[2 * i] = f.x;
        kv[2 * i + 1] = f.y;
        s = fmaf(qv[2 * i], f.x, fmaf(qv[2 * i + 1], f.y, s));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      const float mn = fmaxf(m, s);
      const float alpha = m == -INFINITY ? 0.f : exp2f(m - mn);
      const float pj = exp2f(s - mn);
      l = l * alpha + pj;
#pragma unroll
      for (int i = 0; i < 2 * kVPL; ++i) o[i] = fmaf(pj, kv[i], o[i] * alpha);
      m = mn;
    }
  }
  const int64_t orow = static_cast<int64_t>(t) * a.num_q_heads + h;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float2* dst = reinterpret_cast<float2*>(a.o_own + orow * 512);
#pragma unroll
  for (int i = 0; i < kVPL; ++i) dst[lane + 32 * i] = make_float2(o[2 * i] * inv, o[2 * i + 1] * inv);
  if (lane == 0) a.lse_own[orow] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

int launch_own_token(const OwnArgs& a, int dtype_bf16, cudaStream_t s, cudaError_t* err) {
  const int G = a.num_q_heads / a.num_kv_heads;
  if (a.num_tokens == 0) return CPATTN_OK;
  if (a.head_dim == 576) {  // MLA (the caller checked the shape)
    dim3 grid(a.num_tokens, (a.num_q_heads + kOwnMlaHeads - 1) / kOwnMlaHeads);
    own_token_mla_kernel<<<grid, kOwnMlaHeads * 32, 0, s>>>(a);
    *err = cudaGetLastError();
    return *err == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
  }
  if (dtype_bf16) {
    return launch_own_token_mma(a, s, err);  // tensor cores (own_token_mma.cu)
  } else {
    if (a.head_dim == 128) return own_dispatch_g<float, 128>(a, G, s, err);
    if (a.head_dim == 64) return own_dispatch_g<float, 64>(a, G, s, err);
  }
  return CPATTN_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace cpattn
