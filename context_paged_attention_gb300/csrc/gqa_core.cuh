// Per-warp online-softmax core of the CUDA-core attention kernels
// (cp_paged_attn_partial GQA path and own_token_attn).
//
// A warp handles TPW keys per step.  LPT lanes share one key; each owns CPL
// 16-byte pieces (DL = CPL * VEC dims) of the key and value rows and of the
// G query heads that read this KV head.  Every lane group keeps an
// independent (max, sum, output) state over the keys it saw; groups and warps
// are merged at the end.  Scores live in the log2 domain (q pre-scaled by
// scale * log2 e), so exp2f is the only transcendental in the loop.
#pragma once

#include "common.cuh"

namespace cpattn {

template <typename T, int D, int G>
struct GqaCfg {
  static constexpr int ESZ = sizeof(T);
  static constexpr int VEC = 16 / ESZ;     // elements per 16-byte piece
  static constexpr int CR = D * ESZ / 16;  // 16-byte pieces per row
  static constexpr int CPL_WANT = (64 / (G * VEC)) > 0 ? 64 / (G * VEC) : 1;
  static constexpr int CPL = CPL_WANT < CR ? CPL_WANT : CR;  // pieces per lane
  static constexpr int LPT = CR / CPL;     // lanes per key
  static constexpr int TPW = 32 / LPT;     // keys per warp step
  static constexpr int DL = CPL * VEC;     // dims per lane
  static constexpr int ROWB = D * ESZ;     // bytes per row
  static_assert(CR % CPL == 0 && LPT <= 32, "bad lane split");
};

template <typename T, int D, int G>
struct GqaLaneState {
  using C = GqaCfg<T, D, G>;
  float qf[G][C::DL];
  float m[G], l[G], o[G][C::DL];
  int sub;  // piece index of this lane inside a row
  int grp;  // key slot of this lane inside a warp step

  __device__ __forceinline__ void init(int lane) {
    sub = lane % C::LPT;
    grp = lane / C::LPT;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int e = 0; e < C::DL; ++e) o[g][e] = 0.f;
    }
  }

  // q rows of the G heads, consecutive rows of ROWB bytes; qs = scale * log2 e.
  __device__ __forceinline__ void load_q(const uint8_t* qrows, bool present, float qs) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int cc = 0; cc < C::CPL; ++cc) {
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (present) u = __ldg(reinterpret_cast<const uint4*>(qrows + g * C::ROWB) + sub + cc * C::LPT);
        float f[C::VEC];
        Chunk16<T>::widen(u, f);
#pragma unroll
        for (int e = 0; e < C::VEC; ++e) qf[g][cc * C::VEC + e] = f[e] * qs;
      }
    }
  }

  // One key for this lane group: krow/vrow point at its rows (any address
  // space the generic pointer reaches).  All lanes of the warp must call this
  // together (shuffles); "valid" masks the key of this lane group.  The value
  // row is not touched for an invalid key, so unwritten (NaN) slots never mix
  // into the output.
  template <bool kGlobal>
  __device__ __forceinline__ void step(const uint8_t* krow, const uint8_t* vrow, bool valid) {
    float s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) s[g] = 0.f;
#pragma unroll
    for (int cc = 0; cc < C::CPL; ++cc) {
      uint4 u = make_uint4(0u, 0u, 0u, 0u);
      if (!kGlobal || valid) {
        const uint4* src = reinterpret_cast<const uint4*>(krow + (sub + cc * C::LPT) * 16);
        u = kGlobal ? __ldg(src) : *src;
      }
      float kf[C::VEC];
      Chunk16<T>::widen(u, kf);
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < C::VEC; ++e) s[g] = fmaf(qf[g][cc * C::VEC + e], kf[e], s[g]);
    }
#pragma unroll
    for (int off = 1; off < C::LPT; off <<= 1)
#pragma unroll
      for (int g = 0; g < G; ++g) s[g] += __shfl_xor_sync(0xffffffffu, s[g], off);

    if (valid) {
      float vf[C::DL];
#pragma unroll
      for (int cc = 0; cc < C::CPL; ++cc) {
        const uint4* src = reinterpret_cast<const uint4*>(vrow + (sub + cc * C::LPT) * 16);
        const uint4 u = kGlobal ? __ldg(src) : *src;
        Chunk16<T>::widen(u, vf + cc * C::VEC);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (s[g] > m[g]) {  // new running max: rescale (rare after the first keys)
          const float alpha = exp2f(m[g] - s[g]);
          l[g] *= alpha;
#pragma unroll
          for (int e = 0; e < C::DL; ++e) o[g][e] *= alpha;
          m[g] = s[g];
        }
        const float pe = exp2f(s[g] - m[g]);
        l[g] += pe;
#pragma unroll
        for (int e = 0; e < C::DL; ++e) o[g][e] = fmaf(pe, vf[e], o[g][e]);
      }
    }
  }

  // Merge the TPW lane groups of the warp (they hold the same dims).
  __device__ __forceinline__ void merge_groups() {
#pragma unroll
    for (int off = C::LPT; off < 32; off <<= 1) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m[g], off);
        const float l2 = __shfl_xor_sync(0xffffffffu, l[g], off);
        float mn, fa, fb;
        softmax_merge_factors(m[g], m2, mn, fa, fb);
        l[g] = l[g] * fa + l2 * fb;
#pragma unroll
        for (int e = 0; e < C::DL; ++e) {
          const float o2 = __shfl_xor_sync(0xffffffffu, o[g][e], off);
          o[g][e] = o[g][e] * fa + o2 * fb;
        }
        m[g] = mn;
      }
    }
  }

  // Bytes of shared memory for the cross-warp merge of NW warps.
  static constexpr size_t merge_smem_bytes(int NW) {
    return (static_cast<size_t>(NW) * G * D + 2 * NW * G) * sizeof(float);
  }

  // Lane group 0 of each warp stores its state: o [NW][G][D], m [NW][G], l [NW][G].
  __device__ __forceinline__ void store(float* sm, int NW, int warp) const {
    float* sm_o = sm;
    float* sm_m = sm_o + NW * G * D;
    float* sm_l = sm_m + NW * G;
    if (grp != 0) return;
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int cc = 0; cc < C::CPL; ++cc)
#pragma unroll
        for (int e = 0; e < C::VEC; ++e)
          sm_o[(warp * G + g) * D + (sub + cc * C::LPT) * C::VEC + e] = o[g][cc * C::VEC + e];
      if (sub == 0) {
        sm_m[warp * G + g] = m[g];
        sm_l[warp * G + g] = l[g];
      }
    }
  }
};

// Merge NW stored warp states for (head g, dim d): normalised output and
// natural-log LSE (0 / -inf if no key was seen).
template <int D, int G>
__device__ __forceinline__ void merge_stored(const float* sm, int NW, int g, int d, float& out, float& lse) {
  const float* sm_o = sm;
  const float* sm_m = sm_o + NW * G * D;
  const float* sm_l = sm_m + NW * G;
  float mx = -INFINITY;
  for (int w = 0; w < NW; ++w) mx = fmaxf(mx, sm_m[w * G + g]);
  float lsum = 0.f, acc = 0.f;
  if (mx != -INFINITY) {
    for (int w = 0; w < NW; ++w) {
      const float mw = sm_m[w * G + g];
      const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - mx);
      lsum += sm_l[w * G + g] * f;
      acc += sm_o[(w * G + g) * D + d] * f;
    }
  }
  const bool empty = (lsum == 0.f);
  out = empty ? 0.f : acc / lsum;
  lse = empty ? -INFINITY : (mx + log2f(lsum)) * kLn2;
}

}  // namespace cpattn
