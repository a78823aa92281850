// lse_merge: exact merge of N (output, log-sum-exp) partials over disjoint key
// sets (mstar PR #1124 "Context / Sequence Parallel 1/5", description: the
// partials are merged exactly; vLLM "[Core] Add explicit layer parallel plans",
// _forward_with_dcp, merge_attn_states).
//
// One warp per (token, head): lanes first agree on the weights from the N
// log-sum-exps, then stream the N partial rows with 16-byte loads.  Purely
// bandwidth-bound: N * head_dim_v * 4 bytes read, head_dim_v * out bytes written.
#include "common.cuh"
#include "launch.h"

namespace cpattn {

__global__ void __launch_bounds__(256) lse_merge_kernel(const MergeArgs a) {
  pdl_trigger();
  pdl_wait();
  const int warps_per_block = blockDim.x / 32;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * warps_per_block + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const int64_t items = static_cast<int64_t>(a.num_tokens) * a.num_heads;
  if (item >= items) return;

  const int nvec = a.head_dim_v / 4;
  if (a.num_partials <= 32) {
    // lane i holds partial i's LSE and weight; the value loop takes the
    // weights by shuffle (the same arithmetic and summation order as below)
    const float li = lane < a.num_partials ? __ldg(a.lse_parts + lane * a.stride_lse + item) : -INFINITY;
    float mx = li;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (mx != -INFINITY) {
      const float wi = (li == -INFINITY) ? 0.f : expf(li - mx);
      float wsum = wi;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
      const float inv = 1.f / wsum;
      for (int v = lane; v < nvec; v += 32) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int i = 0; i < a.num_partials; ++i) {
          const float w = __shfl_sync(0xffffffffu, wi, i) * inv;
          if (w != 0.f) {  // an empty partial contributes nothing (its output is not read)
            const float4 o =
                __ldg(reinterpret_cast<const float4*>(a.o_parts + i * a.stride_o + item * a.head_dim_v) + v);
            acc.x = fmaf(w, o.x, acc.x);
            acc.y = fmaf(w, o.y, acc.y);
            acc.z = fmaf(w, o.z, acc.z);
            acc.w = fmaf(w, o.w, acc.w);
          }
        }
        if (a.out_bf16) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
          __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
          uint2 packed;
          packed.x = *reinterpret_cast<uint32_t*>(&lo);
          packed.y = *reinterpret_cast<uint32_t*>(&hi);
          reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + item * a.head_dim_v)[v] = packed;
        } else {
          reinterpret_cast<float4*>(static_cast<float*>(a.out) + item * a.head_dim_v)[v] = acc;
        }
      }
      if (a.lse_out != nullptr && lane == 0) a.lse_out[item] = mx + logf(wsum);
      return;
    }
  }

  float mx = -INFINITY;
  for (int i = lane; i < a.num_partials; i += 32) mx = fmaxf(mx, __ldg(a.lse_parts + i * a.stride_lse + item));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));

  if (mx == -INFINITY) {  // every partial empty: padding merges to zero
    if (a.out_bf16) {
      uint2* o = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + item * a.head_dim_v);
      for (int v = lane; v < nvec; v += 32) o[v] = make_uint2(0u, 0u);
    } else {
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + item * a.head_dim_v);
      for (int v = lane; v < nvec; v += 32) o[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (a.lse_out != nullptr && lane == 0) a.lse_out[item] = -INFINITY;
    return;
  }
  float wsum = 0.f;
  for (int i = lane; i < a.num_partials; i += 32) {
    const float l = __ldg(a.lse_parts + i * a.stride_lse + item);
    wsum += (l == -INFINITY) ? 0.f : expf(l - mx);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
  const float inv = 1.f / wsum;

  for (int v = lane; v < nvec; v += 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < a.num_partials; ++i) {
      const float l = __ldg(a.lse_parts + i * a.stride_lse + item);
      if (l == -INFINITY) continue;  // an empty partial contributes nothing (its output is not read)
      const float w = expf(l - mx) * inv;
      const float4 o = __ldg(reinterpret_cast<const float4*>(a.o_parts + i * a.stride_o + item * a.head_dim_v) + v);
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
    }
    if (a.out_bf16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 packed;
      packed.x = *reinterpret_cast<uint32_t*>(&lo);
      packed.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + item * a.head_dim_v)[v] = packed;
    } else {
      reinterpret_cast<float4*>(static_cast<float*>(a.out) + item * a.head_dim_v)[v] = acc;
    }
  }
  if (a.lse_out != nullptr && lane == 0) a.lse_out[item] = mx + logf(wsum);
}

// The same merge over views: partial i's row of (token t, head h) is
// v[i].o + t * o_st + h * o_sh, its LSE v[i].lse[t * lse_st + h * lse_sh];
// the output row and LSE go to strided places too.  This covers the
// head-major LSE that FlashAttention returns ([H, B]) next to the
// token-major one DCP's combine wants ([B, H]) (vLLM "[Core] Add explicit
// layer parallel plans", _forward_with_dcp), and per-rank head slices.
__global__ void __launch_bounds__(256) lse_merge_views_kernel(const MergeViewArgs a) {
  pdl_trigger();
  pdl_wait();
  const int warps_per_block = blockDim.x / 32;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * warps_per_block + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const int64_t items = static_cast<int64_t>(a.num_tokens) * a.num_heads;
  if (item >= items) return;
  const int t = static_cast<int>(item / a.num_heads);
  const int h = static_cast<int>(item - static_cast<int64_t>(t) * a.num_heads);

  float lse_i = -INFINITY;  // lane i < n holds partial i's LSE
  if (lane < a.n) lse_i = __ldg(a.v[lane].lse + t * a.v[lane].lse_st + h * a.v[lane].lse_sh);
  float mx = lse_i;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  const float w_i = (mx == -INFINITY || lse_i == -INFINITY) ? 0.f : expf(lse_i - mx);
  float wsum = w_i;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
  const bool empty = (wsum == 0.f);  // every partial empty: padding merges to zero
  const float inv = empty ? 0.f : 1.f / wsum;

  const int nvec = a.head_dim_v / 4;
  for (int vv = lane; vv < nvec; vv += 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < a.n; ++i) {
      const float w = __shfl_sync(0xffffffffu, w_i, i) * inv;
      if (w == 0.f) continue;  // an empty partial's row is not read
      const float4 o = __ldg(reinterpret_cast<const float4*>(a.v[i].o + t * a.v[i].o_st + h * a.v[i].o_sh) + vv);
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
    }
    const int64_t orow = t * a.out_st + h * a.out_sh;
    if (a.out_bf16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 packed;
      packed.x = *reinterpret_cast<uint32_t*>(&lo);
      packed.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + orow)[vv] = packed;
    } else {
      reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow)[vv] = acc;
    }
  }
  if (a.lse_out != nullptr && lane == 0)
    a.lse_out[t * a.lse_out_st + h * a.lse_out_sh] = empty ? -INFINITY : mx + logf(wsum);
}

cudaError_t launch_lse_merge_views(const MergeViewArgs& a, cudaStream_t s) {
  const int64_t items = static_cast<int64_t>(a.num_tokens) * a.num_heads;
  if (items == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (items + 7) / 8;
  return launch_pdl(lse_merge_views_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, s, a);
}

cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t s) {
  const int64_t items = static_cast<int64_t>(a.num_tokens) * a.num_heads;
  if (items == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (items + 7) / 8;
  return launch_pdl(lse_merge_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, s, a);
}

}  // namespace cpattn
