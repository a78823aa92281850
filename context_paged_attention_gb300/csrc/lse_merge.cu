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
  const int warps_per_block = blockDim.x / 32;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * warps_per_block + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const int64_t items = static_cast<int64_t>(a.num_tokens) * a.num_heads;
  if (item >= items) return;

  float mx = -INFINITY;
  for (int i = lane; i < a.num_partials; i += 32) mx = fmaxf(mx, __ldg(a.lse_parts + i * a.stride_lse + item));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));

  const int nvec = a.head_dim_v / 4;
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

cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t s) {
  const int64_t items = static_cast<int64_t>(a.num_tokens) * a.num_heads;
  if (items == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (items + 7) / 8;
  lse_merge_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace cpattn
