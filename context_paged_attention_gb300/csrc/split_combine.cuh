// Split-KV bookkeeping shared by the partial-attention kernels.
//
// A partner's stripe of one row may be cut into several chunks, each handled
// by its own CTA.  A CTA of a multi-chunk stripe stores its normalised partial
// (output rows for Hg query heads and their LSE) in the workspace, takes a
// ticket, and the last CTA to arrive merges the chunk partials (exact LSE
// merge, as lse_merge does for partners) into o_part / lse_part.  No
// spin-wait: the last arrival does the work, the others just exit.
//
// Fused calls (cp_paged_attn_fused) go one level further: the partner
// partials live in the workspace, and the CTA that completes a partner's
// partial of a (token, KV head) arrives on a second ticket for the pair; the
// last of the P partners merges them (and an optional precomputed partial,
// e.g. the own-token one) into the final output, as lse_merge would (mstar
// PR #1124 "Context / Sequence Parallel 1/5", description: the partials and
// their LSEs are combined exactly).
#pragma once

#include "common.cuh"
#include "launch.h"

namespace cpattn {

// Returns true in every thread of the CTA that must do the final merge.
// Call after this CTA's workspace stores; all threads must call it.  The
// barrier orders every thread's stores before thread 0's device-scope fence,
// which (being cumulative) publishes them before the ticket; the last CTA's
// thread 0 fences again before the barrier that releases its readers.
__device__ __forceinline__ bool take_ticket(int32_t* counter, int arrivals_needed) {
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int ticket = atomicAdd(counter, 1);
    const bool last = (ticket == arrivals_needed - 1);
    if (last) __threadfence();
    s_last = last;
  }
  __syncthreads();
  return s_last != 0;
}

// Merge nchunks workspace partials of one (token, partner, KV head) slot.
// ws rows: (slot * max_chunks + chunk) * Hg + head, each Dv floats.
// Output rows: o_row0 + head (rows of Dv floats), lse at lse_row0 + head.
__device__ __forceinline__ void merge_chunks(const PartialArgs& a, int64_t slot, int nchunks, int Hg,
                                             int Dv, float* o_out, float* lse_out) {
  for (int idx = threadIdx.x; idx < Hg * Dv; idx += blockDim.x) {
    const int g = idx / Dv;
    const int d = idx - g * Dv;
    float mx = -INFINITY;
    for (int c = 0; c < nchunks; ++c) mx = fmaxf(mx, __ldcg(a.ws_lse + (slot * a.max_chunks + c) * Hg + g));
    float wsum = 0.f, acc = 0.f;
    if (mx != -INFINITY) {
      for (int c = 0; c < nchunks; ++c) {
        const int64_t wrow = (slot * a.max_chunks + c) * Hg + g;
        const float lc = __ldcg(a.ws_lse + wrow);
        if (lc == -INFINITY) continue;  // empty chunk: its output row is not read
        const float w = expf(lc - mx);
        wsum += w;
        acc = fmaf(w, __ldcg(a.ws_o + wrow * Dv + d), acc);
      }
    }
    const bool empty = (wsum == 0.f);
    o_out[static_cast<int64_t>(g) * Dv + d] = empty ? 0.f : acc / wsum;
    if (d == 0) lse_out[g] = empty ? -INFINITY : mx + logf(wsum);
  }
}

// Shared-memory floats merge_partners needs: the Hg x (P + 1) weight table
// and one value per head.
__host__ __device__ __forceinline__ int merge_scratch_floats(int Hg, int P) { return Hg * (P + 1) + Hg; }

// Final output of (token t, KV head h) from the P partner partials (o_part /
// lse_part rows, which fused calls keep in the workspace) and the optional
// extra partial; written as bf16 (round to nearest even) or fp32.
//   1. all threads load the entries' LSEs at once into a [Hg][P + 1] table;
//   2. one warp per head turns them into weights exp(lse - max) and the
//      head's LSE with shuffle reductions;
//   3. each thread sums weight * row over the entries for a float4 group of
//      value dims.
// scratch: merge_scratch_floats(Hg, P) floats of shared memory the CTA no
// longer uses.  Dv % 4 == 0.
__device__ __forceinline__ void merge_partners(const PartialArgs& a, int t, int h, int Hg, int Dv, float* scratch) {
  const int E = a.P + 1;
  float* wt = scratch;              // [Hg][E]
  float* s_inv = scratch + Hg * E;  // [Hg]
  const int64_t hq0 = static_cast<int64_t>(t) * a.num_q_heads + h * Hg;  // first query-head row of the pair
  const int64_t pstride = static_cast<int64_t>(a.num_tokens) * a.num_q_heads;  // rows between partners
  __syncthreads();  // the scratch may still be read from a previous token
  for (int idx = threadIdx.x; idx < Hg * E; idx += blockDim.x) {
    const int g = idx / E;
    const int e = idx - g * E;
    float lse = -INFINITY;
    if (e == E - 1) {
      if (a.extra_lse != nullptr) lse = __ldg(a.extra_lse + hq0 + g);
    } else {
      lse = __ldcg(a.lse_part + e * pstride + hq0 + g);
    }
    wt[idx] = lse;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int g = warp; g < Hg; g += nwarps) {
    float mx = -INFINITY;
    for (int e = lane; e < E; e += 32) mx = fmaxf(mx, wt[g * E + e]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
    for (int e = lane; e < E; e += 32) {
      const float l = wt[g * E + e];
      const float w = (mx == -INFINITY || l == -INFINITY) ? 0.f : expf(l - mx);
      wt[g * E + e] = w;
      sum += w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
      const bool empty = (sum == 0.f);
      s_inv[g] = empty ? 0.f : 1.f / sum;
      if (a.lse_out != nullptr) a.lse_out[hq0 + g] = empty ? -INFINITY : mx + logf(sum);
    }
  }
  __syncthreads();
  const int D4 = Dv / 4;
  for (int idx = threadIdx.x; idx < Hg * D4; idx += blockDim.x) {
    const int g = idx / D4;
    const int d = (idx - g * D4) * 4;
    const float* wg = wt + g * E;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int e = 0; e < E - 1; ++e) {
      const float w = wg[e];
      if (w != 0.f) {  // empty partials' rows are not read
        const float4 v = __ldcg(reinterpret_cast<const float4*>(a.o_part + (e * pstride + hq0 + g) * Dv + d));
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
    }
    if (wg[E - 1] != 0.f) {
      const float w = wg[E - 1];
      const float4 v = __ldg(reinterpret_cast<const float4*>(a.extra_o + (hq0 + g) * Dv + d));
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    const float inv = s_inv[g];
    const int64_t oi = (hq0 + g) * Dv + d;
    if (a.out_bf16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + oi) = pk;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(a.out) + oi) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
  }
}

// Fused calls, after a partner's partial of (token t, KV head h) is complete
// in o_part (written directly, or merged from its chunks by this CTA): arrive
// on the pair's ticket; the last of the P partners merges (all threads call).
__device__ __forceinline__ void pair_finish(const PartialArgs& a, int t, int h, int Hg, int Dv, float* scratch) {
  int32_t* pair = a.ws_pair + static_cast<int64_t>(t) * a.num_kv_heads + h;
  if (!take_ticket(pair, a.P)) return;
  merge_partners(a, t, h, Hg, Dv, scratch);
  if (threadIdx.x == 0) *pair = 0;
}

// Output rows of padding tokens (fused calls): 0 and -inf.
__device__ __forceinline__ void fused_zero_token(const PartialArgs& a, int t, int h, int Hg, int Dv) {
  const int64_t hq0 = static_cast<int64_t>(t) * a.num_q_heads + h * Hg;
  for (int idx = threadIdx.x; idx < Hg * Dv; idx += blockDim.x) {
    if (a.out_bf16) static_cast<__nv_bfloat16*>(a.out)[hq0 * Dv + idx] = __float2bfloat16_rn(0.f);
    else static_cast<float*>(a.out)[hq0 * Dv + idx] = 0.f;
  }
  if (a.lse_out != nullptr)
    for (int g = threadIdx.x; g < Hg; g += blockDim.x) a.lse_out[hq0 + g] = -INFINITY;
}

}  // namespace cpattn
