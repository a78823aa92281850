// Split-KV bookkeeping shared by the partial-attention kernels.
//
// A partner's stripe of one row may be cut into several chunks, each handled
// by its own CTA.  A CTA of a multi-chunk stripe stores its normalised partial
// (output rows for Hg query heads and their LSE) in the workspace, takes a
// ticket, and the last CTA to arrive merges the chunk partials (exact LSE
// merge, as lse_merge does for partners) into o_part / lse_part.  No
// spin-wait: the last arrival does the work, the others just exit.
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

}  // namespace cpattn
