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

// The threads that run a merge together: the whole CTA (CtaGroup), or the
// first kThreads threads of a warp-specialised CTA synchronised by named
// barrier kBarId (WarpsGroup), while its other warps keep working.
struct CtaGroup {
  __device__ static int tid() { return threadIdx.x; }
  __device__ static int size() { return blockDim.x; }
  __device__ static void sync() { __syncthreads(); }
};
template <int kBarId, int kThreads>
struct WarpsGroup {
  __device__ static int tid() { return threadIdx.x; }
  __device__ static int size() { return kThreads; }
  __device__ static void sync() { asm volatile("bar.sync %0, %1;\n" ::"n"(kBarId), "n"(kThreads) : "memory"); }
};

// Page index of stripe slot k (k / ps_l; a shift when ps_l is a power of two).
__device__ __forceinline__ int page_of_slot(const PartialArgs& a, int k) {
  return a.ps_shift >= 0 ? (k >> a.ps_shift) : k / a.ps_l;
}

// Index of the LSE of (partner p, token t, query head hq) in lse_part.
__device__ __forceinline__ int64_t lse_slot(const PartialArgs& a, int p, int t, int hq) {
  return p * a.lse_sp + t * a.lse_st + hq * a.lse_sh;
}

// Returns true in every thread of the CTA that must do the final merge.
// Call after this CTA's workspace stores; all threads must call it.  The
// barrier orders every thread's stores before thread 0's device-scope fence,
// which (being cumulative) publishes them before the ticket; the last CTA's
// thread 0 fences again before the barrier that releases its readers.
template <class Grp = CtaGroup>
__device__ __forceinline__ bool take_ticket(int32_t* counter, int arrivals_needed) {
  __shared__ int s_last;
  Grp::sync();
  if (Grp::tid() == 0) {
    __threadfence();
    const int ticket = atomicAdd(counter, 1);
    const bool last = (ticket == arrivals_needed - 1);
    if (last) __threadfence();
    s_last = last;
  }
  Grp::sync();
  return s_last != 0;
}

// Exact merge of E partials for each of R rows of Dv values (the LSE merge
// of lse_merge).  Row r, entry e: LSE lse_in(r, e) (-inf: empty, its values
// are not read), values at o_in(r, e) (Dv floats, 16-byte aligned).  The
// merged row goes to put(r, d, float4) for d = 0, 4, ..., its LSE to
// put_lse(r, value).  In three phases, all threads busy in each:
//   1. the R x E LSEs are loaded at once into a shared table;
//   2. one warp per row turns them into weights exp(lse - max) / sum and the
//      row's LSE with shuffle reductions;
//   3. each thread sums weight * values over the entries for a float4 group
//      of one row, the loads unrolled so several are in flight; with UNR > 1
//      a thread takes UNR float4 groups (blockDim apart, so a warp's loads
//      stay coalesced) and issues all UNR loads of an entry before it uses
//      them: UNR x 16 bytes in flight a thread, for the wide rows (MLA's 512
//      values x 128 heads) where one CTA merges a megabyte.
// Rows go in batches that fit `scratch` (cap floats of shared memory the
// group no longer uses; cap >= E + 1).  All threads of the group must call.
template <int UNR = 1, class Grp = CtaGroup, class LseIn, class OIn, class Put, class PutLse>
__device__ __forceinline__ void merge_rows(int R, int E, int Dv, LseIn lse_in, OIn o_in, Put put, PutLse put_lse,
                                           float* scratch, int cap) {
  const int RB = max(1, min(R, cap / (E + 1)));
  const int D4 = Dv / 4;
  const int gtid = Grp::tid(), gsize = Grp::size();
  const int warp = gtid >> 5, lane = gtid & 31, nwarps = gsize >> 5;
  for (int r0 = 0; r0 < R; r0 += RB) {
    const int nr = min(RB, R - r0);
    float* wt = scratch;              // [nr][E]
    float* s_ok = scratch + nr * E;   // [nr]: 1 if the row has keys
    Grp::sync();  // the scratch may still be read from the previous batch or caller
    for (int idx = gtid; idx < nr * E; idx += gsize) wt[idx] = lse_in(r0 + idx / E, idx % E);
    Grp::sync();
    for (int r = warp; r < nr; r += nwarps) {
      float mx = -INFINITY;
      for (int e = lane; e < E; e += 32) mx = fmaxf(mx, wt[r * E + e]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float sum = 0.f;
      for (int e = lane; e < E; e += 32) {
        const float l = wt[r * E + e];
        sum += (mx == -INFINITY || l == -INFINITY) ? 0.f : expf(l - mx);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      const bool empty = (sum == 0.f);
      const float inv = empty ? 0.f : 1.f / sum;
      __syncwarp();
      for (int e = lane; e < E; e += 32) {
        const float l = wt[r * E + e];
        wt[r * E + e] = (empty || l == -INFINITY) ? 0.f : expf(l - mx) * inv;
      }
      if (lane == 0) {
        s_ok[r] = empty ? 0.f : 1.f;
        put_lse(r0 + r, empty ? -INFINITY : mx + logf(sum));
      }
    }
    Grp::sync();
    if constexpr (UNR == 1) {
      for (int idx = gtid; idx < nr * D4; idx += gsize) {
        const int r = idx / D4;
        const int d = (idx - r * D4) * 4;
        const float* wr = wt + r * E;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int e = 0; e < E; ++e) {
          const float w = wr[e];
          if (w != 0.f) {  // empty partials' rows are never read
            const float4 v = __ldcg(reinterpret_cast<const float4*>(o_in(r0 + r, e) + d));
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
          }
        }
        put(r0 + r, d, acc);
      }
    } else {
      const int n4 = nr * D4;
      for (int i0 = gtid; i0 < n4; i0 += gsize * UNR) {
        int rr[UNR], dd[UNR];
        float4 acc[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int idx = i0 + u * gsize;
          rr[u] = idx < n4 ? idx / D4 : -1;
          dd[u] = idx < n4 ? (idx - rr[u] * D4) * 4 : 0;
          acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int e = 0; e < E; ++e) {
          float w[UNR];
          float4 v[UNR];
#pragma unroll
          for (int u = 0; u < UNR; ++u) {
            w[u] = rr[u] >= 0 ? wt[rr[u] * E + e] : 0.f;
            v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (w[u] != 0.f) v[u] = __ldcg(reinterpret_cast<const float4*>(o_in(r0 + rr[u], e) + dd[u]));
          }
#pragma unroll
          for (int u = 0; u < UNR; ++u) {
            acc[u].x = fmaf(w[u], v[u].x, acc[u].x);
            acc[u].y = fmaf(w[u], v[u].y, acc[u].y);
            acc[u].z = fmaf(w[u], v[u].z, acc[u].z);
            acc[u].w = fmaf(w[u], v[u].w, acc[u].w);
          }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u)
          if (rr[u] >= 0) put(r0 + rr[u], dd[u], acc[u]);
      }
    }
  }
}

// Merge the nchunks workspace partials of ntok consecutive tokens of one
// (partner p, KV head h): token i's slot is slot0 + i * slot_step; ws rows
// (slot * max_chunks + chunk) * Hg + head, Dv floats each.  Results go to the
// partner partial o_part / lse_part of tokens t0 .. t0 + ntok - 1.
template <int UNR = 1>
__device__ __forceinline__ void merge_chunks(const PartialArgs& a, int p, int h, int t0, int ntok, int64_t slot0,
                                             int64_t slot_step, int nchunks, int Hg, int Dv, float* scratch,
                                             int cap) {
  auto wrow = [&](int r, int e) -> int64_t {
    const int i = r / Hg;
    return ((slot0 + i * slot_step) * a.max_chunks + e) * Hg + (r - i * Hg);
  };
  merge_rows<UNR>(
      ntok * Hg, nchunks, Dv, [&](int r, int e) { return __ldcg(a.ws_lse + wrow(r, e)); },
      [&](int r, int e) { return a.ws_o + wrow(r, e) * Dv; },
      [&](int r, int d, float4 v) {
        const int i = r / Hg;
        const int64_t orow = (static_cast<int64_t>(p) * a.num_tokens + t0 + i) * a.num_q_heads + h * Hg + (r - i * Hg);
        *reinterpret_cast<float4*>(a.o_part + orow * Dv + d) = v;
      },
      [&](int r, float l) {
        const int i = r / Hg;
        a.lse_part[lse_slot(a, p, t0 + i, h * Hg + (r - i * Hg))] = l;
      },
      scratch, cap);
}

// Final output of tokens t0 .. t0 + ntok - 1 for KV head h from the P
// partner partials (o_part / lse_part rows, which fused calls keep in the
// workspace) and the optional extra partial (entry P); written as bf16
// (round to nearest even) or fp32.  Row r = token t0 + r / Hg, head r % Hg.
template <int UNR = 1, class Grp = CtaGroup>
__device__ __forceinline__ void merge_partners(const PartialArgs& a, int t0, int ntok, int h, int Hg, int Dv,
                                               float* scratch, int cap) {
  const int64_t pstride = static_cast<int64_t>(a.num_tokens) * a.num_q_heads;  // rows between partners
  const int E = a.P + (a.extra_lse != nullptr ? 1 : 0);
  // query-head row (token * Hq + head) of merge row r
  auto hq = [&](int r) -> int64_t {
    const int i = r / Hg;
    return static_cast<int64_t>(t0 + i) * a.num_q_heads + h * Hg + (r - i * Hg);
  };
  merge_rows<UNR, Grp>(
      ntok * Hg, E, Dv,
      [&](int r, int e) {
        const int i = r / Hg;
        return e < a.P ? __ldcg(a.lse_part + lse_slot(a, e, t0 + i, h * Hg + (r - i * Hg)))
                       : __ldg(a.extra_lse + hq(r));
      },
      [&](int r, int e) { return e < a.P ? a.o_part + (e * pstride + hq(r)) * Dv : a.extra_o + hq(r) * Dv; },
      [&](int r, int d, float4 v) {
        const int64_t oi = hq(r) * Dv + d;
        if (a.out_bf16) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
          __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
          uint2 pk;
          pk.x = *reinterpret_cast<uint32_t*>(&lo);
          pk.y = *reinterpret_cast<uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + oi) = pk;
        } else {
          *reinterpret_cast<float4*>(static_cast<float*>(a.out) + oi) = v;
        }
      },
      [&](int r, float l) {
        if (a.lse_out != nullptr) a.lse_out[hq(r)] = l;
      },
      scratch, cap);
}

// Fused calls, after a partner's partial of (token t, KV head h) is complete
// in o_part (written directly, or merged from its chunks by this CTA): arrive
// on the pair's ticket; the last of the P partners merges (all threads call).
template <int UNR = 1, class Grp = CtaGroup>
__device__ __forceinline__ void pair_finish(const PartialArgs& a, int t, int h, int Hg, int Dv, float* scratch,
                                            int cap) {
  int32_t* pair = a.ws_pair + static_cast<int64_t>(t) * a.num_kv_heads + h;
  if (!take_ticket<Grp>(pair, a.P)) return;
  merge_partners<UNR, Grp>(a, t, 1, h, Hg, Dv, scratch, cap);
  if (Grp::tid() == 0) *pair = 0;
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
