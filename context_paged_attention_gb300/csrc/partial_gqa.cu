// cp_paged_attn_partial, GQA path on CUDA cores.
//
// Every partner p attends only its own stripe of a row's keys: the logical
// positions j with j % P == p (mstar PR #1124 "Context / Sequence Parallel
// 1/5", description: each partner attends its slots and returns the partial
// with its log-sum-exp).  In partner p's pool those keys are dense: stripe
// slot k (k = 0, 1, ...) is logical position k * P + p and sits in the row's
// page k / (page_size / P) at physical slot k % (page_size / P).  So a partner
// walks its slots as runs of page_size / P contiguous rows per page id, which
// this kernel stages into shared memory with 16-byte cp.async copies.
//
// Work split (flash-decoding style): CTA (chunk c, partner p, KV head h, query
// token t) covers stripe slots [c * chunk, (c + 1) * chunk).  Its 4 warps take
// the chunk's segments (<= 8 rows of one page) round robin, each warp running
// its own NST-deep cp.async ring, so a warp never waits on another.  The lane
// layout and online softmax are in gqa_core.cuh.  A stripe split over several
// chunks is finished by the last CTA to arrive (split_combine.cuh).
#include "gqa_core.cuh"
#include "launch.h"
#include "split_combine.cuh"

namespace cpattn {

constexpr int kGqaWarps = 4;
constexpr int kGqaStages = 6;
constexpr int kSegMax = 8;

template <typename T, int D, int G>
__global__ void __launch_bounds__(kGqaWarps * 32) gqa_partial_kernel(const PartialArgs a) {
  using C = GqaCfg<T, D, G>;
  constexpr int NW = kGqaWarps;
  constexpr int NST = kGqaStages;
  extern __shared__ __align__(16) uint8_t smem[];

  const int c = blockIdx.x;
  const int p = blockIdx.y / a.num_kv_heads;
  const int h = blockIdx.y - p * a.num_kv_heads;
  // token of this grid slot (a dispatch order applies when tokens are rows)
  const int t = a.qo_indptr == nullptr ? ordered_row(a.row_order, blockIdx.z, gridDim.z, a.dev_status) : blockIdx.z;
  if (t < 0) return;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int P = a.P;

  // ---- which row, how many stripe slots
  int b = -1;
  if (a.qo_indptr != nullptr) {
    if (t < __ldg(a.qo_indptr + a.num_rows)) b = find_row(a.qo_indptr, a.num_rows, t);
  } else if (t < a.num_rows) {
    b = t;
  }
  int n_p = 0;
  int L = 0;  // keys of the row (clamped to max_kv_len)
  if (b >= 0) {
    L = __ldg(a.kv_len + b);
    if (L > a.max_kv_len) {
      if (c == 0 && threadIdx.x == 0) report(a.dev_status, CPATTN_DEV_POS_PAST_TABLE);
      L = a.max_kv_len;
    }
    n_p = stripe_len(L, p, P, a.interleave);
  }
  const int nchunks = n_p > 0 ? (n_p + a.chunk - 1) / a.chunk : 1;
  if (c >= nchunks) return;
  const int k_begin = c * a.chunk;
  const int k_end = min(n_p, k_begin + a.chunk);
  const int nseg = k_end > k_begin ? (k_end - k_begin + a.seg - 1) / a.seg : 0;
  const int my_nseg = nseg > warp ? (nseg - warp + NW - 1) / NW : 0;

  GqaLaneState<T, D, G> st;
  st.init(lane);
  st.load_q(static_cast<const uint8_t*>(a.q) + (static_cast<int64_t>(t) * a.num_q_heads + h * G) * C::ROWB,
            b >= 0, a.scale * kLog2e);

  const int32_t* pages = nullptr;
  int npages = 0;
  if (b >= 0) {
    const int pb = __ldg(a.page_indptr + b);
    pages = a.page_indices + pb;
    npages = __ldg(a.page_indptr + b + 1) - pb;
  }
  const int seg_bytes = a.seg * C::ROWB;
  uint8_t* ring = smem + static_cast<size_t>(warp) * NST * seg_bytes * 2;

  // page id holding stripe slot k0, or -1 if the tables do not cover it
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
    if (i < my_nseg) {
      const int k0 = k_begin + (warp + i * NW) * a.seg;
      const int n = min(a.seg, k_end - k0);
      const int pg = page_of(k0, lane == 0);
      if (pg >= 0) {
        const int l0 = k0 % a.ps_l;
        const int64_t row = ((static_cast<int64_t>(p) * a.num_pages + pg) * a.num_kv_heads + h) * a.ps_l + l0;
        const uint8_t* gk = static_cast<const uint8_t*>(a.pool_k) + row * C::ROWB;
        const uint8_t* gv = static_cast<const uint8_t*>(a.pool_v) + row * C::ROWB;
        uint8_t* sk = ring + (i % NST) * seg_bytes * 2;
        uint8_t* sv = sk + seg_bytes;
        const int pieces = n * C::CR;
        for (int x = lane; x < pieces; x += 32) {
          cp_async16(sk + x * 16, gk + x * 16);
          cp_async16(sv + x * 16, gv + x * 16);
        }
      }
    }
    cp_async_commit();
  };

#pragma unroll
  for (int i = 0; i < NST - 1; ++i) issue(i);

  for (int i = 0; i < my_nseg; ++i) {
    cp_async_wait<NST - 2>();
    __syncwarp();
    issue(i + NST - 1);  // refills the stage consumed in step i - 1

    const int k0 = k_begin + (warp + i * NW) * a.seg;
    const int n = min(a.seg, k_end - k0);
    const bool seg_ok = page_of(k0, false) >= 0;
    const uint8_t* sk = ring + (i % NST) * seg_bytes * 2;
    const uint8_t* sv = sk + seg_bytes;
    for (int base = 0; base < n; base += C::TPW) {
      const int tk = base + st.grp;
      const bool valid = seg_ok && tk < n;
      const int row = valid ? tk : 0;
      st.template step<false>(sk + row * C::ROWB, sv + row * C::ROWB, valid);
    }
  }
  cp_async_wait<0>();
  st.merge_groups();

  // ---- merge the warps through shared memory (the ring is free now)
  __syncthreads();
  float* sm = reinterpret_cast<float*>(smem);
  const int scratch_cap = NW * NST * a.seg * C::ROWB * 2 / 4;  // the ring's floats (at most the dynamic smem)
  st.store(sm, NW, warp);
  __syncthreads();

  const int64_t orow0 = (static_cast<int64_t>(p) * a.num_tokens + t) * a.num_q_heads + h * G;
  const int64_t slot = (static_cast<int64_t>(t) * P + p) * a.num_kv_heads + h;  // (t, p, h)
  const bool single = (nchunks == 1);
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int g = idx / D;
    const int d = idx - g * D;
    float out, lse;
    merge_stored<D, G>(sm, NW, g, d, out, lse);
    if (single) {
      a.o_part[(orow0 + g) * D + d] = out;
      if (d == 0) a.lse_part[lse_slot(a, p, t, h * G + g)] = lse;
    } else {
      const int64_t wrow = (slot * a.max_chunks + c) * G + g;
      a.ws_o[wrow * D + d] = out;
      if (d == 0) a.ws_lse[wrow] = lse;
    }
  }
  if (!single) {
    if (!take_ticket(a.ws_cnt + slot, nchunks)) return;
    merge_chunks(a, p, h, t, 1, slot, 0, nchunks, G, D, sm, scratch_cap);
    if (threadIdx.x == 0) a.ws_cnt[slot] = 0;  // ready for the next call
  }
  if (a.fused) pair_finish(a, t, h, G, D, sm, scratch_cap);
}

template <typename T, int D, int G>
static int launch_gqa_t(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  using C = GqaCfg<T, D, G>;
  const size_t ring = static_cast<size_t>(kGqaWarps) * kGqaStages * a.seg * C::ROWB * 2;
  const size_t comb = GqaLaneState<T, D, G>::merge_smem_bytes(kGqaWarps);
  const size_t smem = ring > comb ? ring : comb;
  auto kern = gqa_partial_kernel<T, D, G>;
  if (smem > 32 * 1024) {  // the kernel also has a little static shared memory
    static std::atomic<int> smem_set[64];
    *err = ensure_smem(kern, smem, smem_set);
    if (*err != cudaSuccess) return CPATTN_ERR_CUDA;
  }
  dim3 grid(a.max_chunks, a.P * a.num_kv_heads, a.num_tokens);
  kern<<<grid, kGqaWarps * 32, smem, s>>>(a);
  *err = cudaGetLastError();
  return *err == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

template <typename T, int D>
static int dispatch_g(const PartialArgs& a, int G, cudaStream_t s, cudaError_t* err) {
  switch (G) {
    case 1: return launch_gqa_t<T, D, 1>(a, s, err);
    case 2: return launch_gqa_t<T, D, 2>(a, s, err);
    case 4: return launch_gqa_t<T, D, 4>(a, s, err);
    case 8: return launch_gqa_t<T, D, 8>(a, s, err);
    default: return CPATTN_ERR_UNSUPPORTED_SHAPE;
  }
}

int launch_gqa_partial(const PartialArgs& a, int dtype_bf16, cudaStream_t s, cudaError_t* err) {
  const int G = a.num_q_heads / a.num_kv_heads;
  if (a.head_dim != a.head_dim_v) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  if (dtype_bf16) {
    return launch_gqa_partial_mma(a, s, err);  // bf16 pools: tensor-core path (partial_gqa_mma.cu)
  } else {
    if (a.head_dim == 128) return dispatch_g<float, 128>(a, G, s, err);
    if (a.head_dim == 64) return dispatch_g<float, 64>(a, G, s, err);
  }
  return CPATTN_ERR_UNSUPPORTED_SHAPE;
}

// Largest divisor of ps_l that is at most lim.
static int pick_seg(int ps_l, int lim) {
  for (int s = lim; s >= 1; --s)
    if (ps_l % s == 0) return s;
  return 1;
}

size_t PartialPlan::bytes() const {
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  return al(ws_o_floats * 4) + al(ws_lse_floats * 4) + al(ws_cnt_ints * 4) + al(ws_part_floats * 4) +
         al(ws_part_lse_floats * 4) + al(ws_pair_ints * 4);
}

bool plan_partial(int mla, int fused, int P, int interleave, int page_size, int num_kv_heads, int num_q_heads, int head_dim,
                  int num_tokens, int max_kv_len, int dtype_bytes, PartialPlan* plan) {
  (void)head_dim;
  const int ps_l = page_size / P;
  const int G = num_q_heads / num_kv_heads;
  const int Dv = mla ? 512 : head_dim;
  plan->seg = pick_seg(ps_l, mla ? 16 : kSegMax);
  const int max_stripe = max_stripe_len(max_kv_len, P, interleave);
  if (mla) {
    // the MLA kernel plans on the device (stripes longest first, long ones cut
    // into pieces); the workspace holds the pieces' partials, max_chunks of
    // them at most (0: no stripe can be cut)
    const int grouped = fused && page_size == 64 && num_tokens <= kMlaGroupMaxTokens;  // the kernel's own test
    const int slots = mla_ws_slots(P, interleave, num_tokens, max_kv_len, grouped);
    const size_t stripes = static_cast<size_t>(num_tokens) * P;
    plan->chunk = 64;
    plan->max_chunks = slots;
    plan->ws_o_floats = static_cast<size_t>(slots) * num_q_heads * Dv;
    plan->ws_lse_floats = static_cast<size_t>(slots) * num_q_heads;
    plan->ws_cnt_ints = stripes + (grouped ? 2 * static_cast<size_t>(num_tokens) : 0);  // + per-token records
    if (fused) {
      plan->ws_part_floats = stripes * num_q_heads * Dv;
      plan->ws_part_lse_floats = stripes * num_q_heads;
      plan->ws_pair_ints = static_cast<size_t>(num_tokens);
    } else {
      plan->ws_part_floats = plan->ws_part_lse_floats = plan->ws_pair_ints = 0;
    }
    return true;
  }
  int chunk;
  int unit;
  if (dtype_bytes == 2) {
    // tensor-core paths: 2048-key chunks.  Splitting shorter stripes costs
    // more (a device-scope ticket and a merge of the chunk partials at the end
    // of each CTA) than the balance it buys, now that three decode CTAs share
    // an SM; measured on decode rows of 512-8192 keys (P 4) and on the mixed
    // step, 1024- and 512-key chunks were 2-9% and 14% slower; longer stripes
    // (the 64k-128k rows) lose 0.5% at 4096.
    chunk = 2048;
    unit = 64;
  } else {
    // CUDA-core path: about eight chunks on the longest stripe, within [256, 2048] keys
    chunk = (max_stripe + 7) / 8;
    chunk = chunk < 256 ? 256 : (chunk > 2048 ? 2048 : chunk);
    unit = plan->seg * kGqaWarps;
  }
  chunk = (chunk + unit - 1) / unit * unit;
  plan->chunk = chunk;
  plan->max_chunks = max_stripe > 0 ? (max_stripe + chunk - 1) / chunk : 1;
  // the merges run in shared memory of at least 3000 floats (the fp32
  // kernel's ring at page runs of one row, D 64) and need entries + 1
  if (plan->max_chunks + 1 > 3000 || P + 2 > 3000) return false;
  const size_t slots = static_cast<size_t>(num_tokens) * P * num_kv_heads;
  if (plan->max_chunks > 1) {
    plan->ws_o_floats = slots * plan->max_chunks * G * Dv;
    plan->ws_lse_floats = slots * plan->max_chunks * G;
  } else {
    plan->ws_o_floats = 0;
    plan->ws_lse_floats = 0;
  }
  plan->ws_cnt_ints = slots;
  if (fused) {
    plan->ws_part_floats = slots * G * Dv;
    plan->ws_part_lse_floats = slots * G;
    plan->ws_pair_ints = static_cast<size_t>(num_tokens) * num_kv_heads;
  } else {
    plan->ws_part_floats = plan->ws_part_lse_floats = plan->ws_pair_ints = 0;
  }
  return true;
}

}  // namespace cpattn
