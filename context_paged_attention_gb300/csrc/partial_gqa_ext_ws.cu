// cp_paged_attn_partial, GQA rows with several query tokens over a bf16 or
// E4M3 pool, on the tcgen05 tensor cores with specialised warps.
//
// A non-decode step attends the pool for its context only, and every new
// token of a row sees the same context (mstar PR #1124 "Context / Sequence
// Parallel 1/5", description: context-only plans; vLLM "[Core] Add explicit
// layer parallel plans", _forward_with_dcp: the context partial over the paged
// cache).  The queries of up to 128 / G consecutive tokens of one row and the
// G heads of KV head h form a dense 128-row tile against partner p's stripe
// of that row's context (stripe slot k = logical position k * P + p, at
// physical slot k % (page_size / P) of page k / (page_size / P)):
//   S = Q K^T  (M = 128 query rows, N = 32 keys, K = head_dim)
//   O += P V   (N = head_dim, K = 32 keys)
//
// CTA = (chunk, partner p, KV head h, block of one row's tokens).  Roles:
//   * warps 0-3 (softmax): thread r owns query row r = (token s0 + r / G,
//     head h * G + r % G) and TMEM lane r; it reads S, keeps the online
//     softmax state (running max raised only when it grows by more than 8,
//     so a rescale of O is rare and every probability stays <= 2^8), and
//     writes its row of P as bf16 pairs into tensor memory, where P V reads
//     it as the MMA's A operand (no shared-memory copy, no proxy fence).
//   * warp 4, lane 0 (MMA): S of tile j+2 as soon as its keys landed and S of
//     tile j was read, then P V of tile j once P(j) is written: the tensor
//     core computes the next scores while the softmax warps work.
//   * warps 5-7 (copies): Q once, then K tiles (warps 5 and 7, half the keys
//     each) into a 4-stage ring refilled as soon as S of a stage's tile is
//     done, and V tiles (warp 6) into a 3-stage ring refilled once P V of a
//     stage's tile is done; 16-byte cp.async, a warp instruction covering
//     whole 128-byte blocks of rows.  Keys past the stripe end or on a
//     rejected page are zero-filled, and each tile's valid-key mask is
//     published for the softmax.  E4M3 pools: the copy warps load each key
//     row's codes and store it converted to bf16 (exact); the scores take
//     k_descale and the output v_descale.
// Tensor memory (256 columns, two CTAs an SM): S in two 32-column buffers,
// O at column 64, P in two 16-column buffers after O.  O is normalised by the sum of the bf16-rounded
// probabilities (an exact convex combination of the values); the LSE keeps
// the fp32 sum.  A chunk split of a stripe is merged by the last chunk CTA of
// the segment, its chunk rows brought in by bulk asynchronous copies.  The
// CTAs of chunk 0 also write the padding tokens' 0 / -inf.  Every wait is
// bounded; one that runs out raises the CTA's abort flag, which ends every
// other wait, and the call reports CPATTN_DEV_TC_TIMEOUT.
#include "common.cuh"
#include "launch.h"
#include "mma_sync.cuh"
#include "split_combine.cuh"
#include "tc05.cuh"

namespace cpattn {

namespace {
constexpr int kWTile = 32;      // keys per tile
constexpr int kKStages = 4;     // K ring: a stage is refilled once S of its tile is done
constexpr int kVStages = 3;     // V ring: a stage is refilled once P V of its tile is done
constexpr int kMaskSlots = 8;   // valid-key masks of the tiles in flight
constexpr int kWRows = 128;     // query rows per CTA
constexpr int kWMma = 128;      // lane 0 of warp 4 issues the MMAs
constexpr int kWLoadK = 5;      // warps 5 and 7 copy K tiles (half the keys each), warp 6
constexpr int kWLoadV = 6;      // V tiles; all three copy Q
constexpr int kWLoadK2 = 7;
constexpr int kWThreads = 32 * 8;
constexpr int kWMergeUnroll = 4;

// barrier indices (arrival counts in brackets)
constexpr int W_KFULL = 0;    // [64 K-loader lanes] x4: K tile landed
constexpr int W_KFREE = 4;    // [commit] x4: S of the stage's tile done
constexpr int W_VFULL = 8;    // [32 V-loader lanes] x3: V tile landed
constexpr int W_VFREE = 11;   // [commit] x3: P V of the stage's tile done
constexpr int W_SDONE = 14;   // [commit] x2: S of the buffer's tile done
constexpr int W_SFREE = 16;   // [4 softmax warps] x2: S buffer read
constexpr int W_PFULL = 18;   // [4 softmax warps] x2: P buffer written
constexpr int W_PVDONE = 20;  // [commit] x2: P V of the buffer's tile done
constexpr int W_Q = 22;       // [96 loader lanes]
constexpr int W_FIN = 23;     // [commit]
constexpr int W_MERGE = 24;   // [1 + bytes] x2: chunk rows landed (split-KV merge)
constexpr int W_BARS = 26;

template <int D>
struct WsLayout {
  static constexpr int KB = D / 64;                   // 64-column blocks of a row
  static constexpr int QBLK = kWRows * 128;           // one Q column block
  static constexpr int QBYTES = KB * QBLK;
  static constexpr int BLK = kWTile * 128;            // one column block of a key tile
  static constexpr int TILE = KB * BLK;               // K (or V) tile
  static constexpr int TMEM_COLS = 256;
  static constexpr uint32_t S_COL = 0;                // S buffers at columns 0 and 32
  static constexpr uint32_t O_COL = 64;               // O: D columns
  static constexpr uint32_t P_COL = 64 + D;           // P buffers: 16 columns each (bf16 pairs)
  static constexpr size_t OFF_K = QBYTES;
  static constexpr size_t OFF_V = OFF_K + static_cast<size_t>(kKStages) * TILE;
  static constexpr size_t OFF_BAR = OFF_V + static_cast<size_t>(kVStages) * TILE;
  static constexpr size_t OFF_MASK = OFF_BAR + W_BARS * 8;
  static constexpr size_t OFF_MISC = OFF_MASK + kMaskSlots * 4;  // TMEM base, abort flag
  static constexpr int SCRATCH_FLOATS = static_cast<int>((OFF_BAR - OFF_K) / 4);  // K + V rings, free after the loop
  static constexpr int MERGE_BYTES = static_cast<int>(OFF_BAR);  // Q and the rings: contiguous, free after the loop
  static constexpr size_t OFF_PG = OFF_MISC + 16;
  static size_t smem_bytes(int page_slots) { return 1024 + OFF_PG + static_cast<size_t>(page_slots) * 4; }
};

__device__ __forceinline__ void ws_arrive(uint32_t mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(mbar) : "memory");
}
// each lane arrives once when all of its earlier cp.async copies have landed
__device__ __forceinline__ void ws_cp_arrive(uint32_t mbar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ void ws_cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
// 16 zero bytes through the same copy path (nothing is read)
__device__ __forceinline__ void ws_cp16_zero(uint32_t dst, const void* any_gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, 0;\n" ::"r"(dst), "l"(any_gmem) : "memory");
}
__device__ __forceinline__ void ws_bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(mbar)
               : "memory");
}
// bounded wait on a phase; gives up when the abort flag is raised
__device__ __forceinline__ bool ws_wait(uint32_t mbar, uint32_t parity, const volatile int* abort_flag) {
  for (uint32_t it = 0; it < (1u << 22); ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(mbar), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 63u) == 63u && *abort_flag) return false;
  }
  return false;
}
}  // namespace

// Split-KV merge of the E chunk partials of tokens s0 .. s1-1 (KV head h,
// partner p) into the partner partial: the LSE merge of merge_chunks, with
// each token's G x D chunk rows (2 KB at G 4, D 128) brought into shared
// memory by bulk asynchronous copies, one thread keeping a batch of TB tokens
// x E chunks in flight while the CTA combines the previous batch.  Returns
// false (nothing done) when a batch of one token does not fit; a copy that
// does not land within the poll limit is reported.  All threads call.
template <int D, int G>
__device__ bool ws_merge_chunks_bulk(const PartialArgs& a, int p, int h, int s0, int s1, int E, uint8_t* scratch,
                                     int scratch_bytes, uint32_t mb0) {
  constexpr int ROW = G * D;  // floats of one (token, chunk) block
  const int ntok = s1 - s0;
  const int wt_bytes = ((ntok * G * E * 4) + 15) & ~15;
  int TB = (scratch_bytes - wt_bytes) / (2 * E * ROW * 4);
  if (TB < 1) return false;
  TB = min(TB, ntok);
  const int tid = threadIdx.x;
  const uint32_t buf_bytes = static_cast<uint32_t>(TB * E * ROW * 4);
  float* wt = reinterpret_cast<float*>(scratch + 2 * buf_bytes);  // [ntok][G][E] weights
  const int64_t sstep = static_cast<int64_t>(a.P) * a.num_kv_heads;
  const int64_t slot0 = (static_cast<int64_t>(s0) * a.P + p) * a.num_kv_heads + h;
  if (tid == 0) {
    tc05::mbar_init(mb0, 1);
    tc05::mbar_init(mb0 + 8, 1);
    tc05::mbar_init_fence();
  }
  // weights and merged LSE of each (token, head) row
  for (int r = tid; r < ntok * G; r += blockDim.x) {
    const int i = r / G, g = r - i * G;
    const float* lp = a.ws_lse + ((slot0 + i * sstep) * a.max_chunks) * G + g;
    float mx = -INFINITY;
    for (int e = 0; e < E; ++e) mx = fmaxf(mx, __ldcg(lp + e * G));
    float sum = 0.f;
    for (int e = 0; e < E; ++e) {
      const float l = __ldcg(lp + e * G);
      sum += (mx == -INFINITY || l == -INFINITY) ? 0.f : expf(l - mx);
    }
    const float inv = sum == 0.f ? 0.f : 1.f / sum;
    for (int e = 0; e < E; ++e) {
      const float l = __ldcg(lp + e * G);
      wt[r * E + e] = (sum == 0.f || l == -INFINITY) ? 0.f : expf(l - mx) * inv;
    }
    a.lse_part[lse_slot(a, p, s0 + i, h * G + g)] = sum == 0.f ? -INFINITY : mx + logf(sum);
  }
  __syncthreads();
  const int nbatch = (ntok + TB - 1) / TB;
  auto issue = [&](int k) {
    const uint32_t mb = mb0 + (k & 1) * 8;
    const uint32_t dst = tc05::smem_addr(scratch + (k & 1) * buf_bytes);
    const int t0 = k * TB, nt = min(TB, ntok - t0);
    tc05::mbar_arrive_expect_tx(mb, static_cast<uint32_t>(nt * E * ROW * 4));
    for (int i = 0; i < nt; ++i)
      for (int e = 0; e < E; ++e)
        ws_bulk_g2s(dst + (i * E + e) * ROW * 4, a.ws_o + ((slot0 + (t0 + i) * sstep) * a.max_chunks + e) * ROW,
                    ROW * 4, mb);
  };
  if (tid == 0) {
    // the chunk rows were written by other CTAs' plain stores, published by
    // the ticket; the copies read them through the async proxy
    asm volatile("fence.proxy.async;\n" ::: "memory");
    issue(0);
    if (nbatch > 1) issue(1);
  }
  bool ok = true;
  for (int k = 0; k < nbatch; ++k) {
    ok = __syncthreads_and(tc05::mbar_wait(mb0 + (k & 1) * 8, (k >> 1) & 1)) != 0;
    if (!ok) break;
    const float4* bf = reinterpret_cast<const float4*>(scratch + (k & 1) * buf_bytes);
    const int t0 = k * TB, nt = min(TB, ntok - t0);
    for (int idx = tid; idx < nt * (ROW / 4); idx += blockDim.x) {
      const int i = idx / (ROW / 4), f = idx - i * (ROW / 4);  // token in batch, float4 of its G x D block
      const int g = f / (D / 4);
      const float* w = wt + ((t0 + i) * G + g) * E;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int e = 0; e < E; ++e) {
        const float4 v = bf[(i * E + e) * (ROW / 4) + f];
        if (w[e] != 0.f) {  // empty chunks' rows never enter the sum
          acc.x = fmaf(w[e], v.x, acc.x);
          acc.y = fmaf(w[e], v.y, acc.y);
          acc.z = fmaf(w[e], v.z, acc.z);
          acc.w = fmaf(w[e], v.w, acc.w);
        }
      }
      const int64_t orow0 = (static_cast<int64_t>(p) * a.num_tokens + s0 + t0 + i) * a.num_q_heads + h * G;
      reinterpret_cast<float4*>(a.o_part + orow0 * D)[f] = acc;
    }
    __syncthreads();  // buffer k & 1 consumed
    if (tid == 0 && k + 2 < nbatch) issue(k + 2);
  }
  if (!ok) {
    if (tid == 0) report(a.dev_status, CPATTN_DEV_TC_TIMEOUT);
    for (int k = 0; k < 2 && k < nbatch; ++k) tc05::mbar_wait(mb0 + k * 8, 0, 1u << 20);  // nothing lands later
  }
  return true;
}

// F8: an E4M3 pool.  The copy warps read each key row's codes with 16-byte
// loads, convert them exactly (every E4M3 value is a bf16 value) and store the
// bf16 row into the ring in the MMA layout; the scores take k_descale and the
// output v_descale.  Queries stay bf16.
template <int D, int G, bool F8>
__global__ void __launch_bounds__(kWThreads, 2) gqa_partial_ext_ws_kernel(const PartialArgs a) {
  using Lt = WsLayout<D>;
  constexpr int QB = kWRows / G;  // tokens per block
  constexpr int CH = D / 8;       // 16-byte chunks of a K or V row
  constexpr int RPI = 32 / CH;    // rows a warp instruction copies
  static_assert(G >= 1 && G <= 16 && (D == 64 || D == 128), "shape");
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_scan[kWThreads / 32];  // one partial sum a warp
  __shared__ int s_row[3];  // row, first token, end token of this CTA's block
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sK = base + Lt::OFF_K;
  uint8_t* sV = base + Lt::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + Lt::OFF_BAR);
  uint32_t* smask = reinterpret_cast<uint32_t*>(base + Lt::OFF_MASK);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + Lt::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(base + Lt::OFF_MISC + 4);
  int* spg = reinterpret_cast<int*>(base + Lt::OFF_PG);

  const int c = blockIdx.x;
  const int p = blockIdx.y / a.num_kv_heads;
  const int h = blockIdx.y - p * a.num_kv_heads;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int P = a.P;
  const int z = blockIdx.z;
  const int t_real = __ldg(a.qo_indptr + a.num_rows);

  // ---- block z of padding tokens past the last row: 0 / -inf (chunk 0's CTAs)
  if (c == 0) {
    const int lo = t_real + z * QB, hi = min(lo + QB, a.num_tokens);
    if (a.fused) {
      if (p == 0)
        for (int tok = lo; tok < hi; ++tok) fused_zero_token(a, tok, h, G, D);
    } else {
      for (int tok = lo; tok < hi; ++tok) {
        const int64_t orow0 = (static_cast<int64_t>(p) * a.num_tokens + tok) * a.num_q_heads + h * G;
        for (int x = tid; x < G * D; x += blockDim.x) a.o_part[orow0 * D + x] = 0.f;
        if (tid < G) a.lse_part[lse_slot(a, p, tok, h * G + tid)] = -INFINITY;
      }
    }
  }
  // ---- row block z: the rows of >= 2 tokens in order, ceil(n / QB) blocks
  // each; found with a block-wide prefix sum over the rows (one-token rows
  // are the decode kernel's)
  if (tid == 0) s_row[0] = -1;
  {
    int done_blocks = 0;
    for (int r0 = 0; r0 < a.num_rows; r0 += blockDim.x) {
      const int r = r0 + tid;
      int nb = 0, first = 0, n = 0;
      if (r < a.num_rows) {
        first = __ldg(a.qo_indptr + r);
        n = __ldg(a.qo_indptr + r + 1) - first;
        nb = n >= 2 ? (n + QB - 1) / QB : 0;
      }
      int incl = nb;  // inclusive scan within the warp
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      __syncthreads();  // s_scan of the previous round is read
      if (lane == 31) s_scan[warp] = incl;
      __syncthreads();
      int before = done_blocks, total = done_blocks;
      for (int w = 0; w < kWThreads / 32; ++w) {
        if (w < warp) before += s_scan[w];
        total += s_scan[w];
      }
      const int lo = before + incl - nb;
      if (nb > 0 && z >= lo && z < lo + nb) {
        s_row[0] = r;
        s_row[1] = first + (z - lo) * QB;
        s_row[2] = min(first + n, first + (z - lo) * QB + QB);
      }
      done_blocks = total;
    }
    __syncthreads();
  }
  const int b = s_row[0];
  if (b < 0) return;
  const int s0 = s_row[1], s1 = s_row[2];
  int L = __ldg(a.kv_len + b);
  if (L > a.max_kv_len) {
    if (c == 0 && tid == 0) report(a.dev_status, CPATTN_DEV_POS_PAST_TABLE);
    L = a.max_kv_len;
  }
  const int n_p = stripe_len(L, p, P, a.interleave);
  const int nchunks = n_p > 0 ? (n_p + a.chunk - 1) / a.chunk : 1;
  if (c >= nchunks) return;
  const int k_begin = c * a.chunk;
  const int k_end = min(n_p, k_begin + a.chunk);
  const int ntiles = k_end > k_begin ? (k_end - k_begin + kWTile - 1) / kWTile : 0;
  const bool single = (nchunks == 1);
  const int my_tok = s0 + tid / G;  // softmax threads
  const bool my_ok = tid < kWRows && my_tok < s1;
  const int my_g = tid % G;

  bool done = true;  // this CTA holds the partner's complete partial of the segment
  if (ntiles == 0) {  // empty stripe of this row for this partner: 0 / -inf
    if (my_ok) {
      const int64_t orow = (static_cast<int64_t>(p) * a.num_tokens + my_tok) * a.num_q_heads + h * G + my_g;
      float4* d4 = reinterpret_cast<float4*>(a.o_part + orow * D);
      for (int e = 0; e < D / 4; ++e) d4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      a.lse_part[lse_slot(a, p, my_tok, h * G + my_g)] = -INFINITY;
    }
  } else {
    // ---- page ids of the chunk, checked once
    const int j0 = k_begin / a.ps_l;
    {
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
    auto bar = [&](int i) { return tc05::smem_addr(&bars[i]); };
    if (tid == 0) {
      for (int i = 0; i < W_MERGE; ++i) {  // the merge initialises its own two
        uint32_t cnt = 1;
        if (i < W_KFREE) cnt = 64;                    // the two K warps' lanes
        if (i >= W_VFULL && i < W_VFREE) cnt = 32;    // the V warp's lanes
        if (i == W_Q) cnt = 96;
        if (i >= W_SFREE && i < W_SFREE + 4) cnt = 4;  // sfree, pfull: one arrival a softmax warp
        tc05::mbar_init(bar(i), cnt);
      }
      *s_abort = 0;
      tc05::mbar_init_fence();
    }
    if (warp == 0) tc05::tmem_alloc(tc05::smem_addr(tmem_slot), Lt::TMEM_COLS);
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    const uint32_t tbase = *tmem_slot;

    bool alive = true;
    if (warp >= kWLoadK) {
      // ================= copies: Q (all three), then K tiles (warps 5, 7) or V tiles (warp 6) =================
      const bool is_k = (warp != kWLoadV);
      const int khalf = (warp == kWLoadK2) ? 1 : 0;  // K warps: which half of each tile's keys
      {
        const uint8_t* q = static_cast<const uint8_t*>(a.q);
        const uint32_t q0 = tc05::smem_addr(sQ);
        for (int x = (warp - kWLoadK) * 32 + lane; x < kWRows * CH; x += 96) {
          const int r = x / CH, cc = x - r * CH;
          const int tok = s0 + r / G;
          const uint32_t dst = q0 + (cc >> 3) * Lt::QBLK + tc05::sw128(r, cc & 7);
          if (tok < s1)
            ws_cp16(dst, q + ((static_cast<int64_t>(tok) * a.num_q_heads + h * G + r % G) * D + cc * 8) * 2);
          else
            ws_cp16_zero(dst, q);
        }
        ws_cp_arrive(bar(W_Q));
      }
      const uint8_t* pool = static_cast<const uint8_t*>(is_k ? a.pool_k : a.pool_v);
      const int nst = is_k ? kKStages : kVStages;
      const uint32_t ring = tc05::smem_addr(is_k ? sK : sV);
      const int b_full = is_k ? W_KFULL : W_VFULL, b_free = is_k ? W_KFREE : W_VFREE;
      const int64_t head_row0 = static_cast<int64_t>(p) * a.num_pages * a.num_kv_heads + h;
      const int ro = lane / CH, cc = lane - (lane / CH) * CH;
      const uint32_t coff = (cc >> 3) * Lt::BLK;
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % nst;
        if (i >= nst) {
          const bool ok = ws_wait(bar(b_free + st), ((i - nst) / nst) & 1, s_abort);
          if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
        }
        int myrow = -1;  // lane k: pool row of key k of the tile (the launch checks rows fit 31 bits)
        {
          const int k = k_begin + i * kWTile + lane;
          if (k < k_end) {
            const int j = page_of_slot(a, k);
            const int pg = spg[j - j0];
            if (pg >= 0)
              myrow = static_cast<int>((head_row0 + static_cast<int64_t>(pg) * a.num_kv_heads) * a.ps_l + (k - j * a.ps_l));
          }
        }
        if (is_k && khalf == 0) {
          // keys of the tile that hold data, for the softmax mask: written
          // before the tile's copies; its slot is rewritten kMaskSlots tiles
          // later, when the softmax has long read it
          const uint32_t vm = __ballot_sync(0xffffffffu, myrow >= 0);
          if (lane == 0) {
            smask[i % kMaskSlots] = vm;
            __threadfence_block();
          }
        }
        const uint32_t dst0 = ring + st * Lt::TILE;
        if constexpr (F8) {
          // lane: 16 codes (chunk c8 of a key row) -> two bf16 chunks; the
          // warp's loads all go out before any conversion
          constexpr int CH8 = D / 16, RPI8 = 32 / CH8;
          constexpr int NK = kWTile / RPI8;  // keys a lane takes in the V warp (half that in a K warp)
          const int ro8 = lane / CH8, c8 = lane - (lane / CH8) * CH8;
          const int kstep8 = is_k ? 2 * RPI8 : RPI8;
          uint4 codes[NK];
#pragma unroll
          for (int u = 0; u < NK; ++u) {
            const int key = ro8 + (is_k ? khalf * RPI8 : 0) + u * kstep8;
            const int row = __shfl_sync(0xffffffffu, myrow, key & 31);
            codes[u] = make_uint4(0u, 0u, 0u, 0u);  // masked key: zero row
            if (key < kWTile && row >= 0)
              codes[u] = __ldg(reinterpret_cast<const uint4*>(pool + static_cast<int64_t>(row) * D + c8 * 16));
          }
#pragma unroll
          for (int u = 0; u < NK; ++u) {
            const int key = ro8 + (is_k ? khalf * RPI8 : 0) + u * kstep8;
            if (key >= kWTile) continue;
            const uint32_t w[4] = {codes[u].x, codes[u].y, codes[u].z, codes[u].w};
            uint32_t bf[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              bf[2 * q] = e4m3x2_to_bf16x2(w[q]);
              bf[2 * q + 1] = e4m3x2_to_bf16x2(w[q] >> 16);
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int cb = 2 * c8 + hh;  // bf16 chunk of the row (8 values)
              *reinterpret_cast<uint4*>(base + (dst0 - tc05::smem_addr(base)) + (cb >> 3) * Lt::BLK +
                                        tc05::sw128(key, cb & 7)) =
                  make_uint4(bf[4 * hh], bf[4 * hh + 1], bf[4 * hh + 2], bf[4 * hh + 3]);
            }
          }
          tc05::fence_smem_to_async();  // the tensor core reads what this lane wrote
          ws_arrive(bar(b_full + st));
        } else {
          // unrolled: the shuffles and addresses of all the warp's rows are
          // formed before the copies issue (one chain a row is latency-bound)
          const int kstep = is_k ? 2 * RPI : RPI;  // the K warps split the keys
#pragma unroll 8
          for (int key = ro + khalf * RPI; key < kWTile; key += kstep) {
            const int row = __shfl_sync(0xffffffffu, myrow, key);
            const uint32_t dst = dst0 + coff + tc05::sw128(key, cc & 7);
            if (row >= 0) ws_cp16(dst, pool + (static_cast<int64_t>(row) * D + cc * 8) * 2);
            else ws_cp16_zero(dst, pool);  // masked key: zero row (finite scores, zero values)
          }
          ws_cp_arrive(bar(b_full + st));
        }
      }
      cp_async_wait<0>();  // nothing lands after the CTA moves on
      if (!alive) *s_abort = 1;
    } else if (tid == kWMma) {
      // ================= MMA issue =================
      const uint64_t dq = tc05::desc_k128(tc05::smem_addr(sQ));
      const uint32_t id_s = tc05::idesc_bf16(128, kWTile, false, false);
      const uint32_t id_o = tc05::idesc_bf16(128, D, false, true);
      int batches = 0;
      auto issue_s = [&](int i) -> bool {
        const int bb = i & 1, st = i % kKStages;
        if (!ws_wait(bar(W_KFULL + st), (i / kKStages) & 1, s_abort)) return false;
        if (i >= 2 && !ws_wait(bar(W_SFREE + bb), ((i >> 1) - 1) & 1, s_abort)) return false;
        // the copies landed through the generic proxy; the tensor core reads them
        tc05::fence_smem_to_async();
        tc05::fence_after_sync();
        const uint64_t dk = tc05::desc_k128(tc05::smem_addr(sK + st * Lt::TILE));
#pragma unroll
        for (int s = 0; s < D / 16; ++s)
          tc05::mma_ss(tbase + Lt::S_COL + 32 * bb, tc05::desc_add(dq, (s >> 2) * Lt::QBLK + (s & 3) * 32),
                       tc05::desc_add(dk, (s >> 2) * Lt::BLK + (s & 3) * 32), id_s, s > 0);
        tc05::commit(bar(W_SDONE + bb));
        tc05::commit(bar(W_KFREE + st));
        ++batches;
        return true;
      };
      alive = ws_wait(bar(W_Q), 0, s_abort);
      if (alive) alive = issue_s(0);
      if (alive && ntiles > 1) alive = issue_s(1);
      for (int j = 0; j < ntiles && alive; ++j) {
        const int bb = j & 1, st = j % kVStages;
        if (j + 2 < ntiles && !issue_s(j + 2)) { alive = false; break; }
        if (!ws_wait(bar(W_PFULL + bb), (j >> 1) & 1, s_abort)) { alive = false; break; }
        if (!ws_wait(bar(W_VFULL + st), (j / kVStages) & 1, s_abort)) { alive = false; break; }
        tc05::fence_smem_to_async();
        tc05::fence_after_sync();
        const uint64_t dv = tc05::desc_mn128(tc05::smem_addr(sV + st * Lt::TILE), Lt::BLK);
#pragma unroll
        for (int s = 0; s < kWTile / 16; ++s)  // P from tensor memory: 8 columns a 16-key step
          tc05::mma_ts(tbase + Lt::O_COL, tbase + Lt::P_COL + 16 * bb + 8 * s, tc05::desc_add(dv, s * 16 * 128),
                       id_o, j > 0 || s > 0);
        tc05::commit(bar(W_PVDONE + bb));
        tc05::commit(bar(W_VFREE + st));
        ++batches;
      }
      if (!alive) {
        *s_abort = 1;
        if (batches > 0) {  // no MMA may still run when the tensor memory is released
          tc05::commit(bar(W_FIN));
          tc05::mbar_wait(bar(W_FIN), 0, 1u << 20);
        }
      }
    } else if (tid < kWRows) {
      // ================= softmax rows =================
      const uint32_t my_lane = tc05::taddr(tbase, warp * 32, 0);
      const float sl = a.scale * kLog2e * (F8 ? a.k_descale : 1.f);
      float m = -INFINITY, l = 0.f, lr = 0.f;  // running max (log2), fp32 sum, sum of bf16-rounded p
      for (int i = 0; i < ntiles; ++i) {
        const int bb = i & 1;
        bool ok = ws_wait(bar(W_SDONE + bb), (i >> 1) & 1, s_abort);
        if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
        tc05::fence_after_sync();
        const uint32_t vmask = smask[i % kMaskSlots];  // written before tile i's K copies
        float sv[32];
        {
          // both halves of the row's scores in flight at once
          float v0[16], v1[16];
          tc05::ld_x16(my_lane + Lt::S_COL + 32 * bb, v0);
          tc05::ld_x16(my_lane + Lt::S_COL + 32 * bb + 16, v1);
          tc05::ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            sv[e] = v0[e];
            sv[16 + e] = v1[e];
          }
        }
        tc05::fence_before_sync();
        __syncwarp();
        if (lane == 0) ws_arrive(bar(W_SFREE + bb));
        // keys without data: -inf (probability 0); scores stay unscaled, the
        // running max is in log2 units; the max as a tree, not a chain
        if (vmask != 0xffffffffu) {
#pragma unroll
          for (int e = 0; e < 32; ++e) sv[e] = ((vmask >> e) & 1u) ? sv[e] : -INFINITY;
        }
        float mx[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) mx[e] = fmaxf(sv[e], sv[16 + e]);
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
          for (int e = 0; e < w; ++e) mx[e] = fmaxf(mx[e], mx[e + w]);
        const float bm = mx[0] * sl;
        const bool up = bm > m + 8.f;
        if (__any_sync(0xffffffffu, up) && i > 0) {
          // rescale O rows whose max rose; P V of the previous tile must be done
          ok = ws_wait(bar(W_PVDONE + ((i - 1) & 1)), ((i - 1) >> 1) & 1, s_abort);
          if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
          tc05::fence_after_sync();
          const float alpha = up ? exp2f(m - bm) : 1.f;
#pragma unroll
          for (int col = 0; col < D; col += 16) {
            float v[16];
            tc05::ld_x16(my_lane + Lt::O_COL + col, v);
            tc05::ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] *= alpha;
            tc05::st_x16(my_lane + Lt::O_COL + col, v);
          }
          tc05::st_wait();
          l *= alpha;
          lr *= alpha;
        }
        if (up) m = bm;
        // P(i) into its buffer once P V of tile i-2 no longer reads it
        if (i >= 2) {
          ok = ws_wait(bar(W_PVDONE + bb), ((i - 2) >> 1) & 1, s_abort);
          if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
        }
        {
          // p = 2^(s * scale * log2 e - m): one FMA and one ex2 a key (-inf
          // gives 0; while every key so far is masked m is -inf and every p
          // is 0); four partial sums of p and of bf16(p) each
          const float nm = m == -INFINITY ? 0.f : -m;
          float ls[4] = {0.f, 0.f, 0.f, 0.f}, lrs[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t pk[16];  // bf16 pairs of keys 2e, 2e+1: row `tid` of P, as the MMA reads it from TMEM
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float pa = ex2_approx(fmaf(sv[2 * e], sl, nm));
            const float pb = ex2_approx(fmaf(sv[2 * e + 1], sl, nm));
            ls[e & 3] += pa + pb;
            __nv_bfloat162 h2 = __floats2bfloat162_rn(pa, pb);
            pk[e] = *reinterpret_cast<uint32_t*>(&h2);
            lrs[e & 3] += __uint_as_float(pk[e] << 16) + __uint_as_float(pk[e] & 0xffff0000u);
          }
          l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
          lr += (lrs[0] + lrs[1]) + (lrs[2] + lrs[3]);
          tc05::st_x16_u32(my_lane + Lt::P_COL + 16 * bb, pk);
          asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
        }
        tc05::fence_before_sync();
        __syncwarp();
        if (lane == 0) ws_arrive(bar(W_PFULL + bb));
      }
      if (alive) {
        const int last = ntiles - 1;
        const bool ok = ws_wait(bar(W_PVDONE + (last & 1)), (last >> 1) & 1, s_abort);
        alive = __all_sync(0xffffffffu, ok);
      }
      if (!alive) {
        *s_abort = 1;
      } else {
        // ---- row `tid`: normalised output and LSE, to o_part or the chunk workspace
        tc05::fence_after_sync();
        const float inv = lr > 0.f ? (F8 ? a.v_descale : 1.f) / lr : 0.f;  // E4M3: value = code * v_descale
        const float lse = l == 0.f ? -INFINITY : (m + log2f(l)) * kLn2;
        float* dst = nullptr;
        float* ldst = nullptr;
        if (single) {
          const int64_t orow = (static_cast<int64_t>(p) * a.num_tokens + my_tok) * a.num_q_heads + h * G + my_g;
          dst = a.o_part + orow * D;
          ldst = a.lse_part + lse_slot(a, p, my_tok, h * G + my_g);
        } else {
          const int64_t slot = (static_cast<int64_t>(my_tok) * P + p) * a.num_kv_heads + h;
          const int64_t wrow = (slot * a.max_chunks + c) * G + my_g;
          dst = a.ws_o + wrow * D;
          ldst = a.ws_lse + wrow;
        }
#pragma unroll
        for (int col = 0; col < D; col += 16) {
          float v[16];
          tc05::ld_x16(my_lane + Lt::O_COL + col, v);  // warp-collective: every lane loads
          tc05::ld_wait();
          if (my_ok) {
            float4* d4 = reinterpret_cast<float4*>(dst + col);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              d4[e] = make_float4(v[4 * e] * inv, v[4 * e + 1] * inv, v[4 * e + 2] * inv, v[4 * e + 3] * inv);
          }
        }
        if (my_ok) *ldst = lse;
      }
    }
    tc05::fence_before_sync();
    __syncthreads();
    const bool ok_all = *s_abort == 0;
    if (warp == 0) tc05::tmem_dealloc(tbase, Lt::TMEM_COLS);
    if (!ok_all) {
      if (tid == 0) report(a.dev_status, CPATTN_DEV_TC_TIMEOUT);
      return;
    }
    if (!single) {
      const int64_t slot0 = (static_cast<int64_t>(s0) * P + p) * a.num_kv_heads + h;
      done = take_ticket(a.ws_cnt + slot0, nchunks);
      if (done) {
        if (!ws_merge_chunks_bulk<D, G>(a, p, h, s0, s1, nchunks, base, Lt::MERGE_BYTES,
                                        tc05::smem_addr(&bars[W_MERGE])))
          merge_chunks<kWMergeUnroll>(a, p, h, s0, s1 - s0, slot0, static_cast<int64_t>(P) * a.num_kv_heads,
                                      nchunks, G, D, reinterpret_cast<float*>(sK), Lt::SCRATCH_FLOATS);
        if (tid == 0) a.ws_cnt[slot0] = 0;
      }
    }
  }
  if (a.fused && done) {
    // fused: the last of the P partners of (segment, KV head) merges them
    int32_t* pair = a.ws_pair + static_cast<int64_t>(s0) * a.num_kv_heads + h;
    if (take_ticket(pair, P)) {
      merge_partners<kWMergeUnroll>(a, s0, s1 - s0, h, G, D, reinterpret_cast<float*>(sK), Lt::SCRATCH_FLOATS);
      if (tid == 0) *pair = 0;
    }
  }
}

template <int D, int G, bool F8>
static int launch_ext_ws_t(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  constexpr int QB = kWRows / G;
  const int page_slots = a.chunk / a.ps_l + 2;
  const size_t smem = WsLayout<D>::smem_bytes(page_slots);
  if (smem > 227 * 1024) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  // the copy warps exchange pool row indices as 32-bit values
  if (static_cast<int64_t>(a.P) * a.num_pages * a.num_kv_heads * a.ps_l >= (int64_t{1} << 31))
    return CPATTN_ERR_UNSUPPORTED_SHAPE;
  auto kern = gqa_partial_ext_ws_kernel<D, G, F8>;
  static std::atomic<int> smem_set[64];
  *err = ensure_smem(kern, smem, smem_set);
  if (*err != cudaSuccess) return CPATTN_ERR_CUDA;
  // row blocks: at most one partial block a row beyond T / QB full ones (the
  // first T / QB of them also cover the blocks of padding tokens)
  const int qblocks = (a.num_tokens + QB - 1) / QB;
  dim3 grid(a.max_chunks, a.P * a.num_kv_heads, a.num_rows + qblocks);
  kern<<<grid, kWThreads, smem, s>>>(a);
  *err = cudaGetLastError();
  return *err == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

template <int D, bool F8>
static int ext_ws_dispatch_g(const PartialArgs& a, int G, cudaStream_t s, cudaError_t* err) {
  switch (G) {
    case 1: return launch_ext_ws_t<D, 1, F8>(a, s, err);
    case 2: return launch_ext_ws_t<D, 2, F8>(a, s, err);
    case 4: return launch_ext_ws_t<D, 4, F8>(a, s, err);
    case 8: return launch_ext_ws_t<D, 8, F8>(a, s, err);
    case 16: return launch_ext_ws_t<D, 16, F8>(a, s, err);
    default: return CPATTN_ERR_UNSUPPORTED_SHAPE;
  }
}

int launch_gqa_partial_ext(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  return launch_gqa_partial_ext_ws(a, s, err);
}

int launch_gqa_partial_ext_ws(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  const int G = a.num_q_heads / a.num_kv_heads;
  if (a.kv_fp8) {
    if (a.head_dim == 128) return ext_ws_dispatch_g<128, true>(a, G, s, err);
    if (a.head_dim == 64) return ext_ws_dispatch_g<64, true>(a, G, s, err);
    return CPATTN_ERR_UNSUPPORTED_SHAPE;
  }
  if (a.head_dim == 128) return ext_ws_dispatch_g<128, false>(a, G, s, err);
  if (a.head_dim == 64) return ext_ws_dispatch_g<64, false>(a, G, s, err);
  return CPATTN_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace cpattn
