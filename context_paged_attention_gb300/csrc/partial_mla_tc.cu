// cp_paged_attn_partial, MLA path on the tcgen05 tensor cores.
//
// MLA's one latent KV head is striped like a GQA head (mstar PR #1124
// "Context / Sequence Parallel 1/5", description: MLA's one latent head
// included; copy_slots indexes the token axis): partner p's stripe slot k is
// logical position k * P + p at physical slot k % (page_size / P) of page
// k / (page_size / P).  All 128 query heads of a token share the latent rows,
// so the partial is a dense contraction with M = 128 heads:
//   S = Q K^T   (K = 576 latent + rope values)
//   O += P V    (V = the first 512 values of the same latent rows)
//
// CTA = (chunk, partner, token), 4 warps; thread i owns head i (TMEM lane i),
// so the online softmax needs no cross-thread reduction.  Shared memory (all
// 1024-byte aligned): Q [128 x 576] K-major with the 128-byte swizzle (9
// column blocks, resident), two stages of 32 latent rows (9 blocks of
// 32 x 128 B; the same bytes are read K-major for S and M/N-major for P V),
// and P [128 x 32] bf16 K-major with the 64-byte swizzle.  Tensor memory (512
// columns): O for value dims 0..447 accumulates in columns 0..447; columns
// 448..511 hold S (two 32-column accumulation chains, summed on read-back)
// and, after the softmax, the P V product of dims 448..511, which the threads
// add into registers -- O (512 x 128 fp32) and S together would need more
// than the 512 columns.
//
// Loads: with page runs that tile the 32-key tile evenly, thread 32 (while
// thread 0 issues the S MMAs) copies each run of latent rows with TMA (tensor-map bulk copies, 128-byte swizzle,
// completion counted in bytes on the stage's mbarrier) -- 9 copies of 64
// columns per run -- and Q the same way.  Other page sizes use 16-byte
// cp.async copies.  Rows of keys past the stripe end are zeroed before P V
// (their S is masked to -inf), so unwritten pool slots never reach the output.
//
// Per 32-key tile: wait for the tile, one thread issues the 36 S MMAs and the
// next tile's copies, the threads read S, update the running max (raised only
// when it grows by more than 8 in log2 units, so rescaling O in TMEM is rare
// and every probability stays <= 2^8), write P as bf16, and one thread issues
// the P V MMAs.  O is normalised by the sum of the bf16-rounded probabilities
// (an exact convex combination of the values); the LSE uses the fp32 sum.
// Every wait is bounded; a wait that runs out reports CPATTN_DEV_TC_TIMEOUT,
// and the CTA stops, frees its tensor memory and returns.
#include <cuda.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "split_combine.cuh"
#include "tc05.cuh"

namespace cpattn {

namespace {
constexpr int kHeads = 128;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kBlocks = kDqk / 64;          // 9 column blocks of 64 values
constexpr int kTile = 32;                   // keys per tile
constexpr int kRowB = kDqk * 2;             // 1152 bytes per latent row
constexpr int kChunks = kRowB / 16;         // 72 16-byte chunks per row
constexpr int kQBytes = kBlocks * kHeads * 128;   // 147456
constexpr int kBlkB = kTile * 128;                // 4096: one column block of a tile
constexpr int kTileBytes = kBlocks * kBlkB;       // 36864
constexpr int kPBytes = kHeads * 64;              // 8192
constexpr int kMainCols = 448;              // O columns kept in TMEM
constexpr int kTailCol = 448;               // S, then the P V tail
constexpr int kPageSlots = 256;             // staged page ids per CTA
constexpr int kBars = 7;                    // tile stage 0 / 1 full, Q full, S done, P V done, 2 merge buffers
constexpr int kMergeUnroll = 8;             // float4 loads in flight a thread in the chunk / partner merges
constexpr int kTmaThread = 32;              // issues the TMA copies (warp 1), beside thread 0's MMAs
constexpr size_t kSmemBytes = 1024 /*align*/ + kQBytes + 2 * kTileBytes + kPBytes + kPageSlots * 4 + kBars * 8 + 8;
constexpr int kScratchB = kQBytes + 2 * kTileBytes + kPBytes;  // contiguous shared memory free after the key loop

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(mbar)
               : "memory");
}

// Split-KV merge of the E chunk partials of (token t, partner p) into the
// partner partial: the LSE merge, as merge_chunks does, with the chunk rows
// brought into shared memory by bulk asynchronous copies (one thread keeps
// E x HB x 2 KB in flight; two buffers, batches of HB heads), so that one CTA
// reads the E x 256 KB at copy speed.  Returns false when the shared memory
// cannot hold two batches of one head (the caller falls back to merge_chunks)
// or a copy did not land within the poll limit (reported).  All threads call.
__device__ bool mla_merge_chunks_bulk(const PartialArgs& a, int p, int t, int64_t slot, int E, uint8_t* scratch,
                                      uint64_t* mb2) {
  int HB = 8;
  while (HB > 0 && 2 * E * HB * (kDv * 4) + E * kHeads * 4 > kScratchB) HB >>= 1;
  if (HB == 0) return false;
  const int tid = threadIdx.x;
  const uint32_t buf_bytes = static_cast<uint32_t>(E * HB * kDv * 4);
  uint8_t* buf0 = scratch;
  float* wt = reinterpret_cast<float*>(scratch + 2 * buf_bytes);  // [E][128] weights
  const uint32_t mb0 = tc05::smem_addr(&mb2[0]);
  if (tid == 0) {
    tc05::mbar_init(mb0, 1);
    tc05::mbar_init(mb0 + 8, 1);
    tc05::mbar_init_fence();
  }
  // weights of head `tid` (128 threads, one head each) and its merged LSE
  {
    const int h = tid;
    const float* lp = a.ws_lse + (slot * a.max_chunks) * kHeads + h;
    float mx = -INFINITY;
    for (int e = 0; e < E; ++e) mx = fmaxf(mx, __ldcg(lp + e * kHeads));
    float sum = 0.f;
    for (int e = 0; e < E; ++e) {
      const float l = __ldcg(lp + e * kHeads);
      sum += (mx == -INFINITY || l == -INFINITY) ? 0.f : expf(l - mx);
    }
    const float inv = sum == 0.f ? 0.f : 1.f / sum;
    for (int e = 0; e < E; ++e) {
      const float l = __ldcg(lp + e * kHeads);
      wt[e * kHeads + h] = (sum == 0.f || l == -INFINITY) ? 0.f : expf(l - mx) * inv;
    }
    a.lse_part[lse_slot(a, p, t, h)] = sum == 0.f ? -INFINITY : mx + logf(sum);
  }
  __syncthreads();
  const int nbatch = kHeads / HB;
  auto issue = [&](int k) {
    const uint32_t mb = mb0 + (k & 1) * 8;
    const uint32_t dst = tc05::smem_addr(buf0 + (k & 1) * buf_bytes);
    tc05::mbar_arrive_expect_tx(mb, buf_bytes);
    for (int e = 0; e < E; ++e)
      bulk_g2s(dst + e * HB * kDv * 4, a.ws_o + ((slot * a.max_chunks + e) * kHeads + k * HB) * kDv, HB * kDv * 4, mb);
  };
  if (tid == 0) {
    // the chunk rows were written by other CTAs' plain stores, published by
    // the ticket; the copies read them through the async proxy
    asm volatile("fence.proxy.async;\n" ::: "memory");
    issue(0);
    if (nbatch > 1) issue(1);
  }
  const int64_t orow0 = (static_cast<int64_t>(p) * a.num_tokens + t) * a.num_q_heads;
  bool ok = true;
  for (int k = 0; k < nbatch; ++k) {
    ok = __syncthreads_and(tc05::mbar_wait(mb0 + (k & 1) * 8, (k >> 1) & 1)) != 0;
    if (!ok) break;
    const float4* bf = reinterpret_cast<const float4*>(buf0 + (k & 1) * buf_bytes);
    for (int idx = tid; idx < HB * (kDv / 4); idx += blockDim.x) {
      const int hl = idx / (kDv / 4);
      const int h = k * HB + hl;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int e = 0; e < E; ++e) {
        const float w = wt[e * kHeads + h];
        const float4 v = bf[e * HB * (kDv / 4) + idx];
        if (w != 0.f) {  // empty chunks' rows never enter the sum
          acc.x = fmaf(w, v.x, acc.x);
          acc.y = fmaf(w, v.y, acc.y);
          acc.z = fmaf(w, v.z, acc.z);
          acc.w = fmaf(w, v.w, acc.w);
        }
      }
      reinterpret_cast<float4*>(a.o_part + (orow0 + h) * kDv)[idx - hl * (kDv / 4)] = acc;
    }
    __syncthreads();  // buffer k & 1 consumed
    if (tid == 0 && k + 2 < nbatch) issue(k + 2);
  }
  if (!ok) {
    if (tid == 0) report(a.dev_status, CPATTN_DEV_TC_TIMEOUT);
    // nothing may land after the CTA exits: wait (bounded) for both buffers' copies
    for (int k = 0; k < 2 && k < nbatch; ++k) tc05::mbar_wait(mb0 + k * 8, 0, 1u << 20);
  }
  return true;
}
}  // namespace

template <bool kTma>
__global__ void __launch_bounds__(128, 1)
    mla_partial_tc_kernel(const PartialArgs a, const __grid_constant__ CUtensorMap tmap_kv,
                          const __grid_constant__ CUtensorMap tmap_q, int box_rows) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sKV = sQ + kQBytes;  // two stages
  uint8_t* sP = sKV + 2 * kTileBytes;
  int* spg = reinterpret_cast<int*>(sP + kPBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(spg + kPageSlots);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBars);

  const int c = blockIdx.x;
  const int p = blockIdx.y;
  // token of this grid slot (a dispatch order applies when tokens are rows)
  const int t = a.qo_indptr == nullptr ? ordered_row(a.row_order, blockIdx.z, gridDim.z, a.dev_status) : blockIdx.z;
  if (t < 0) return;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int P = a.P;

  // ---- row, stripe length, chunk bounds (same rules as the other partial kernels)
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
      if (c == 0 && tid == 0) report(a.dev_status, CPATTN_DEV_POS_PAST_TABLE);
      L = a.max_kv_len;
    }
    n_p = stripe_len(L, p, P, a.interleave);
  }
  const int nchunks = n_p > 0 ? (n_p + a.chunk - 1) / a.chunk : 1;
  if (c >= nchunks) return;
  const int k_begin = c * a.chunk;
  const int k_end = min(n_p, k_begin + a.chunk);
  const int ntiles = k_end > k_begin ? (k_end - k_begin + kTile - 1) / kTile : 0;

  const int64_t orow = (static_cast<int64_t>(p) * a.num_tokens + t) * a.num_q_heads + tid;  // head tid
  const int64_t slot = static_cast<int64_t>(t) * P + p;
  if (ntiles == 0) {  // empty stripe (or padding token): 0 / -inf
    float4* dst = reinterpret_cast<float4*>(a.o_part + orow * kDv);
    for (int e = 0; e < kDv / 4; ++e) dst[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    a.lse_part[lse_slot(a, p, t, tid)] = -INFINITY;
    if (a.fused) pair_finish<kMergeUnroll>(a, t, 0, kHeads, kDv, reinterpret_cast<float*>(sQ), kQBytes / 4);
    return;
  }

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
  // pool row of stripe slot k (k < k_end), or -1 on a rejected page
  auto pool_row = [&](int k) -> int64_t {
    const int jj = page_of_slot(a, k);
    const int pg = spg[jj - j0];
    if (pg < 0) return -1;
    return (static_cast<int64_t>(p) * a.num_pages + pg) * a.ps_l + (k - jj * a.ps_l);
  };

  if (tid == 0) {
    for (int i = 0; i < kBars; ++i) tc05::mbar_init(tc05::smem_addr(&bars[i]), 1);
    tc05::mbar_init_fence();
  }
  if (warp == 0) tc05::tmem_alloc(tc05::smem_addr(tmem_slot), 512);
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  const uint32_t tbase = *tmem_slot;
  const uint32_t mb_full0 = tc05::smem_addr(&bars[0]);
  const uint32_t mb_q = tc05::smem_addr(&bars[2]);
  const uint32_t mb_s = tc05::smem_addr(&bars[3]);
  const uint32_t mb_pv = tc05::smem_addr(&bars[4]);
  const uint32_t my_lane = tc05::taddr(tbase, warp * 32, 0);

  const uint8_t* pool = static_cast<const uint8_t*>(a.pool_k);
  // ---- copies of tile i into stage i & 1
  auto load_tile = [&](int i) {
    uint8_t* st = sKV + (i & 1) * kTileBytes;
    const int k0 = k_begin + i * kTile;
    if constexpr (kTma) {
      if (tid == kTmaThread) {
        const int runs = kTile / box_rows;
        uint32_t bytes = 0;
        for (int r = 0; r < runs; ++r) {
          const int kr = k0 + r * box_rows;
          if (kr < k_end && pool_row(kr) >= 0) bytes += kBlocks * box_rows * 128;
        }
        const uint32_t mb = mb_full0 + (i & 1) * 8;
        tc05::mbar_arrive_expect_tx(mb, bytes);
        for (int r = 0; r < runs; ++r) {
          const int kr = k0 + r * box_rows;
          if (kr >= k_end) break;
          const int64_t row = pool_row(kr);
          if (row < 0) continue;
          const uint32_t dst = tc05::smem_addr(st + r * box_rows * 128);
#pragma unroll
          for (int kb = 0; kb < kBlocks; ++kb)
            tc05::tma_load_2d(dst + kb * kBlkB, &tmap_kv, kb * 64, static_cast<int>(row), mb);
        }
      }
    } else {
      // each warp resolves the 32 keys' row addresses (lane = key), its threads
      // pick them up with shuffles: no division in the copy loop
      const uint8_t* myrow = nullptr;
      {
        const int k = k0 + lane;
        if (k < k_end) {
          const int64_t row = pool_row(k);
          if (row >= 0) myrow = pool + row * kRowB;
        }
      }
#pragma unroll 2
      for (int x = tid; x < kTile * kChunks; x += blockDim.x) {
        const int key = x / kChunks;
        const int cc = x - key * kChunks;
        const uint8_t* src =
            reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(myrow), key));
        uint8_t* dst = st + (cc >> 3) * kBlkB + tc05::sw128(key, cc & 7);
        if (src != nullptr) {
          cp_async16(dst, src + cc * 16);
        } else {
          *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      cp_async_commit();
    }
  };

  // ---- Q (all heads of token t) and the first tile
  if constexpr (kTma) {
    if (tid == 0) {
      tc05::mbar_arrive_expect_tx(mb_q, kQBytes);
#pragma unroll
      for (int kb = 0; kb < kBlocks; ++kb)
        tc05::tma_load_2d(tc05::smem_addr(sQ + kb * (kHeads * 128)), &tmap_q, kb * 64, t * kHeads, mb_q);
    }
  } else {
    const uint8_t* qsrc = static_cast<const uint8_t*>(a.q) + static_cast<int64_t>(t) * a.num_q_heads * kRowB;
    for (int x = tid; x < kHeads * kChunks; x += blockDim.x) {
      const int h = x / kChunks;
      const int cc = x - h * kChunks;
      cp_async16(sQ + (cc >> 3) * (kHeads * 128) + tc05::sw128(h, cc & 7), qsrc + h * kRowB + cc * 16);
    }
  }
  load_tile(0);

  const uint32_t id_s = tc05::idesc_bf16(128, kTile, false, false);
  const uint32_t id_256 = tc05::idesc_bf16(128, 256, false, true);
  const uint32_t id_192 = tc05::idesc_bf16(128, 192, false, true);
  const uint32_t id_64 = tc05::idesc_bf16(128, 64, false, true);
  const uint64_t dq = tc05::desc_k128(tc05::smem_addr(sQ));
  const uint64_t dp = tc05::desc_k64(tc05::smem_addr(sP));
  const float sl = a.scale * kLog2e;

  float m = -INFINITY, l = 0.f, lr = 0.f;  // running max (log2), fp32 sum, sum of bf16-rounded p
  float tail[64];
#pragma unroll
  for (int e = 0; e < 64; ++e) tail[e] = 0.f;
  bool alive = true;
  if constexpr (kTma) alive = __syncthreads_and(tc05::mbar_wait(mb_q, 0)) != 0;

  for (int i = 0; i < ntiles && alive; ++i) {
    uint8_t* st = sKV + (i & 1) * kTileBytes;
    const int k0 = k_begin + i * kTile;
    // keys of this tile that hold real data (inside the stripe, on an accepted page)
    uint32_t vmask;
    {
      const int k = k0 + lane;
      vmask = __ballot_sync(0xffffffffu, k < k_end && pool_row(k) >= 0);
    }
    if constexpr (kTma) {
      alive = __syncthreads_and(tc05::mbar_wait(mb_full0 + (i & 1) * 8, (i >> 1) & 1)) != 0;
      if (!alive) break;
    } else {
      cp_async_wait<0>();
    }
    if (vmask != 0xffffffffu) {  // zero the value rows of masked keys (never NaN into P V)
      for (int x = tid; x < kTile * kChunks; x += blockDim.x) {
        const int key = x / kChunks;
        if ((vmask >> key) & 1u) continue;
        const int cc = x - key * kChunks;
        *reinterpret_cast<uint4*>(st + (cc >> 3) * kBlkB + tc05::sw128(key, cc & 7)) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    tc05::fence_smem_to_async();
    __syncthreads();
    const uint32_t kv0 = tc05::smem_addr(st);

    // S = Q K^T as two independent accumulation chains (k-steps 0..17 into
    // columns 448..479, 18..35 into 480..511), summed after the read-back
    if (tid == 0) {
      tc05::fence_after_sync();
      const uint64_t dk = tc05::desc_k128(kv0);
#pragma unroll
      for (int s = 0; s < kDqk / 32; ++s) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int ks = h2 * (kDqk / 32) + s;
          const uint32_t off = (ks & 3) * 32;
          tc05::mma_ss(tbase + kTailCol + 32 * h2, tc05::desc_add(dq, (ks >> 2) * (kHeads * 128) + off),
                       tc05::desc_add(dk, (ks >> 2) * kBlkB + off), id_s, s > 0);
        }
      }
      tc05::commit(mb_s);
    }
    // the next tile's copies overlap this tile (its stage was freed by tile
    // i-1's P V wait)
    if (i + 1 < ntiles) load_tile(i + 1);
    alive = __syncthreads_and(tc05::mbar_wait(mb_s, i & 1)) != 0;  // every thread leaves together
    if (!alive) break;
    tc05::fence_after_sync();
    float sv[32];
    {
      float v16[16], w16[16];
      tc05::ld_x16(my_lane + kTailCol, v16);
      tc05::ld_x16(my_lane + kTailCol + 32, w16);
      tc05::ld_wait();
#pragma unroll
      for (int e = 0; e < 16; ++e) sv[e] = v16[e] + w16[e];
      tc05::ld_x16(my_lane + kTailCol + 16, v16);
      tc05::ld_x16(my_lane + kTailCol + 48, w16);
      tc05::ld_wait();
#pragma unroll
      for (int e = 0; e < 16; ++e) sv[16 + e] = v16[e] + w16[e];
    }
    float bm = -INFINITY;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      sv[e] = ((vmask >> e) & 1u) ? sv[e] * sl : -INFINITY;
      bm = fmaxf(bm, sv[e]);
    }
    const bool up = bm > m + 8.f;
    if (__any_sync(0xffffffffu, up) && i > 0) {
      // rescale O (TMEM columns 0..447) of the rows whose max rose; P V of the
      // previous tile has completed (waited below), so nothing else writes O now
      const float alpha = up ? exp2f(m - bm) : 1.f;
      for (int col = 0; col < kMainCols; col += 16) {
        float v[16];
        tc05::ld_x16(my_lane + col, v);
        tc05::ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] *= alpha;
        tc05::st_x16(my_lane + col, v);
      }
      tc05::st_wait();
#pragma unroll
      for (int e = 0; e < 64; ++e) tail[e] *= alpha;
      l *= alpha;
      lr *= alpha;
    }
    if (up) m = bm;
    // probabilities -> bf16 P rows (K-major, 64-byte swizzle)
    {
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float p0f = sv[2 * e] == -INFINITY ? 0.f : ex2_approx(sv[2 * e] - m);  // masked: 0
        const float p1f = sv[2 * e + 1] == -INFINITY ? 0.f : ex2_approx(sv[2 * e + 1] - m);
        l += p0f + p1f;
        __nv_bfloat162 pb = __floats2bfloat162_rn(p0f, p1f);
        lr += __low2float(pb) + __high2float(pb);
        pk[e] = *reinterpret_cast<uint32_t*>(&pb);
      }
#pragma unroll
      for (int cidx = 0; cidx < 4; ++cidx)
        *reinterpret_cast<uint4*>(sP + tc05::sw64(tid, cidx)) =
            make_uint4(pk[4 * cidx], pk[4 * cidx + 1], pk[4 * cidx + 2], pk[4 * cidx + 3]);
    }
    tc05::fence_smem_to_async();
    tc05::fence_before_sync();
    __syncthreads();

    // O[:, 0:448] += P V ; tail (columns 448..511) = P V[:, 448:512]
    if (tid == 0) {
      tc05::fence_after_sync();
      const uint64_t dv = tc05::desc_mn128(kv0, kBlkB);
#pragma unroll
      for (int s = 0; s < kTile / 16; ++s) {
        const uint64_t ad = tc05::desc_add(dp, s * 32);
        const uint32_t vrow = s * 16 * 128;
        tc05::mma_ss(tbase, ad, tc05::desc_add(dv, vrow), id_256, i > 0 || s > 0);
        tc05::mma_ss(tbase + 256, ad, tc05::desc_add(dv, vrow + 4 * kBlkB), id_192, i > 0 || s > 0);
        tc05::mma_ss(tbase + kTailCol, ad, tc05::desc_add(dv, vrow + 7 * kBlkB), id_64, s > 0);
      }
      tc05::commit(mb_pv);
    }
    alive = __syncthreads_and(tc05::mbar_wait(mb_pv, i & 1)) != 0;
    if (!alive) break;
    tc05::fence_after_sync();
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      float v[16];
      tc05::ld_x16(my_lane + kTailCol + 16 * q4, v);
      tc05::ld_wait();
#pragma unroll
      for (int e = 0; e < 16; ++e) tail[16 * q4 + e] += v[e];
    }
    tc05::fence_before_sync();
  }
  if constexpr (!kTma) cp_async_wait<0>();

  if (!alive) {
    if (tid == 0) report(a.dev_status, CPATTN_DEV_TC_TIMEOUT);
  } else {
    // ---- normalised partial of head `tid`: to o_part directly, or to the workspace
    const bool single = (nchunks == 1);
    const float inv = lr > 0.f ? 1.f / lr : 0.f;
    const float lse = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    float* dst = single ? a.o_part + orow * kDv : a.ws_o + ((slot * a.max_chunks + c) * kHeads + tid) * kDv;
    tc05::fence_after_sync();
    for (int col = 0; col < kMainCols; col += 16) {
      float v[16];
      tc05::ld_x16(my_lane + col, v);
      tc05::ld_wait();
      float4* d4 = reinterpret_cast<float4*>(dst + col);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        d4[e] = make_float4(v[4 * e] * inv, v[4 * e + 1] * inv, v[4 * e + 2] * inv, v[4 * e + 3] * inv);
    }
    {
      float4* d4 = reinterpret_cast<float4*>(dst + kMainCols);
#pragma unroll
      for (int e = 0; e < 16; ++e)
        d4[e] = make_float4(tail[4 * e] * inv, tail[4 * e + 1] * inv, tail[4 * e + 2] * inv, tail[4 * e + 3] * inv);
    }
    if (single) {
      a.lse_part[lse_slot(a, p, t, tid)] = lse;
    } else {
      a.ws_lse[(slot * a.max_chunks + c) * kHeads + tid] = lse;
    }
  }
  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc05::tmem_dealloc(tbase, 512);
  if (!alive) return;
  if (nchunks > 1) {
    if (!take_ticket(a.ws_cnt + slot, nchunks)) return;
    if (!mla_merge_chunks_bulk(a, p, t, slot, nchunks, sQ, bars + 5))
      merge_chunks<kMergeUnroll>(a, p, 0, t, 1, slot, 0, nchunks, kHeads, kDv, reinterpret_cast<float*>(sQ),
                                 kQBytes / 4);
    if (tid == 0) a.ws_cnt[slot] = 0;
  }
  if (a.fused) pair_finish<kMergeUnroll>(a, t, 0, kHeads, kDv, reinterpret_cast<float*>(sQ), kQBytes / 4);
}

int mla_tc_chunk(int ps_l) {
  // keys per CTA: a multiple of the 32-key tile whose pages fit the staged table
  int chunk = 2048;
  while (chunk > kTile && chunk / ps_l + 2 > kPageSlots) chunk -= kTile;
  return chunk;
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 2-D bf16 view [rows][576] with 1152-byte rows, 64-column boxes of `box_rows` rows, 128-byte swizzle.
bool encode_rows(CUtensorMap* map, const void* ptr, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || rows == 0) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDqk), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRowB)};
  const cuuint32_t box[2] = {64u, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_mla_partial(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  if (a.num_q_heads != kHeads || a.head_dim != kDqk || a.head_dim_v != kDv || a.num_kv_heads != 1 ||
      a.chunk % kTile != 0 || a.chunk / a.ps_l + 2 > kPageSlots)
    return CPATTN_ERR_UNSUPPORTED_SHAPE;
  // TMA when the page runs tile the 32-key tile evenly (every tile starts on a
  // run) and a run is at least 8 rows, so each box lands on a 1024-byte
  // boundary of the 128-byte swizzle pattern
  int box_rows = 0;
  if (a.ps_l >= 8 && a.ps_l <= kTile && kTile % a.ps_l == 0) box_rows = a.ps_l;
  else if (a.ps_l % kTile == 0) box_rows = kTile;
  CUtensorMap map_kv, map_q;
  std::memset(&map_kv, 0, sizeof(map_kv));
  std::memset(&map_q, 0, sizeof(map_q));
  bool tma = box_rows > 0 && a.chunk % box_rows == 0;
  if (tma) {
    tma = encode_rows(&map_kv, a.pool_k, static_cast<uint64_t>(a.P) * a.num_pages * a.ps_l, box_rows) &&
          encode_rows(&map_q, a.q, static_cast<uint64_t>(a.num_tokens) * kHeads, kHeads);
  }
  auto kern = tma ? mla_partial_tc_kernel<true> : mla_partial_tc_kernel<false>;
  static std::atomic<int> smem_set[2][64];
  *err = ensure_smem(kern, kSmemBytes, smem_set[tma ? 1 : 0]);
  if (*err != cudaSuccess) return CPATTN_ERR_CUDA;
  dim3 grid(a.max_chunks, a.P, a.num_tokens);
  kern<<<grid, 128, kSmemBytes, s>>>(a, map_kv, map_q, box_rows);
  *err = cudaGetLastError();
  return *err == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

}  // namespace cpattn
