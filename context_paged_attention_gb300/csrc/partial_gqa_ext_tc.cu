// cp_paged_attn_partial, GQA rows with several query tokens on the tcgen05
// tensor cores, E4M3 pools (bf16 pools take the warp-specialised kernel of
// partial_gqa_ext_ws.cu).
//
// A non-decode step attends the pool for its context only, and every new
// token of a row sees the same context (mstar PR #1124 "Context / Sequence
// Parallel 1/5", description: context-only plans; vLLM "[Core] Add explicit
// layer parallel plans", _forward_with_dcp: the context partial over the paged
// cache).  The queries of 128 / G consecutive tokens of a row and the G heads
// of KV head h form a dense 128-row tile against partner p's stripe of that
// context (stripe slot k = logical position k * P + p, at physical slot
// k % (page_size / P) of page k / (page_size / P)):
//   S = Q K^T  (M = 128 query rows, N = 32 keys, K = head_dim)
//   O += P V   (N = head_dim, K = 32 keys)
//
// CTA = (chunk, partner p, KV head h, token block j), 4 warps; thread r owns
// query row r = (token j * 128 / G + r / G, head h * G + r % G) and TMEM lane r,
// so the online softmax is thread-local.  Shared memory: Q [128 x D] K-major
// with the 128-byte swizzle; a ring of four stages of E4M3 code rows of 32
// keys (K then V, [key][D] bytes; tile i + 2 is requested as soon as tile i
// has landed); each landed tile is converted exactly (every E4M3 value is a
// bf16 value) into one of two bf16 tiles in the MMA layout (the same bytes
// serve K-major for S and M/N-major for P V); the scores take k_descale and
// the output v_descale.  P [128 x 32] bf16 K-major with the 64-byte swizzle;
// O is normalised by the sum of the bf16-rounded probabilities (an exact
// convex combination of the values; the LSE keeps the fp32 sum).
// Tensor memory: 32 columns of S and D columns of O (256 allocated, two CTAs
// per SM).  The S MMAs of a tile overlap the P V MMAs of the one before.  A
// chunk split of a stripe is merged by the last CTA to arrive, per token.
// Rows of one token are left to the decode kernel; this kernel also writes the
// padding tokens past the last row.  Waits are bounded (CPATTN_DEV_TC_TIMEOUT).
#include "common.cuh"
#include "launch.h"
#include "mma_sync.cuh"
#include "split_combine.cuh"
#include "tc05.cuh"

namespace cpattn {

namespace {
constexpr int kXTile = 32;    // keys per tile
constexpr int kXStages = 4;
constexpr int kXRows = 128;   // query rows per CTA
}  // namespace

template <int D>
struct ExtTcLayout {
  static constexpr int KB = D / 64;                   // 64-column blocks of a row
  static constexpr int QBYTES = KB * kXRows * 128;    // Q tile
  static constexpr int BLK = kXTile * 128;            // one column block of a key tile
  static constexpr int TILE = KB * BLK;               // K (or V) tile
  static constexpr int STAGE = 2 * TILE;              // K + V
  static constexpr int PBYTES = kXRows * 64;          // one P tile (bf16, 32 keys)
  static constexpr int TMEM_COLS = 256;
  static constexpr int S_COL = 0;                     // S: columns 0..31
  static constexpr int O_COL = 64;                    // O: columns 64..64+D
  // the code rows of a tile land in a ring of kXStages stages (K then V,
  // [key][D] bytes) and are converted into one of two bf16 tiles
  static constexpr int RING8 = 2 * kXTile * D;        // one E4M3 stage (K + V)
  static size_t smem_bytes(int page_slots) {
    const size_t tiles = 2 * static_cast<size_t>(STAGE) + kXStages * static_cast<size_t>(RING8);
    return 1024 + QBYTES + tiles + PBYTES + 64 + static_cast<size_t>(page_slots) * 4;
  }
};

template <int D, int G>
__global__ void __launch_bounds__(128, 2) gqa_partial_ext_tc_kernel(const PartialArgs a) {
  using Lt = ExtTcLayout<D>;
  constexpr int QB = kXRows / G;  // tokens per block
  static_assert(G >= 1 && G <= 16 && (D == 64 || D == 128), "shape");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sKV = sQ + Lt::QBYTES;  // bf16 tiles the MMAs read: kXStages stages, or (E4M3) two
  uint8_t* sRing8 = sKV + 2 * Lt::STAGE;  // E4M3 code stages
  uint8_t* sPh = sRing8 + kXStages * Lt::RING8;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sPh + Lt::PBYTES);  // [0] S done, [1] P V done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
  int* spg = reinterpret_cast<int*>(bars + 4);

  const int c = blockIdx.x;
  const int p = blockIdx.y / a.num_kv_heads;
  const int h = blockIdx.y - p * a.num_kv_heads;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int P = a.P;

  const int t_lo = blockIdx.z * QB;
  const int t_real = __ldg(a.qo_indptr + a.num_rows);
  const int t_hi = min(t_lo + QB, t_real);
  if (c == 0 && a.fused) {
    // padding tokens past the last row: final output 0 / -inf (written once, by partner 0)
    if (p == 0)
      for (int tok = max(t_lo, t_real); tok < min(t_lo + QB, a.num_tokens); ++tok) fused_zero_token(a, tok, h, G, D);
  } else if (c == 0) {
    // padding tokens past the last row: this (partner, KV head)'s 0 / -inf
    for (int tok = max(t_lo, t_real); tok < min(t_lo + QB, a.num_tokens); ++tok) {
      const int64_t orow0 = (static_cast<int64_t>(p) * a.num_tokens + tok) * a.num_q_heads + h * G;
      for (int x = tid; x < G * D; x += blockDim.x) a.o_part[orow0 * D + x] = 0.f;
      if (tid < G) a.lse_part[lse_slot(a, p, tok, h * G + tid)] = -INFINITY;
    }
  }
  if (t_lo >= t_hi) return;
  // is there any row of >= 2 tokens in this block with keys in chunk c?  (uniform)
  {
    bool any = false;
    for (int b = find_row(a.qo_indptr, a.num_rows, t_lo); b < a.num_rows; ++b) {
      const int r0 = __ldg(a.qo_indptr + b);
      if (r0 >= t_hi) break;
      if (__ldg(a.qo_indptr + b + 1) - r0 >= 2) {
        any = true;
        break;
      }
    }
    if (!any) return;
  }

  if (tid == 0) {
    tc05::mbar_init(tc05::smem_addr(&bars[0]), 1);
    tc05::mbar_init(tc05::smem_addr(&bars[1]), 1);
    tc05::mbar_init_fence();
  }
  if (warp == 0) tc05::tmem_alloc(tc05::smem_addr(tmem_slot), Lt::TMEM_COLS);
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  const uint32_t tbase = *tmem_slot;
  const uint32_t mb_s = tc05::smem_addr(&bars[0]);
  const uint32_t mb_pv = tc05::smem_addr(&bars[1]);
  const uint32_t my_lane = tc05::taddr(tbase, warp * 32, 0);
  const uint64_t dq = tc05::desc_k128(tc05::smem_addr(sQ));
  const uint64_t dph = tc05::desc_k64(tc05::smem_addr(sPh));
  const uint32_t id_s = tc05::idesc_bf16(128, kXTile, false, false);
  const uint32_t id_o = tc05::idesc_bf16(128, D, false, true);
  const uint8_t* poolk = static_cast<const uint8_t*>(a.pool_k);
  const uint8_t* poolv = static_cast<const uint8_t*>(a.pool_v);
  const float sl = a.scale * kLog2e * a.k_descale;
  uint32_t s_phase = 0, pv_phase = 0;  // completed phases of the two mbarriers
  bool alive = true;

  for (int b = find_row(a.qo_indptr, a.num_rows, t_lo); b < a.num_rows && alive; ++b) {
    const int r0 = __ldg(a.qo_indptr + b);
    if (r0 >= t_hi) break;
    const int r1 = __ldg(a.qo_indptr + b + 1);
    if (r1 - r0 < 2) continue;  // one-token rows: the decode kernel's
    const int s0 = max(r0, t_lo), s1 = min(r1, t_hi);
    if (s1 <= s0) continue;
    int L = __ldg(a.kv_len + b);
    if (L > a.max_kv_len) {
      if (c == 0 && tid == 0) report(a.dev_status, CPATTN_DEV_POS_PAST_TABLE);
      L = a.max_kv_len;
    }
    const int n_p = stripe_len(L, p, P, a.interleave);
    const int nchunks = n_p > 0 ? (n_p + a.chunk - 1) / a.chunk : 1;
    if (c >= nchunks) continue;
    const int k_begin = c * a.chunk;
    const int k_end = min(n_p, k_begin + a.chunk);
    const int ntiles = k_end > k_begin ? (k_end - k_begin + kXTile - 1) / kXTile : 0;

    // ---- Q rows of the segment (rows past the segment: zero), page ids of the chunk
    const int my_tok = s0 + tid / G;
    const bool my_ok = my_tok < s1;
    {
      const uint8_t* qrow = static_cast<const uint8_t*>(a.q) +
                            (static_cast<int64_t>(my_ok ? my_tok : s0) * a.num_q_heads + h * G + tid % G) * (D * 2);
#pragma unroll
      for (int cc = 0; cc < D / 8; ++cc) {
        uint8_t* dst = sQ + (cc >> 3) * (kXRows * 128) + tc05::sw128(tid, cc & 7);
        if (my_ok) cp_async16(dst, qrow + cc * 16);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    const int j0 = k_begin / a.ps_l;
    if (ntiles > 0) {
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
    __syncthreads();
    const int64_t head_row0 = static_cast<int64_t>(p) * a.num_pages * a.num_kv_heads + h;
    auto row_of = [&](int k) -> int64_t {
      if (k >= k_end) return -1;
      const int j = page_of_slot(a, k);
      const int pg = spg[j - j0];
      if (pg < 0) return -1;
      return (head_row0 + static_cast<int64_t>(pg) * a.num_kv_heads) * a.ps_l + (k - j * a.ps_l);
    };
    // copies of tile i (K and V rows) into stage i % kXStages; each warp
    // resolves the 32 keys' rows once (lane = key) and shares them by shuffle
    auto load_tile = [&](int i) {
      if (i < ntiles) {
        const int64_t myrow = row_of(k_begin + i * kXTile + lane);
        // code rows, [key][D] bytes per K / V
        uint8_t* rk = sRing8 + (i % kXStages) * Lt::RING8;
        uint8_t* rv = rk + kXTile * D;
        constexpr int CH8 = D / 16;
        for (int x = tid; x < kXTile * CH8; x += blockDim.x) {
          const int key = x / CH8;
          const int cc = x - key * CH8;
          const int64_t row = __shfl_sync(0xffffffffu, myrow, key);
          if (row >= 0) {
            cp_async16(rk + x * 16, poolk + row * D + cc * 16);
            cp_async16(rv + x * 16, poolv + row * D + cc * 16);
          } else {
            *reinterpret_cast<uint4*>(rv + x * 16) = make_uint4(0u, 0u, 0u, 0u);  // masked keys: value 0
          }
        }
      }
      cp_async_commit();
    };
    // E4M3: the codes of tile i -> bf16 tile i % 2 in the MMA layout (exact:
    // every E4M3 value is a bf16 value); the tile it overwrites (i - 2) was
    // last read by P V of tile i - 2, which has completed
    auto convert_tile = [&](int i) {
      const uint8_t* rk = sRing8 + (i % kXStages) * Lt::RING8;
      uint8_t* wk = sKV + (i & 1) * Lt::STAGE;
      constexpr int CH8 = D / 16;
      for (int x = tid; x < 2 * kXTile * CH8; x += blockDim.x) {
        const int kv = x / (kXTile * CH8);  // 0: K, 1: V
        const int y = x - kv * (kXTile * CH8);
        const int key = y / CH8;
        const int c16 = y - key * CH8;  // codes of dims 16 c16 .. 16 c16 + 15
        const uint4 w = *reinterpret_cast<const uint4*>(rk + kv * kXTile * D + y * 16);
        const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
        uint32_t bf[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          bf[2 * q] = e4m3x2_to_bf16x2(wd[q]);
          bf[2 * q + 1] = e4m3x2_to_bf16x2(wd[q] >> 16);
        }
        uint8_t* dst = wk + kv * Lt::TILE;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int cc = 2 * c16 + hh;  // 8-dim chunk of the bf16 row
          *reinterpret_cast<uint4*>(dst + (cc >> 3) * Lt::BLK + tc05::sw128(key, cc & 7)) =
              make_uint4(bf[4 * hh], bf[4 * hh + 1], bf[4 * hh + 2], bf[4 * hh + 3]);
        }
      }
    };
    load_tile(0);
    load_tile(1);

    float m = -INFINITY, l = 0.f, lr = 0.f;  // running max (log2), fp32 sum, sum of the bf16-rounded p
    bool have_pv = false;  // a P V MMA of this segment is in flight (or done but unwaited)
    for (int i = 0; i < ntiles; ++i) {
      cp_async_wait<1>();  // tile i (and Q) landed for this thread
      __syncthreads();  // every thread's codes of tile i landed
      convert_tile(i);
      tc05::fence_smem_to_async();
      __syncthreads();
      const uint32_t kv0 = tc05::smem_addr(sKV + (i & 1) * Lt::STAGE);
      load_tile(i + 2);  // into the stage of tile i - 2, whose P V completed before this tile
      uint32_t vmask;
      {
        const int k = k_begin + i * kXTile + lane;
        vmask = __ballot_sync(0xffffffffu, row_of(k) >= 0);
      }
      if (tid == 0) {
        tc05::fence_after_sync();
        const uint64_t dk = tc05::desc_k128(kv0);
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t off = (s >> 2) * (kXRows * 128) + (s & 3) * 32;
          const uint32_t koff = (s >> 2) * Lt::BLK + (s & 3) * 32;
          tc05::mma_ss(tbase + Lt::S_COL, tc05::desc_add(dq, off), tc05::desc_add(dk, koff), id_s, s > 0);
        }
        tc05::commit(mb_s);  // also covers the previous tile's P V
      }
      if (have_pv) {  // P V of tile i-1 done: its stage and P are free, O is stable
        alive = __syncthreads_and(tc05::mbar_wait(mb_pv, pv_phase & 1)) != 0;
        ++pv_phase;
        have_pv = false;
        if (!alive) break;
      }
      alive = __syncthreads_and(tc05::mbar_wait(mb_s, s_phase & 1)) != 0;
      ++s_phase;
      if (!alive) break;
      tc05::fence_after_sync();
      float sv[32];
      {
        float v16[16];
        tc05::ld_x16(my_lane + Lt::S_COL, v16);
        tc05::ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) sv[e] = v16[e];
        tc05::ld_x16(my_lane + Lt::S_COL + 16, v16);
        tc05::ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) sv[16 + e] = v16[e];
      }
      float bm = -INFINITY;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        sv[e] = ((vmask >> e) & 1u) ? sv[e] * sl : -INFINITY;
        bm = fmaxf(bm, sv[e]);
      }
      const bool up = bm > m + 8.f;
      if (__any_sync(0xffffffffu, up) && i > 0) {  // rescale O rows whose max rose (rare)
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
      {
        uint32_t hi[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float pa = sv[2 * e] == -INFINITY ? 0.f : ex2_approx(sv[2 * e] - m);  // masked: 0, also while m is -inf
          const float pb = sv[2 * e + 1] == -INFINITY ? 0.f : ex2_approx(sv[2 * e + 1] - m);
          l += pa + pb;
          __nv_bfloat162 h2 = __floats2bfloat162_rn(pa, pb);
          lr += __low2float(h2) + __high2float(h2);
          hi[e] = *reinterpret_cast<uint32_t*>(&h2);
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          *reinterpret_cast<uint4*>(sPh + tc05::sw64(tid, q4)) =
              make_uint4(hi[4 * q4], hi[4 * q4 + 1], hi[4 * q4 + 2], hi[4 * q4 + 3]);
      }
      tc05::fence_smem_to_async();
      tc05::fence_before_sync();
      __syncthreads();
      if (tid == 0) {
        tc05::fence_after_sync();
        const uint64_t dv = tc05::desc_mn128(kv0 + Lt::TILE, Lt::BLK);
#pragma unroll
        for (int s = 0; s < kXTile / 16; ++s)
          tc05::mma_ss(tbase + Lt::O_COL, tc05::desc_add(dph, s * 32), tc05::desc_add(dv, s * 16 * 128), id_o,
                       i > 0 || s > 0);
        tc05::commit(mb_pv);
      }
      have_pv = true;
    }
    if (have_pv && alive) {
      alive = __syncthreads_and(tc05::mbar_wait(mb_pv, pv_phase & 1)) != 0;
      ++pv_phase;
    }
    cp_async_wait<0>();
    __syncthreads();
    if (!alive) break;

    // ---- row `tid`: normalised output and LSE, to o_part or the workspace.
    // Every lane runs the (warp-collective) TMEM loads; only valid rows store.
    const bool single = (nchunks == 1);
    {
      const bool empty = (l == 0.f);
      const float inv = lr > 0.f ? a.v_descale / lr : 0.f;  // E4M3: value = code * v_descale
      const float lse = empty ? -INFINITY : (m + log2f(l)) * kLn2;
      const int g = tid % G;
      float* dst = nullptr;
      float* ldst = nullptr;
      if (single) {
        const int64_t orow = (static_cast<int64_t>(p) * a.num_tokens + my_tok) * a.num_q_heads + h * G + g;
        dst = a.o_part + orow * D;
        ldst = a.lse_part + lse_slot(a, p, my_tok, h * G + g);
      } else {
        const int64_t slot = (static_cast<int64_t>(my_tok) * P + p) * a.num_kv_heads + h;
        const int64_t wrow = (slot * a.max_chunks + c) * G + g;
        dst = a.ws_o + wrow * D;
        ldst = a.ws_lse + wrow;
      }
      tc05::fence_after_sync();
#pragma unroll
      for (int col = 0; col < D; col += 16) {
        float v[16];
        if (ntiles > 0) {  // uniform across the CTA
          tc05::ld_x16(my_lane + Lt::O_COL + col, v);
          tc05::ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0.f;
        }
        if (my_ok) {
          float4* d4 = reinterpret_cast<float4*>(dst + col);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            d4[e] = make_float4(v[4 * e] * inv, v[4 * e + 1] * inv, v[4 * e + 2] * inv, v[4 * e + 3] * inv);
        }
      }
      if (my_ok) *ldst = lse;
    }
    tc05::fence_before_sync();
    bool done = true;  // this CTA holds the partner's complete partial of the segment
    if (!single) {
      const int64_t slot0 = (static_cast<int64_t>(s0) * P + p) * a.num_kv_heads + h;
      done = take_ticket(a.ws_cnt + slot0, nchunks);
      if (done) {
        merge_chunks<4>(a, p, h, s0, s1 - s0, slot0, static_cast<int64_t>(P) * a.num_kv_heads, nchunks, G, D,
                     reinterpret_cast<float*>(sKV), 2 * Lt::STAGE / 4);
        if (tid == 0) a.ws_cnt[slot0] = 0;
      }
    }
    if (a.fused && done) {
      // fused: the last of the P partners of (segment, KV head) merges them
      int32_t* pair = a.ws_pair + static_cast<int64_t>(s0) * a.num_kv_heads + h;
      if (take_ticket(pair, P)) {
        merge_partners<4>(a, s0, s1 - s0, h, G, D, reinterpret_cast<float*>(sKV), 2 * Lt::STAGE / 4);
        if (tid == 0) *pair = 0;
      }
    }
    __syncthreads();  // Q, the ring and the page table are reused by the next row
  }
  if (!alive && tid == 0) report(a.dev_status, CPATTN_DEV_TC_TIMEOUT);
  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc05::tmem_dealloc(tbase, Lt::TMEM_COLS);
}

template <int D, int G>
static int launch_ext_tc_t(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  constexpr int QB = kXRows / G;
  const int page_slots = a.chunk / a.ps_l + 2;
  const size_t smem = ExtTcLayout<D>::smem_bytes(page_slots);
  if (smem > 227 * 1024) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  auto kern = gqa_partial_ext_tc_kernel<D, G>;
  static std::atomic<int> smem_set[64];
  *err = ensure_smem(kern, smem, smem_set);
  if (*err != cudaSuccess) return CPATTN_ERR_CUDA;
  dim3 grid(a.max_chunks, a.P * a.num_kv_heads, (a.num_tokens + QB - 1) / QB);
  kern<<<grid, 128, smem, s>>>(a);
  *err = cudaGetLastError();
  return *err == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

template <int D>
static int ext_tc_dispatch_g(const PartialArgs& a, int G, cudaStream_t s, cudaError_t* err) {
  switch (G) {
    case 1: return launch_ext_tc_t<D, 1>(a, s, err);
    case 2: return launch_ext_tc_t<D, 2>(a, s, err);
    case 4: return launch_ext_tc_t<D, 4>(a, s, err);
    case 8: return launch_ext_tc_t<D, 8>(a, s, err);
    case 16: return launch_ext_tc_t<D, 16>(a, s, err);
    default: return CPATTN_ERR_UNSUPPORTED_SHAPE;
  }
}

int launch_gqa_partial_ext(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  // bf16 pools: the warp-specialised kernel (partial_gqa_ext_ws.cu); E4M3
  // pools: this kernel, which converts each tile of codes before its MMAs
  if (!a.kv_fp8) return launch_gqa_partial_ext_ws(a, s, err);
  const int G = a.num_q_heads / a.num_kv_heads;
  if (a.head_dim == 128) return ext_tc_dispatch_g<128>(a, G, s, err);
  if (a.head_dim == 64) return ext_tc_dispatch_g<64>(a, G, s, err);
  return CPATTN_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace cpattn
