// cp_paged_attn_partial, GQA rows of one token with groups of 1..8 query
// heads: the transposed tensor-core formulation.
//
// Same work split, partner addressing and split-KV merge as the kernel in
// partial_gqa_mma.cu (CTA = chunk of partner p's stripe of row b for KV head
// h; stripe slot k at page k / (page_size / P), slot k % (page_size / P) -- mstar
// PR #1124 "Context / Sequence Parallel 1/5", description).  A decode group
// has at most 8 query heads, so the heads go on the N side of mma.sync
// m16n8k16 and the 16 keys of a stage on the M side:
//   S^T = K Q^T   (A = K rows by ldmatrix, B = the query heads; D / 16 k-steps)
//   O^T += V^T P^T (A = V rows by ldmatrix.trans, one m-tile a 16 dims; B = P^T)
// which takes half the MMAs of the head-rows form (a group of 4 fills half an
// n-tile instead of a quarter of an m-tile) and half the accumulator
// registers.  P^T is built from the S^T accumulators
// (key rows, head columns) with movmatrix.trans, as a 16-bit hi + lo pair so
// P V keeps fp32-grade probabilities.  Softmax state (running max and sum) is
// per head: each lane holds heads 2 (lane % 4) and 2 (lane % 4) + 1 for keys
// lane / 4 and lane / 4 + 8, and reduces over keys with three xor shuffles.
//
// Loads: 16-byte cp.async copies, each warp instruction covering whole rows,
// into an XOR-swizzled ring (chunk c of key r at c ^ (r & 7); E4M3 rows of
// 64 bytes at c ^ ((r >> 1) & 3)).  E4M3 pools: the fragments are ldmatrix-ed as code
// bytes and converted in registers (float16 MMAs; the K fragment's k order is
// dims 4 (lane % 4) .. + 3, which the query fragment follows; V's code bytes
// split into even- and odd-dim rows of the m-tile).
#include "gqa_core.cuh"
#include "launch.h"
#include "mma_sync.cuh"
#include "split_combine.cuh"

namespace cpattn {

namespace {
constexpr int kTWarps = 4;
constexpr int kTKeys = 16;  // keys a stage
}  // namespace

// Shared memory of one CTA: the warps' cp.async rings.  bf16: 2 stages (64 KB
// at D 128, three CTAs an SM at <= 170 registers: 96 KB of K/V in flight an
// SM, and while one CTA starts or finishes -- page table and first copies;
// cross-warp merge, partial write, split-KV ticket -- two keep streaming;
// 3 stages at two CTAs an SM ran 3% slower on short rows); E4M3: 3 stages of
// half-size rows (48 KB, four CTAs an SM at <= 128 registers, 16 warps).
template <int D, bool F8>
struct TSmem {
  static constexpr int NST = F8 ? 3 : 2;
  static constexpr int SRC_ROWB = F8 ? D : 2 * D;
  static constexpr int RING_STAGE = kTKeys * SRC_ROWB;
  static constexpr size_t MAIN = static_cast<size_t>(kTWarps) * NST * RING_STAGE * 2;
};

template <int CHR>
__device__ __forceinline__ int swz_t(int c, int r) {
  if constexpr (CHR >= 8) return c ^ (r & 7);
  else return c ^ ((r >> 1) & (CHR - 1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

template <int D, int G, bool F8>
__global__ void __launch_bounds__(kTWarps * 32, F8 ? 4 : 3) gqa_partial_mmat_kernel(const PartialArgs a) {
  using SM = TSmem<D, F8>;
  constexpr int NW = kTWarps;
  constexpr int NST = SM::NST;
  constexpr int KT = kTKeys;
  constexpr int SRC_ROWB = SM::SRC_ROWB;
  constexpr int SRC_CH = SRC_ROWB / 16;  // 16-byte chunks of a pool row
  constexpr int ITERS = KT * SRC_CH / 32;  // copy instructions a stage (K and V each)
  constexpr int RING_STAGE = SM::RING_STAGE;
  constexpr int KSTEPS = D / 16;         // k-steps of S^T
  constexpr int MT = D / 16;             // m-tiles of O^T (16 dims each)
  static_assert(G >= 1 && G <= 8, "group size");
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint32_t s_vmask[NW][NST];  // bit k: key k of the stage was copied

  const int c = blockIdx.x;
  const int p = blockIdx.y / a.num_kv_heads;
  const int h = blockIdx.y - p * a.num_kv_heads;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int P = a.P;
  const int g8 = lane >> 2;  // key row (S^T) / dim row (O^T) / head column of B fragments
  const int qi = lane & 3;   // heads 2 qi, 2 qi + 1 of the accumulators

  pdl_trigger();
  pdl_wait();  // every input may come from the kernels before this one
  const int b = ordered_row(a.row_order, blockIdx.z, gridDim.z, a.dev_status);
  if (b < 0) return;
  int t = b;
  if (a.qo_indptr != nullptr) {
    t = __ldg(a.qo_indptr + b);
    if (__ldg(a.qo_indptr + b + 1) - t != 1) return;
  }
  int L = __ldg(a.kv_len + b);
  if (L > a.max_kv_len) {
    if (c == 0 && threadIdx.x == 0) report(a.dev_status, CPATTN_DEV_POS_PAST_TABLE);
    L = a.max_kv_len;
  }
  const int n_p = stripe_len(L, p, P, a.interleave);
  const int nchunks = n_p > 0 ? (n_p + a.chunk - 1) / a.chunk : 1;
  if (c >= nchunks) return;
  const int k_begin = c * a.chunk;
  const int k_end = min(n_p, k_begin + a.chunk);
  const int nstage = k_end > k_begin ? (k_end - k_begin + KT - 1) / KT : 0;
  const int my_n = nstage > warp ? (nstage - warp + NW - 1) / NW : 0;

  // ---- Q^T as the B operand: head g8, dims of k-step s (see the header comment)
  uint32_t qb[KSTEPS][2];
  {
    const bool ok = g8 < G;
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(
        static_cast<const uint8_t*>(a.q) + (static_cast<int64_t>(t) * a.num_q_heads + h * G + (ok ? g8 : 0)) * (2 * D));
#pragma unroll
    for (int s = 0; s < KSTEPS; ++s) {
      const int w0 = F8 ? s * 8 + 2 * qi : s * 8 + qi;
      const int w1 = F8 ? w0 + 1 : w0 + 4;
      qb[s][0] = ok ? __ldg(qw + w0) : 0u;
      qb[s][1] = ok ? __ldg(qw + w1) : 0u;
      if constexpr (F8) {
        qb[s][0] = bf16x2_to_f16x2(qb[s][0]);
        qb[s][1] = bf16x2_to_f16x2(qb[s][1]);
      }
    }
  }

  uint8_t* ring = smem + static_cast<size_t>(warp) * NST * RING_STAGE * 2;
  const uint8_t* poolk = static_cast<const uint8_t*>(a.pool_k);
  const uint8_t* poolv = static_cast<const uint8_t*>(a.pool_v);

  // page ids of the chunk, checked once and staged in shared memory
  int* spg = reinterpret_cast<int*>(smem + SM::MAIN);
  const int j0 = k_begin / a.ps_l;
  if (nstage > 0) {
    const int j1 = (k_end - 1) / a.ps_l;
    const int pb = __ldg(a.page_indptr + b);
    const int npages = __ldg(a.page_indptr + b + 1) - pb;
    for (int x = threadIdx.x; x <= j1 - j0; x += blockDim.x) {
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

  // stage i of this warp: each copy instruction covers whole rows (32 lanes
  // = 32 consecutive 16-byte chunks), the rows resolved once a stage by lanes
  // 0-15 (and 16-31) and shared by shuffle
  auto issue = [&](int i) {
    if (i < my_n) {
      const int k0 = k_begin + (warp + i * NW) * KT;
      const int64_t myrow = row_of(k0 + (lane & (KT - 1)));
      const uint32_t vm = __ballot_sync(0xffffffffu, myrow >= 0) & 0xffffu;  // bit k: key k copied
      if (lane == 0) s_vmask[warp][i % NST] = vm;
      uint8_t* sk = ring + (i % NST) * RING_STAGE * 2;
      uint8_t* sv = sk + RING_STAGE;
#pragma unroll
      for (int it = 0; it < ITERS; ++it) {
        const int idx = it * 32 + lane;
        const int key = idx / SRC_CH;
        const int ch = idx - key * SRC_CH;
        const int64_t row = __shfl_sync(0xffffffffu, myrow, key);
        const int soff = (key * SRC_CH + swz_t<SRC_CH>(ch, key)) * 16;
        if (row >= 0) {
          cp_async16(sk + soff, poolk + row * SRC_ROWB + ch * 16);
          cp_async16(sv + soff, poolv + row * SRC_ROWB + ch * 16);
        } else {
          *reinterpret_cast<uint4*>(sv + soff) = make_uint4(0u, 0u, 0u, 0u);  // masked keys: value 0, never NaN
        }
      }
    }
    cp_async_commit();
  };

  float o[MT][4];
#pragma unroll
  for (int u = 0; u < MT; ++u) o[u][0] = o[u][1] = o[u][2] = o[u][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2 qi, 2 qi + 1
  const float sl = a.scale * kLog2e * (F8 ? a.k_descale : 1.f);
  const int mrow = lane & 7;
  const int mi = lane >> 3;

#pragma unroll
  for (int i = 0; i < NST - 1; ++i) issue(i);

  for (int i = 0; i < my_n; ++i) {
    cp_async_wait<NST - 2>();
    __syncwarp();
    issue(i + NST - 1);  // refills the stage consumed in step i - 1

    const uint32_t sk = smem_u32(ring + (i % NST) * RING_STAGE * 2);
    const uint32_t sv = sk + RING_STAGE;
    const uint32_t vm = s_vmask[warp][i % NST];

    // ---- S^T = K Q^T: rows = the 16 keys, columns = heads; even / odd k-steps in two chains
    float st[4] = {0.f, 0.f, 0.f, 0.f}, st2[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int key = (mi & 1) * 8 + mrow;
      if constexpr (F8) {
#pragma unroll
        for (int s = 0; s < KSTEPS; s += 2) {
          const int ch = s + (mi >> 1);  // a chunk of codes is one k-step
          uint32_t r0, r1, r2, r3;
          ldsm_x4(sk + (key * SRC_CH + swz_t<SRC_CH>(ch, key)) * 16, r0, r1, r2, r3);
          const uint32_t fa[4] = {e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r0 >> 16),
                                  e4m3x2_to_f16x2(r1 >> 16)};
          const uint32_t fb[4] = {e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r2 >> 16),
                                  e4m3x2_to_f16x2(r3 >> 16)};
          mma_f16(st, fa, qb[s][0], qb[s][1]);
          mma_f16(st2, fb, qb[s + 1][0], qb[s + 1][1]);
        }
      } else {
#pragma unroll
        for (int s = 0; s < KSTEPS; ++s) {
          const int ch = 2 * s + (mi >> 1);
          uint32_t fa[4];
          ldsm_x4(sk + (key * SRC_CH + swz_t<SRC_CH>(ch, key)) * 16, fa[0], fa[1], fa[2], fa[3]);
          if (s & 1) mma_bf16(st2, fa, qb[s][0], qb[s][1]);
          else mma_bf16(st, fa, qb[s][0], qb[s][1]);
        }
      }
    }
    // ---- mask keys past the stripe end (or on a rejected page), per-head block max
    const bool ka = (vm >> g8) & 1u;        // key g8
    const bool kb = (vm >> (g8 + 8)) & 1u;  // key g8 + 8
    float v[4];
    v[0] = ka ? (st[0] + st2[0]) * sl : -INFINITY;  // key g8,     head 2 qi
    v[1] = ka ? (st[1] + st2[1]) * sl : -INFINITY;  // key g8,     head 2 qi + 1
    v[2] = kb ? (st[2] + st2[2]) * sl : -INFINITY;  // key g8 + 8, head 2 qi
    v[3] = kb ? (st[3] + st2[3]) * sl : -INFINITY;  // key g8 + 8, head 2 qi + 1
    float bm0 = fmaxf(v[0], v[2]), bm1 = fmaxf(v[1], v[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
      bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
    }
    const bool up0 = bm0 > m0 + 8.f;
    const bool up1 = bm1 > m1 + 8.f;
    if (__any_sync(0xffffffffu, up0 || up1)) {
      const float a0 = up0 ? exp2f(m0 - bm0) : 1.f;
      const float a1 = up1 ? exp2f(m1 - bm1) : 1.f;
      if (up0) m0 = bm0;
      if (up1) m1 = bm1;
      l0 *= a0;
      l1 *= a1;
#pragma unroll
      for (int u = 0; u < MT; ++u) {
        o[u][0] *= a0;
        o[u][1] *= a1;
        o[u][2] *= a0;
        o[u][3] *= a1;
      }
    }
    const float p0 = v[0] == -INFINITY ? 0.f : exp2f(v[0] - m0);
    const float p1 = v[1] == -INFINITY ? 0.f : exp2f(v[1] - m1);
    const float p2 = v[2] == -INFINITY ? 0.f : exp2f(v[2] - m0);
    const float p3 = v[3] == -INFINITY ? 0.f : exp2f(v[3] - m1);
    l0 += p0 + p2;
    l1 += p1 + p3;
    // ---- P^T as the B operand: the key-row / head-column pairs transposed by movmatrix
    uint32_t ph0, pl0, ph1, pl1;
    split16<F8>(p0, p1, ph0, pl0);  // keys 0-7
    split16<F8>(p2, p3, ph1, pl1);  // keys 8-15
    const uint32_t bh0 = movmatrix_t(ph0), bh1 = movmatrix_t(ph1);
    const uint32_t bl0 = movmatrix_t(pl0), bl1 = movmatrix_t(pl1);

    // ---- O^T += V^T P^T: one m-tile a 16 dims
    if constexpr (F8) {
      // code bytes by ldmatrix.trans: keys 0-7 / 8-15 x chunks ch, ch + 1; the
      // even bytes of a register are the even dims of the m-tile (rows 0-7),
      // the odd bytes its odd dims (rows 8-15)
      const int vkey = (mi & 1) * 8 + mrow;
#pragma unroll
      for (int ch0 = 0; ch0 < MT; ch0 += 2) {
        const int ch = ch0 + (mi >> 1);
        uint32_t r[4];
        ldsm_x4_t(sv + (vkey * SRC_CH + swz_t<SRC_CH>(ch, vkey)) * 16, r[0], r[1], r[2], r[3]);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t lo = r[2 * hh], hi = r[2 * hh + 1];  // keys 0-7, keys 8-15 of chunk ch0 + hh
          const uint32_t fa[4] = {e4m3x2_to_f16x2(__byte_perm(lo, 0u, 0x4420u)),
                                  e4m3x2_to_f16x2(__byte_perm(lo, 0u, 0x4431u)),
                                  e4m3x2_to_f16x2(__byte_perm(hi, 0u, 0x4420u)),
                                  e4m3x2_to_f16x2(__byte_perm(hi, 0u, 0x4431u))};
          mma_f16(o[ch0 + hh], fa, bh0, bh1);
          mma_f16(o[ch0 + hh], fa, bl0, bl1);
        }
      }
    } else {
      // ldmatrix.trans: keys 0-7 x dims lo 8, keys 0-7 x dims hi 8, keys 8-15 x lo, keys 8-15 x hi
      const int vkey = (mi >> 1) * 8 + mrow;
      uint32_t fa[MT][4];
#pragma unroll
      for (int u = 0; u < MT; ++u) {
        const int ch = 2 * u + (mi & 1);
        ldsm_x4_t(sv + (vkey * SRC_CH + swz_t<SRC_CH>(ch, vkey)) * 16, fa[u][0], fa[u][1], fa[u][2], fa[u][3]);
      }
#pragma unroll
      for (int u = 0; u < MT; ++u) mma_bf16(o[u], fa[u], bh0, bh1);
#pragma unroll
      for (int u = 0; u < MT; ++u) mma_bf16(o[u], fa[u], bl0, bl1);
    }
  }
  cp_async_wait<0>();

  if constexpr (F8) {  // value = code * v_descale
#pragma unroll
    for (int u = 0; u < MT; ++u) {
      o[u][0] *= a.v_descale;
      o[u][1] *= a.v_descale;
      o[u][2] *= a.v_descale;
      o[u][3] *= a.v_descale;
    }
  }
  // ---- per-warp state -> shared memory (heads < G), then the cross-warp merge
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  __syncthreads();
  float* sm = reinterpret_cast<float*>(smem);
  float* sm_o = sm;                 // [NW][G][D]
  float* sm_m = sm_o + NW * G * D;  // [NW][G]
  float* sm_l = sm_m + NW * G;      // [NW][G]
  const int h0 = 2 * qi, h1 = 2 * qi + 1;
  // dims of accumulator rows g8 and g8 + 8 of m-tile u
  auto dim_a = [&](int u) { return F8 ? 16 * u + 2 * g8 : 16 * u + g8; };
  auto dim_b = [&](int u) { return F8 ? 16 * u + 2 * g8 + 1 : 16 * u + g8 + 8; };
  if (h0 < G) {
#pragma unroll
    for (int u = 0; u < MT; ++u) {
      sm_o[(warp * G + h0) * D + dim_a(u)] = o[u][0];
      sm_o[(warp * G + h0) * D + dim_b(u)] = o[u][2];
    }
    if (g8 == 0) {
      sm_m[warp * G + h0] = m0;
      sm_l[warp * G + h0] = l0;
    }
  }
  if (h1 < G) {
#pragma unroll
    for (int u = 0; u < MT; ++u) {
      sm_o[(warp * G + h1) * D + dim_a(u)] = o[u][1];
      sm_o[(warp * G + h1) * D + dim_b(u)] = o[u][3];
    }
    if (g8 == 0) {
      sm_m[warp * G + h1] = m1;
      sm_l[warp * G + h1] = l1;
    }
  }
  __syncthreads();

  const int64_t orow0 = (static_cast<int64_t>(p) * a.num_tokens + t) * a.num_q_heads + h * G;
  const int64_t slot = (static_cast<int64_t>(t) * P + p) * a.num_kv_heads + h;
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
    merge_chunks(a, p, h, t, 1, slot, 0, nchunks, G, D, sm, static_cast<int>(SM::MAIN / 4));
    if (threadIdx.x == 0) a.ws_cnt[slot] = 0;  // ready for the next call
  }
  if (a.fused) pair_finish(a, t, h, G, D, sm, static_cast<int>(SM::MAIN / 4));
}

template <int D, int G, bool F8>
static int launch_mmat_t(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  using SM = TSmem<D, F8>;
  const size_t comb = (static_cast<size_t>(kTWarps) * G * D + 2 * kTWarps * G) * sizeof(float);
  const size_t pages = (static_cast<size_t>(a.chunk) / a.ps_l + 2) * sizeof(int);
  const size_t smem = (SM::MAIN > comb ? SM::MAIN : comb) + pages;
  auto kern = gqa_partial_mmat_kernel<D, G, F8>;
  static std::atomic<int> smem_set[64];
  *err = ensure_smem(kern, smem, smem_set);
  if (*err != cudaSuccess) return CPATTN_ERR_CUDA;
  dim3 grid(a.max_chunks, a.P * a.num_kv_heads, a.qo_indptr != nullptr ? a.num_rows : a.num_tokens);
  *err = launch_pdl(kern, grid, dim3(kTWarps * 32), smem, s, a);
  return *err == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

template <int D, bool F8>
static int mmat_dispatch_g(const PartialArgs& a, int G, cudaStream_t s, cudaError_t* err) {
  switch (G) {
    case 1: return launch_mmat_t<D, 1, F8>(a, s, err);
    case 2: return launch_mmat_t<D, 2, F8>(a, s, err);
    case 4: return launch_mmat_t<D, 4, F8>(a, s, err);
    case 8: return launch_mmat_t<D, 8, F8>(a, s, err);
    default: return CPATTN_ERR_UNSUPPORTED_SHAPE;
  }
}

// Rows of one token, group size <= 8: the transposed kernel.
int launch_gqa_partial_mmat(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  const int G = a.num_q_heads / a.num_kv_heads;
  if (a.kv_fp8) {
    if (a.head_dim == 128) return mmat_dispatch_g<128, true>(a, G, s, err);
    if (a.head_dim == 64) return mmat_dispatch_g<64, true>(a, G, s, err);
  } else {
    if (a.head_dim == 128) return mmat_dispatch_g<128, false>(a, G, s, err);
    if (a.head_dim == 64) return mmat_dispatch_g<64, false>(a, G, s, err);
  }
  return CPATTN_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace cpattn
