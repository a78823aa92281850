// cp_paged_attn_partial, GQA path on tensor cores (bf16 pools), rows of one
// query token (rows of several tokens: partial_gqa_ext.cu).
//
// Same work split and partner addressing as the CUDA-core path (see
// partial_gqa.cu): CTA = (chunk, partner p, KV head h, query token t); partner
// p's stripe slot k is logical position k * P + p at physical slot
// k % (page_size / P) of the row's page k / (page_size / P) (mstar PR #1124
// "Context / Sequence Parallel 1/5", description: logical slot s on partner
// s % P at physical slot s / P, page ids logical).
//
// The chunk's page ids are checked once and staged in shared memory.  Per
// warp: stages of 16 keys (gathered from as many page runs as needed) are
// copied with 16-byte cp.async into an XOR-swizzled ring (chunk c of row r at
// c ^ (r & 7), so ldmatrix rows never share banks).  The G query heads of the
// KV head form the rows of a 16-row A tile (rows >= G are zero), so
//   S = Q K^T  : 2 n-tiles (8 keys) x D/16 k-steps of mma.m16n8k16 (bf16 -> f32)
//   O += P V   : D/8 n-tiles x 1 k-step (16 keys), P re-packed from the S
//                accumulators in registers (their layout is the A layout) as
//                a bf16 hi + lo pair, so P V keeps fp32-grade accuracy.
// The tile is only G/16 full: decode reads each key once, so the contraction
// is tiny and the kernel stays bound by HBM; the tensor cores only take the
// multiply-adds off the issue slots (tcgen05 needs M >= 64 rows, a decode group
// has 1..16).  Online softmax in the log2 domain with a lazily raised running
// max (raised only when a block exceeds it by more than 8, which keeps every
// probability <= 2^8 and the result exact).
#include "gqa_core.cuh"
#include "launch.h"
#include "mma_sync.cuh"
#include "split_combine.cuh"

namespace cpattn {

constexpr int kMmaWarps = 4;
constexpr int kMmaStages = 3;
constexpr int kMmaStagesF8 = 5;  // E4M3 pools: half the bytes a stage, deeper ring
constexpr int kMmaKeys = 16;  // keys per stage

// Shared memory of one CTA: the warps' cp.async rings of pool rows.
template <int D, bool F8>
struct MmaSmem {
  static constexpr int NST = F8 ? kMmaStagesF8 : kMmaStages;
  static constexpr int SRC_ROWB = F8 ? D : 2 * D;                    // bytes of a pool row
  static constexpr int RING_STAGE = kMmaKeys * SRC_ROWB;             // K (or V) bytes per ring stage
  static constexpr size_t MAIN = static_cast<size_t>(kMmaWarps) * NST * RING_STAGE * 2;
};

// 16-byte chunk c of row r of a stage sits at chunk position swz(c, r), so
// the 8 rows an ldmatrix phase reads hit distinct banks: bf16 rows (2 D
// bytes) and E4M3 rows of 128 bytes XOR with r & 7; E4M3 rows of 64 bytes
// (4 chunks) XOR with (r >> 1) & 3.
template <int CHR>
__device__ __forceinline__ int swz(int c, int r) {
  if constexpr (CHR >= 8) return c ^ (r & 7);
  else return c ^ ((r >> 1) & (CHR - 1));
}

template <int D, int G, bool F8>
__global__ void __launch_bounds__(kMmaWarps * 32, 2) gqa_partial_mma_kernel(const PartialArgs a) {
  using SM = MmaSmem<D, F8>;
  constexpr int NW = kMmaWarps;
  constexpr int NST = SM::NST;
  constexpr int KT = kMmaKeys;
  constexpr int ROWB = D * 2;            // bytes of a bf16 row (query rows)
  constexpr int SRC_ROWB = SM::SRC_ROWB;
  constexpr int SRC_CH = SRC_ROWB / 16;  // 16-byte chunks per pool row
  constexpr int RING_STAGE = SM::RING_STAGE;
  constexpr int KSTEPS = D / 16;
  constexpr int NT = D / 8;              // n-tiles of the output
  constexpr int ITERS = KT * SRC_CH / 32;  // cp.async rounds per stage
  static_assert(G >= 1 && G <= 16, "group size");
  static_assert(NT % 4 == 0, "head dim");
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint32_t s_vmask[NW][NST];  // which of a stage's 16 keys were copied

  const int c = blockIdx.x;
  const int p = blockIdx.y / a.num_kv_heads;
  const int h = blockIdx.y - p * a.num_kv_heads;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int P = a.P;
  const int quad = lane >> 2;  // row of the accumulator fragments
  const int qi = lane & 3;

  // one CTA column per row: with a token -> row map only rows of exactly one
  // token are handled here (rows of two or more tokens: partial_gqa_ext.cu,
  // which also writes the padding tokens past the last row); without a map
  // row b is token b
  const int b = ordered_row(a.row_order, blockIdx.z, gridDim.z, a.dev_status);
  if (b < 0) return;
  int t = b;
  if (a.qo_indptr != nullptr) {
    t = __ldg(a.qo_indptr + b);
    if (__ldg(a.qo_indptr + b + 1) - t != 1) return;
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
  const int nstage = k_end > k_begin ? (k_end - k_begin + KT - 1) / KT : 0;
  const int my_n = nstage > warp ? (nstage - warp + NW - 1) / NW : 0;

  // ---- Q fragments (A operand), rows = the G heads of this KV head
  uint32_t qa[KSTEPS][4];
  {
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(a.q) +
                                                           (static_cast<int64_t>(t) * a.num_q_heads + h * G) * ROWB);
    const bool r0ok = b >= 0 && quad < G;
    const bool r1ok = b >= 0 && quad + 8 < G;
#pragma unroll
    for (int s = 0; s < KSTEPS; ++s) {
      // bf16: MMA k index = dim (words of dims 16s + 2qi, +1 and +8, +9).
      // E4M3: the K fragment comes from an ldmatrix of code bytes, whose k
      // order is dims 16s + 4qi, +1 (k 2qi, 2qi+1) and +2, +3 (k 2qi+8, +9);
      // the query takes the same order (float16 operands).
      const int w0 = F8 ? s * 8 + 2 * qi : s * 8 + qi;
      const int w1 = F8 ? w0 + 1 : w0 + 4;
      qa[s][0] = r0ok ? __ldg(qw + quad * (D / 2) + w0) : 0u;
      qa[s][1] = r1ok ? __ldg(qw + (quad + 8) * (D / 2) + w0) : 0u;
      qa[s][2] = r0ok ? __ldg(qw + quad * (D / 2) + w1) : 0u;
      qa[s][3] = r1ok ? __ldg(qw + (quad + 8) * (D / 2) + w1) : 0u;
      if constexpr (F8) {
#pragma unroll
        for (int r = 0; r < 4; ++r) qa[s][r] = bf16x2_to_f16x2(qa[s][r]);
      }
    }
  }

  uint8_t* ring = smem + static_cast<size_t>(warp) * NST * RING_STAGE * 2;
  const uint8_t* poolk = static_cast<const uint8_t*>(a.pool_k);
  const uint8_t* poolv = static_cast<const uint8_t*>(a.pool_v);

  // The chunk's page ids, checked once and staged in shared memory (-1 = not
  // covered by the row's table or outside the pool), so issuing a stage never
  // waits on a dependent global load.
  int* spg = reinterpret_cast<int*>(smem + SM::MAIN);
  const int j0 = k_begin / a.ps_l;
  if (nstage > 0) {
    const int j1 = (k_end - 1) / a.ps_l;
    int pb = 0, npages = 0;
    if (b >= 0) {
      pb = __ldg(a.page_indptr + b);
      npages = __ldg(a.page_indptr + b + 1) - pb;
    }
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

  // pool row of stripe slot k, or -1 if past the stripe or on a rejected page
  auto row_of = [&](int k) -> int64_t {
    if (k >= k_end) return -1;
    const int j = page_of_slot(a, k);
    const int pg = spg[j - j0];
    if (pg < 0) return -1;
    return (head_row0 + static_cast<int64_t>(pg) * a.num_kv_heads) * a.ps_l + (k - j * a.ps_l);
  };

  auto issue = [&](int i) {
    if (i < my_n) {
      const int k0 = k_begin + (warp + i * NW) * KT;
      const int64_t myrow = row_of(k0 + (lane & (KT - 1)));  // lanes 0..15 and 16..31 both cover the 16 keys
      const uint32_t vm = __ballot_sync(0xffffffffu, myrow >= 0) & 0xffffu;
      if (lane == 0) s_vmask[warp][i % NST] = vm;
      uint8_t* sk = ring + (i % NST) * RING_STAGE * 2;
      uint8_t* sv = sk + RING_STAGE;
#pragma unroll
      for (int it = 0; it < ITERS; ++it) {
        const int idx = it * 32 + lane;
        const int key = idx / SRC_CH;
        const int ch = idx - key * SRC_CH;
        const int64_t row = __shfl_sync(0xffffffffu, myrow, key);
        const int soff = (key * SRC_CH + swz<SRC_CH>(ch, key)) * 16;
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

  float o[NT][4];
#pragma unroll
  for (int u = 0; u < NT; ++u) o[u][0] = o[u][1] = o[u][2] = o[u][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float sl = a.scale * kLog2e * (F8 ? a.k_descale : 1.f);
  const int mrow = lane & 7;
  const int mi = lane >> 3;  // which of the 4 matrices of an ldmatrix.x4 this lane addresses

#pragma unroll
  for (int i = 0; i < NST - 1; ++i) issue(i);

  for (int i = 0; i < my_n; ++i) {
    cp_async_wait<NST - 2>();
    __syncwarp();
    issue(i + NST - 1);  // refills the stage consumed in step i - 1

    const uint32_t sk = smem_u32(ring + (i % NST) * RING_STAGE * 2);
    const uint32_t sv = sk + RING_STAGE;
    const uint32_t vm = s_vmask[warp][i % NST];

    // S = Q K^T for the 16 keys (two n-tiles), even / odd k-steps in two MMA chains
    float s[2][4], s_alt[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[j][e] = s_alt[j][e] = 0.f;
    if constexpr (F8) {
      // one ldmatrix.x4 of code bytes: keys 0-7 / 8-15 x chunks s2, s2 + 1
      // (a 16-byte chunk of E4M3 codes is one 16-dim k-step); each register's
      // 4 codes become the b0 / b1 float16 pairs of that k-step
      const int key = (mi & 1) * 8 + mrow;
#pragma unroll
      for (int s2 = 0; s2 < KSTEPS; s2 += 2) {
        const int ch = s2 + (mi >> 1);
        uint32_t r0, r1, r2, r3;
        ldsm_x4(sk + (key * SRC_CH + swz<SRC_CH>(ch, key)) * 16, r0, r1, r2, r3);
        mma_f16(s[0], qa[s2], e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r0 >> 16));
        mma_f16(s[1], qa[s2], e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r1 >> 16));
        mma_f16(s_alt[0], qa[s2 + 1], e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r2 >> 16));
        mma_f16(s_alt[1], qa[s2 + 1], e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r3 >> 16));
      }
    } else {
#pragma unroll
      for (int s2 = 0; s2 < KSTEPS; s2 += 2) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int key = j * 8 + mrow;
          const int ch = s2 * 2 + mi;  // chunks 2*s2 .. 2*s2+3 cover k-steps s2, s2+1
          uint32_t b0, b1, b2, b3;
          ldsm_x4(sk + (key * SRC_CH + swz<SRC_CH>(ch, key)) * 16, b0, b1, b2, b3);
          mma_bf16(s[j], qa[s2], b0, b1);
          mma_bf16(s_alt[j], qa[s2 + 1], b2, b3);
        }
      }
    }
    // mask keys past the stripe end (or on a rejected page), scale into the log2 domain
    float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool ok = (vm >> (j * 8 + 2 * qi + e)) & 1u;
        s[j][e] = ok ? (s[j][e] + s_alt[j][e]) * sl : -INFINITY;
        s[j][e + 2] = ok ? (s[j][e + 2] + s_alt[j][e + 2]) * sl : -INFINITY;
        bm0 = fmaxf(bm0, s[j][e]);
        bm1 = fmaxf(bm1, s[j][e + 2]);
      }
    }
    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 1));
    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 2));
    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 1));
    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 2));
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
      for (int u = 0; u < NT; ++u) {
        o[u][0] *= a0;
        o[u][1] *= a0;
        o[u][2] *= a1;
        o[u][3] *= a1;
      }
    }
    uint32_t pa[4], pl[4];
    {
      const float p00 = exp2f(s[0][0] - m0), p01 = exp2f(s[0][1] - m0);
      const float p02 = exp2f(s[0][2] - m1), p03 = exp2f(s[0][3] - m1);
      const float p10 = exp2f(s[1][0] - m0), p11 = exp2f(s[1][1] - m0);
      const float p12 = exp2f(s[1][2] - m1), p13 = exp2f(s[1][3] - m1);
      l0 += (p00 + p01) + (p10 + p11);
      l1 += (p02 + p03) + (p12 + p13);
      split16<F8>(p00, p01, pa[0], pl[0]);
      split16<F8>(p02, p03, pa[1], pl[1]);
      split16<F8>(p10, p11, pa[2], pl[2]);
      split16<F8>(p12, p13, pa[3], pl[3]);
    }
    // O += P V  (V rows via ldmatrix.trans)
    const int vkey = (mi & 1) * 8 + mrow;
    if constexpr (F8) {
      // ldmatrix.trans of code bytes: matrices keys 0-7 / 8-15 x chunks ch,
      // ch + 1 (16 dims each); a register holds keys (2qi, 2qi+1) of the
      // code pairs of dims 2n, 2n+1 (n = lane / 4), so its even bytes are
      // the b pair of dim 2n and its odd bytes that of dim 2n + 1: n-tile
      // 2 ch gathers a chunk's even dims, n-tile 2 ch + 1 its odd dims
#pragma unroll
      for (int ch0 = 0; ch0 < SRC_CH; ch0 += 2) {
        const int ch = ch0 + (mi >> 1);
        uint32_t r[4];
        ldsm_x4_t(sv + (vkey * SRC_CH + swz<SRC_CH>(ch, vkey)) * 16, r[0], r[1], r[2], r[3]);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // chunk ch0 + hh: registers 2 hh (keys 0-7), 2 hh + 1 (keys 8-15)
          const uint32_t lo = r[2 * hh], hi = r[2 * hh + 1];
          const uint32_t ev0 = e4m3x2_to_f16x2(__byte_perm(lo, 0u, 0x4420u));
          const uint32_t ev1 = e4m3x2_to_f16x2(__byte_perm(hi, 0u, 0x4420u));
          const uint32_t od0 = e4m3x2_to_f16x2(__byte_perm(lo, 0u, 0x4431u));
          const uint32_t od1 = e4m3x2_to_f16x2(__byte_perm(hi, 0u, 0x4431u));
          const int u = 2 * (ch0 + hh);
          mma_f16(o[u], pa, ev0, ev1);
          mma_f16(o[u + 1], pa, od0, od1);
          mma_f16(o[u], pl, ev0, ev1);
          mma_f16(o[u + 1], pl, od0, od1);
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < NT; u += 4) {
        uint32_t bv[2][4];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int ch = u + 2 * hh + (mi >> 1);  // 16-byte chunk = 8-dim group
          ldsm_x4_t(sv + (vkey * SRC_CH + swz<SRC_CH>(ch, vkey)) * 16, bv[hh][0], bv[hh][1], bv[hh][2], bv[hh][3]);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          mma_bf16(o[u + 2 * hh], pa, bv[hh][0], bv[hh][1]);
          mma_bf16(o[u + 2 * hh + 1], pa, bv[hh][2], bv[hh][3]);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          mma_bf16(o[u + 2 * hh], pl, bv[hh][0], bv[hh][1]);
          mma_bf16(o[u + 2 * hh + 1], pl, bv[hh][2], bv[hh][3]);
        }
      }
    }
  }
  cp_async_wait<0>();

  if constexpr (F8) {  // value = code * v_descale
#pragma unroll
    for (int u = 0; u < NT; ++u) {
      o[u][0] *= a.v_descale;
      o[u][1] *= a.v_descale;
      o[u][2] *= a.v_descale;
      o[u][3] *= a.v_descale;
    }
  }
  // ---- per-warp state -> shared memory (rows < G only), then the cross-warp merge
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  __syncthreads();
  float* sm = reinterpret_cast<float*>(smem);
  float* sm_o = sm;                       // [NW][G][D]
  float* sm_m = sm_o + NW * G * D;        // [NW][G]
  float* sm_l = sm_m + NW * G;            // [NW][G]
  // dim of accumulator column 2 qi + e of n-tile u: bf16 8 u + 2 qi + e;
  // E4M3 (n-tiles of a chunk's even / odd dims) 16 (u / 2) + 4 qi + 2 e + u % 2
  auto odim = [&](int u, int e) { return F8 ? 16 * (u >> 1) + 4 * qi + 2 * e + (u & 1) : u * 8 + 2 * qi + e; };
  if (quad < G) {
#pragma unroll
    for (int u = 0; u < NT; ++u) {
      sm_o[(warp * G + quad) * D + odim(u, 0)] = o[u][0];
      sm_o[(warp * G + quad) * D + odim(u, 1)] = o[u][1];
    }
    if (qi == 0) {
      sm_m[warp * G + quad] = m0;
      sm_l[warp * G + quad] = l0;
    }
  }
  if (quad + 8 < G) {
#pragma unroll
    for (int u = 0; u < NT; ++u) {
      sm_o[(warp * G + quad + 8) * D + odim(u, 0)] = o[u][2];
      sm_o[(warp * G + quad + 8) * D + odim(u, 1)] = o[u][3];
    }
    if (qi == 0) {
      sm_m[warp * G + quad + 8] = m1;
      sm_l[warp * G + quad + 8] = l1;
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
static int launch_mma_t(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  using SM = MmaSmem<D, F8>;
  const size_t comb = (static_cast<size_t>(kMmaWarps) * G * D + 2 * kMmaWarps * G) * sizeof(float);
  const size_t pages = (static_cast<size_t>(a.chunk) / a.ps_l + 2) * sizeof(int);
  const size_t smem = (SM::MAIN > comb ? SM::MAIN : comb) + pages;
  auto kern = gqa_partial_mma_kernel<D, G, F8>;
  static std::atomic<int> smem_set[64];
  *err = ensure_smem(kern, smem, smem_set);
  if (*err != cudaSuccess) return CPATTN_ERR_CUDA;
  dim3 grid(a.max_chunks, a.P * a.num_kv_heads, a.qo_indptr != nullptr ? a.num_rows : a.num_tokens);
  kern<<<grid, kMmaWarps * 32, smem, s>>>(a);
  *err = cudaGetLastError();
  return *err == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

template <int D, bool F8>
static int mma_dispatch_g(const PartialArgs& a, int G, cudaStream_t s, cudaError_t* err) {
  switch (G) {
    case 1: return launch_mma_t<D, 1, F8>(a, s, err);
    case 2: return launch_mma_t<D, 2, F8>(a, s, err);
    case 4: return launch_mma_t<D, 4, F8>(a, s, err);
    case 8: return launch_mma_t<D, 8, F8>(a, s, err);
    case 16: return launch_mma_t<D, 16, F8>(a, s, err);
    default: return CPATTN_ERR_UNSUPPORTED_SHAPE;
  }
}

int launch_gqa_partial_mma(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  const int G = a.num_q_heads / a.num_kv_heads;
  if (a.head_dim != a.head_dim_v) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  int st = CPATTN_ERR_UNSUPPORTED_SHAPE;
  // groups of up to 8 heads: the transposed kernel (partial_gqa_mmat.cu);
  // groups of 16: the head-rows kernel above
  if (a.kv_fp8) {
    if (G <= 8) {
      st = launch_gqa_partial_mmat(a, s, err);
    } else {
      if (a.head_dim == 128) st = mma_dispatch_g<128, true>(a, G, s, err);
      if (a.head_dim == 64) st = mma_dispatch_g<64, true>(a, G, s, err);
    }
  } else if (G <= 8) {
    st = launch_gqa_partial_mmat(a, s, err);
  } else {
    if (a.head_dim == 128) st = mma_dispatch_g<128, false>(a, G, s, err);
    if (a.head_dim == 64) st = mma_dispatch_g<64, false>(a, G, s, err);
  }
  // ragged rows may hold several tokens: those rows go to the multi-token kernel
  if (st == CPATTN_OK && a.qo_indptr != nullptr) st = launch_gqa_partial_ext(a, s, err);
  return st;
}

}  // namespace cpattn
