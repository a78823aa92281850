// own_token_attn, bf16 on tensor cores: causal attention of a step's new
// tokens over the row's own new K/V (mstar PR #1124 "Context / Sequence
// Parallel 1/5", description: a step that is not one token a row attends its
// own tokens apart; vLLM "[Core] Add explicit layer parallel plans",
// _forward_with_dcp: flash_attn_varlen_func with cu_seqlens_k = cu_seqlens_q,
// causal).
//
// CTA = (block of TQ = 4 * 16 / G tokens of row b, KV head h), 4 warps.  Warp
// w owns 16 query rows: tokens q0 + w * 16 / G + r / G, heads h * G + r % G
// (r = 0..15), so each row's online softmax stays inside its warp and no
// cross-warp merge is needed.  The row's new keys 0 .. (last token of the
// block) stream through a CTA-wide 3-stage cp.async ring of 16 keys (K and V
// rows, 16-byte chunk c of key r at c ^ (r & 7)); every warp runs
//   S = Q K^T  (mma.sync m16n8k16, 2 n-tiles of 8 keys, D / 16 k-steps)
//   O += P V   (P re-packed from the accumulators as a bf16 hi + lo pair)
// on the tiles up to its own last token, with keys after a row's token masked
// (causal; the diagonal is kept).  Rows of padding rows (b >= num_real_rows)
// and tokens past the last row get O = 0, LSE = -inf without any K/V read.
#include "launch.h"
#include "mma_sync.cuh"

namespace cpattn {

namespace {
constexpr int kOwnMmaWarps = 4;
constexpr int kOwnKeys = 16;
constexpr int kOwnStages = 3;
}  // namespace

template <int D, int G>
__global__ void __launch_bounds__(kOwnMmaWarps * 32) own_token_mma_kernel(const OwnArgs a) {
  constexpr int NW = kOwnMmaWarps;
  constexpr int KT = kOwnKeys;
  constexpr int NST = kOwnStages;
  constexpr int TPW = 16 / G;     // tokens a warp
  constexpr int TQ = NW * TPW;    // tokens a CTA
  constexpr int ROWB = D * 2;
  constexpr int CH = ROWB / 16;   // 16-byte chunks a row
  constexpr int STAGE_B = KT * ROWB;
  constexpr int KSTEPS = D / 16;
  constexpr int NT = D / 8;
  static_assert(G >= 1 && G <= 16 && 16 % G == 0, "group size");
  extern __shared__ __align__(128) uint8_t smem[];

  const int x = blockIdx.x;
  const int h = blockIdx.y;
  const int z = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int quad = lane >> 2;
  const int qi = lane & 3;
  const int Hq = a.num_q_heads;

  // token range of this z slice: row z, or (z == num_rows_bucket) the tokens past the last row
  int r0, r1;
  if (z < a.num_rows_bucket) {
    r0 = __ldg(a.qo_indptr + z);
    r1 = __ldg(a.qo_indptr + z + 1);
  } else {
    r0 = __ldg(a.qo_indptr + a.num_rows_bucket);
    r1 = a.num_tokens;
  }
  r0 = max(0, min(r0, a.num_tokens));
  r1 = max(r0, min(r1, a.num_tokens));
  if (z >= a.num_real_rows) {
    // padding row or tokens of no row: 0 / -inf, keys never read
    for (int t = r0 + x * TQ; t < r1; t += gridDim.x * TQ) {
      for (int tt = t; tt < min(t + TQ, r1); ++tt) {
        const int64_t row0 = static_cast<int64_t>(tt) * Hq + h * G;
        for (int i = threadIdx.x; i < G * D; i += blockDim.x) a.o_own[row0 * D + i] = 0.f;
        if (threadIdx.x < G) a.lse_own[row0 + threadIdx.x] = -INFINITY;
      }
    }
    return;
  }
  // blocks of TQ tokens, x, x + gridDim.x, ... (max_q_len sizes the grid; longer rows loop)
  for (int q0 = r0 + x * TQ; q0 < r1; q0 += gridDim.x * TQ) {
    __syncthreads();  // the ring of the previous block is no longer read
    const int q_end = min(q0 + TQ, r1);                // tokens of the block: [q0, q_end)
    const int nkeys = q_end - r0;                      // keys r0 .. q_end - 1
    const int ntiles = (nkeys + KT - 1) / KT;
    const int w_first = q0 + warp * TPW;               // this warp's first token
    const int w_last = min(w_first + TPW, q_end) - 1;  // its last valid token (< w_first if none)
    const int my_tiles = w_last >= w_first ? (w_last - r0) / KT + 1 : 0;

    // ---- Q fragments: rows r -> token w_first + r / G, head h * G + r % G
    uint32_t qa[KSTEPS][4];
    const int tok0 = w_first + quad / G, tok1 = w_first + (quad + 8) / G;
    const bool ok0 = tok0 <= w_last, ok1 = tok1 <= w_last;
    {
      const uint32_t* q0w = reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(a.q) +
                                                              (static_cast<int64_t>(tok0) * Hq + h * G + quad % G) * ROWB);
      const uint32_t* q1w = reinterpret_cast<const uint32_t*>(
          static_cast<const uint8_t*>(a.q) + (static_cast<int64_t>(tok1) * Hq + h * G + (quad + 8) % G) * ROWB);
#pragma unroll
      for (int s = 0; s < KSTEPS; ++s) {
        const int w0 = s * 8 + qi;
        qa[s][0] = ok0 ? __ldg(q0w + w0) : 0u;
        qa[s][1] = ok1 ? __ldg(q1w + w0) : 0u;
        qa[s][2] = ok0 ? __ldg(q0w + w0 + 4) : 0u;
        qa[s][3] = ok1 ? __ldg(q1w + w0 + 4) : 0u;
      }
    }

    // ---- CTA-wide ring of key tiles (K then V of a stage)
    const uint8_t* kb = static_cast<const uint8_t*>(a.k_new);
    const uint8_t* vb = static_cast<const uint8_t*>(a.v_new);
    auto issue = [&](int i) {
      if (i < ntiles) {
        uint8_t* sk = smem + (i % NST) * STAGE_B * 2;
        uint8_t* sv = sk + STAGE_B;
        for (int idx = threadIdx.x; idx < KT * CH; idx += blockDim.x) {
          const int key = idx / CH;
          const int ch = idx - key * CH;
          const int j = i * KT + key;  // key index within the row
          const int soff = (key * CH + (ch ^ (key & 7))) * 16;
          if (j < nkeys) {
            const int64_t src = (static_cast<int64_t>(r0 + j) * a.num_kv_heads + h) * ROWB + ch * 16;
            cp_async16(sk + soff, kb + src);
            cp_async16(sv + soff, vb + src);
          } else {
            *reinterpret_cast<uint4*>(sv + soff) = make_uint4(0u, 0u, 0u, 0u);  // past the keys: value 0
          }
        }
      }
      cp_async_commit();
    };

    float o[NT][4];
#pragma unroll
    for (int u = 0; u < NT; ++u) o[u][0] = o[u][1] = o[u][2] = o[u][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const float sl = a.scale * kLog2e;
    const int mrow = lane & 7;
    const int mi = lane >> 3;
    const int pos0 = tok0 - r0, pos1 = tok1 - r0;  // causal limits (key index <= position)

#pragma unroll
    for (int i = 0; i < NST - 1; ++i) issue(i);
    for (int i = 0; i < ntiles; ++i) {
      cp_async_wait<NST - 2>();
      __syncthreads();        // tile i landed for every thread; tile i - 1 is no longer read
      issue(i + NST - 1);
      if (i < my_tiles) {
        const uint32_t sk = smem_u32(smem + (i % NST) * STAGE_B * 2);
        const uint32_t sv = sk + STAGE_B;
        float s[2][4], s_alt[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[j][e] = s_alt[j][e] = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < KSTEPS; s2 += 2) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int key = j * 8 + mrow;
            const int ch = s2 * 2 + mi;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(sk + (key * CH + (ch ^ (key & 7))) * 16, b0, b1, b2, b3);
            mma_bf16(s[j], qa[s2], b0, b1);
            mma_bf16(s_alt[j], qa[s2 + 1], b2, b3);
          }
        }
        // causal mask (key index <= the row's position; also < nkeys) and scale
        float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int kj = i * KT + j * 8 + 2 * qi + e;
            const bool v0 = ok0 && kj <= pos0;
            const bool v1 = ok1 && kj <= pos1;
            s[j][e] = v0 ? (s[j][e] + s_alt[j][e]) * sl : -INFINITY;
            s[j][e + 2] = v1 ? (s[j][e + 2] + s_alt[j][e + 2]) * sl : -INFINITY;
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
          // masked entries give exp2(-inf - m) = 0, also while m is still -inf for a row with no key yet
          auto ex = [](float sv, float m) { return sv == -INFINITY ? 0.f : exp2f(sv - m); };
          const float p00 = ex(s[0][0], m0), p01 = ex(s[0][1], m0);
          const float p02 = ex(s[0][2], m1), p03 = ex(s[0][3], m1);
          const float p10 = ex(s[1][0], m0), p11 = ex(s[1][1], m0);
          const float p12 = ex(s[1][2], m1), p13 = ex(s[1][3], m1);
          l0 += (p00 + p01) + (p10 + p11);
          l1 += (p02 + p03) + (p12 + p13);
          split_bf16(p00, p01, pa[0], pl[0]);
          split_bf16(p02, p03, pa[1], pl[1]);
          split_bf16(p10, p11, pa[2], pl[2]);
          split_bf16(p12, p13, pa[3], pl[3]);
        }
        const int vkey = (mi & 1) * 8 + mrow;
#pragma unroll
        for (int u = 0; u < NT; u += 4) {
          uint32_t bv[2][4];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int ch = u + 2 * hh + (mi >> 1);
            ldsm_x4_t(sv + (vkey * CH + (ch ^ (vkey & 7))) * 16, bv[hh][0], bv[hh][1], bv[hh][2], bv[hh][3]);
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

    // ---- rows of this lane: quad (c0, c1) and quad + 8 (c2, c3)
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
    const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    if (ok0) {
      const int64_t row = static_cast<int64_t>(tok0) * Hq + h * G + quad % G;
#pragma unroll
      for (int u = 0; u < NT; ++u)
        *reinterpret_cast<float2*>(a.o_own + row * D + u * 8 + 2 * qi) = make_float2(o[u][0] * inv0, o[u][1] * inv0);
      if (qi == 0) a.lse_own[row] = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
    }
    if (ok1) {
      const int64_t row = static_cast<int64_t>(tok1) * Hq + h * G + (quad + 8) % G;
#pragma unroll
      for (int u = 0; u < NT; ++u)
        *reinterpret_cast<float2*>(a.o_own + row * D + u * 8 + 2 * qi) = make_float2(o[u][2] * inv1, o[u][3] * inv1);
      if (qi == 0) a.lse_own[row] = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
    }
  }
}

template <int D, int G>
static int launch_own_mma_t(const OwnArgs& a, cudaStream_t s, cudaError_t* err) {
  constexpr int TQ = kOwnMmaWarps * (16 / G);
  const size_t smem = static_cast<size_t>(kOwnStages) * kOwnKeys * D * 2 * 2;
  auto kern = own_token_mma_kernel<D, G>;
  static std::atomic<int> smem_set[64];
  *err = ensure_smem(kern, smem, smem_set);
  if (*err != cudaSuccess) return CPATTN_ERR_CUDA;
  const int blocks = (a.max_q_len + TQ - 1) / TQ > 0 ? (a.max_q_len + TQ - 1) / TQ : 1;
  dim3 grid(blocks, a.num_kv_heads, a.num_rows_bucket + 1);
  kern<<<grid, kOwnMmaWarps * 32, smem, s>>>(a);
  *err = cudaGetLastError();
  return *err == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

int launch_own_token_mma(const OwnArgs& a, cudaStream_t s, cudaError_t* err) {
  const int G = a.num_q_heads / a.num_kv_heads;
  if (a.head_dim != 128 && a.head_dim != 64) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  switch (G) {
    case 1: return a.head_dim == 128 ? launch_own_mma_t<128, 1>(a, s, err) : launch_own_mma_t<64, 1>(a, s, err);
    case 2: return a.head_dim == 128 ? launch_own_mma_t<128, 2>(a, s, err) : launch_own_mma_t<64, 2>(a, s, err);
    case 4: return a.head_dim == 128 ? launch_own_mma_t<128, 4>(a, s, err) : launch_own_mma_t<64, 4>(a, s, err);
    case 8: return a.head_dim == 128 ? launch_own_mma_t<128, 8>(a, s, err) : launch_own_mma_t<64, 8>(a, s, err);
    case 16: return a.head_dim == 128 ? launch_own_mma_t<128, 16>(a, s, err) : launch_own_mma_t<64, 16>(a, s, err);
    default: return CPATTN_ERR_UNSUPPORTED_SHAPE;
  }
}

}  // namespace cpattn
