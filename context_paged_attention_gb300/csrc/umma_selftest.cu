// cpattn_umma_selftest: one 128-row tcgen05 GEMM tile in the operand layouts
// the attention kernels use, so a test can compare it with a plain matmul.
// Not part of the method; it checks the tensor-core plumbing (descriptors,
// TMEM allocation, commit, tcgen05.ld) on the device.
#include <cuda_bf16.h>

#include "common.cuh"
#include "cpattn_selftest.h"
#include "tc05.cuh"

namespace cpattn {

constexpr int kSelfTestSmem = 200 * 1024;  // operands + 1 KB alignment slack

__global__ void __launch_bounds__(128) umma_selftest_kernel(int variant, const __nv_bfloat16* A,
                                                            const __nv_bfloat16* B, float* D, int N, int K,
                                                            int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t mbar;
  __shared__ uint32_t tmem_base_sh;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- operands into their swizzled shared-memory layouts
  uint8_t* sA = base;
  uint8_t* sB;
  const uint4* gA = reinterpret_cast<const uint4*>(A);
  const uint4* gB = reinterpret_cast<const uint4*>(B);
  if (variant == 5) {
    sB = sA;  // no operands: the completion wait below is on a barrier nothing arrives at
  } else if (variant == 0 || variant == 4) {
    // A [128][K], B [N][K], both K-major SW128 in 64-element column blocks
    // (variant 4 reads A from tensor memory instead, written below)
    sB = sA + 128 * K * 2;
    const int kc = K / 8;
    for (int i = tid; i < 128 * kc; i += blockDim.x) {
      const int r = i / kc, c = i % kc;
      *reinterpret_cast<uint4*>(sA + (c / 8) * (128 * 128) + tc05::sw128(r, c % 8)) = gA[i];
    }
    for (int i = tid; i < N * kc; i += blockDim.x) {
      const int r = i / kc, c = i % kc;
      *reinterpret_cast<uint4*>(sB + (c / 8) * (N * 128) + tc05::sw128(r, c % 8)) = gB[i];
    }
  } else {
    // A [128][32] K-major SW64 (variant 3: A goes to tensor memory below);
    // B [K][N] MN-major SW128 in 64-element N blocks
    sB = sA + 128 * 64;
    for (int i = tid; i < 128 * 4; i += blockDim.x) {
      const int r = i / 4, c = i % 4;
      *reinterpret_cast<uint4*>(sA + tc05::sw64(r, c)) = gA[i];
    }
    const int nc = N / 8;
    for (int i = tid; i < K * nc; i += blockDim.x) {
      const int k = i / nc, c = i % nc;
      *reinterpret_cast<uint4*>(sB + (c / 8) * (K * 128) + tc05::sw128(k, c % 8)) = gB[i];
    }
  }
  tc05::fence_smem_to_async();
  __syncthreads();  // operands complete before the allocation and the MMAs
  const uint32_t ncols = variant >= 3 ? 512 : 256;  // variants 3, 4: A at column 256
  if (warp == 0) tc05::tmem_alloc(tc05::smem_addr(&tmem_base_sh), ncols);
  if (tid == 0) {
    tc05::mbar_init(tc05::smem_addr(&mbar), 1);
    tc05::mbar_init_fence();
  }
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  const uint32_t tbase = tmem_base_sh;
  const uint32_t mb = tc05::smem_addr(&mbar);
  if (variant == 4) {
    // row tid of A (K bf16 = K/2 words) -> lane tid, columns 256 .. 256 + K/2
    const uint4* row = gA + tid * (K / 8);
    for (int c0 = 0; c0 < K / 2; c0 += 16) {
      uint32_t w[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = row[c0 / 4 + q];
        w[4 * q] = u.x;
        w[4 * q + 1] = u.y;
        w[4 * q + 2] = u.z;
        w[4 * q + 3] = u.w;
      }
      tc05::st_x16_u32(tc05::taddr(tbase, warp * 32, 256 + c0), w);
    }
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
  }
  if (variant == 3) {
    // row tid of A (32 bf16 = 16 words, element 2j in the low half of word j) -> lane tid, columns 256..271
    uint32_t w[16];
    const uint4* row = gA + tid * 4;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = row[q];
      w[4 * q] = u.x;
      w[4 * q + 1] = u.y;
      w[4 * q + 2] = u.z;
      w[4 * q + 3] = u.w;
    }
    tc05::st_x16_u32(tc05::taddr(tbase, warp * 32, 256), w);
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
  }

  if (tid == 0 && variant != 5) {
    const uint32_t a0 = tc05::smem_addr(sA), b0 = tc05::smem_addr(sB);
    if (variant == 0) {
      const uint32_t id = tc05::idesc_bf16(128, N, false, false);
      for (int s = 0; s < K / 16; ++s) {
        const uint32_t off = (s % 4) * 32;
        const uint64_t ad = tc05::desc_k128(a0 + (s / 4) * (128 * 128) + off);
        const uint64_t bd = tc05::desc_k128(b0 + (s / 4) * (N * 128) + off);
        tc05::mma_ss(tbase, ad, bd, id, s > 0);
      }
    } else if (variant == 4) {
      const uint32_t id = tc05::idesc_bf16(128, N, false, false);
      for (int s = 0; s < K / 16; ++s) {
        const uint64_t bd = tc05::desc_k128(b0 + (s / 4) * (N * 128) + (s % 4) * 32);
        tc05::mma_ts(tbase, tbase + 256 + s * 8, bd, id, s > 0);
      }
    } else if (variant == 3) {
      const uint32_t id = tc05::idesc_bf16(128, N, false, true);
      for (int s = 0; s < K / 16; ++s)
        tc05::mma_ts(tbase, tbase + 256 + s * 8, tc05::desc_mn128(b0 + s * 16 * 128, K * 128), id, s > 0);
    } else {
      const uint32_t id = tc05::idesc_bf16(128, N, false, true);
      for (int s = 0; s < K / 16; ++s) {
        const uint64_t ad = tc05::desc_k64(a0 + s * 32);
        const uint32_t bs = b0 + s * 16 * 128;
        const uint64_t bd = variant == 1 ? tc05::desc_mn128(bs, K * 128)
                                         : tc05::make_desc(bs, 1024, K * 128, tc05::kSwizzle128);
        tc05::mma_ss(tbase, ad, bd, id, s > 0);
      }
    }
    tc05::commit(mb);
  }
  // variant 5: no MMA is issued and nothing commits, so the wait runs out
  // after a short poll limit and takes the timeout path (status, TMEM freed)
  const bool ok = tc05::mbar_wait(mb, 0, variant == 5 ? (1u << 12) : (1u << 24));
  tc05::fence_after_sync();
  if (ok) {
    for (int col = 0; col < N; col += 16) {
      float v[16];
      tc05::ld_x16(tc05::taddr(tbase, warp * 32, col), v);
      tc05::ld_wait();
      float* dst = D + static_cast<int64_t>(warp * 32 + lane) * N + col;
#pragma unroll
      for (int i = 0; i < 16; ++i) dst[i] = v[i];
    }
  } else if (tid == 0) {
    report(status, CPATTN_DEV_TC_TIMEOUT);
  }
  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc05::tmem_dealloc(tbase, ncols);
}

}  // namespace cpattn

extern "C" int cpattn_umma_selftest(int variant, const void* A, const void* B, float* D, int N, int K,
                                    int32_t* dev_status, cudaStream_t stream) {
  using namespace cpattn;
  if (A == nullptr || B == nullptr || D == nullptr) return CPATTN_ERR_INVALID_ARG;
  if (variant == 0 || variant == 4) {
    if (N < 16 || N > 256 || N % 16 != 0 || K < 64 || K > 256 || K % 64 != 0) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  } else if (variant == 1 || variant == 2 || variant == 3) {
    if (N < 64 || N > 256 || N % 64 != 0 || K != 32) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  } else if (variant == 5) {
    N = 16;  // nothing is read or written but the status
    K = 64;
  } else {
    return CPATTN_ERR_INVALID_ARG;
  }
  // both operand tiles plus the 1 KB alignment slack must fit the shared-memory allocation
  const size_t need = (variant == 0 || variant == 4 ? static_cast<size_t>(128 + N) * K * 2 : 128 * 64 + static_cast<size_t>(K) * N * 2) + 1024;
  if (need > static_cast<size_t>(kSelfTestSmem)) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  if (cudaFuncSetAttribute(umma_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelfTestSmem) !=
      cudaSuccess)
    return CPATTN_ERR_CUDA;
  umma_selftest_kernel<<<1, 128, kSelfTestSmem, stream>>>(variant, static_cast<const __nv_bfloat16*>(A),
                                                         static_cast<const __nv_bfloat16*>(B), D, N, K, dev_status);
  return cudaGetLastError() == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}
