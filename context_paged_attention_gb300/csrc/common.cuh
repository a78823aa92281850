// Internal helpers shared by the libcpattn kernels (not part of the C ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cpattn.h"

namespace cpattn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Programmatic dependent launch.  A kernel launched by launch_pdl may start
// while the previous kernel on its stream is still running: it calls
// pdl_wait() before it reads anything written before it on the stream (the
// wait returns once that work is complete and visible; without a
// programmatic launch it returns at once), and pdl_trigger() lets the next
// such kernel be scheduled (it only starts its own prologue early).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Record the first device-detected inconsistency (0 stays 0 until something happens).
__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Two bfloat16 values packed in a 32-bit word -> float (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// A 16-byte chunk of elements of type T, widened to float.
template <typename T>
struct Chunk16;

template <>
struct Chunk16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void widen(const uint4& u, float* f) {
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
    f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
    f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
  }
};

template <>
struct Chunk16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void widen(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
};

// 16-byte asynchronous global -> shared copy (bypasses L1).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Row of token t: the b in [0, num_rows) with indptr[b] <= t < indptr[b+1]
// (indptr non-decreasing, t < indptr[num_rows]).  Empty rows are skipped.
__device__ __forceinline__ int find_row(const int32_t* __restrict__ indptr, int num_rows, int t) {
  int lo = 0, hi = num_rows - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(indptr + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32: relative error
// about 2^-22, results below 2^-126 flushed to zero).  Used where the
// probability is rounded to bf16 right after (relative step 2^-9).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Keys of a row of L positions that partner p holds when runs of I
// consecutive positions go round the P partners (I = 1: positions p, p + P, ...).
// Those keys fill the partner's physical slots 0 .. n - 1 in stripe order.
__host__ __device__ __forceinline__ int stripe_len(int L, int p, int P, int I) {
  const int groups = L / I;  // whole runs
  const int mine = groups > p ? (groups - p + P - 1) / P : 0;
  return mine * I + (groups % P == p ? L - groups * I : 0);
}

// Upper bound of stripe_len over the partners (exact for I = 1).
__host__ __device__ __forceinline__ int max_stripe_len(int L, int P, int I) {
  const int runs = (L + I * P - 1) / (I * P);
  return runs * I < L ? runs * I : L;
}

// Row (or token) that grid slot z works on under an optional dispatch order;
// an entry outside [0, n) is reported (CPATTN_DEV_BAD_INDPTR) and gives -1.
__device__ __forceinline__ int ordered_row(const int32_t* __restrict__ order, int z, int n, int32_t* dev_status) {
  if (order == nullptr) return z;
  const int b = __ldg(order + z);
  if (b < 0 || b >= n) {
    if (threadIdx.x == 0) report(dev_status, CPATTN_DEV_BAD_INDPTR);
    return -1;
  }
  return b;
}

// Online-softmax state merge in the log2 domain: (m, l) absorbs (m2, l2);
// returns the factors the two accumulators are scaled by.
__device__ __forceinline__ void softmax_merge_factors(float m, float m2, float& mn, float& a, float& b) {
  mn = fmaxf(m, m2);
  a = (m == -INFINITY) ? 0.f : exp2f(m - mn);
  b = (m2 == -INFINITY) ? 0.f : exp2f(m2 - mn);
}

}  // namespace cpattn
