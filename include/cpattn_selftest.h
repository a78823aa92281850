/*
 * cpattn_selftest.h -- device self-test of libcpattn's tensor-core plumbing.
 *
 * The pages have no counterpart: this checks, against a plain matmul in a
 * test, that the shared-memory operand layouts, tcgen05 descriptors, TMEM
 * allocation and tcgen05.ld read-back used by the attention kernels produce
 * the product they are meant to.  Same conventions as cpattn.h (device
 * pointers, caller's stream, negative status on bad arguments).
 */
#ifndef CPATTN_SELFTEST_H_
#define CPATTN_SELFTEST_H_

#include <stdint.h>

#include "cpattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * One 128-row tile, bf16 inputs (row-major in global memory), fp32 output
 * D [128][N] (row-major):
 *   variant 0: D = A B^T, A [128][K], B [N][K]; both staged K-major with the
 *              128-byte swizzle (the Q K^T pattern).  N in 16..256 step 16,
 *              K in {64, 128, 192, 256}.
 *   variant 1: D = A B, A [128][32] K-major with the 64-byte swizzle, B [32][N]
 *              read M/N-major from 128-byte-swizzled rows (the P V pattern).
 *              N in {64, 128, 192, 256}.
 *   variant 2: variant 1 with the two descriptor strides exchanged (a check
 *              of which field carries which stride).
 *   variant 3: variant 1 with A read from tensor memory (row m in lane m, two
 *              bf16 K elements a 32-bit column), written there by tcgen05.st.
 *   variant 4: variant 0 with A read from tensor memory the same way (the
 *              Q K^T pattern with Q held in TMEM, K/16 k-steps of 8 columns).
 *   variant 5: the timeout path.  No MMA is issued and nothing arrives on the
 *              completion barrier, so its wait gives up after a short poll
 *              limit; the kernel stores CPATTN_DEV_TC_TIMEOUT, frees its
 *              tensor memory and returns (A, B, D are not read or written,
 *              N and K are ignored).  The context stays usable.
 * A completion wait that times out stores 4 in *dev_status (if not NULL).
 */
CPATTN_API int cpattn_umma_selftest(int variant, const void* A, const void* B, float* D, int N, int K,
                                    int32_t* dev_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_SELFTEST_H_ */
