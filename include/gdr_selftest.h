/*
 * gdr_selftest.h -- diagnostic entry points of libgdr.so.  They exercise, on
 * the GPU, the tensor-core building blocks the fused forward path uses, so a
 * test can compare them with a library matmul before trusting the fused
 * kernels.  The pages describe no counterpart (they are tests of this
 * implementation's own operand layouts).  Device pointers; work enqueued on
 * `stream`; `status` (device int32, may be NULL) receives GDR_ERR_TIMEOUT if
 * a bounded wait expires.  Return GDR_OK or a GDR_ERR_* code (gdr.h).
 */
#ifndef GDR_SELFTEST_H_
#define GDR_SELFTEST_H_

#include <stdint.h>

#include "gdr.h"

#ifdef __cplusplus
extern "C" {
#endif

/* D[128][N] (FP32, row-major) = A[128][Kd] * B[N][Kd]^T with A, B BF16
 * row-major, computed by tcgen05.mma (kind::f16) with A staged K-major
 * (a_mn = 0) or MN-major (a_mn = 1) in shared memory, or in tensor memory
 * (a_mn = 2: row m on lane m, two BF16 per 32-bit column, the lower K index
 * in the low half), and B K-major or MN-major (b_mn) in shared memory, all
 * shared-memory operands with the 128-byte swizzle.  N in {64, 128}, Kd in
 * {64, 128}. */
int gdr_selftest_umma(const void *A, const void *B, float *D, int N, int Kd,
                      int a_mn, int b_mn, int32_t *status, gdr_stream_t stream);

/* out[64][64] (BF16) = src[t0 + r][h][k0 + c] for r, c < 64 (zero past T),
 * src a BF16 [T][H][K] tensor, loaded as one TMA box with the 128-byte
 * swizzle and read back through the library's swizzle address map.
 * k0 a multiple of 8 with k0 + 64 <= K. */
int gdr_selftest_tma(const void *src, int64_t T, int64_t H, int64_t K, int t0,
                     int h, int k0, void *out, int32_t *status,
                     gdr_stream_t stream);

/* T[64][64] (FP32, row-major) = (I + A)^-1 for the strictly lower part of
 * A[64][64] (FP32, row-major; entries on and above the diagonal are
 * ignored), by the blocked triangular inverse the tensor-core path uses (FP32
 * diagonal blocks, warp-level 3xTF32 products off the diagonal).  Entries
 * above the diagonal of T are written as 0. */
int gdr_selftest_inverse(const float *A, float *T, gdr_stream_t stream);

/* Waits on an mbarrier that nothing will complete, with the library's
 * bounded wait limited to `limit_ns` (at most 0.1 s): the wait gives up,
 * writes GDR_ERR_TIMEOUT to *status (device int32, caller zeroes it) and the
 * kernel exits normally, writing 2 to *done (1 would mean the wait was
 * satisfied).  This exercises the failure path of every time-bounded wait
 * without faulting or hanging the GPU. */
int gdr_selftest_timeout(int32_t *status, uint64_t limit_ns, int32_t *done,
                         gdr_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDR_SELFTEST_H_ */
