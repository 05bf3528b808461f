// simt_tile.cuh -- register-tiled products of 64-row FP32 tiles in shared
// memory for the CUDA-core kernels (256 threads a CTA).
#pragma once

namespace gdr {

// Eight (four for FP32) consecutive input elements from one 16-byte load.
__device__ __forceinline__ void unpack16(const uint4 &raw, const __nv_bfloat16 *, float *x) {
    const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(b[e]);
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}
__device__ __forceinline__ void unpack16(const uint4 &raw, const __half *, float *x) {
    const __half2 *b = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(b[e]);
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}
__device__ __forceinline__ void unpack16(const uint4 &raw, const float *, float *x) {
    x[0] = __uint_as_float(raw.x);
    x[1] = __uint_as_float(raw.y);
    x[2] = __uint_as_float(raw.z);
    x[3] = __uint_as_float(raw.w);
}

// Register-tiled products on shared-memory tiles.  Thread t owns the rows
// 4 (t >> 4) + r (r < 4) and the columns (t & 15) + 16 s (s < NS) of a
// 64 x 16 NS result: per reduction step it loads 4 + NS values for 4 NS
// multiply-adds.  A warp reads two rows of the left operand (two addresses)
// and sixteen consecutive rows or columns of the right one, so no step has a
// bank conflict with 65-float rows.  The reduction runs in ascending order
// for every output, so each element has one fixed summation order.
template <int NS>
__device__ __forceinline__ void acc_zero(float (&a)[4][NS]) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s = 0; s < NS; ++s) a[r][s] = 0.f;
}

// a += A B^T over n:  A[i][c] (row stride lda), B[j][c] (ldb)
template <int NS>
__device__ __forceinline__ void mm_abT(float (&a)[4][NS], const float *A, int lda, const float *B,
                                       int ldb, int n, int tid) {
    const int i0 = 4 * (tid >> 4), j0 = tid & 15;
#pragma unroll 4
    for (int c = 0; c < n; ++c) {
        float x[4], y[NS];
#pragma unroll
        for (int r = 0; r < 4; ++r) x[r] = A[(i0 + r) * lda + c];
#pragma unroll
        for (int s = 0; s < NS; ++s) y[s] = B[(j0 + 16 * s) * ldb + c];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int s = 0; s < NS; ++s) a[r][s] = fmaf(x[r], y[s], a[r][s]);
    }
}

// a += A^T B over n:  A[m][i] (lda), B[m][j] (ldb)
template <int NS>
__device__ __forceinline__ void mm_atb(float (&a)[4][NS], const float *A, int lda, const float *B,
                                       int ldb, int n, int tid) {
    const int i0 = 4 * (tid >> 4), j0 = tid & 15;
#pragma unroll 4
    for (int m = 0; m < n; ++m) {
        float x[4], y[NS];
#pragma unroll
        for (int r = 0; r < 4; ++r) x[r] = A[m * lda + i0 + r];
#pragma unroll
        for (int s = 0; s < NS; ++s) y[s] = B[m * ldb + j0 + 16 * s];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int s = 0; s < NS; ++s) a[r][s] = fmaf(x[r], y[s], a[r][s]);
    }
}

// a += A B over n:  A[i][m] (lda), B[m][j] (ldb)
template <int NS>
__device__ __forceinline__ void mm_ab(float (&a)[4][NS], const float *A, int lda, const float *B,
                                      int ldb, int n, int tid) {
    const int i0 = 4 * (tid >> 4), j0 = tid & 15;
#pragma unroll 4
    for (int m = 0; m < n; ++m) {
        float x[4], y[NS];
#pragma unroll
        for (int r = 0; r < 4; ++r) x[r] = A[(i0 + r) * lda + m];
#pragma unroll
        for (int s = 0; s < NS; ++s) y[s] = B[m * ldb + j0 + 16 * s];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int s = 0; s < NS; ++s) a[r][s] = fmaf(x[r], y[s], a[r][s]);
    }
}

#define FOR_TILE(NS)                                                      \
    _Pragma("unroll") for (int r = 0; r < 4; ++r)                         \
        _Pragma("unroll") for (int s = 0; s < NS; ++s)

}  // namespace gdr
