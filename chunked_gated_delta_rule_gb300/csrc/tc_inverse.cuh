// tc_inverse.cuh -- T = (I + A)^-1 for a strictly lower-triangular 64 x 64
// FP32 matrix A in shared memory (row stride kInvLd), by one CTA of 256
// threads (A4 of the chunked form: the UT transform's triangular inverse).
//
//   1. The four 16 x 16 diagonal blocks T_bb = (I + A_bb)^-1 in FP32: one
//      thread per (block, column) solves (I + A_bb) x = e_m by right-looking
//      forward substitution (after x_j is known, every later row's partial
//      sum takes its A_rj x_j term), so the dependent chain is 16 steps long.
//   2. Off-diagonal blocks by distance d = 1, 2, 3 (standard block forward
//      substitution):  T_ij = -T_ii * sum_{k=j}^{i-1} A_ik T_kj,  i = j + d.
//      Each 16 x 8 column tile of each block is one warp's job: the products
//      run on warp-level tensor cores as three TF32 products (x = hi + lo;
//      a_hi b_hi + a_hi b_lo + a_lo b_hi, each in its own accumulator), which
//      keeps close to FP32 accuracy with short dependent chains.
//
// T's entries above the diagonal of each diagonal block are written as 0;
// blocks above the block diagonal are not written (callers mask j > i).
#pragma once

#include "tc_common.cuh"

namespace gdr {
namespace tc {

constexpr int kInvLd = 68;   // row stride of A and T (floats; rows 16-B aligned)
constexpr int kInvXLd = 8;   // row stride of a warp's 16 x 8 scratch tile
constexpr int kInvScratchFloats = 6 * 16 * kInvXLd;

// acc_* (16 x 8, mma accumulator layout) += A(16 x 16) * B(16 x 8), both
// row-major FP32 in shared memory, split into TF32 hi/lo parts.
__device__ __forceinline__ void warp_gemm16x8_3xtf32(float (&hh)[4], float (&hl)[4],
                                                     float (&lh)[4], const float *A, int lda,
                                                     const float *B, int ldb, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const float av[4] = {A[g * lda + 8 * ks + t], A[(g + 8) * lda + 8 * ks + t],
                             A[g * lda + 8 * ks + t + 4], A[(g + 8) * lda + 8 * ks + t + 4]};
        const float bv[2] = {B[(8 * ks + t) * ldb + g], B[(8 * ks + t + 4) * ldb + g]};
        uint32_t ahi[4], alo[4], bhi[2], blo[2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ahi[i] = to_tf32(av[i]);
            alo[i] = to_tf32(av[i] - __uint_as_float(ahi[i]));
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            bhi[i] = to_tf32(bv[i]);
            blo[i] = to_tf32(bv[i] - __uint_as_float(bhi[i]));
        }
        mma_tf32_16x8x8(hh, ahi, bhi);
        mma_tf32_16x8x8(hl, ahi, blo);
        mma_tf32_16x8x8(lh, alo, bhi);
    }
}

// sX: kInvScratchFloats floats of scratch.  All 256 threads call this.
__device__ __forceinline__ void invert_unit_lower64(const float *sA, float *sT, float *sX,
                                                    int tid) {
    if (tid < 64) {
        const int b = tid >> 4, m = tid & 15, o = 16 * b;
        float s[16], x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) s[r] = 0.f;
        // Columns before m are exactly zero, so their (finite) updates add
        // exact zeros: the loop runs unpredicated, as straight-line code.
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            x[j] = j < m ? 0.f : (j == m ? 1.f : -s[j]);
#pragma unroll
            for (int r = j + 1; r < 16; ++r)
                s[r] = fmaf(sA[(o + r) * kInvLd + o + j], x[j], s[r]);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(o + r) * kInvLd + o + m] = x[r];
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    for (int d = 1; d <= 3; ++d) {
        if (warp < 2 * (4 - d)) {
            const int j = warp >> 1, nt = warp & 1, i = j + d;
            float hh[4] = {0.f, 0.f, 0.f, 0.f}, hl[4] = {0.f, 0.f, 0.f, 0.f},
                  lh[4] = {0.f, 0.f, 0.f, 0.f};
            for (int k = j; k < i; ++k)
                warp_gemm16x8_3xtf32(hh, hl, lh, sA + (16 * i) * kInvLd + 16 * k, kInvLd,
                                     sT + (16 * k) * kInvLd + 16 * j + 8 * nt, kInvLd, lane);
            float *X = sX + warp * 16 * kInvXLd;
            X[g * kInvXLd + 2 * t] = (lh[0] + hl[0]) + hh[0];
            X[g * kInvXLd + 2 * t + 1] = (lh[1] + hl[1]) + hh[1];
            X[(g + 8) * kInvXLd + 2 * t] = (lh[2] + hl[2]) + hh[2];
            X[(g + 8) * kInvXLd + 2 * t + 1] = (lh[3] + hl[3]) + hh[3];
            __syncwarp();
            float th[4] = {0.f, 0.f, 0.f, 0.f}, tl[4] = {0.f, 0.f, 0.f, 0.f},
                  tm[4] = {0.f, 0.f, 0.f, 0.f};
            warp_gemm16x8_3xtf32(th, tl, tm, sT + (16 * i) * kInvLd + 16 * i, kInvLd, X,
                                 kInvXLd, lane);
            float *Tij = sT + (16 * i) * kInvLd + 16 * j + 8 * nt;
            Tij[g * kInvLd + 2 * t] = -((tm[0] + tl[0]) + th[0]);
            Tij[g * kInvLd + 2 * t + 1] = -((tm[1] + tl[1]) + th[1]);
            Tij[(g + 8) * kInvLd + 2 * t] = -((tm[2] + tl[2]) + th[2]);
            Tij[(g + 8) * kInvLd + 2 * t + 1] = -((tm[3] + tl[3]) + th[3]);
        }
        __syncthreads();
    }
}

}  // namespace tc
}  // namespace gdr
