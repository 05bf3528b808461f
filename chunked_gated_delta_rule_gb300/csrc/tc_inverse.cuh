// tc_inverse.cuh -- T = (I + A)^-1 for a strictly lower-triangular 64 x 64
// FP32 matrix A in shared memory (row stride kInvLd), by one CTA of >= 128
// threads (A4 of the chunked form: the UT transform's triangular inverse).
//
//   1. The four 16 x 16 diagonal blocks T_bb = (I + A_bb)^-1 in FP32: one
//      thread per (block, column) solves (I + A_bb) x = e_m by right-looking
//      forward substitution (after x_j is known, every later row's partial
//      sum takes its A_rj x_j term), so the dependent chain is 16 steps long.
//   2. Off-diagonal blocks by distance d = 1, 2, 3 (standard block forward
//      substitution):  T_ij = -T_ii * sum_{k=j}^{i-1} A_ik T_kj,  i = j + d,
//      one warp per block pair, each 16 x 16 x 16 product on warp-level
//      tensor cores with three TF32 products (hi/lo split, ~FP32 accuracy).
//
// T's entries above the diagonal of each diagonal block are written as 0;
// blocks above the block diagonal are not written (callers mask j > i).
#pragma once

#include "tc_common.cuh"

namespace gdr {
namespace tc {

constexpr int kInvLd = 65;   // row stride of A and T (floats)
constexpr int kInvXLd = 24;  // row stride of the per-warp 16 x 16 scratch

// sX: 3 x 16 x kInvXLd floats of scratch.  All threads of the CTA call this.
__device__ __forceinline__ void invert_unit_lower64(const float *sA, float *sT, float *sX,
                                                    int tid) {
    if (tid < 64) {
        const int b = tid >> 4, m = tid & 15, o = 16 * b;
        float s[16], x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) s[r] = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            x[j] = j < m ? 0.f : (j == m ? 1.f : -s[j]);
            if (j >= m) {
#pragma unroll
                for (int r = j + 1; r < 16; ++r)
                    s[r] = fmaf(sA[(o + r) * kInvLd + o + j], x[j], s[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(o + r) * kInvLd + o + m] = x[r];
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    for (int d = 1; d <= 3; ++d) {
        if (warp < 4 - d) {
            const int j = warp, i = warp + d;
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int k = j; k < i; ++k)
                warp_gemm16_3xtf32(acc, sA + (16 * i) * kInvLd + 16 * k, kInvLd,
                                   sT + (16 * k) * kInvLd + 16 * j, kInvLd, lane);
            float *X = sX + warp * 16 * kInvXLd;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                X[g * kInvXLd + 8 * nt + 2 * t] = acc[nt][0];
                X[g * kInvXLd + 8 * nt + 2 * t + 1] = acc[nt][1];
                X[(g + 8) * kInvXLd + 8 * nt + 2 * t] = acc[nt][2];
                X[(g + 8) * kInvXLd + 8 * nt + 2 * t + 1] = acc[nt][3];
            }
            __syncwarp();
            float tij[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            warp_gemm16_3xtf32(tij, sT + (16 * i) * kInvLd + 16 * i, kInvLd, X, kInvXLd, lane);
            float *Tij = sT + (16 * i) * kInvLd + 16 * j;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                Tij[g * kInvLd + 8 * nt + 2 * t] = -tij[nt][0];
                Tij[g * kInvLd + 8 * nt + 2 * t + 1] = -tij[nt][1];
                Tij[(g + 8) * kInvLd + 8 * nt + 2 * t] = -tij[nt][2];
                Tij[(g + 8) * kInvLd + 8 * nt + 2 * t + 1] = -tij[nt][3];
            }
        }
        __syncthreads();
    }
}

}  // namespace tc
}  // namespace gdr
