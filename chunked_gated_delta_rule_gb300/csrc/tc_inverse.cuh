// tc_inverse.cuh -- T = (I + A)^-1 for a strictly lower-triangular 64 x 64
// FP32 matrix A in shared memory (row stride kInvLd), by one CTA of 256
// threads (A4 of the chunked form: the UT transform's triangular inverse),
// in place: the array holds A on entry and T on exit.
//
//   1. invert_diag16: the four 16 x 16 diagonal blocks T_bb = (I + A_bb)^-1
//      in FP32, one thread per (block, column) (64 threads): right-looking
//      forward substitution (after x_j is known, every later row's partial
//      sum takes its A_rj x_j term), a dependent chain of 16 steps.
//   2. invert_merge, standard recursive block inversion of
//      [[T_1, 0], [A_21, T_2]]:  T_21 = -T_2 (A_21 T_1), first for the 16 x 16
//      blocks (1, 0) and (3, 2), then for the 32 x 32 block of rows 32-63,
//      columns 0-31.  Every 16 x 8 output tile of a product is one warp's
//      job on warp-level tensor cores, as three TF32 products (x = hi + lo;
//      a_hi b_hi + a_hi b_lo + a_lo b_hi, each in its own accumulator), which
//      keeps close to FP32 accuracy; tiles of a triangular factor that are
//      zero are skipped.
//
// Every block is read as A before it is written as T: each step forms its
// products from A (and blocks of T already final), then a barrier, then the
// writes.  T's entries above the diagonal of each diagonal block are written
// as 0; blocks above the block diagonal keep A's zeros.
#pragma once

#include "tc_common.cuh"

namespace gdr {
namespace tc {

constexpr int kInvLd = 68;   // row stride of A and T (floats; rows 16-B aligned)
constexpr int kInvXLd = 8;   // row stride of a warp's 16 x 8 scratch tile
constexpr int kInvYLd = 40;  // row stride of the 32 x 32 scratch product
constexpr int kInvScratchFloats = 32 * kInvYLd;  // covers 4 warps x 16 x 8 too

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

// Stores sign * (sum of the three accumulators) as a 16 x 8 row-major tile.
__device__ __forceinline__ void warp_store16x8(float *D, int ldd, const float (&hh)[4],
                                               const float (&hl)[4], const float (&lh)[4],
                                               float sign, int lane) {
    const int g = lane >> 2, t = lane & 3;
    D[g * ldd + 2 * t] = sign * ((lh[0] + hl[0]) + hh[0]);
    D[g * ldd + 2 * t + 1] = sign * ((lh[1] + hl[1]) + hh[1]);
    D[(g + 8) * ldd + 2 * t] = sign * ((lh[2] + hl[2]) + hh[2]);
    D[(g + 8) * ldd + 2 * t + 1] = sign * ((lh[3] + hl[3]) + hh[3]);
}

// Step 1: threads 0..63 only (block tid / 16, column tid % 16); named
// barrier 2 among them.
__device__ __forceinline__ void invert_diag16(float *sAT, int tid) {
    const float *sA = sAT;
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
        for (int r = j + 1; r < 16; ++r) s[r] = fmaf(sA[(o + r) * kInvLd + o + j], x[j], s[r]);
    }
    asm volatile("bar.sync 2, 64;" ::: "memory");  // every column has read A_bb
#pragma unroll
    for (int r = 0; r < 16; ++r) sAT[(o + r) * kInvLd + o + m] = x[r];
}

// Step 2: all 256 threads; the diagonal blocks must be complete (and
// visible: a barrier after step 1).  sX: kInvScratchFloats floats.  Named
// barrier 3 among warps 0-3; ends with a barrier.
__device__ __forceinline__ void invert_merge(float *sAT, float *sX, int tid) {
    const float *sA = sAT;
    float *sT = sAT;
    const int warp = tid >> 5, lane = tid & 31;
    // 16 x 16 blocks (1, 0) and (3, 2): warp = 2 (block pair) + column tile
    if (warp < 4) {
        const int j = 2 * (warp >> 1), i = j + 1, nt = warp & 1;
        float hh[4] = {0.f, 0.f, 0.f, 0.f}, hl[4] = {0.f, 0.f, 0.f, 0.f},
              lh[4] = {0.f, 0.f, 0.f, 0.f};
        warp_gemm16x8_3xtf32(hh, hl, lh, sA + (16 * i) * kInvLd + 16 * j, kInvLd,
                             sT + (16 * j) * kInvLd + 16 * j + 8 * nt, kInvLd, lane);
        float *X = sX + warp * 16 * kInvXLd;
        warp_store16x8(X, kInvXLd, hh, hl, lh, 1.f, lane);
        asm volatile("bar.sync 3, 128;" ::: "memory");  // A_ij read by both column tiles
        float th[4] = {0.f, 0.f, 0.f, 0.f}, tl[4] = {0.f, 0.f, 0.f, 0.f},
              tm[4] = {0.f, 0.f, 0.f, 0.f};
        warp_gemm16x8_3xtf32(th, tl, tm, sT + (16 * i) * kInvLd + 16 * i, kInvLd, X, kInvXLd,
                             lane);
        warp_store16x8(sT + (16 * i) * kInvLd + 16 * j + 8 * nt, kInvLd, th, tl, tm, -1.f, lane);
    }
    __syncthreads();
    // 32 x 32 block: Y = A[32:64, 0:32] T[0:32, 0:32], then T[32:64, 0:32] =
    // -T[32:64, 32:64] Y.  Warp = row block rb (16 rows) x column tile nt (8).
    const int rb = warp >> 2, nt = warp & 3;
    {
        float hh[4] = {0.f, 0.f, 0.f, 0.f}, hl[4] = {0.f, 0.f, 0.f, 0.f},
              lh[4] = {0.f, 0.f, 0.f, 0.f};
        // T[0:32, 0:32] is lower triangular: rows 0-15 vanish in columns 16-31
        for (int kb = nt >= 2 ? 1 : 0; kb < 2; ++kb)
            warp_gemm16x8_3xtf32(hh, hl, lh, sA + (32 + 16 * rb) * kInvLd + 16 * kb, kInvLd,
                                 sT + (16 * kb) * kInvLd + 8 * nt, kInvLd, lane);
        warp_store16x8(sX + (16 * rb) * kInvYLd + 8 * nt, kInvYLd, hh, hl, lh, 1.f, lane);
    }
    __syncthreads();
    {
        float hh[4] = {0.f, 0.f, 0.f, 0.f}, hl[4] = {0.f, 0.f, 0.f, 0.f},
              lh[4] = {0.f, 0.f, 0.f, 0.f};
        // T[32:64, 32:64] is lower triangular: row block 0 ends at column 15
        for (int kb = 0; kb <= rb; ++kb)
            warp_gemm16x8_3xtf32(hh, hl, lh, sT + (32 + 16 * rb) * kInvLd + 32 + 16 * kb, kInvLd,
                                 sX + (16 * kb) * kInvYLd + 8 * nt, kInvYLd, lane);
        warp_store16x8(sT + (32 + 16 * rb) * kInvLd + 8 * nt, kInvLd, hh, hl, lh, -1.f, lane);
    }
    __syncthreads();
}

// Both steps, for callers with nothing to overlap with step 1.
__device__ __forceinline__ void invert_unit_lower64(float *sAT, float *sX, int tid) {
    if (tid < 64) invert_diag16(sAT, tid);
    __syncthreads();
    invert_merge(sAT, sX, tid);
}

}  // namespace tc
}  // namespace gdr
