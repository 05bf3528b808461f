// tc_chunk.cuh -- pieces shared by the tensor-core prep and scan kernels:
// the per-chunk record the prep kernel leaves for the scan kernel, BF16
// packing, and the per-chunk gate vectors.
#pragma once

#include "tc_common.cuh"

namespace gdr {
namespace tc {

constexpr int kD = 128;  // K = V = 128 on the tensor-core path

// One record per (chunk, head): the byte image of the scan kernel's
// shared-memory stage, so that bulk copies load it.  BF16 tiles of 64
// columns in the 128-byte swizzled layout (sw128_off, 64 rows per 8 KB
// block unless noted):
//   [0, 16 KB)      W^T, 128 rows: row k holds W[t][k] for t = 0..63 (the
//                   MN-major B operand of h^T W^T)
//   [16 KB, 32 KB)  Q~ block 0 | Q~ block 1: row t of block b holds
//                   Q~[t][64 b .. 64 b + 63] (K-major), Q~ = scale e^{G_t} q_t
//   [32 KB, 48 KB)  not written: the scan kernel loads k there and forms
//                   K~ = e^{G_last - G_t} k_t in place
//   [48 KB, 56 KB)  scale P: row i holds scale P[i][j] for j = 0..63, where
//                   P = (Q K^T * e^{G_i - G_j}, j <= i)
//   [56 KB, 72 KB)  U^T, 128 rows: row v holds U[t][v] for t = 0..63
//   [72 KB, +272 B) FP32 G_last, e^{G_last}, two unused floats, then
//                   e^{G_last - G_t} for t = 0..63
// Padded tokens (past a sequence end) have zero W, Q~, U and P entries and
// zero decay: every later product with them adds exact zeros.
constexpr uint32_t kImgW = 0, kImgQ = 16384, kImgK = 32768, kImgP = 49152, kImgU = 57344, kImgVec = 73728;
constexpr uint32_t kImgDec = kImgVec + 16;      // the 64 decay factors
constexpr uint32_t kImgBytes = kImgDec + 256;   // bytes of one stage image (74,000)
constexpr uint32_t kRecBytes = 74752;           // record stride (1 KB aligned); gdr_api.cu sizes it
constexpr int kImgGamLast = 1;                  // float index of e^{G_last} at kImgVec

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint8_t *p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(a, b, c, d);
}

// Eight FP32 values -> one 16-byte chunk of BF16 at `p` (shared or global).
__device__ __forceinline__ void st_bf16x8(void *p, const float *x) {
    *reinterpret_cast<uint4 *>(p) =
        make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                   pack_bf16x2(x[6], x[7]));
}

// Eight FP32 values -> the BF16 chunk of their rounded values at `hi` and of
// the rounded remainders x - hi at `lo` (shared or global): the pair carries
// about 16 significant bits of x.
__device__ __forceinline__ void st_split_bf16x8(void *hi, void *lo, const float *x) {
    float h[8], l[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        h[u] = __bfloat162float(__float2bfloat16_rn(x[u]));
        l[u] = x[u] - h[u];
    }
    st_bf16x8(hi, h);
    st_bf16x8(lo, l);
}

// Eight BF16 of a 16-byte chunk -> FP32.
__device__ __forceinline__ void ld_bf16x8(const void *p, float *x) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
        const float2 f = __bfloat1622float2(b);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

// Per-chunk gate vectors (A2) from one warp: lane l holds the log gates and
// betas of tokens 2l and 2l + 1 (zero past `len`).  Fixed-order scan: pair
// sums scanned across lanes.  Layout of v (kGateFloats floats):
//   [0,64) G   [64,128) beta   [128,192) beta e^G   [192,256) e^{G_last - G}
//   [256,320) e^G   [320,384) e^{G - G_last}
//   [384] G_last  [385] e^{G_last}  [386] 1 if every |G_t - G_last| < 80
//   (then e^{G_i - G_j} = e^{G_i - G_last} e^{G_last - G_j} neither
//   overflows nor underflows), else 0.
constexpr int kGateFloats = 392;

__device__ __forceinline__ void gate_vectors(float *v, const float (&g2)[2], const float (&b2)[2],
                                             int len, int lane_id) {
    float *sG = v, *sBeta = v + 64, *sBG = v + 128, *sDec = v + 192, *sGam = v + 256,
          *sEP = v + 320, *sScal = v + 384;
    float x = g2[0] + g2[1];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane_id >= off) x += y;
    }
    float excl = __shfl_up_sync(0xffffffffu, x, 1);
    if (lane_id == 0) excl = 0.f;
    const float G0 = excl + g2[0], G1 = G0 + g2[1];
    sG[2 * lane_id] = G0;
    sG[2 * lane_id + 1] = G1;
    sBeta[2 * lane_id] = b2[0];
    sBeta[2 * lane_id + 1] = b2[1];
    __syncwarp();
    const float glast = sG[len - 1];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int tok = 2 * lane_id + u;
        const float Gt = u ? G1 : G0;
        const float gm = __expf(Gt);
        sGam[tok] = gm;
        sBG[tok] = b2[u] * gm;
        sDec[tok] = __expf(glast - Gt);
        sEP[tok] = __expf(Gt - glast);
    }
    float spread = fmaxf(fabsf(G0 - glast), fabsf(G1 - glast));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        spread = fmaxf(spread, __shfl_xor_sync(0xffffffffu, spread, off));
    if (lane_id == 0) {
        sScal[0] = glast;
        sScal[1] = __expf(glast);
        sScal[2] = spread < 80.f ? 1.f : 0.f;
    }
    __syncwarp();
}

}  // namespace tc
}  // namespace gdr
