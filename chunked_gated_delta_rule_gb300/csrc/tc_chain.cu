// tc_chain.cu -- tensor-core path (sm_103a) of the chunked gated-delta-rule
// forward pass for BF16 q/k/v with K = V = 128, delta rule.
//
// One CTA of 256 threads runs one chain: all chunks of one (sequence, head)
// (serial scan), or of one (sequence, head, segment) (segment pre-scan and
// segment output pass).  Per 64-token chunk, everything happens on chip:
//
//   prep    D1 = [K; Q] K^T on tcgen05 (M = 128: rows 0-63 are K K^T, rows
//           64-127 are Q K^T);  A_ij = beta_i e^{G_i - G_j} (k_i . k_j), i > j;
//           T = (I + A)^-1 in FP32 (tc_inverse.cuh);
//           W^T = K^T (T diag(beta e^G))^T and U^T = V^T (T diag(beta))^T on
//           tcgen05 (A operand MN-major straight from the TMA tiles);
//           P = (Q K^T) * e^{G_i - G_j}, j <= i (BF16 operand).
//   scan    v_new^T = U^T - h^T W^T (tcgen05, A = BF16 mirror of h^T);
//           h^T <- e^{G_last} h^T + (v_new e^{G_last - G})^T K (tcgen05; the
//           canonical state is FP32 in registers).
//   output  O^T = scale [(h^T Q^T) * e^G + v_new^T P^T] (tcgen05, two FP32
//           accumulators), staged through shared memory, stored coalesced.
//
// The formulation is the transposed one (h^T, with value columns as TMEM
// lanes), so every MMA has M = 128.  Thread layout: warp w reads TMEM lanes
// 32 (w % 4) .. + 31 (its "row") and handles column half w / 4 of every
// epilogue; the state column v = row is held as 64 keys by each of the two
// threads that own row v.  Inputs arrive by TMA with 128-byte swizzle into a
// two-stage ring (the next chunk loads while this one runs); the next
// chunk's gates are prefetched into registers.  TMEM: 256 columns, regions
// reused across phases.  Waits are time-bounded: on expiry the CTA records
// GDR_ERR_TIMEOUT in the status word and leaves.
//
// Chunked form: the project statement; the state scan of fla's
// chunk_gated_delta_rule_fwd_kernel_h_blockdim64 (Kev PR #259 intro); the
// BF16 mirror used only as MMA operand with the state canonical in FP32 and
// the segment pre-scan with a K x K transition (cuLA PR #127 "Summary",
// "Root cause and implementation").
#include "gdr_internal.cuh"
#include "tc_common.cuh"
#include "tc_inverse.cuh"
#include "tma_host.cuh"

namespace gdr {
namespace {

using namespace tc;

enum TcMode { kModeSerial = 0, kModePre = 1, kModeSegOut = 2 };

struct TcArgs {
    Problem p;
    Workspace ws;
    CUtensorMap tq, tk, tv;
};

constexpr int kThreads = 256;
constexpr int kD = 128;  // K = V = 128

// Shared memory (bytes from a 1024-aligned base).
constexpr uint32_t kStage = 49152;                 // [Kb0|Qb0|Kb1|Qb1] + [Vb0|Vb1]
constexpr uint32_t kOffW = 2 * kStage;             // W tile 16 KB; B_W, B_U before it
constexpr uint32_t kOffBU = kOffW + 8192;
constexpr uint32_t kOffHm = kOffW + 16384;         // h^T mirror, K-major, 32 KB
constexpr uint32_t kOffAT = kOffHm + 32768;        // sA, sT (FP32, ld 65); then vn, vd
constexpr uint32_t kOffT = kOffAT + 64 * kInvLd * 4;
constexpr uint32_t kOffVn = kOffAT;
constexpr uint32_t kOffVd = kOffAT + 16384;
constexpr uint32_t kOffP = kOffAT + 33792;         // P tile 8 KB
constexpr uint32_t kOffX = kOffP + 8192;           // inverse scratch 3 x 16 x 24 FP32
constexpr uint32_t kOffVec = kOffX + 5120;         // per-token vectors
constexpr uint32_t kOffBar = kOffVec + 2048;
constexpr uint32_t kSmemLaunch = kOffBar + 256 + 1024;

// TMEM columns (256 allocated).
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColD1 = 0, kColO2 = 0;
constexpr uint32_t kColW = 64, kColO1 = 64;
constexpr uint32_t kColU = 128, kColH = 128;
constexpr uint32_t kColVn = 192;

constexpr uint32_t kIdescKK64 = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t kIdescMK64 = idesc_bf16(128, 64, 1, 0);
constexpr uint32_t kIdescKM64 = idesc_bf16(128, 64, 0, 1);
constexpr uint32_t kIdescKM128 = idesc_bf16(128, 128, 0, 1);

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint8_t *p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(a, b, c, d);
}

// Eight FP32 values -> one 16-byte chunk of BF16 at `p`.
__device__ __forceinline__ void st_bf16x8(uint8_t *p, const float *x) {
    st_shared_v4(p, pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                 pack_bf16x2(x[6], x[7]));
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) k_tc_chain(const __grid_constant__ TcArgs args) {
    const Problem &p = args.p;
    const Workspace &ws = args.ws;
    constexpr bool kOut = MODE != kModePre;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    float *sPart = reinterpret_cast<float *>(sm + kOffVec);
    float *sG = sPart + 64, *sBeta = sG + 64, *sBG = sBeta + 64, *sDec = sBG + 64,
          *sGam = sDec + 64;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);  // full0, full1, mma, a, h, o
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + kOffBar + 64);
    float *sA = reinterpret_cast<float *>(sm + kOffAT);
    float *sT = reinterpret_cast<float *>(sm + kOffT);
    float *sX = reinterpret_cast<float *>(sm + kOffX);

    const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int row = 32 * quad + lane_id;  // TMEM lane = matrix row
    const int H = (int)p.H;
    const int S = MODE == kModeSerial ? 1 : ws.n_segments;
    const bool trans = MODE == kModePre && blockIdx.z == 1;  // transition (M) chain
    const int s = (int)(blockIdx.x % S);
    const int64_t n = blockIdx.x / S;
    const int h = blockIdx.y;
    const int c_begin = ws.seq_chunk0[n];
    const int nc = ws.seq_chunk0[n + 1] - c_begin;
    int s0 = 0, s1 = nc;
    if (MODE != kModeSerial) {
        const int per = (nc + S - 1) / S;
        s0 = s * per;
        s1 = min(nc, s0 + per);
        if (s0 >= s1) return;
    }
    const bool needQ = kOut;
    const bool needV = !trans;
    const int4 *tab = reinterpret_cast<const int4 *>(ws.chunk_tab);

    if (warp == 0) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < 6; ++b) mbar_init(&bars[b], 1);
        mbar_init_fence();
        tma_prefetch_desc(&args.tk);
        if (needQ) tma_prefetch_desc(&args.tq);
        if (needV) tma_prefetch_desc(&args.tv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t lane = (uint32_t)(32 * quad) << 16;

    // Canonical state: column v = row of h, keys [64 half, 64 half + 64).
    const int64_t seg_base = (n * H + h) * (int64_t)S + s;
    const int kbase = 64 * half;
    float hr[64];
#pragma unroll
    for (int kk = 0; kk < 64; ++kk) {
        const int key = kbase + kk;
        float x = 0.f;
        if (MODE == kModeSerial) {
            if (p.h0) x = p.h0[((n * H + h) * kD + key) * kD + row];
        } else if (MODE == kModeSegOut) {
            x = ws.segH[(seg_base * kD + key) * kD + row];
        } else if (trans) {
            x = key == row ? 1.f : 0.f;
        }
        hr[kk] = x;
    }
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8)
        st_bf16x8(sm + kOffHm + sw128_off(row, kbase + 8 * c8, 128), hr + 8 * c8);
    fence_async_smem();

    auto issue_tma = [&](int cc, int stage) {
        const int tt = tab[c_begin + cc].y;
        uint64_t *bar = &bars[stage];
        uint8_t *dst = sm + stage * kStage;
        mbar_arrive_expect_tx(bar, 32768u - (needQ ? 0u : 16384u) + (needV ? 16384u : 0u));
        tma_load_3d(dst, &args.tk, bar, 0, h, tt);
        tma_load_3d(dst + 16384, &args.tk, bar, 64, h, tt);
        if (needQ) {
            tma_load_3d(dst + 8192, &args.tq, bar, 0, h, tt);
            tma_load_3d(dst + 24576, &args.tq, bar, 64, h, tt);
        }
        if (needV) {
            tma_load_3d(dst + 32768, &args.tv, bar, 0, h, tt);
            tma_load_3d(dst + 40960, &args.tv, bar, 64, h, tt);
        }
    };
    // gates of the first chunk; later chunks' gates are prefetched one chunk
    // ahead in registers
    float g_next = 0.f, b_next = 0.f;
    if (s0 < s1 && tid < 64) {
        const int4 e0 = tab[c_begin + s0];
        if (tid < e0.z) {
            g_next = p.g[((int64_t)e0.y + tid) * H + h];
            b_next = p.beta[((int64_t)e0.y + tid) * H + h];
        }
    }
    if (tid == 0 && s0 < s1) issue_tma(s0, 0);
    uint32_t ph_mma = 0, ph_a = 0, ph_h = 0, ph_o = 0;
    bool failed = false;
    __syncthreads();

    for (int cc = s0; cc < s1; ++cc) {
        const int it = cc - s0, stage = it & 1;
        const int4 e = tab[c_begin + cc];
        const int64_t t0 = e.y;
        const int len = e.z;
        uint8_t *st = sm + stage * kStage;
        const uint32_t sta = sb + stage * kStage;
        if (tid == 0 && cc + 1 < s1) issue_tma(cc + 1, stage ^ 1);

        // A2: chunk-local inclusive cumsum of the log gate (padded: g = beta = 0),
        // a fixed-order warp scan over tokens 0-31 and 32-63.
        const float gcur = g_next, bcur = b_next;
        if (tid < 64) {
            if (cc + 1 < s1) {
                const int4 en = tab[c_begin + cc + 1];
                g_next = tid < en.z ? p.g[((int64_t)en.y + tid) * H + h] : 0.f;
                b_next = tid < en.z ? p.beta[((int64_t)en.y + tid) * H + h] : 0.f;
            }
            float x = gcur;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane_id >= off) x += y;
            }
            sPart[tid] = x;
            sBeta[tid] = bcur;
        }
        __syncthreads();
        if (tid < 64) sG[tid] = tid < 32 ? sPart[tid] : sPart[tid] + sPart[31];
        __syncthreads();
        const float gl = sG[len - 1];
        if (tid < 64) {
            const float gm = __expf(sG[tid]);
            sGam[tid] = gm;
            sBG[tid] = sBeta[tid] * gm;
            sDec[tid] = __expf(gl - sG[tid]);
        }
        const float gam_last = __expf(gl);

        bool ok = mbar_wait(&bars[stage], (uint32_t)(it >> 1) & 1u, p.status);
        if (__syncthreads_or(!ok)) { failed = true; break; }
        if (len < 64) {  // rows past the sequence end belong to the next one: zero them
            const int rows = 64 - len;
            for (int idx = tid; idx < rows * 6 * 8; idx += kThreads) {
                const int r = len + idx / 48, blk = (idx / 8) % 6, c16 = idx & 7;
                st_shared_v4(st + blk * 8192 + r * 128 + c16 * 16, 0u, 0u, 0u, 0u);
            }
            fence_async_smem();
        }
        __syncthreads();

        // A3 (+ Q K^T): D1 = [K; Q] K^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a = sta + (kk >> 2) * 16384 + (kk & 3) * 32;
                umma_bf16(tmem + kColD1, sdesc_sw128(a, 16, 1024), sdesc_sw128(a, 16, 1024),
                          kIdescKK64, kk > 0);
            }
            umma_commit(&bars[2]);
        }
        ok = mbar_wait(&bars[2], ph_mma, p.status);
        ph_mma ^= 1;
        if (__syncthreads_or(!ok)) { failed = true; break; }
        tc_fence_after();
        if (quad < 2 || kOut) {
            float f[32];
            tmem_load32f(tmem + lane + kColD1 + 32 * half, f);
            const int i = row & 63;
            const float gi = sG[i];
            if (quad < 2) {  // row i of A (strictly lower)
                const float bi = sBeta[i];
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int j = 32 * half + u;
                    sA[i * kInvLd + j] = j < i ? bi * __expf(gi - sG[j]) * f[u] : 0.f;
                }
            } else {  // row i of P (lower, diagonal included)
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int j = 32 * half + u;
                    f[u] = j <= i ? f[u] * __expf(gi - sG[j]) : 0.f;
                }
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8)
                    st_bf16x8(sm + kOffP + sw128_off(i, 32 * half + 8 * c8, 64), f + 8 * c8);
            }
        }
        tc_fence_before();
        __syncthreads();

        // A4: T = (I + A)^-1
        invert_unit_lower64(sA, sT, sX, tid);

        // A5 operands: rows of T diag(beta e^G) (rows 0-63) and T diag(beta)
        // (rows 64-127), BF16, columns [32 half, 32 half + 32).
        if (quad < 2 || !trans) {
            const int i = row & 63;
            const float *scale_vec = quad < 2 ? sBG : sBeta;
            uint8_t *dst = sm + (quad < 2 ? kOffW : kOffBU);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                float x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = 32 * half + 8 * c8 + u;
                    x[u] = j <= i ? sT[i * kInvLd + j] * scale_vec[j] : 0.f;
                }
                st_bf16x8(dst + sw128_off(i, 32 * half + 8 * c8, 64), x);
            }
        }
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                umma_bf16(tmem + kColW, sdesc_sw128(sta + kk * 2048, 16384, 1024),
                          sdesc_sw128(sb + kOffW + kk * 32, 16, 1024), kIdescMK64, kk > 0);
            if (!trans) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(tmem + kColU, sdesc_sw128(sta + 32768 + kk * 2048, 8192, 1024),
                              sdesc_sw128(sb + kOffBU + kk * 32, 16, 1024), kIdescMK64, kk > 0);
            }
            umma_commit(&bars[2]);
        }
        ok = mbar_wait(&bars[2], ph_mma, p.status);
        ph_mma ^= 1;
        if (__syncthreads_or(!ok)) { failed = true; break; }
        tc_fence_after();
        {  // W tile, MN-major [key][t]: row = key, t in [32 half, 32 half + 32)
            float f[32];
            tmem_load32f(tmem + lane + kColW + 32 * half, f);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8)
                st_bf16x8(sm + kOffW + sw128_off(row, 32 * half + 8 * c8, 128), f + 8 * c8);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // A6: v_new^T = U^T - h^T W^T   (and O1 = h^T Q^T for the output)
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                umma_bf16(tmem + kColVn,
                          sdesc_sw128(sb + kOffHm + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                          sdesc_sw128(sb + kOffW + kk * 2048, 8192, 1024), kIdescKM64, kk > 0);
            umma_commit(&bars[3]);
            if (kOut) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_bf16(tmem + kColO1,
                              sdesc_sw128(sb + kOffHm + (kk >> 2) * 16384 + (kk & 3) * 32, 16,
                                          1024),
                              sdesc_sw128(sta + 8192 + (kk >> 2) * 16384 + (kk & 3) * 32, 16,
                                          1024),
                              kIdescKK64, kk > 0);
            }
        }
        ok = mbar_wait(&bars[3], ph_a, p.status);
        ph_a ^= 1;
        if (__syncthreads_or(!ok)) { failed = true; break; }
        tc_fence_after();
        {
            float w[32], u[32];
            tmem_load32f(tmem + lane + kColVn + 32 * half, w);
            if (!trans) {
                tmem_load32f(tmem + lane + kColU + 32 * half, u);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) u[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                u[i] -= w[i];                        // v_new
                w[i] = u[i] * sDec[32 * half + i];   // v_new e^{G_last - G}
            }
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                st_bf16x8(sm + kOffVn + sw128_off(row, 32 * half + 8 * c8, 128), u + 8 * c8);
                st_bf16x8(sm + kOffVd + sw128_off(row, 32 * half + 8 * c8, 128), w + 8 * c8);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // h^T update product, and O2 = v_new^T P^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                umma_bf16(tmem + kColH, sdesc_sw128(sb + kOffVd + kk * 32, 16, 1024),
                          sdesc_sw128(sta + kk * 2048, 16384, 1024), kIdescKM128, kk > 0);
            umma_commit(&bars[4]);
            if (kOut) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(tmem + kColO2, sdesc_sw128(sb + kOffVn + kk * 32, 16, 1024),
                              sdesc_sw128(sb + kOffP + kk * 32, 16, 1024), kIdescKK64, kk > 0);
                umma_commit(&bars[5]);
            }
        }
        ok = mbar_wait(&bars[4], ph_h, p.status);
        ph_h ^= 1;
        if (__syncthreads_or(!ok)) { failed = true; break; }
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float f[32];
            tmem_load32f(tmem + lane + kColH + kbase + 32 * q, f);
#pragma unroll
            for (int i = 0; i < 32; ++i) hr[32 * q + i] = fmaf(gam_last, hr[32 * q + i], f[i]);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8)
                st_bf16x8(sm + kOffHm + sw128_off(row, kbase + 32 * q + 8 * c8, 128),
                          hr + 32 * q + 8 * c8);
        }
        fence_async_smem();

        // A7: output rows of this chunk.
        if (kOut) {
            ok = mbar_wait(&bars[5], ph_o, p.status);
            ph_o ^= 1;
            if (__syncthreads_or(!ok)) { failed = true; break; }
            tc_fence_after();
            uint8_t *stage_o = st + 32768;  // V tile is free after the U product
            {
                float o1[32], o2[32];
                tmem_load32f(tmem + lane + kColO1 + 32 * half, o1);
                tmem_load32f(tmem + lane + kColO2 + 32 * half, o2);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int t = 32 * half + i;
                    const float y = p.scale * fmaf(sGam[t], o1[i], o2[i]);
                    *reinterpret_cast<__nv_bfloat16 *>(stage_o + t * 256 + row * 2) =
                        __float2bfloat16_rn(y);
                }
            }
            tc_fence_before();
            __syncthreads();
            __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int idx = tid + kThreads * r;
                const int t = idx >> 4, c16 = idx & 15;
                if (t < len)
                    *reinterpret_cast<uint4 *>(o + ((t0 + t) * H + h) * (int64_t)kD + c16 * 8) =
                        *reinterpret_cast<const uint4 *>(stage_o + t * 256 + c16 * 16);
            }
            fence_async_smem();
        }
        tc_fence_before();
        __syncthreads();
    }

    if (!failed) {
        if (MODE == kModeSerial && p.ht) {
#pragma unroll
            for (int kk = 0; kk < 64; ++kk)
                p.ht[((n * H + h) * kD + kbase + kk) * kD + row] = hr[kk];
        } else if (MODE == kModePre && trans) {  // M_s stored transposed: row `row`
            float4 *dst =
                reinterpret_cast<float4 *>(ws.segM + (seg_base * kD + row) * kD + kbase);
#pragma unroll
            for (int k4 = 0; k4 < 16; ++k4)
                dst[k4] = make_float4(hr[4 * k4], hr[4 * k4 + 1], hr[4 * k4 + 2], hr[4 * k4 + 3]);
        } else if (MODE == kModePre) {
#pragma unroll
            for (int kk = 0; kk < 64; ++kk)
                ws.segC[(seg_base * kD + kbase + kk) * kD + row] = hr[kk];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int MODE>
cudaError_t launch_chain(const TcArgs &args, dim3 grid, cudaStream_t st) {
    cudaError_t err = cudaFuncSetAttribute(k_tc_chain<MODE>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemLaunch);
    if (err != cudaSuccess) return err;
    k_tc_chain<MODE><<<grid, kThreads, kSmemLaunch, st>>>(args);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(const Problem &p) {
    auto al = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
    return p.dtype == GDR_BF16 && p.K == kD && p.V == kD && p.beta != nullptr && al(p.q) &&
           al(p.k) && al(p.v) && al(p.o);
}

cudaError_t tc_chain(const Problem &p, const Workspace &ws, int mode, cudaStream_t st) {
    TcArgs args;
    args.p = p;
    args.ws = ws;
    const uint64_t rows = (uint64_t)p.B * (uint64_t)p.T;
    const uint64_t H = (uint64_t)p.H;
    if (!make_tmap_bf16_3d(&args.tq, p.q, kD, H, rows, kD * 2, H * kD * 2, 64, 1, 64) ||
        !make_tmap_bf16_3d(&args.tk, p.k, kD, H, rows, kD * 2, H * kD * 2, 64, 1, 64) ||
        !make_tmap_bf16_3d(&args.tv, p.v, kD, H, rows, kD * 2, H * kD * 2, 64, 1, 64))
        return cudaErrorInvalidValue;
    const int S = mode == 0 ? 1 : ws.n_segments;
    dim3 grid((unsigned)(p.N * S), (unsigned)p.H, mode == 1 ? 2u : 1u);
    switch (mode) {
    case 0: return launch_chain<kModeSerial>(args, grid, st);
    case 1: return launch_chain<kModePre>(args, grid, st);
    case 2: return launch_chain<kModeSegOut>(args, grid, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdr
