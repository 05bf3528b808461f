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
//           canonical state is FP32 in TMEM).
//   output  O^T = scale [(h^T Q^T) * e^G + v_new^T P^T] (tcgen05, two FP32
//           accumulators), staged through shared memory, stored coalesced.
//
// The formulation is the transposed one (h^T, with value columns as TMEM
// lanes), so every MMA has M = 128.  Thread layout: warp w reads TMEM lanes
// 32 (w % 4) .. + 31 (its "row") and handles column half w / 4 of every
// epilogue; the state column v = row is TMEM lane v, 64 keys per thread.  Inputs arrive by TMA with 128-byte swizzle into a
// two-stage ring (the next chunk loads while this one runs); the next
// chunk's gates are prefetched into registers.  TMEM: accumulator regions
// reused across phases, plus the FP32 state.  Waits are time-bounded: on expiry the CTA records
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
constexpr uint32_t kOffAT = kOffHm + 32768;        // sA, sT (FP32, ld 68); then vn, vd
constexpr uint32_t kOffT = kOffAT + 64 * kInvLd * 4;
constexpr uint32_t kOffVn = kOffAT;
constexpr uint32_t kOffVd = kOffAT + 16384;
constexpr uint32_t kOffP = kOffAT + 34816;         // P tile 8 KB
constexpr uint32_t kOffX = kOffP + 8192;           // inverse scratch (3 KB)
constexpr uint32_t kOffVec = kOffX + 5120;         // per-token vectors, 2 buffers
constexpr int kVecFloats = 392;                    // 6 x 64 + 8 scalars
constexpr uint32_t kOffBar = kOffVec + 4096;
constexpr uint32_t kSmemLaunch = kOffBar + 256 + 1024;

// TMEM columns (512 allocated; one CTA per SM).  The canonical FP32 state
// h^T lives in columns [256, 384): lane v, column key.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColD1 = 0, kColO2 = 0;
constexpr uint32_t kColW = 64, kColO1 = 64;
constexpr uint32_t kColU = 128, kColH = 128;
constexpr uint32_t kColVn = 192;
constexpr uint32_t kColS = 256;

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

// Gate vectors of one chunk from one warp: lane l holds the log gates and
// betas of tokens 2l and 2l + 1 (zero past `len`).  Fixed-order scan: pair
// sums scanned across lanes.  Writes G, beta, beta e^G, e^{G_last - G},
// e^G, e^{G - G_last} and [G_last, e^{G_last}, factorisation flag].
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
}

// One chain of the work list: (sequence n, segment s, head h[, transition]).
struct Chain {
    int64_t n;
    int h, s;
    bool trans;
    int c_begin, s0, s1;
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) k_tc_chain(const __grid_constant__ TcArgs args) {
    const Problem &p = args.p;
    const Workspace &ws = args.ws;
    constexpr bool kOut = MODE != kModePre;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    float *vecbase = reinterpret_cast<float *>(sm + kOffVec);  // 2 x kVecFloats
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);  // full0, full1, mma, a, h, o
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + kOffBar + 64);
    int *s_ctl = reinterpret_cast<int *>(sm + kOffBar + 128);  // current, next chain
    float *sA = reinterpret_cast<float *>(sm + kOffAT);
    float *sT = reinterpret_cast<float *>(sm + kOffT);
    float *sX = reinterpret_cast<float *>(sm + kOffX);

    const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int row = 32 * quad + lane_id;  // TMEM lane = matrix row
    const int H = (int)p.H;
    const int S = MODE == kModeSerial ? 1 : ws.n_segments;
    const int kinds = MODE == kModePre ? 2 : 1;
    const int total = (int)(p.N * S * H * kinds);
    int32_t *counter = ws.n_chunks + 1 + MODE;
    const int4 *tab = reinterpret_cast<const int4 *>(ws.chunk_tab);

    // Work list: heads fastest, then (transition kind), segment, and the
    // sequences longest first.
    auto decode = [&](int id, Chain &c) {
        int r = id;
        c.h = r % H;
        r /= H;
        c.trans = false;
        if (MODE == kModePre) {
            c.trans = (r & 1) != 0;
            r >>= 1;
        }
        c.s = r % S;
        r /= S;
        c.n = ws.seq_order[r];
        c.c_begin = ws.seq_chunk0[c.n];
        const int nc = ws.seq_chunk0[c.n + 1] - c.c_begin;
        c.s0 = 0;
        c.s1 = nc;
        if (MODE != kModeSerial) {
            const int per = (nc + S - 1) / S;
            c.s0 = c.s * per;
            c.s1 = min(nc, c.s0 + per);
        }
    };
    // Thread 0: next chain with work (empty segments are skipped), or total.
    auto fetch = [&]() -> int {
        while (true) {
            const int id = atomicAdd(counter, 1);
            if (id >= total) return total;
            Chain c;
            decode(id, c);
            if (c.s0 < c.s1) return id;
        }
    };

    if (warp == 0) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < 6; ++b) mbar_init(&bars[b], 1);
        mbar_init_fence();
        tma_prefetch_desc(&args.tk);
        if (kOut) tma_prefetch_desc(&args.tq);
        tma_prefetch_desc(&args.tv);
        s_ctl[0] = fetch();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t lane = (uint32_t)(32 * quad) << 16;
    const int kbase = 64 * half;

    auto issue_tma = [&](const Chain &c, int cc, int stage) {
        const int tt = tab[c.c_begin + cc].y;
        const bool needQ = kOut, needV = !c.trans;
        uint64_t *bar = &bars[stage];
        uint8_t *dst = sm + stage * kStage;
        mbar_arrive_expect_tx(bar, 32768u - (needQ ? 0u : 16384u) + (needV ? 16384u : 0u));
        tma_load_3d(dst, &args.tk, bar, 0, c.h, tt);
        tma_load_3d(dst + 16384, &args.tk, bar, 64, c.h, tt);
        if (needQ) {
            tma_load_3d(dst + 8192, &args.tq, bar, 0, c.h, tt);
            tma_load_3d(dst + 24576, &args.tq, bar, 64, c.h, tt);
        }
        if (needV) {
            tma_load_3d(dst + 32768, &args.tv, bar, 0, c.h, tt);
            tma_load_3d(dst + 40960, &args.tv, bar, 64, c.h, tt);
        }
    };
    // gates of a chunk into registers (a warp: tokens 2 lane, 2 lane + 1)
    float gq[2] = {0.f, 0.f}, bq[2] = {0.f, 0.f};
    auto load_gates = [&](const Chain &c, int cc) {
        const int4 en = tab[c.c_begin + cc];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int tok = 2 * lane_id + u;
            gq[u] = tok < en.z ? p.g[((int64_t)en.y + tok) * H + c.h] : 0.f;
            bq[u] = tok < en.z ? p.beta[((int64_t)en.y + tok) * H + c.h] : 0.f;
        }
    };

    int cur = s_ctl[0];
    uint32_t gk = 0;  // chunks processed by this CTA: stage, parity, vector buffer
    uint32_t ph_mma = 0, ph_a = 0, ph_h = 0, ph_o = 0;
    bool failed = false;
    if (cur < total) {  // first chunk of the first chain: tiles and gate vectors
        Chain c;
        decode(cur, c);
        if (tid == 0) issue_tma(c, c.s0, 0);
        if (warp == 0) {
            load_gates(c, c.s0);
            gate_vectors(vecbase, gq, bq, tab[c.c_begin + c.s0].z, lane_id);
        }
    }

    while (cur < total) {
        Chain C;
        decode(cur, C);
        if (tid == 0) s_ctl[1] = fetch();
        const int h = C.h;
        const bool trans = C.trans;
        const int64_t seg_base = (C.n * H + h) * (int64_t)S + C.s;

        // Canonical state: column v = row of h, keys [64 half, 64 half + 64),
        // FP32 in TMEM; its BF16 mirror (the MMA operand) in shared memory.
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float hv[32];
#pragma unroll
            for (int kk = 0; kk < 32; ++kk) {
                const int key = kbase + 32 * q + kk;
                float x = 0.f;
                if (MODE == kModeSerial) {
                    if (p.h0) x = p.h0[((C.n * H + h) * kD + key) * kD + row];
                } else if (MODE == kModeSegOut) {
                    x = ws.segH[(seg_base * kD + key) * kD + row];
                } else if (trans) {
                    x = key == row ? 1.f : 0.f;
                }
                hv[kk] = x;
            }
            tmem_store32f(tmem + lane + kColS + kbase + 32 * q, hv);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8)
                st_bf16x8(sm + kOffHm + sw128_off(row, kbase + 32 * q + 8 * c8, 128),
                          hv + 8 * c8);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        const int nxt = s_ctl[1];
        Chain Cn;
        if (nxt < total) decode(nxt, Cn);

        for (int cc = C.s0; cc < C.s1; ++cc, ++gk) {
            const int stage = gk & 1;
            const int4 e = tab[C.c_begin + cc];
            const int64_t t0 = e.y;
            const int len = e.z;
            uint8_t *st = sm + stage * kStage;
            const uint32_t sta = sb + stage * kStage;
            const float *vb = vecbase + (gk & 1) * kVecFloats;
            const float *sG = vb, *sBeta = vb + 64, *sBG = vb + 128, *sDec = vb + 192,
                        *sGam = vb + 256, *sEP = vb + 320, *sScal = vb + 384;
            // the chunk after this one: next in this chain, or the next chain's first
            const bool follow_here = cc + 1 < C.s1;
            const bool has_follow = follow_here || nxt < total;
            const Chain *F = follow_here ? &C : &Cn;
            const int fcc = follow_here ? cc + 1 : Cn.s0;
            if (warp == 1 && has_follow) load_gates(*F, fcc);

            bool ok = mbar_wait(&bars[stage], (gk >> 1) & 1u, p.status);
            if (__syncthreads_or(!ok)) { failed = true; break; }
            const float gam_last = sScal[1];
            // e^{G_i - G_j} = e^{G_i - G_last} e^{G_last - G_j} when every
            // |G_i - G_last| of the chunk is below 80 (no overflow or
            // underflow); otherwise the direct exponential.
            const bool fact = sScal[2] != 0.f;
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
                if (has_follow) issue_tma(*F, fcc, stage ^ 1);
            }
            ok = mbar_wait(&bars[2], ph_mma, p.status);
            ph_mma ^= 1;
            if (__syncthreads_or(!ok)) { failed = true; break; }
            tc_fence_after();
            if (quad < 2 || kOut) {
                float f[32];
                tmem_load32f(tmem + lane + kColD1 + 32 * half, f);
                const int i = row & 63;
                const int j0 = 32 * half;
                // A rows keep j < i (beta_i folded in); P rows keep j <= i.
                const int jlim = quad < 2 ? i : i + 1;
                const float rowf = quad < 2 ? sBeta[i] : 1.f;
                if (fact) {
                    const float ri = rowf * sEP[i];
    #pragma unroll
                    for (int u = 0; u < 32; ++u)
                        f[u] = (j0 + u < jlim) ? f[u] * (ri * sDec[j0 + u]) : 0.f;
                } else {
                    const float gi = sG[i];
    #pragma unroll
                    for (int u = 0; u < 32; ++u)
                        f[u] = (j0 + u < jlim) ? f[u] * (rowf * __expf(gi - sG[j0 + u])) : 0.f;
                }
                if (quad < 2) {  // row i of A (strictly lower), FP32
    #pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4)
                        *reinterpret_cast<float4 *>(sA + i * kInvLd + j0 + 4 * c4) =
                            make_float4(f[4 * c4], f[4 * c4 + 1], f[4 * c4 + 2], f[4 * c4 + 3]);
                } else {  // row i of P (lower, diagonal included), BF16
    #pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8)
                        st_bf16x8(sm + kOffP + sw128_off(i, j0 + 8 * c8, 64), f + 8 * c8);
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
                    const int j0 = 32 * half + 8 * c8;
                    const float4 t0 = *reinterpret_cast<const float4 *>(sT + i * kInvLd + j0);
                    const float4 t1 = *reinterpret_cast<const float4 *>(sT + i * kInvLd + j0 + 4);
                    const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
                    float x[8];
    #pragma unroll
                    for (int u = 0; u < 8; ++u)
                        x[u] = j0 + u <= i ? tv[u] * scale_vec[j0 + u] : 0.f;
                    st_bf16x8(dst + sw128_off(i, j0, 64), x);
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
            // Gate vectors of the following chunk (warp 1, while v_new's product runs).
            if (warp == 1 && has_follow) {
                const int4 ef = tab[F->c_begin + fcc];
                gate_vectors(vecbase + ((gk + 1) & 1) * kVecFloats, gq, bq, ef.z, lane_id);
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
                float f[32], hv[32];
                tmem_load32f(tmem + lane + kColH + kbase + 32 * q, f);
                tmem_load32f(tmem + lane + kColS + kbase + 32 * q, hv);
    #pragma unroll
                for (int i = 0; i < 32; ++i) hv[i] = fmaf(gam_last, hv[i], f[i]);
                tmem_store32f(tmem + lane + kColS + kbase + 32 * q, hv);
    #pragma unroll
                for (int c8 = 0; c8 < 4; ++c8)
                    st_bf16x8(sm + kOffHm + sw128_off(row, kbase + 32 * q + 8 * c8, 128),
                              hv + 8 * c8);
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
            if (failed) break;
            if ((MODE != kModeSegOut) && (MODE != kModeSerial || p.ht)) {
            tc_fence_after();
    #pragma unroll
            for (int q = 0; q < 2; ++q) {
                float hv[32];
                tmem_load32f(tmem + lane + kColS + kbase + 32 * q, hv);
                if (MODE == kModeSerial) {
    #pragma unroll
                    for (int kk = 0; kk < 32; ++kk)
                        p.ht[((C.n * H + h) * kD + kbase + 32 * q + kk) * kD + row] = hv[kk];
                } else if (trans) {  // M_s stored transposed: row `row`
                    float4 *dst = reinterpret_cast<float4 *>(ws.segM + (seg_base * kD + row) * kD +
                                                             kbase + 32 * q);
    #pragma unroll
                    for (int k4 = 0; k4 < 8; ++k4)
                        dst[k4] = make_float4(hv[4 * k4], hv[4 * k4 + 1], hv[4 * k4 + 2],
                                              hv[4 * k4 + 3]);
                } else {
    #pragma unroll
                    for (int kk = 0; kk < 32; ++kk)
                        ws.segC[(seg_base * kD + kbase + 32 * q + kk) * kD + row] = hv[kk];
                }
            }
        }
        cur = nxt;
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
    const int64_t chains = p.N * S * p.H * (mode == 1 ? 2 : 1);
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    dim3 grid((unsigned)(chains < sms ? chains : sms));
    switch (mode) {
    case 0: return launch_chain<kModeSerial>(args, grid, st);
    case 1: return launch_chain<kModePre>(args, grid, st);
    case 2: return launch_chain<kModeSegOut>(args, grid, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdr
