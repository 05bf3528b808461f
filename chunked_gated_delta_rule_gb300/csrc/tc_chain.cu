// tc_chain.cu -- A6/A7 (and A8/A10 of the segment split) on the tensor-core
// path (BF16, K = V = 128, delta rule): the serial state scan and the output.
//
// Persistent CTAs (one per SM, 256 threads) pull chains -- all chunks of one
// (sequence, head), or of one (sequence, segment, head) -- longest first from
// an atomic counter.  Everything that does not depend on the state was done
// by tc_prep.cu for all chunks in parallel and left in one record per
// (chunk, head); here, per chunk, in order:
//
//   v_new^T = U^T - h^T W^T           (tcgen05, A = BF16 mirror of h^T)
//   h^T <- e^{G_last} h^T + (v_new e^{G_last - G})^T K   (tcgen05; the
//                                      canonical state is FP32 in TMEM)
//   O^T = scale [(h^T Q^T) * e^G + v_new^T P^T]   (tcgen05, staged, stored)
//
// The formulation is the transposed one (value columns are TMEM lanes), so
// every MMA has M = 128.  Warp w reads TMEM lanes 32 (w % 4) .. + 31 (its
// "row") and handles column half w / 4 of every epilogue.  K, Q and the
// record's W, U^T, P and decay vectors arrive by TMA / bulk copy with
// 128-byte swizzle into a two-stage ring (the next chunk, possibly of the
// next chain, loads while this one runs).  Waits are time-bounded: on expiry
// the CTA records GDR_ERR_TIMEOUT in the status word and leaves.
//
// Chunked form: the project statement; the state scan of fla's
// chunk_gated_delta_rule_fwd_kernel_h_blockdim64 (Kev PR #259 intro); the
// BF16 mirror used only as MMA operand with the state canonical in FP32 and
// the segment pre-scan with a K x K transition (cuLA PR #127 "Summary",
// "Root cause and implementation").
#include "gdr_internal.cuh"
#include "tc_chunk.cuh"
#include "tma_host.cuh"

namespace gdr {
namespace {

using namespace tc;

enum TcMode { kModeSerial = 0, kModePre = 1, kModeSegOut = 2 };

struct TcArgs {
    Problem p;
    Workspace ws;
    CUtensorMap tq, tk, trec128, trec64;
};

constexpr int kThreads = 256;

// Shared memory (bytes from a 1024-aligned base).  One stage:
//   [Kb0|Qb0|Kb1|Qb1] 32 KB, W 16 KB, U^T 16 KB, P 8 KB, vectors 1 KB.
constexpr uint32_t kStW = 32768, kStU = 49152, kStP = 65536, kStVec = 73728;
constexpr uint32_t kStage = 75776;
constexpr uint32_t kOffHm = 2 * kStage;            // h^T mirror, K-major, 32 KB
constexpr uint32_t kOffVn = kOffHm + 32768;        // v_new^T tile; output staging after
constexpr uint32_t kOffVd = kOffVn + 16384;        // (v_new e^{G_last - G})^T tile
constexpr uint32_t kOffBar = kOffVd + 16384;
constexpr uint32_t kSmemLaunch = kOffBar + 256 + 1024;

// TMEM columns (512 allocated; one CTA per SM).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColVn = 0, kColO2 = 0;  // O2 after v_new is read
constexpr uint32_t kColO1 = 64;
constexpr uint32_t kColH = 128;             // 128 columns
constexpr uint32_t kColS = 256;             // FP32 state h^T, 128 columns

constexpr uint32_t kIdescKK64 = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t kIdescKM64 = idesc_bf16(128, 64, 0, 1);
constexpr uint32_t kIdescKM128 = idesc_bf16(128, 128, 0, 1);

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
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);  // full0, full1, a, h, o
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + kOffBar + 64);
    int *s_ctl = reinterpret_cast<int *>(sm + kOffBar + 128);  // current, next chain

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
        for (int b = 0; b < 5; ++b) mbar_init(&bars[b], 1);
        mbar_init_fence();
        tma_prefetch_desc(&args.tk);
        if (kOut) tma_prefetch_desc(&args.tq);
        tma_prefetch_desc(&args.trec128);
        if (kOut) tma_prefetch_desc(&args.trec64);
        s_ctl[0] = fetch();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t lane = (uint32_t)(32 * quad) << 16;
    const int kbase = 64 * half;

    // K (and Q) tiles of a chunk plus its record (W, U^T, P, vectors).
    auto issue_tma = [&](const Chain &c, int cc, int stage) {
        const int gc = c.c_begin + cc;
        const int tt = tab[gc].y;
        const int64_t rid = (int64_t)gc * H + c.h;
        const int rrow = (int)(rid * kRecRows);  // the host keeps this below 2^31
        const uint8_t *rec = ws.rec + rid * kRecBytes;
        uint64_t *bar = &bars[stage];
        uint8_t *dst = sm + stage * kStage;
        uint32_t bytes = 16384u + 16384u + 1024u;  // K, W, vectors
        if (kOut) bytes += 16384u + 8192u;          // Q, P
        if (!c.trans) bytes += 16384u;              // U^T
        mbar_arrive_expect_tx(bar, bytes);
        tma_load_3d(dst, &args.tk, bar, 0, c.h, tt);
        tma_load_3d(dst + 16384, &args.tk, bar, 64, c.h, tt);
        if (kOut) {
            tma_load_3d(dst + 8192, &args.tq, bar, 0, c.h, tt);
            tma_load_3d(dst + 24576, &args.tq, bar, 64, c.h, tt);
        }
        tma_load_2d(dst + kStW, &args.trec128, bar, 0, rrow + kRecW);
        if (!c.trans) tma_load_2d(dst + kStU, &args.trec128, bar, 0, rrow + kRecU);
        if (kOut) tma_load_2d(dst + kStP, &args.trec64, bar, 0, rrow + kRecP);
        bulk_load(dst + kStVec, rec + kRecVec * 128, 1024u, bar);
    };

    int cur = s_ctl[0];
    uint32_t gk = 0;  // chunks processed by this CTA: stage and parity
    uint32_t ph_a = 0, ph_h = 0, ph_o = 0;
    bool failed = false;
    if (cur < total && tid == 0) {
        Chain c;
        decode(cur, c);
        issue_tma(c, c.s0, 0);
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
                st_bf16x8(sm + kOffHm + sw128_off(row, kbase + 32 * q + 8 * c8, 128), hv + 8 * c8);
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
            const float *sDec = reinterpret_cast<const float *>(st + kStVec);
            const float *sGam = sDec + 64;
            // the chunk after this one: next in this chain, or the next chain's first
            if (tid == 0) {
                if (cc + 1 < C.s1)
                    issue_tma(C, cc + 1, stage ^ 1);
                else if (nxt < total)
                    issue_tma(Cn, Cn.s0, stage ^ 1);
            }
            bool ok = mbar_wait(&bars[stage], (gk >> 1) & 1u, p.status);
            if (__syncthreads_or(!ok)) { failed = true; break; }
            const float gam_last = sDec[128];
            if (len < 64) {  // K rows past the sequence end belong to the next one: zero them
                const int rows = 64 - len;
                for (int idx = tid; idx < rows * 2 * 8; idx += kThreads) {
                    const int r = len + idx / 16, blk = (idx / 8) & 1, c16 = idx & 7;
                    st_shared_v4(st + blk * 16384 + r * 128 + c16 * 16, 0u, 0u, 0u, 0u);
                }
                fence_async_smem();
            }
            __syncthreads();

            // A6: v_new^T = U^T - h^T W^T   (and O1 = h^T Q^T for the output)
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_bf16(tmem + kColVn,
                              sdesc_sw128(sb + kOffHm + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                              sdesc_sw128(sta + kStW + kk * 2048, 8192, 1024), kIdescKM64, kk > 0);
                umma_commit(&bars[2]);
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
            ok = mbar_wait(&bars[2], ph_a, p.status);
            ph_a ^= 1;
            if (__syncthreads_or(!ok)) { failed = true; break; }
            tc_fence_after();
            {
                float w[32], u[32];
                tmem_load32f(tmem + lane + kColVn + 32 * half, w);
                if (!trans) {
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8)
                        ld_bf16x8(st + kStU + sw128_off(row, 32 * half + 8 * c8, 128), u + 8 * c8);
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
                umma_commit(&bars[3]);
                if (kOut) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + kColO2, sdesc_sw128(sb + kOffVn + kk * 32, 16, 1024),
                                  sdesc_sw128(sta + kStP + kk * 32, 16, 1024), kIdescKK64, kk > 0);
                    umma_commit(&bars[4]);
                }
            }
            ok = mbar_wait(&bars[3], ph_h, p.status);
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

            // A7: output rows of this chunk, staged over the v_new tile.
            if (kOut) {
                ok = mbar_wait(&bars[4], ph_o, p.status);
                ph_o ^= 1;
                if (__syncthreads_or(!ok)) { failed = true; break; }
                tc_fence_after();
                uint8_t *stage_o = sm + kOffVn;
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
            }
            fence_async_smem();
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
    const uint64_t rec_rows = (uint64_t)ws.max_chunks * H * kRecRows;
    if (!make_tmap_bf16_3d(&args.tq, p.q, kD, H, rows, kD * 2, H * kD * 2, 64, 1, 64) ||
        !make_tmap_bf16_3d(&args.tk, p.k, kD, H, rows, kD * 2, H * kD * 2, 64, 1, 64) ||
        !make_tmap_bf16_2d(&args.trec128, ws.rec, 64, rec_rows, 128, 64, 128) ||
        !make_tmap_bf16_2d(&args.trec64, ws.rec, 64, rec_rows, 128, 64, 64))
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
