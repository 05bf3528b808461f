// tc_gla.cu -- A11, the beta-free mode (pure gated linear attention state
// scan, S_t = alpha_t S_{t-1} + v_t k_t^T) on the tensor-core path, for BF16
// q/k/v with K in {128, 256} and V a multiple of 128.
//
// Persistent CTAs (one per SM, 256 threads) pull chains -- one (sequence,
// segment, head, 128-wide value tile) each -- longest sequences first.  Per
// 64-token chunk, with h^T (value rows x keys) the FP32 state in TMEM:
//
//   D1 = [K; Q] K^T (tcgen05; rows 64-127 are Q K^T),
//   P = (Q K^T) * e^{G_i - G_j}, j <= i                 (BF16 operand)
//   O1 = h_pre^T Q^T        (tcgen05, A = BF16 mirror of h^T)
//   h^T <- e^{G_last} h^T   (in TMEM), then h^T += (V e^{G_last - G})^T K
//                           (tcgen05, accumulating onto the state)
//   O2 = V^T P^T;  O^T = scale (O1 * e^G + O2)
//
// The chunk's transition is the scalar e^{G_last} (the diagonal affine chunk
// transform of flash-linear-attention issue #23 "Proposed Dataflow"), so the
// segment pre-scan only emits the local state c_s and the product of the
// chunk decays; the ordered composition is h_{s+1} = d_s h_s + c_s.
// Inputs arrive by TMA (128-byte swizzle) into one buffer; the next chunk's
// load is issued as soon as this chunk's last product has read its tiles.
// Waits are time-bounded (GDR_ERR_TIMEOUT in the status word on expiry).
#include "gdr_internal.cuh"
#include "tc_chunk.cuh"
#include "tma_host.cuh"

namespace gdr {
namespace {

using namespace tc;

enum GlaMode { kModeSerial = 0, kModePre = 1, kModeSegOut = 2 };

struct GlaArgs {
    Problem p;
    Workspace ws;
    CUtensorMap tq, tk, tv;
};

constexpr int kThreads = 256;

template <int KD>
struct GlaLayout {
    static constexpr uint32_t kKB = KD / 64;               // 64-key blocks
    static constexpr uint32_t kInQK = kKB * 16384;         // [Kb | Qb] per key block
    static constexpr uint32_t kInV = kInQK;                // V tile [Vb0 | Vb1]
    static constexpr uint32_t kOffHm = kInQK + 16384;      // h^T mirror, K-major
    static constexpr uint32_t kOffVd = kOffHm + kKB * 16384;  // (V e^{G_last-G})^T; output staging
    static constexpr uint32_t kOffP = kOffVd + 16384;
    static constexpr uint32_t kOffVec = kOffP + 8192;
    static constexpr uint32_t kOffBar = kOffVec + 1600;
    static constexpr uint32_t kSmem = kOffBar + 256 + 1024;
    // TMEM: state [0, KD), D1, O1, O2
    static constexpr uint32_t kColS = 0, kColD1 = KD, kColO1 = KD + 64, kColO2 = KD + 128;
};

struct GlaChain {
    int64_t n, tstart, tlen;  // the sequence's first token row and length
    int h, s, vt;
    int c_begin, s0, s1;
};

template <int KD, int MODE>
__global__ void __launch_bounds__(kThreads, 1) k_tc_gla(const __grid_constant__ GlaArgs args) {
    using L = GlaLayout<KD>;
    const Problem &p = args.p;
    const Workspace &ws = args.ws;
    constexpr bool kOut = MODE != kModePre;
    constexpr uint32_t kTmemCols = 512;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    float *vec = reinterpret_cast<float *>(sm + L::kOffVec);
    const float *sG = vec, *sDec = vec + 192, *sGam = vec + 256, *sEP = vec + 320,
                *sScal = vec + 384;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kOffBar);  // full, d1o1, ho2
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + L::kOffBar + 64);
    int *s_ctl = reinterpret_cast<int *>(sm + L::kOffBar + 128);

    const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int row = 32 * quad + lane_id;  // TMEM lane = value row of the tile
    const int H = (int)p.H, V = (int)p.V;
    const int VT = V / 128;
    const int S = MODE == kModeSerial ? 1 : ws.n_segments;
    const int total = (int)(p.N * S * H * VT);
    int32_t *counter = ws.n_chunks + 1 + MODE;
    constexpr int kHalfKeys = KD / 2;
    const int kbase = kHalfKeys * half;

    auto decode = [&](int id, GlaChain &c) {
        int r = id;
        c.vt = r % VT;
        r /= VT;
        c.h = r % H;
        r /= H;
        c.s = r % S;
        r /= S;
        c.n = ws.seq_order[r];
        c.c_begin = ws.seq_chunk0[c.n];
        const int nc = ws.seq_chunk0[c.n + 1] - c.c_begin;
        c.tstart = p.cu ? (int64_t)p.cu[c.n] : c.n * p.T;
        c.tlen = (p.cu ? (int64_t)p.cu[c.n + 1] : (c.n + 1) * p.T) - c.tstart;
        c.s0 = 0;
        c.s1 = nc;
        if (MODE != kModeSerial) {
            const int per = (nc + S - 1) / S;
            c.s0 = c.s * per;
            c.s1 = min(nc, c.s0 + per);
        }
    };
    auto fetch = [&]() -> int {
        while (true) {
            const int id = atomicAdd(counter, 1);
            if (id >= total) return total;
            GlaChain c;
            decode(id, c);
            if (c.s0 < c.s1) return id;
        }
    };

    if (warp == 0) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        // the two product barriers count one commit per issuing thread
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], kOut ? 2 : 1);
        mbar_init(&bars[2], kOut ? 2 : 1);
        mbar_init_fence();
        tma_prefetch_desc(&args.tk);
        tma_prefetch_desc(&args.tq);
        tma_prefetch_desc(&args.tv);
        s_ctl[0] = fetch();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t lane = (uint32_t)(32 * quad) << 16;

    auto issue_tma = [&](const GlaChain &c, int cc) {
        const int tt = (int)(c.tstart + (int64_t)kChunk * cc);
        uint64_t *bar = &bars[0];
        mbar_arrive_expect_tx(bar, L::kInQK + 16384u);
#pragma unroll
        for (int kb = 0; kb < (int)L::kKB; ++kb) {
            tma_load_3d(sm + kb * 16384, &args.tk, bar, 64 * kb, c.h, tt);
            tma_load_3d(sm + kb * 16384 + 8192, &args.tq, bar, 64 * kb, c.h, tt);
        }
        tma_load_3d(sm + L::kInV, &args.tv, bar, 128 * c.vt, c.h, tt);
        tma_load_3d(sm + L::kInV + 8192, &args.tv, bar, 128 * c.vt + 64, c.h, tt);
    };
    float gq[2] = {0.f, 0.f};
    const float bone[2] = {1.f, 1.f};
    auto load_gates = [&](const GlaChain &c, int cc) {
        const int64_t t0 = c.tstart + (int64_t)kChunk * cc;
        const int64_t len = c.tlen - (int64_t)kChunk * cc;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int tok = 2 * lane_id + u;
            gq[u] = tok < len ? p.g[(t0 + tok) * H + c.h] : 0.f;
        }
    };

    int cur = s_ctl[0];
    uint32_t gk = 0;
    uint32_t ph1 = 0, ph2 = 0;
    bool failed = false;
    if (cur < total) {
        GlaChain c;
        decode(cur, c);
        if (tid == 32) issue_tma(c, c.s0);
        if (warp == 0) load_gates(c, c.s0);
    }
    while (cur < total) {
        GlaChain C;
        decode(cur, C);
        if (tid == 0) s_ctl[1] = fetch();
        const int h = C.h, v0 = 128 * C.vt;
        const int64_t seg_base = (C.n * H + h) * (int64_t)S + C.s;
        // state h^T rows (value v0 + row), keys [kbase, kbase + KD/2), FP32 in TMEM
#pragma unroll 1
        for (int q = 0; q < kHalfKeys / 32; ++q) {
            float hv[32];
#pragma unroll
            for (int kk = 0; kk < 32; ++kk) {
                const int key = kbase + 32 * q + kk;
                float x = 0.f;
                if (MODE == kModeSerial) {
                    if (p.h0) x = p.h0[((C.n * H + h) * KD + key) * (int64_t)V + v0 + row];
                } else if (MODE == kModeSegOut) {
                    x = ws.segH[(seg_base * KD + key) * V + v0 + row];
                }
                hv[kk] = x;
            }
            tmem_store32f(tmem + lane + L::kColS + kbase + 32 * q, hv);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8)
                st_bf16x8(sm + L::kOffHm + sw128_off(row, kbase + 32 * q + 8 * c8, 128),
                          hv + 8 * c8);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        const int nxt = s_ctl[1];
        GlaChain Cn;
        if (nxt < total) decode(nxt, Cn);
        float dprod = 1.f;  // product of the chunk decays (pre-scan summary)

        for (int cc = C.s0; cc < C.s1; ++cc, ++gk) {
            const int64_t t0 = C.tstart + (int64_t)kChunk * cc;
            const int64_t rem = C.tlen - (int64_t)kChunk * cc;
            const int len = rem < kChunk ? (int)rem : kChunk;
            if (warp == 0) gate_vectors(vec, gq, bone, len, lane_id);
            bool ok = mbar_wait(&bars[0], gk & 1u, p.status);
            if (__syncthreads_or(!ok)) { failed = true; break; }
            const float gam_last = sScal[1];
            const bool fact = sScal[2] != 0.f;
            dprod *= gam_last;
            if (len < 64) {  // rows past the sequence end belong to the next one: zero them
                const int rows = 64 - len;
                const int nblk = 2 * (int)L::kKB + 2;
                for (int idx = tid; idx < rows * nblk * 8; idx += kThreads) {
                    const int r = len + idx / (nblk * 8), blk = (idx / 8) % nblk, c16 = idx & 7;
                    st_shared_v4(sm + blk * 8192 + r * 128 + c16 * 16, 0u, 0u, 0u, 0u);
                }
                fence_async_smem();
            }
            __syncthreads();
            // D1 = [K; Q] K^T (thread 0) and O1 = h_pre^T Q^T (thread 128), issued
            // side by side, each committed by its own thread
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < KD / 16; ++kk) {
                    const uint32_t a = sb + (kk >> 2) * 16384 + (kk & 3) * 32;
                    umma_bf16(tmem + L::kColD1, sdesc_sw128(a, 16, 1024), sdesc_sw128(a, 16, 1024),
                              idesc_bf16(128, 64, 0, 0), kk > 0);
                }
                umma_commit(&bars[1]);
            }
            if (kOut && tid == 128) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < KD / 16; ++kk)
                    umma_bf16(tmem + L::kColO1,
                              sdesc_sw128(sb + L::kOffHm + (kk >> 2) * 16384 + (kk & 3) * 32, 16,
                                          1024),
                              sdesc_sw128(sb + (kk >> 2) * 16384 + 8192 + (kk & 3) * 32, 16, 1024),
                              idesc_bf16(128, 64, 0, 0), kk > 0);
                umma_commit(&bars[1]);
            }
            {  // state <- e^{G_last} state; (V e^{G_last - G})^T tile, t in [32 half, +32)
#pragma unroll 1
                for (int q = 0; q < kHalfKeys / 32; ++q) {
                    float hv[32];
                    tmem_load32f(tmem + lane + L::kColS + kbase + 32 * q, hv);
#pragma unroll
                    for (int i = 0; i < 32; ++i) hv[i] *= gam_last;
                    tmem_store32f(tmem + lane + L::kColS + kbase + 32 * q, hv);
                }
                float vd[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int t = 32 * half + i;
                    const __nv_bfloat16 x = *reinterpret_cast<const __nv_bfloat16 *>(
                        sm + L::kInV + sw128_off(t, row, 64));
                    vd[i] = __bfloat162float(x) * sDec[t];
                }
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8)
                    st_bf16x8(sm + L::kOffVd + sw128_off(row, 32 * half + 8 * c8, 128), vd + 8 * c8);
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            ok = mbar_wait(&bars[1], ph1, p.status);
            ph1 ^= 1;
            if (__syncthreads_or(!ok)) { failed = true; break; }
            tc_fence_after();
            if (kOut && quad >= 2) {  // row i of P (lower, diagonal included)
                float f[32];
                tmem_load32f(tmem + lane + L::kColD1 + 32 * half, f);
                const int i = row - 64, j0 = 32 * half;
                if (fact) {
                    const float ri = sEP[i];
#pragma unroll
                    for (int u = 0; u < 32; ++u)
                        f[u] = (j0 + u <= i) ? f[u] * (ri * sDec[j0 + u]) : 0.f;
                } else {
                    const float gi = sG[i];
#pragma unroll
                    for (int u = 0; u < 32; ++u)
                        f[u] = (j0 + u <= i) ? f[u] * __expf(gi - sG[j0 + u]) : 0.f;
                }
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8)
                    st_bf16x8(sm + L::kOffP + sw128_off(i, j0 + 8 * c8, 64), f + 8 * c8);
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            // state += vd^T K (thread 0) and O2 = V^T P^T (thread 128)
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(tmem + L::kColS, sdesc_sw128(sb + L::kOffVd + kk * 32, 16, 1024),
                              sdesc_sw128(sb + kk * 2048, 16384, 1024), idesc_bf16(128, KD, 0, 1),
                              1u);
                umma_commit(&bars[2]);
            }
            if (kOut && tid == 128) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(tmem + L::kColO2, sdesc_sw128(sb + L::kInV + kk * 2048, 8192, 1024),
                              sdesc_sw128(sb + L::kOffP + kk * 32, 16, 1024),
                              idesc_bf16(128, 64, 1, 0), kk > 0);
                umma_commit(&bars[2]);
            }
            ok = mbar_wait(&bars[2], ph2, p.status);
            ph2 ^= 1;
            if (__syncthreads_or(!ok)) { failed = true; break; }
            tc_fence_after();
            // every product has read this chunk's tiles: load the next chunk now
            {
                const bool here = cc + 1 < C.s1;
                if (here || nxt < total) {
                    const GlaChain &F = here ? C : Cn;
                    const int fcc = here ? cc + 1 : Cn.s0;
                    if (tid == 32) issue_tma(F, fcc);  // off the MMA issuers' warps
                    if (warp == 0) load_gates(F, fcc);
                }
            }
            // mirror of the updated state
#pragma unroll 1
            for (int q = 0; q < kHalfKeys / 32; ++q) {
                float hv[32];
                tmem_load32f(tmem + lane + L::kColS + kbase + 32 * q, hv);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8)
                    st_bf16x8(sm + L::kOffHm + sw128_off(row, kbase + 32 * q + 8 * c8, 128),
                              hv + 8 * c8);
            }
            if (kOut) {  // output rows, staged over the vd tile
                uint8_t *stage_o = sm + L::kOffVd;
                float o1[32], o2[32];
                tmem_load32f(tmem + lane + L::kColO1 + 32 * half, o1);
                tmem_load32f(tmem + lane + L::kColO2 + 32 * half, o2);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int t = 32 * half + i;
                    const float y = p.scale * fmaf(sGam[t], o1[i], o2[i]);
                    *reinterpret_cast<__nv_bfloat16 *>(stage_o + t * 256 + row * 2) =
                        __float2bfloat16_rn(y);
                }
                tc_fence_before();
                __syncthreads();
                __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int idx = tid + kThreads * r;
                    const int t = idx >> 4, c16 = idx & 15;
                    if (t < len)
                        *reinterpret_cast<uint4 *>(o + ((t0 + t) * H + h) * (int64_t)V + v0 +
                                                   c16 * 8) =
                            *reinterpret_cast<const uint4 *>(stage_o + t * 256 + c16 * 16);
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
        }
        if (failed) break;
        if (MODE != kModeSegOut && (MODE != kModeSerial || p.ht)) {
            tc_fence_after();
#pragma unroll 1
            for (int q = 0; q < kHalfKeys / 32; ++q) {
                float hv[32];
                tmem_load32f(tmem + lane + L::kColS + kbase + 32 * q, hv);
#pragma unroll
                for (int kk = 0; kk < 32; ++kk) {
                    const int key = kbase + 32 * q + kk;
                    if (MODE == kModeSerial)
                        p.ht[((C.n * H + h) * KD + key) * (int64_t)V + v0 + row] = hv[kk];
                    else
                        ws.segC[(seg_base * KD + key) * V + v0 + row] = hv[kk];
                }
            }
            if (MODE == kModePre && C.vt == 0 && tid == 0) ws.segD[seg_base] = dprod;
        }
        cur = nxt;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int KD, int MODE>
cudaError_t launch_gla(const GlaArgs &args, unsigned grid, cudaStream_t st) {
    const int smem = (int)GlaLayout<KD>::kSmem;
    cudaError_t err =
        cudaFuncSetAttribute(k_tc_gla<KD, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    k_tc_gla<KD, MODE><<<grid, kThreads, smem, st>>>(args);
    return cudaGetLastError();
}

}  // namespace

bool tc_gla_supported(const Problem &p) {
    auto al = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
    return p.dtype == GDR_BF16 && p.beta == nullptr && (p.K == 128 || p.K == 256) &&
           p.V % 128 == 0 && p.V <= kMaxV && al(p.q) && al(p.k) && al(p.v) && al(p.o);
}

cudaError_t tc_gla(const Problem &p, const Workspace &ws, int mode, cudaStream_t st) {
    GlaArgs args;
    args.p = p;
    args.ws = ws;
    const uint64_t rows = (uint64_t)p.B * (uint64_t)p.T;
    const uint64_t H = (uint64_t)p.H, K = (uint64_t)p.K, V = (uint64_t)p.V;
    if (!make_tmap_bf16_3d(&args.tq, p.q, K, H, rows, K * 2, H * K * 2, 64, 1, 64) ||
        !make_tmap_bf16_3d(&args.tk, p.k, K, H, rows, K * 2, H * K * 2, 64, 1, 64) ||
        !make_tmap_bf16_3d(&args.tv, p.v, V, H, rows, V * 2, H * V * 2, 64, 1, 64))
        return cudaErrorInvalidValue;
    const int S = mode == 0 ? 1 : ws.n_segments;
    const int64_t chains = p.N * S * p.H * (p.V / 128);
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const unsigned grid = (unsigned)(chains < sms ? chains : sms);
    if (p.K == 128) {
        switch (mode) {
        case 0: return launch_gla<128, kModeSerial>(args, grid, st);
        case 1: return launch_gla<128, kModePre>(args, grid, st);
        case 2: return launch_gla<128, kModeSegOut>(args, grid, st);
        }
    } else {
        switch (mode) {
        case 0: return launch_gla<256, kModeSerial>(args, grid, st);
        case 1: return launch_gla<256, kModePre>(args, grid, st);
        case 2: return launch_gla<256, kModeSegOut>(args, grid, st);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdr
