// tc_gla.cu -- A11, the beta-free mode (pure gated linear attention state
// scan, S_t = alpha_t S_{t-1} + v_t k_t^T) on the tensor-core path, for BF16
// q/k/v with K in {128, 256} and V a multiple of 128.
//
// Persistent CTAs (one per SM) pull chains -- one (sequence, segment, head,
// 128-wide value tile) each -- longest sequences first.  Per 64-token chunk,
// with h^T (value rows x keys) the FP32 state in TMEM:
//
//   D1 = [K; Q] K^T (tcgen05; rows 64-127 are Q K^T),
//   P = (Q K^T) * e^{G_i - G_j}, j <= i                 (BF16 operand)
//   O1 = h_pre^T Q^T        (tcgen05, A = BF16 mirror of h^T held in TMEM)
//   h^T <- e^{G_last} h^T (in TMEM), then h^T += (e^{G_last - G} V)^T K
//   O2 = V^T P^T;  O^T = scale (O1 * e^G + O2)
//
// The chunk's transition is the scalar e^{G_last} (the diagonal affine chunk
// transform of flash-linear-attention issue #23 "Proposed Dataflow"), so the
// segment pre-scan only emits the local state c_s and the product of the
// chunk decays; the ordered composition is h_{s+1} = d_s h_s + c_s.
//
// The warps specialise (as the delta-rule scan in tc_chain.cu):
//   warps 0-3  state path: the BF16 mirror of h^T into TMEM and h^T scaled
//              by e^{G_last}, per chunk (the serial dependency);
//   warps 4-7  side path: (e^{G_last - G} V) into its own tile, P from D1,
//              then the chunk's output (staged, stored; TMA for whole chunks);
//   warp 8     control: every tcgen05 MMA;
//   warp 9     producer: claims and decodes chains, loads K, Q and the value
//              tile by TMA into a two-stage ring and computes the chunk's gate
//              vectors (one warp, shuffle scan) beside them.
// Every wait is time-bounded: on expiry the CTA records GDR_ERR_TIMEOUT in
// the status word, the other roles leave too, and the CTA exits.
#include "gdr_internal.cuh"
#include "gdr_segments.cuh"
#include "tc_chunk.cuh"
#include "tma_host.cuh"

namespace gdr {
namespace {

using namespace tc;

enum GlaMode { kModeSerial = 0, kModePre = 1, kModeSegOut = 2 };

struct GlaArgs {
    Problem p;
    Workspace ws;
    CUtensorMap tq, tk, tv, to;
};

constexpr int kThreads = 320;  // warps 0-3 state, 4-7 side, 8 control, 9 producer
constexpr int kRing = 3;       // decoded chains handed out ahead

// One chain of the work list, decoded; valid == 0 ends the list; whole: an
// output-pass chain over a whole unsplit sequence (common segment length),
// from h0 to ht.
struct GlaDesc {
    int64_t n, tstart, tlen;  // the sequence's first token row and length
    int h, s, vt, c_begin, s0, s1, valid, whole;
};
static_assert(sizeof(GlaDesc) == 56, "chain descriptor layout");

template <int KD>
struct GlaLayout {
    // one stage: [Kb | Qb] per 64-key block, the value tile [Vb0 | Vb1], the
    // gate vectors
    static constexpr uint32_t kKB = KD / 64;
    static constexpr uint32_t kStV = kKB * 16384;
    static constexpr uint32_t kStVec = kStV + 16384;
    static constexpr uint32_t kStage = kStVec + 2048;
    static constexpr uint32_t kOffVd = 2 * kStage;        // e^{G_last - G} V, V's layout
    static constexpr uint32_t kOffP = kOffVd + 16384;     // P, K-major
    static constexpr uint32_t kOffOs = kOffP + 8192;      // output staging
    static constexpr uint32_t kOffGam = kOffOs + 16384;   // e^G of the chunk (side path copy)
    static constexpr uint32_t kOffRing = kOffGam + 256;
    static constexpr uint32_t kOffBar = kOffRing + 64 * kRing;
    // TMEM: state [0, KD), BF16 mirror, D1 (then O2), O1
    static constexpr uint32_t kColS = 0, kColM = KD, kColD = KD + KD / 2, kColO = kColD + 64;
};

enum : int {
    kGFull = 0,     // [2] stage landed: TMA bytes + the gate vectors (2 arrivals)
    kGD1 = 2,       // D1 done (commit)
    kGSready = 3,   // mirror written, state scaled (state path, 128)
    kGVready = 4,   // e^{G_last - G} V written (side path, 128)
    kGPready = 5,   // P written (side path, 128)
    kGHdone = 6,    // state update done (commit)
    kGO2 = 7,       // O2 done (commit)
    kGOfree = 8,    // O1 / O2 read (side path, 128)
    kGFree = 9,     // [2] stage free (commit)
    kGDrain = 11,   // every issued MMA done (commit, at the end)
    kGCfull = 12,   // [kRing] chain posted (producer)
    kGCempty = 12 + kRing,  // [kRing] chain read (state, side, control: 257)
    kGNumBars = 12 + 2 * kRing
};

__device__ __forceinline__ void side_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool side_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok)
        : "memory");
    return r != 0;
}

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
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + L::kOffBar + 8 * kGNumBars);
    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + L::kOffBar + 8 * kGNumBars + 4);
    GlaDesc *ring = reinterpret_cast<GlaDesc *>(sm + L::kOffRing);
    float *s_gam = reinterpret_cast<float *>(sm + L::kOffGam);

    const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
    const int row = 32 * (warp & 3) + lane_id;  // TMEM lane = value row of the tile
    const uint32_t lane = (uint32_t)(32 * (warp & 3)) << 16;
    const int H = (int)p.H, V = (int)p.V;
    const int VT = V / 128;
    const int S = MODE == kModeSerial ? 1 : ws.n_segments;

    auto wait = [&](int b, uint32_t parity) -> bool {
        return mbar_wait_or_abort(&bars[b], parity & 1u, p.status, s_abort);
    };
    auto take = [&](int k, GlaDesc &c) -> bool {
        const int slot = k % kRing;
        if (!wait(kGCfull + slot, (uint32_t)(k / kRing))) return false;
        c = ring[slot];
        mbar_arrive(&bars[kGCempty + slot]);
        return true;
    };

    pdl_trigger();
    if (warp == 0) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < kGNumBars; ++b) {
            uint32_t cnt = 1;
            if (b == kGFull || b == kGFull + 1) cnt = 2;
            if (b == kGSready || b == kGVready || b == kGPready || b == kGOfree) cnt = 128;
            if (b >= kGCempty) cnt = 257;
            mbar_init(&bars[b], cnt);
        }
        *s_abort = 0;
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    pdl_wait();  // the workspace and outputs, once the kernels before have finished

    if (warp == 9) {
        // ------------------------------------------------------------ producer
        const int total = (int)(p.N * S * H * VT);
        int32_t *counter = ws.n_chunks + (MODE == 0 ? kCtrSerial : MODE == 1 ? kCtrPre : kCtrSegOut);
        int issued = 0;
        bool ok = true;
        for (int posted = 0; ok; ++posted) {
            GlaDesc c{};
            if (lane_id == 0) {  // the next chain with chunks (heads, value tiles fastest)
                while (true) {
                    const int id = atomicAdd(counter, 1);
                    if (id >= total) break;
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
                    c.s0 = 0;
                    c.s1 = nc;
                    c.whole = 0;
                    if (MODE != kModeSerial) {
                        const int per = seg_per(ws, nc);
                        c.s0 = c.s * per;
                        c.s1 = min(nc, c.s0 + per);
                        // with one segment length, a sequence no longer than it
                        // has no pre-scan chain; its output chain runs it whole
                        if (seg_len(ws) && nc <= per) {
                            if (MODE == kModePre) {
                                // and so do all after it in the exact order
                                if (whole_from_here(ws, nc, per)) {
                                    atomicMax(counter, total);
                                    break;
                                }
                                c.s1 = c.s0;
                            } else {
                                c.whole = 1;
                            }
                        }
                    }
                    // the serial scan also takes a sequence without tokens
                    // (its final state is its initial one), and so does the
                    // output chain of a whole one
                    if (c.s0 < c.s1 || MODE == kModeSerial || (c.whole && c.s == 0)) {
                        c.tstart = seq_start(p, c.n);
                        c.tlen = seq_end(p, c.n) - c.tstart;
                        c.valid = 1;
                        break;
                    }
                    // the sequence's later ids are empty too: skip them for all
                    atomicMax(counter, (r + 1) * S * H * VT);
                }
                const int slot = posted % kRing;
                if (posted >= kRing && !wait(kGCempty + slot, (uint32_t)(posted / kRing - 1))) {
                    ok = false;
                } else {
                    ring[slot] = c;
                    mbar_arrive(&bars[kGCfull + slot]);
                }
            }
            // the lanes learn the chain through the ring slot
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            __syncwarp();
            c = ring[posted % kRing];
            if (!c.valid) break;
            for (int cc = c.s0; cc < c.s1; ++cc, ++issued) {
                const int stage = issued & 1;
                uint64_t *bar = &bars[kGFull + stage];
                uint8_t *dst = sm + stage * L::kStage;
                const int64_t t0 = c.tstart + (int64_t)kChunk * cc;
                const int64_t rem = c.tlen - (int64_t)kChunk * cc;
                const int len = rem < kChunk ? (int)rem : kChunk;
                bool free_ok = true;
                if (lane_id == 0 && issued >= 2)
                    free_ok = wait(kGFree + stage, (uint32_t)((issued >> 1) - 1));
                if (!__shfl_sync(0xffffffffu, free_ok ? 1 : 0, 0)) {
                    ok = false;
                    break;
                }
                if (lane_id == 0) {
                    const uint32_t bytes = L::kKB * (kOut ? 16384u : 8192u) + 16384u;
                    mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
                    for (int kb = 0; kb < (int)L::kKB; ++kb) {
                        tma_load_3d(dst + kb * 16384, &args.tk, bar, 64 * kb, c.h, (int)t0);
                        if (kOut)
                            tma_load_3d(dst + kb * 16384 + 8192, &args.tq, bar, 64 * kb, c.h,
                                        (int)t0);
                    }
                    tma_load_3d(dst + L::kStV, &args.tv, bar, 128 * c.vt, c.h, (int)t0);
                    tma_load_3d(dst + L::kStV + 8192, &args.tv, bar, 128 * c.vt + 64, c.h, (int)t0);
                }
                // gates of the chunk (padded tokens: g = 0), then their vectors
                float g2[2];
                const float one2[2] = {1.f, 1.f};
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int tok = 2 * lane_id + u;
                    g2[u] = tok < len ? p.g[(t0 + tok) * H + c.h] : 0.f;
                }
                gate_vectors(reinterpret_cast<float *>(dst + L::kStVec), g2, one2, len, lane_id);
                if (lane_id == 0) mbar_arrive(bar);
            }
        }
        __syncwarp();
    } else if (warp == 8) {
        // ------------------------------------------------------------ control
        if (lane_id == 0) {
            int k = 0, gk = 0;
            bool ok = true;
            while (ok) {
                GlaDesc C;
                if (!take(k++, C) || !C.valid) break;
                for (int cc = C.s0; cc < C.s1; ++cc, ++gk) {
                    const int b = gk & 1;
                    const uint32_t sta = sb + b * L::kStage;
                    if (!wait(kGFull + b, gk >> 1) || (kOut && gk > 0 && !wait(kGOfree, gk - 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (kOut) {  // D1 = [K; Q] K^T
#pragma unroll
                        for (int kk = 0; kk < KD / 16; ++kk) {
                            const uint32_t a = sta + (kk >> 2) * 16384 + (kk & 3) * 32;
                            umma_bf16(tmem + L::kColD, sdesc_sw128(a, 16, 1024),
                                      sdesc_sw128(a, 16, 1024), idesc_bf16(128, 64, 0, 0), kk > 0);
                        }
                        umma_commit(&bars[kGD1]);
                    }
                    if (!wait(kGSready, gk)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (kOut) {  // O1 = h_pre^T Q^T, A = the BF16 mirror in TMEM
#pragma unroll
                        for (int kk = 0; kk < KD / 16; ++kk)
                            umma_bf16_ts(tmem + L::kColO, tmem + L::kColM + 8 * kk,
                                         sdesc_sw128(sta + (kk >> 2) * 16384 + 8192 + (kk & 3) * 32,
                                                     16, 1024),
                                         idesc_bf16(128, 64, 0, 0), kk > 0);
                    }
                    if (!wait(kGVready, gk)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // h^T += (e^{G_last - G} V)^T K
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + L::kColS,
                                  sdesc_sw128(sb + L::kOffVd + kk * 2048, 8192, 1024),
                                  sdesc_sw128(sta + kk * 2048, 16384, 1024),
                                  idesc_bf16(128, KD, 1, 1), 1u);
                    umma_commit(&bars[kGHdone]);
                    if (kOut) {  // O2 = V^T P^T, over D1 (read by now)
                        if (!wait(kGPready, gk)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_bf16(tmem + L::kColD,
                                      sdesc_sw128(sta + L::kStV + kk * 2048, 8192, 1024),
                                      sdesc_sw128(sb + L::kOffP + kk * 32, 16, 1024),
                                      idesc_bf16(128, 64, 1, 0), kk > 0);
                        umma_commit(&bars[kGO2]);
                    }
                    umma_commit(&bars[kGFree + b]);
                }
            }
            umma_commit(&bars[kGDrain]);
            mbar_wait(&bars[kGDrain], 0, p.status, 100000000ull);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------------ state path
        int k = 0, gk = 0;
        bool ok = true;
        while (ok) {
            GlaDesc C;
            if (!take(k++, C) || !C.valid) break;
            const int h = C.h, v0 = 128 * C.vt;
            const int64_t seg_base = (C.n * H + h) * (int64_t)S + C.s;
            // h0 / ht column v0 + row of this (sequence, head): element `key`
            // at st_base + key * st_step, in either state layout
            const int64_t st_base = state_off(p, C.n * H + h, 0, v0 + row);
            const int64_t st_step = p.state_vk ? 1 : V;
            float dprod = 1.f;
            for (int cc = C.s0; cc < C.s1; ++cc, ++gk) {
                const int b = gk & 1;
                const float *vec = reinterpret_cast<const float *>(sm + b * L::kStage + L::kStVec);
                if (!wait(kGFull + b, gk >> 1)) { ok = false; break; }
                tc_fence_after();  // the state written by the previous update
                const float gam_last = vec[385];
                dprod *= gam_last;
                // h_pre -> BF16 mirror (O1's A operand, in TMEM); the FP32 state
                // scaled by e^{G_last} for the update.
#pragma unroll 1
                for (int q = 0; q < KD / 64; ++q) {
                    uint32_t r0[32], r1[32];
                    if (cc == C.s0) {  // the chain's initial state, value column v0 + row
#pragma unroll
                        for (int kk = 0; kk < 64; ++kk) {
                            const int key = 64 * q + kk;
                            float x = 0.f;
                            if (MODE == kModeSerial || C.whole) {
                                if (p.h0) x = p.h0[st_base + key * st_step];
                            } else if (MODE == kModeSegOut) {
                                x = ws.segH[(seg_base * KD + key) * V + v0 + row];
                            }
                            if (kk < 32) r0[kk] = __float_as_uint(x);
                            else r1[kk - 32] = __float_as_uint(x);
                        }
                    } else {
                        tmem_ld32(tmem + lane + L::kColS + 64 * q, r0);
                        tmem_ld32(tmem + lane + L::kColS + 64 * q + 32, r1);
                        tmem_wait_ld();
                        reg_fence(r0);
                        reg_fence(r1);
                    }
                    if (kOut) {
                        uint32_t m[32];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            m[i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
                            m[16 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]),
                                                    __uint_as_float(r1[2 * i + 1]));
                        }
                        tmem_st32(tmem + lane + L::kColM + 32 * q, m);
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        r0[i] = __float_as_uint(__uint_as_float(r0[i]) * gam_last);
                        r1[i] = __float_as_uint(__uint_as_float(r1[i]) * gam_last);
                    }
                    tmem_st32(tmem + lane + L::kColS + 64 * q, r0);
                    tmem_st32(tmem + lane + L::kColS + 64 * q + 32, r1);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars[kGSready]);
                if (!wait(kGHdone, gk)) { ok = false; break; }
            }
            if (!ok) break;
            if ((MODE == kModeSerial || C.whole) && C.s0 == C.s1) {  // no tokens: ht = h0 (or 0)
                if (p.ht) {
                    for (int key = 0; key < KD; ++key) {
                        const int64_t idx = st_base + key * st_step;
                        p.ht[idx] = p.h0 ? p.h0[idx] : 0.f;
                    }
                }
                continue;
            }
            const bool to_ht = (MODE == kModeSerial || C.whole) && p.ht;
            if (MODE == kModePre || to_ht) {
                tc_fence_after();
#pragma unroll 1
                for (int q = 0; q < KD / 32; ++q) {
                    float hv[32];
                    tmem_load32f(tmem + lane + L::kColS + 32 * q, hv);
#pragma unroll
                    for (int kk = 0; kk < 32; ++kk) {
                        const int key = 32 * q + kk;
                        if (to_ht)
                            p.ht[st_base + key * st_step] = hv[kk];
                        else
                            ws.segC[(seg_base * KD + key) * V + v0 + row] = hv[kk];
                    }
                }
                if (MODE == kModePre && C.vt == 0 && tid == 0) ws.segD[seg_base] = dprod;
            }
        }
    } else {
        // ------------------------------------------------------------ side path
        const int tb = tid - 128;
        const int q4 = warp & 3;  // lane quarter: rows 32 q4 .. 32 q4 + 31
        int k = 0, gk = 0;
        bool ok = true, stores = false;
        uint8_t *os = sm + L::kOffOs;  // [t][v] as two swizzled 64-column blocks
        while (ok) {
            GlaDesc C;
            if (!take(k++, C) || !C.valid) break;
            const int h = C.h, v0 = 128 * C.vt;
            for (int cc = C.s0; cc < C.s1; ++cc, ++gk) {
                const int b = gk & 1;
                const uint8_t *st = sm + b * L::kStage;
                const float *vec = reinterpret_cast<const float *>(st + L::kStVec);
                const float *sG = vec, *sDec = vec + 192, *sGam = vec + 256, *sEP = vec + 320;
                const int64_t t0 = C.tstart + (int64_t)kChunk * cc;
                const int64_t rem = C.tlen - (int64_t)kChunk * cc;
                const int len = rem < kChunk ? (int)rem : kChunk;
                if (!wait(kGFull + b, gk >> 1)) { ok = false; break; }
                // (e^{G_last - G} V) in V's layout; rows past the sequence end
                // (they belong to the next one) become zero.  Every read is
                // issued before the first write (the compiler cannot reorder
                // shared-memory reads past writes it cannot tell apart).
                uint4 raw[8];
                float dv[8];
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int idx = tb + 128 * r;
                    const int t = (idx >> 3) & 63;
                    const uint32_t off = (idx >> 9) * 8192 + t * 128 + (idx & 7) * 16;
                    raw[r] = *reinterpret_cast<const uint4 *>(st + L::kStV + off);
                    dv[r] = t < len ? sDec[t] : 0.f;
                }
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int idx = tb + 128 * r;
                    const int t = (idx >> 3) & 63;
                    const uint32_t off = (idx >> 9) * 8192 + t * 128 + (idx & 7) * 16;
                    if (t < len) {
                        float x[8];
                        ld_bf16x8(&raw[r], x);
#pragma unroll
                        for (int u = 0; u < 8; ++u) x[u] *= dv[r];
                        st_bf16x8(sm + L::kOffVd + off, x);
                    } else {
                        st_shared_v4(sm + L::kOffVd + off, 0u, 0u, 0u, 0u);
                    }
                }
                if (kOut && tb < 64) s_gam[tb] = sGam[tb];
                fence_async_smem();
                mbar_arrive(&bars[kGVready]);
                if (!kOut) {
                    // the tile is read by the update product: the next chunk's
                    // waits for it (the output below orders this otherwise)
                    if (!wait(kGHdone, gk)) { ok = false; break; }
                    continue;
                }
                // P from D1 (rows 64-127 of D1 are Q K^T): warps of lane quarters 2, 3
                if (!side_all(wait(kGD1, gk))) { ok = false; break; }
                tc_fence_after();
                if (q4 >= 2) {
                    const int i = row - 64;
                    const bool fact = vec[386] != 0.f;
                    // row i of Q K^T (both halves) in one TMEM wait
                    uint32_t d0[32], d1[32];
                    tmem_ld32(tmem + lane + L::kColD, d0);
                    tmem_ld32(tmem + lane + L::kColD + 32, d1);
                    tmem_wait_ld();
                    reg_fence(d0);
                    reg_fence(d1);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        float f[32];
#pragma unroll
                        for (int u = 0; u < 32; ++u) f[u] = __uint_as_float(hh ? d1[u] : d0[u]);
                        const int j0 = 32 * hh;
                        if (fact) {
                            // the 32 column factors as eight 16-byte shared-memory reads
                            const float ri = sEP[i];
                            float dj[32];
#pragma unroll
                            for (int v4 = 0; v4 < 8; ++v4) {
                                const float4 t4 = *reinterpret_cast<const float4 *>(sDec + j0 + 4 * v4);
                                dj[4 * v4] = t4.x;
                                dj[4 * v4 + 1] = t4.y;
                                dj[4 * v4 + 2] = t4.z;
                                dj[4 * v4 + 3] = t4.w;
                            }
#pragma unroll
                            for (int u = 0; u < 32; ++u)
                                f[u] = (j0 + u <= i && j0 + u < len) ? f[u] * (ri * dj[u]) : 0.f;
                        } else {
                            const float gi = sG[i];
#pragma unroll
                            for (int u = 0; u < 32; ++u)
                                f[u] = (j0 + u <= i && j0 + u < len) ? f[u] * __expf(gi - sG[j0 + u])
                                                                      : 0.f;
                        }
#pragma unroll
                        for (int c8 = 0; c8 < 4; ++c8)
                            st_bf16x8(sm + L::kOffP + sw128_off(i, j0 + 8 * c8, 64), f + 8 * c8);
                    }
                }
                fence_async_smem();
                tc_fence_before();
                mbar_arrive(&bars[kGPready]);
                // the chunk's output once O2 is done: O^T = scale (O1 * e^G + O2)
                if (tb == 0 && stores) bulk_wait_read();  // the staging tile is free again
                if (!side_all(wait(kGO2, gk))) { ok = false; break; }
                tc_fence_after();
                uint8_t *col = os + (row >> 6) * 8192;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t o1[32], o2[32];
                    tmem_ld32(tmem + lane + L::kColO + 32 * hh, o1);
                    tmem_ld32(tmem + lane + L::kColD + 32 * hh, o2);
                    tmem_wait_ld();
                    reg_fence(o1);
                    reg_fence(o2);
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        const int t = 32 * hh + u;
                        const float y = p.scale * fmaf(s_gam[t], __uint_as_float(o1[u]),
                                                       __uint_as_float(o2[u]));
                        *reinterpret_cast<__nv_bfloat16 *>(col + sw128_off(t, row & 63, 64)) =
                            __float2bfloat16_rn(y);
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars[kGOfree]);
                if (len == kChunk) {
                    fence_async_smem();
                    side_sync();
                    if (tb == 0) {
                        tma_store_3d(&args.to, os, v0, h, (int)t0);
                        tma_store_3d(&args.to, os + 8192, v0 + 64, h, (int)t0);
                        bulk_commit();
                        stores = true;
                    }
                } else {  // a sequence's last chunk: rows past its end belong to the next
                    side_sync();
                    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int idx = tb + 128 * r;
                        const int t = idx >> 4, c16 = idx & 15;
                        if (t < len)
                            *reinterpret_cast<uint4 *>(o + tok_at(p.so, t0 + t, h) + v0 +
                                                       c16 * 8) =
                                *reinterpret_cast<const uint4 *>(os + (c16 >> 3) * 8192 +
                                                                 sw128_off(t, (c16 & 7) * 8, 64));
                    }
                }
                // s_gam and the staging tile are reused by the next chunk
                side_sync();
            }
        }
        if (tb == 0 && stores) bulk_wait_read();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int KD, int MODE>
cudaError_t launch_gla(const GlaArgs &args, unsigned grid, cudaStream_t st) {
    const int smem = (int)(GlaLayout<KD>::kOffBar + 8 * kGNumBars + 16 + 1024);
    cudaError_t err =
        cudaFuncSetAttribute(k_tc_gla<KD, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(k_tc_gla<KD, MODE>, grid, dim3(kThreads), smem, st, args);
}

}  // namespace

bool tc_gla_supported(const Problem &p) {
    // TMA and the 16-byte stores of partial chunks: aligned bases and strides
    return p.dtype == GDR_BF16 && p.beta == nullptr && (p.K == 128 || p.K == 256) &&
           p.V % 128 == 0 && p.V <= kMaxV && rows_aligned16(p.q, p.sq, 2) &&
           rows_aligned16(p.k, p.sk, 2) && rows_aligned16(p.v, p.sv, 2) &&
           rows_aligned16(p.o, p.so, 2);
}

cudaError_t tc_gla(const Problem &p, const Workspace &ws, int mode, cudaStream_t st) {
    GlaArgs args;
    args.p = p;
    args.ws = ws;
    const uint64_t rows = (uint64_t)p.B * (uint64_t)p.T;
    const uint64_t H = (uint64_t)p.H, K = (uint64_t)p.K, V = (uint64_t)p.V;
    if (!make_tmap_bf16_3d(&args.tq, p.q, K, H, rows, p.sq.h * 2, p.sq.t * 2, 64, 1, 64) ||
        !make_tmap_bf16_3d(&args.tk, p.k, K, H, rows, p.sk.h * 2, p.sk.t * 2, 64, 1, 64) ||
        !make_tmap_bf16_3d(&args.tv, p.v, V, H, rows, p.sv.h * 2, p.sv.t * 2, 64, 1, 64) ||
        !make_tmap_bf16_3d(&args.to, p.o, V, H, rows, p.so.h * 2, p.so.t * 2, 64, 1, 64))
        return cudaErrorInvalidValue;
    const int S = mode == 0 ? 1 : ws.n_segments;
    const int64_t chains = p.N * S * p.H * (p.V / 128);
    const unsigned grid = (unsigned)persistent_grid(p, chains, 1);
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
