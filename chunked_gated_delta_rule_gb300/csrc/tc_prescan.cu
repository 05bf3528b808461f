// tc_prescan.cu -- A8 on the tensor-core path (BF16, K = V = 128, delta
// rule): the segment pre-scan, both summaries of a (sequence, segment, head)
// in one CTA.  From the segment's first chunk, per chunk in order:
//
//   local state  c:  h_c^T <- e^{G_last} h_c^T + (U^T - h_c^T W^T) K~   (from 0)
//   transition   M:  h_t^T <- e^{G_last} h_t^T - (h_t^T W^T) K~          (from I)
//
// with K~ = diag(e^{G_last - G}) K; the segment's summaries are c_s = h_c and
// M_s^T = h_t (the K x K transition of cuLA PR #127 "Root cause and
// implementation", kept in FP32).  The two chains share every load and the
// K~ pass, and their BF16 mirrors (the first product's A operand) and v_new
// tiles (the update's A operand, written over the columns of h^T W^T it was
// formed from) live in tensor memory, so shared memory holds only the
// two-stage ring of record images, and an MMA reads only its B tile there.
//
// The two recurrences are independent, so each has its own warps and
// barriers and runs at the latency of one chain: warps 0-3 (local state) and
// 4-7 (transition) write their state's mirror, scale it by e^{G_last}, form
// half of K~ and then their v_new tile; warps 8 and 9 issue the MMAs of the
// local state and of the transition (a commit tracks the MMAs of the thread
// that issued them); warp 10 is the producer (chain claims and decoding,
// the record images and k tiles, as in tc_chain.cu).  They meet only at the
// stage: its K~ (both halves) before either update, and its release after
// both.  Every wait is time-bounded: on expiry the CTA records
// GDR_ERR_TIMEOUT in the status word, the other roles leave too, and the
// CTA exits.
#include "gdr_internal.cuh"
#include "gdr_segments.cuh"
#include "tc_chunk.cuh"
#include "tma_host.cuh"

namespace gdr {
namespace {

using namespace tc;

struct PreArgs {
    Problem p;
    Workspace ws;
    CUtensorMap tk;
};

constexpr int kThreads = 352;  // warps 0-3, 4-7 state paths; 8, 9 their MMAs; 10 producer
constexpr int kRing = 3;

// Shared memory (bytes from a 1024-aligned base): two record-image stages
// (only W, the k tile, U^T and the vectors are loaded).
constexpr uint32_t kStage = kRecBytes;
constexpr uint32_t kOffRing = 2 * kStage;
enum : int {
    kPFull = 0,     // [2] stage landed
    kPKready = 2,   // [2] K~ formed in the stage (both paths: 256)
    kPFree = 4,     // [2] stage free (both MMA warps' commits: 2)
    kPMready = 6,   // [2] per state: mirror written, state scaled (128)
    kPAdone = 8,    // [2] per state: h^T W^T done (commit)
    kPVready = 10,  // [2] per state: v_new tile written (128)
    kPHdone = 12,   // [2] per state: update done (commit)
    kPDrain = 14,   // [2] per state: every issued MMA done (commit, at the end)
    kPCfull = 16,   // [kRing] chain posted (producer)
    kPCempty = 16 + kRing,  // [kRing] chain read (paths and MMA warps: 258)
    kPNumBars = 16 + 2 * kRing
};

struct PreDesc {
    int64_t n, tstart, tlen;
    int h, s, c_begin, s0, s1, valid, pad0, pad1;
};
static_assert(sizeof(PreDesc) == 56, "chain descriptor layout");
constexpr uint32_t kOffBar = kOffRing + 64 * kRing;
constexpr uint32_t kSmemLaunch = kOffBar + 8 * kPNumBars + 16 + 1024;

// TMEM (512 columns): h W^T of both states (then v_new^T over its first 32
// columns, two BF16 tokens per column), both FP32 states, both mirrors (two
// BF16 keys per column).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColA = 0;     // [2] 64 columns each
constexpr uint32_t kColS = 128;   // [2] 128 columns each
constexpr uint32_t kColM = 384;   // [2] 64 columns each

constexpr uint32_t kIdescA = idesc_bf16(128, 64, 0, 1);  // B = W^T, MN-major
constexpr uint32_t kIdescH = idesc_bf16(128, 128, 0, 1);

__global__ void __launch_bounds__(kThreads, 1) k_tc_prescan(const __grid_constant__ PreArgs args) {
    const Problem &p = args.p;
    const Workspace &ws = args.ws;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + kOffBar + 8 * kPNumBars);
    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + kOffBar + 8 * kPNumBars + 4);
    PreDesc *ring = reinterpret_cast<PreDesc *>(sm + kOffRing);

    const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
    const int row = 32 * (warp & 3) + lane_id;  // TMEM lane = matrix row
    const uint32_t lane = (uint32_t)(32 * (warp & 3)) << 16;
    const int H = (int)p.H;
    const int S = ws.n_segments;

    auto wait = [&](int b, uint32_t parity) -> bool {
        return mbar_wait_or_abort(&bars[b], parity & 1u, p.status, s_abort);
    };
    auto take = [&](int k, PreDesc &c) -> bool {
        const int slot = k % kRing;
        if (!wait(kPCfull + slot, (uint32_t)(k / kRing))) return false;
        c = ring[slot];
        mbar_arrive(&bars[kPCempty + slot]);
        return true;
    };

    pdl_trigger();
    if (warp == 0) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < kPNumBars; ++b) {
            uint32_t cnt = 1;
            if (b == kPKready || b == kPKready + 1) cnt = 256;
            if (b == kPFree || b == kPFree + 1) cnt = 2;
            if ((b >= kPMready && b < kPAdone) || (b >= kPVready && b < kPHdone)) cnt = 128;
            if (b >= kPCempty) cnt = 258;
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

    if (warp == 10) {
        // ------------------------------------------------------------ producer
        if (lane_id == 0) {
            const int total = (int)(p.N * S * H);
            int32_t *counter = ws.n_chunks + kCtrPre;
            tma_prefetch_desc(&args.tk);
            int issued = 0;
            for (int posted = 0;; ++posted) {
                PreDesc c{};
                while (true) {  // heads fastest, then segments; longest sequences first
                    const int id = atomicAdd(counter, 1);
                    if (id >= total) break;
                    int r = id;
                    c.h = r % H;
                    r /= H;
                    c.s = r % S;
                    r /= S;
                    c.n = ws.seq_order[r];
                    c.c_begin = ws.seq_chunk0[c.n];
                    const int nc = ws.seq_chunk0[c.n + 1] - c.c_begin;
                    const int per = seg_per(ws, nc);
                    c.s0 = c.s * per;
                    c.s1 = min(nc, c.s0 + per);
                    // a sequence within the common segment length runs whole in
                    // the output pass, and so do all after it in the exact order
                    if (whole_from_here(ws, nc, per)) {
                        atomicMax(counter, total);
                        break;
                    }
                    if (seg_len(ws) && nc <= per) c.s1 = c.s0;
                    if (c.s0 < c.s1) {
                        c.tstart = seq_start(p, c.n);
                        c.tlen = seq_end(p, c.n) - c.tstart;
                        c.valid = 1;
                        break;
                    }
                    // the sequence's later ids are empty too: skip them for all
                    atomicMax(counter, (r + 1) * S * H);
                }
                const int slot = posted % kRing;
                if (posted >= kRing && !wait(kPCempty + slot, (uint32_t)(posted / kRing - 1)))
                    break;
                ring[slot] = c;
                mbar_arrive(&bars[kPCfull + slot]);
                if (!c.valid) break;
                bool ok = true;
                for (int cc = c.s0; cc < c.s1; ++cc, ++issued) {
                    const int stage = issued & 1;
                    if (issued >= 2 && !wait(kPFree + stage, (uint32_t)((issued >> 1) - 1))) {
                        ok = false;
                        break;
                    }
                    const int64_t rid = (int64_t)(c.c_begin + cc) * H + c.h;
                    const uint8_t *rec = ws.rec + rid * kRecBytes;
                    const int tt = (int)(c.tstart + (int64_t)kChunk * cc);
                    uint64_t *bar = &bars[kPFull + stage];
                    uint8_t *dst = sm + stage * kStage;
                    mbar_arrive_expect_tx(bar, 16384u + 16384u + 16384u + (kImgBytes - kImgVec));
                    bulk_load(dst + kImgW, rec + kImgW, 16384u, bar);
                    tma_load_3d(dst + kImgK, &args.tk, bar, 0, c.h, tt);
                    tma_load_3d(dst + kImgK + 8192, &args.tk, bar, 64, c.h, tt);
                    bulk_load(dst + kImgU, rec + kImgU, 16384u, bar);
                    bulk_load(dst + kImgVec, rec + kImgVec, kImgBytes - kImgVec, bar);
                }
                if (!ok) break;
            }
        }
        __syncwarp();
    } else if (warp >= 8) {
        // ------------------------------------------------------------ MMAs of state warp - 8
        if (lane_id == 0) {
            const int q = warp - 8;
            const uint32_t cA = tmem + kColA + 64 * q, cS = tmem + kColS + 128 * q;
            const uint32_t cM = tmem + kColM + 64 * q;
            int k = 0, gk = 0;
            bool ok = true;
            while (ok) {
                PreDesc C;
                if (!take(k++, C) || !C.valid) break;
                for (int cc = C.s0; cc < C.s1; ++cc, ++gk) {
                    const int b = gk & 1;
                    const uint32_t sta = sb + b * kStage;
                    if (!wait(kPFull + b, gk >> 1) || !wait(kPMready + q, gk)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // h^T W^T, A = the state's BF16 mirror in TMEM
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_bf16_ts(cA, cM + 8 * kk, sdesc_sw128(sta + kImgW + kk * 2048, 16384, 1024),
                                     kIdescA, kk > 0);
                    umma_commit(&bars[kPAdone + q]);
                    if (!wait(kPVready + q, gk) || !wait(kPKready + b, gk >> 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // h^T += v_new^T K~ (A = v_new^T in TMEM; the next chunk's h^T W^T,
                    // issued after this by the same thread, overwrites it only
                    // once this product has read it)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16_ts(cS, cA + 8 * kk,
                                     sdesc_sw128(sta + kImgK + kk * 2048, 8192, 1024), kIdescH, 1u);
                    umma_commit(&bars[kPHdone + q]);
                    umma_commit(&bars[kPFree + b]);
                }
            }
            // nothing of this CTA may still run on the tensor cores at exit
            umma_commit(&bars[kPDrain + q]);
            mbar_wait(&bars[kPDrain + q], 0, p.status, 100000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ state paths
        const int path = warp >> 2;  // 0: local state from 0, 1: transition from I
        const int pt = tid & 127;
        const uint32_t cS = kColS + 128 * path, cM = kColM + 64 * path, cA = kColA + 64 * path;
        int k = 0, gk = 0;
        bool ok = true;
        while (ok) {
            PreDesc C;
            if (!take(k++, C) || !C.valid) break;
            const int64_t seg_base = (C.n * H + C.h) * (int64_t)S + C.s;
            for (int cc = C.s0; cc < C.s1; ++cc, ++gk) {
                const int b = gk & 1;
                uint8_t *st = sm + b * kStage;
                const int64_t rem = C.tlen - (int64_t)kChunk * cc;
                const int len = rem < kChunk ? (int)rem : kChunk;
                if (!wait(kPFull + b, gk >> 1)) { ok = false; break; }
                tc_fence_after();  // the state written by the previous update
                const float *vec = reinterpret_cast<const float *>(st + kImgVec);
                const float gam_last = vec[kImgGamLast];
                // the state before the chunk, column `row` of keys [64 hq, 64 hq + 64)
                auto state_half = [&](int hq, uint32_t (&r0)[32], uint32_t (&r1)[32]) {
                    if (cc == C.s0) {
#pragma unroll
                        for (int kk = 0; kk < 32; ++kk) {
                            r0[kk] = __float_as_uint(path && 64 * hq + kk == row ? 1.f : 0.f);
                            r1[kk] = __float_as_uint(path && 64 * hq + 32 + kk == row ? 1.f : 0.f);
                        }
                    } else {
                        tmem_ld32(tmem + lane + cS + 64 * hq, r0);
                        tmem_ld32(tmem + lane + cS + 64 * hq + 32, r1);
                        tmem_wait_ld();
                        reg_fence(r0);
                        reg_fence(r1);
                    }
                };
                // -> BF16 mirror in TMEM (two keys per column): the chain's
                // critical path, so it goes first
#pragma unroll 1
                for (int hq = 0; hq < 2; ++hq) {
                    uint32_t r0[32], r1[32], m[32];
                    state_half(hq, r0, r1);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        m[i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
                        m[16 + i] =
                            pack_bf16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
                    }
                    tmem_st32(tmem + lane + cM + 32 * hq, m);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars[kPMready + path]);
                // then the FP32 state scaled by e^{G_last}, while h^T W^T runs
#pragma unroll 1
                for (int hq = 0; hq < 2; ++hq) {
                    uint32_t r0[32], r1[32];
                    state_half(hq, r0, r1);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        r0[i] = __float_as_uint(__uint_as_float(r0[i]) * gam_last);
                        r1[i] = __float_as_uint(__uint_as_float(r1[i]) * gam_last);
                    }
                    tmem_st32(tmem + lane + cS + 64 * hq, r0);
                    tmem_st32(tmem + lane + cS + 64 * hq + 32, r1);
                }
                // half of K~ = diag(e^{G_last - G}) K in place (rows past the
                // sequence end, which belong to the next one, become zero)
                const float *dec = reinterpret_cast<const float *>(st + kImgDec);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int c = pt + 128 * (2 * r + path);
                    const int t = c >> 4;
                    uint8_t *ptr = st + kImgK + ((c >> 3) & 1) * 8192 + t * 128 + (c & 7) * 16;
                    if (t < len) {
                        float x[8];
                        ld_bf16x8(ptr, x);
                        const float d = dec[t];
#pragma unroll
                        for (int u = 0; u < 8; ++u) x[u] *= d;
                        st_bf16x8(ptr, x);
                    } else {
                        st_shared_v4(ptr, 0u, 0u, 0u, 0u);
                    }
                }
                fence_async_smem();
                mbar_arrive(&bars[kPKready + b]);
                if (!wait(kPAdone + path, gk)) { ok = false; break; }
                tc_fence_after();
                {  // v_new^T = U^T - h^T W^T (the transition: U = 0), as BF16 over
                   // the first 32 columns of h^T W^T once those are read
                    uint32_t w0[32], w1[32], vv[32];
                    tmem_ld32(tmem + lane + cA, w0);
                    tmem_ld32(tmem + lane + cA + 32, w1);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        float u[32];
                        if (path == 0) {
#pragma unroll
                            for (int c8 = 0; c8 < 4; ++c8)
                                ld_bf16x8(st + kImgU + sw128_off(row, 32 * hh + 8 * c8, 128),
                                          u + 8 * c8);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) u[i] = 0.f;
                        }
                        if (hh == 0) {
                            tmem_wait_ld();
                            reg_fence(w0);
                            reg_fence(w1);
                        }
#pragma unroll
                        for (int i = 0; i < 32; ++i) u[i] -= __uint_as_float(hh ? w1[i] : w0[i]);
#pragma unroll
                        for (int i = 0; i < 16; ++i) vv[16 * hh + i] = pack_bf16x2(u[2 * i], u[2 * i + 1]);
                    }
                    tmem_st32(tmem + lane + cA, vv);
                }
                tmem_wait_st();  // v_new and the scaled state, before the update product
                tc_fence_before();
                mbar_arrive(&bars[kPVready + path]);
                if (!wait(kPHdone + path, gk)) { ok = false; break; }
            }
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float hv[32];
                tmem_load32f(tmem + lane + cS + 32 * q, hv);
                if (path == 1) {  // M_s stored transposed: row `row`, as the
                    // tensor-core composition's B images when it runs, FP32 rows for
                    // the CUDA-core composition and the backward's maps
                    if (ws.segMimg) {
                        uint8_t *img = ws.segMimg + seg_base * 65536;
#pragma unroll
                        for (int c8 = 0; c8 < 4; ++c8) {
                            const uint32_t o = sw128_off(row, 32 * q + 8 * c8, 128);
                            st_split_bf16x8(img + o, img + 32768 + o, hv + 8 * c8);
                        }
                    }
                    if (ws.bwd_tc || !ws.segMimg) {
                        float4 *dst = reinterpret_cast<float4 *>(ws.segM + (seg_base * kD + row) * kD +
                                                                 32 * q);
#pragma unroll
                        for (int k4 = 0; k4 < 8; ++k4)
                            dst[k4] = make_float4(hv[4 * k4], hv[4 * k4 + 1], hv[4 * k4 + 2],
                                                  hv[4 * k4 + 3]);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 32; ++kk)
                        ws.segC[(seg_base * kD + 32 * q + kk) * kD + row] = hv[kk];
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t tc_prescan(const Problem &p, const Workspace &ws, cudaStream_t st) {
    PreArgs args;
    args.p = p;
    args.ws = ws;
    const uint64_t rows = (uint64_t)p.B * (uint64_t)p.T;
    const uint64_t H = (uint64_t)p.H;
    if (!make_tmap_bf16_3d(&args.tk, p.k, kD, H, rows, p.sk.h * 2, p.sk.t * 2, 64, 1, 64))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(k_tc_prescan,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemLaunch);
    if (err != cudaSuccess) return err;
    const int64_t chains = p.N * ws.n_segments * p.H;
    return launch_pdl(k_tc_prescan, dim3((unsigned)persistent_grid(p, chains, 1)),
                      dim3(kThreads), kSmemLaunch, st, args);
}

}  // namespace gdr
