// tc_bwd_scan.cu -- the reverse state-gradient scan of the backward pass on
// the tensor cores (BF16, K = V = 128, delta rule, serial over the chunks of
// a sequence): the reverse dH recurrence the flash-linear-attention ABC
// issue #23 pages run chunk by chunk ("Problem": chunk_abc_bwd_kernel_dh;
// "Proposed Dataflow" step 4), for the gated delta rule's chunked form.
//
// With E the gradient of the loss with respect to the state at a chunk's
// end (K x V), the chunk's step, last chunk first, is
//
//   dV' = scale M^T dO + diag(lam) K E        (64 x V; M = causal(Q K^T * D))
//   E  <- e^{G_last} E + scale (diag(gamma) Q)^T dO - W^T dV'
//
// (lam_t = e^{G_last - G_t}, gamma_t = e^{G_t}).  Every operand but dO is
// part of the record the forward preparation kernel (tc_prep.cu) leaves per
// (chunk, head): W^T, Q~ = scale diag(gamma) Q, scale P (P = M), and the
// decay vectors; K~ = diag(lam) K is formed in place from the k tile, as the
// forward scan does.  In the transposed formulation (value columns are TMEM
// lanes, every MMA has M = 128), per chunk:
//
//   D  = dO^T (scale P)          tcgen05, A = the dO tile (MN-major)
//   D += E^T K~^T                tcgen05, A = the BF16 mirror of E^T;
//                                D = dV'^T, read back in FP32
//   E^T <- e^{G_last} E^T        (state path, in TMEM)
//   E^T += dO^T Q~               tcgen05
//   E^T += (-dV'^T) W            tcgen05, A = BF16 -dV'^T
//
// dV'^T is stored as a pair of BF16 images (hi + lo) and the E^T mirror as
// its byte image, for the per-chunk gradients (tc_bwd_grad.cu); dh0 is E
// after the sequence's first chunk.  The state stays FP32 in TMEM; its BF16 mirror,
// dV' and dO are the MMA operands (the route's tolerance covers them).  The
// mirror and -dV'^T, the A operands the state path forms, are written to
// tensor memory, so those products read only their B tiles from shared
// memory.
//
// Warps: 0-3 state path (the serial dependency: E mirror and image, decay,
// dV'), 4-7 side path (K~ in place; rows past a sequence's end zeroed in
// the k and dO tiles), 8 control (every MMA), 9 producer (chains longest
// first, record and tile loads into a two-stage ring, last chunk first).
// Every wait is time-bounded; on expiry the CTA records GDR_ERR_TIMEOUT in
// the status word and every role leaves.
#include "gdr_internal.cuh"
#include "tc_chunk.cuh"
#include "tma_host.cuh"

namespace gdr {
namespace {

using namespace tc;

struct BwdScanArgs {
    Problem p;
    Workspace ws;
    uint8_t *lkimg;     // [chunks][H][kLkImgBytes]: the E^T and dV'^T images written here
    const float *dht;   // state layout of h0, or nullptr
    float *dh0;         // state layout of h0, or nullptr
    CUtensorMap tk;     // k, loaded into the stage for K~
    CUtensorMap tdo;    // dO [rows][H][V]
};

constexpr int kThreads = 320;
constexpr int kRing = 3;

// Shared memory: two stages of the record image (layout in tc_chunk.cuh),
// with the dO tile in the U^T slot (two 64-column blocks, 128-byte
// swizzled rows of 64 tokens); chain ring, barriers.
constexpr uint32_t kStage = kRecBytes;
constexpr uint32_t kImgDo = kImgU;
constexpr uint32_t kOffRing = 2 * kStage;
enum : int {
    kBFull = 0,     // [2] stage landed
    kBMready = 2,   // mirror of E^T written (state path, 128)
    kBAdone = 3,    // D = dV'^T complete (commit)
    kBVready = 4,   // -dV'^T written, E^T decayed (state path, 128)
    kBHdone = 5,    // E^T update done (commit)
    kBDrain = 6,    // every issued MMA done (commit, at the end)
    kBFree = 7,     // [2] every product reading the stage done (commit)
    kBKready = 9,   // [2] K~ formed, padded rows zeroed (side path, 128)
    kBCfull = 11,   // [kRing] chain posted (producer)
    kBCempty = 11 + kRing,  // [kRing] chain read (state, side, control: 257)
    kNumBars = 11 + 2 * kRing
};

// One chain: (sequence n, head h, segment s) over the sequence's chunks
// [s0, s0 + nc), last first.
struct ChainDesc {
    int64_t n, tstart, tlen;
    int h, c_begin, nc, valid, s, s0, nseg, pad0;  // nseg: non-empty segments of the sequence
};
static_assert(sizeof(ChainDesc) == 56, "chain descriptor layout");
constexpr uint32_t kOffBar = kOffRing + 64 * kRing;
constexpr uint32_t kOffMisc = kOffBar + 8 * kNumBars;
constexpr uint32_t kSmemLaunch = kOffMisc + 16 + 1024;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColD = 0;    // two buffers of dV'^T (64 columns), 128 apart
constexpr uint32_t kColE = 256;  // FP32 E^T, 128 columns
constexpr uint32_t kColM = 384;  // BF16 mirror of E^T, two keys a column, 64 columns
constexpr uint32_t kColV = 448;  // BF16 -dV'^T, two tokens a column, 32 columns

constexpr uint32_t kIdescDP = idesc_bf16(128, 64, 1, 1);    // dO^T (scale P)
constexpr uint32_t kIdescEK = idesc_bf16(128, 64, 0, 0);    // E^T K~^T
constexpr uint32_t kIdescDQ = idesc_bf16(128, 128, 1, 1);   // dO^T Q~
constexpr uint32_t kIdescVW = idesc_bf16(128, 128, 0, 0);   // (-dV'^T) W

// MODE 0: serial, from dht at each sequence's end to dh0; 1: segment
// pre-scan, from E = 0 at each segment's end, storing only E at its start
// (the segment's offset; segment s of a sequence's nseg non-empty segments
// in slot nseg - 1 - s of the summaries, for the composition from the last
// segment to the first); 2: segment output pass, from the composed E at
// each segment's end (the same slot).  Modes 0 and 2 store the images.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) k_tc_bwd_scan(const __grid_constant__ BwdScanArgs args) {
    const Problem &p = args.p;
    const Workspace &ws = args.ws;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + kOffMisc);
    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
    ChainDesc *ring = reinterpret_cast<ChainDesc *>(sm + kOffRing);

    const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
    const int row = 32 * (warp & 3) + lane_id;  // TMEM lane = value column v
    const uint32_t lane = (uint32_t)(32 * (warp & 3)) << 16;
    const int H = (int)p.H;
    const int S = MODE == 0 ? 1 : ws.n_segments;
    constexpr bool kImages = MODE != 1;

    auto wait = [&](int b, uint32_t parity) -> bool {
        return mbar_wait_or_abort(&bars[b], parity & 1u, p.status, s_abort);
    };
    auto take = [&](int k, ChainDesc &c) -> bool {
        const int slot = k % kRing;
        if (!wait(kBCfull + slot, (uint32_t)(k / kRing))) return false;
        c = ring[slot];
        mbar_arrive(&bars[kBCempty + slot]);
        return true;
    };

    pdl_trigger();
    if (warp == 0) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) {
            uint32_t cnt = 1;
            if (b == kBMready || b == kBVready || b == kBKready || b == kBKready + 1) cnt = 128;
            if (b >= kBCempty) cnt = 257;
            mbar_init(&bars[b], cnt);
        }
        *s_abort = 0;
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    pdl_wait();

    if (warp == 9) {
        // ------------------------------------------------------------ producer
        // Chains: (sequence, head, segment), heads fastest, then segments,
        // sequences longest first; serially a sequence without chunks is
        // posted too (dh0 = dht), split an empty segment is skipped.  Chunks
        // of a chain load last first.
        if (lane_id == 0) {
            const int total = (int)(p.N * S * H);
            int32_t *counter =
                ws.n_chunks + (MODE == 0 ? kCtrBwdSerial : MODE == 1 ? kCtrBwdPre : kCtrBwdSegOut);
            int issued = 0;
            for (int posted = 0;; ++posted) {
                ChainDesc c{};
                while (true) {
                    const int id = atomicAdd(counter, 1);
                    if (id >= total) break;
                    c.h = id % H;
                    c.s = (id / H) % S;
                    c.n = ws.seq_order[id / H / S];
                    c.c_begin = ws.seq_chunk0[c.n];
                    const int nseq = ws.seq_chunk0[c.n + 1] - c.c_begin;
                    const int per = (nseq + S - 1) / S;  // the forward's segment bounds
                    c.s0 = min(nseq, c.s * per);
                    c.nc = min(nseq, c.s0 + per) - c.s0;
                    c.nseg = per ? (nseq + per - 1) / per : 0;
                    if (c.nc > 0 || MODE == 0) {
                        c.tstart = seq_start(p, c.n);
                        c.tlen = seq_end(p, c.n) - c.tstart;
                        c.valid = 1;
                        break;
                    }
                    // the sequence's later ids are empty too: skip them for all
                    atomicMax(counter, (id / H / S + 1) * S * H);
                }
                const int slot = posted % kRing;
                if (posted >= kRing && !wait(kBCempty + slot, (uint32_t)(posted / kRing - 1)))
                    break;
                ring[slot] = c;
                mbar_arrive(&bars[kBCfull + slot]);
                if (!c.valid) break;
                bool ok = true;
                for (int j = 0; j < c.nc; ++j, ++issued) {
                    const int cc = c.s0 + c.nc - 1 - j;
                    const int stage = issued & 1;
                    if (issued >= 2 && !wait(kBFree + stage, (uint32_t)((issued >> 1) - 1))) {
                        ok = false;
                        break;
                    }
                    const int64_t rid = (int64_t)(c.c_begin + cc) * H + c.h;
                    const uint8_t *rec = ws.rec + rid * kRecBytes;
                    uint64_t *bar = &bars[kBFull + stage];
                    uint8_t *dst = sm + stage * kStage;
                    const int tt = (int)(c.tstart + (int64_t)kChunk * cc);
                    mbar_arrive_expect_tx(bar, kImgBytes);
                    bulk_load(dst, rec, kImgK, bar);  // W^T, Q~
                    tma_load_3d(dst + kImgK, &args.tk, bar, 0, c.h, tt);
                    tma_load_3d(dst + kImgK + 8192, &args.tk, bar, 64, c.h, tt);
                    bulk_load(dst + kImgP, rec + kImgP, 8192u, bar);  // scale P
                    tma_load_3d(dst + kImgDo, &args.tdo, bar, 0, c.h, tt);
                    tma_load_3d(dst + kImgDo + 8192, &args.tdo, bar, 64, c.h, tt);
                    bulk_load(dst + kImgVec, rec + kImgVec, kImgBytes - kImgVec, bar);
                }
                if (!ok) break;
            }
        }
        __syncwarp();
    } else if (warp == 8) {
        // ------------------------------------------------------------ control
        if (lane_id == 0) {
            int k = 0, gk = 0;
            bool ok = true;
            while (ok) {
                ChainDesc C;
                if (!take(k++, C) || !C.valid) break;
                for (int j = 0; j < C.nc; ++j, ++gk) {
                    const int b = gk & 1;
                    const uint32_t sta = sb + b * kStage;
                    const uint32_t dcol = tmem + kColD + 128 * b;
                    // the stage, with K~ formed and the dO rows past a
                    // sequence's end zeroed
                    if (!wait(kBFull + b, gk >> 1) || !wait(kBKready + b, gk >> 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // D = dO^T (scale P), before E is known
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(dcol, sdesc_sw128(sta + kImgDo + kk * 2048, 8192, 1024),
                                  sdesc_sw128(sta + kImgP + kk * 2048, 8192, 1024), kIdescDP,
                                  kk > 0);
                    if (!wait(kBMready, gk)) { ok = false; break; }
                    tc_fence_after();
                    // D += E^T K~^T
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_bf16_ts(dcol, tmem + kColM + 8 * kk,
                                     sdesc_sw128(sta + kImgK + (kk >> 2) * 8192 + (kk & 3) * 32, 16,
                                                 1024),
                                     kIdescEK, 1u);
                    umma_commit(&bars[kBAdone]);
                    if (!wait(kBVready, gk)) { ok = false; break; }
                    tc_fence_after();
                    // E^T += dO^T Q~, then E^T += (-dV'^T) W
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + kColE, sdesc_sw128(sta + kImgDo + kk * 2048, 8192, 1024),
                                  sdesc_sw128(sta + kImgQ + kk * 2048, 8192, 1024), kIdescDQ, 1u);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16_ts(tmem + kColE, tmem + kColV + 8 * kk,
                                     sdesc_sw128(sta + kImgW + kk * 32, 16, 1024), kIdescVW, 1u);
                    umma_commit(&bars[kBHdone]);
                    umma_commit(&bars[kBFree + b]);
                }
            }
            umma_commit(&bars[kBDrain]);
            mbar_wait(&bars[kBDrain], 0, p.status, 100000000ull);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------------ state path
        int k = 0, gk = 0;
        bool ok = true;
        while (ok) {
            ChainDesc C;
            if (!take(k++, C) || !C.valid) break;
            const int h = C.h;
            // dht / dh0 column `row` of this (sequence, head): key at
            // st_base + key * kst, by the state layout
            const int64_t st_base = state_off(p, C.n * H + h, 0, row);
            const int64_t kst = p.state_vk ? 1 : kD;
            // the segment's summary slot: segment s of the sequence's nseg
            // non-empty ones in slot nseg - 1 - s, so that the composition
            // runs from the last segment to the first
            const int64_t slot = (C.n * H + h) * (int64_t)S + (C.nseg - 1 - C.s);
            for (int j = 0; j < C.nc; ++j, ++gk) {
                const int cc = C.s0 + C.nc - 1 - j;
                const int b = gk & 1;
                const uint8_t *st = sm + b * kStage;
                const int64_t item = (int64_t)(C.c_begin + cc) * H + h;
                if (!wait(kBFull + b, gk >> 1)) { ok = false; break; }
                tc_fence_after();  // E^T written by the previous update
                const float gam_last = reinterpret_cast<const float *>(st + kImgVec)[kImgGamLast];
                // E at the chunk's end, keys [64 hq, 64 hq + 64) of column `row`
                auto state_half = [&](int hq, uint32_t (&r0)[32], uint32_t (&r1)[32]) {
                    if (j == 0) {  // the chain's end: dht (or 0), 0, or the composed E
#pragma unroll
                        for (int kk = 0; kk < 64; ++kk) {
                            const int key = 64 * hq + kk;
                            float v = 0.f;
                            if (MODE == 0) {
                                if (args.dht) v = args.dht[st_base + key * kst];
                            } else if (MODE == 2) {
                                v = ws.segH[(slot * kD + key) * kD + row];
                            }
                            if (kk < 32) r0[kk] = __float_as_uint(v);
                            else r1[kk - 32] = __float_as_uint(v);
                        }
                    } else {
                        tmem_ld32(tmem + lane + kColE + 64 * hq, r0);
                        tmem_ld32(tmem + lane + kColE + 64 * hq + 32, r1);
                        tmem_wait_ld();
                        reg_fence(r0);
                        reg_fence(r1);
                    }
                };
                // E's BF16 mirror (the A operand of E^T K~^T), and its image
                // for the per-chunk gradients: the chain's critical path goes first
                uint8_t *limg = args.lkimg + item * kLkImgBytes;
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
                    tmem_st32(tmem + lane + kColM + 32 * hq, m);
                    if (kImages) {
#pragma unroll
                        for (int c8 = 0; c8 < 4; ++c8) {
                            const uint32_t ox = sw128_off(row, 64 * hq + 8 * c8, 128);
                            const uint32_t oy = sw128_off(row, 64 * hq + 32 + 8 * c8, 128);
                            *reinterpret_cast<uint4 *>(limg + kLkImgE + ox) =
                                make_uint4(m[4 * c8], m[4 * c8 + 1], m[4 * c8 + 2], m[4 * c8 + 3]);
                            *reinterpret_cast<uint4 *>(limg + kLkImgE + oy) =
                                make_uint4(m[16 + 4 * c8], m[16 + 4 * c8 + 1], m[16 + 4 * c8 + 2],
                                           m[16 + 4 * c8 + 3]);
                        }
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars[kBMready]);
                // E^T decayed by e^{G_last} in TMEM, while D is formed
#pragma unroll 1
                for (int hq = 0; hq < 2; ++hq) {
                    uint32_t r0[32], r1[32];
                    state_half(hq, r0, r1);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        r0[i] = __float_as_uint(__uint_as_float(r0[i]) * gam_last);
                        r1[i] = __float_as_uint(__uint_as_float(r1[i]) * gam_last);
                    }
                    tmem_st32(tmem + lane + kColE + 64 * hq, r0);
                    tmem_st32(tmem + lane + kColE + 64 * hq + 32, r1);
                }
                if (!wait(kBAdone, gk)) { ok = false; break; }
                tc_fence_after();
                {  // dV'^T: its hi + lo images for the gradients, -dV'^T in BF16 for the update
                    uint32_t w0[32], w1[32];
                    tmem_ld32(tmem + lane + kColD + 128 * b, w0);
                    tmem_ld32(tmem + lane + kColD + 128 * b + 32, w1);
                    tmem_wait_ld();
                    reg_fence(w0);
                    reg_fence(w1);
                    uint8_t *dimg = args.lkimg + item * kLkImgBytes;
                    uint32_t vv[32];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                        for (int c8 = 0; c8 < 4; ++c8) {
                            float d[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                d[i] = __uint_as_float(hh ? w1[8 * c8 + i] : w0[8 * c8 + i]);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                vv[16 * hh + 4 * c8 + i] = pack_bf16x2(-d[2 * i], -d[2 * i + 1]);
                            if (kImages) {
                                const uint32_t ou = sw128_off(row, 32 * hh + 8 * c8, 128);
                                st_split_bf16x8(dimg + kLkImgDh + ou, dimg + kLkImgDl + ou, d);
                            }
                        }
                    }
                    tmem_st32(tmem + lane + kColV, vv);
                }
                tmem_wait_st();  // -dV'^T and the decayed state, before the update products
                tc_fence_before();
                mbar_arrive(&bars[kBVready]);
                if (!wait(kBHdone, gk)) { ok = false; break; }
            }
            if (!ok) break;
            if (MODE == 1) {  // E at the segment's start: its offset
                tc_fence_after();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float hv[32];
                    tmem_load32f(tmem + lane + kColE + 32 * q, hv);
#pragma unroll
                    for (int kk = 0; kk < 32; ++kk)
                        ws.segC[(slot * kD + 32 * q + kk) * kD + row] = hv[kk];
                }
            } else if (MODE == 0 && args.dh0) {
                if (C.nc == 0) {  // no tokens: dh0 = dht (or 0)
                    for (int key = 0; key < kD; ++key) {
                        const int64_t idx = st_base + key * kst;
                        args.dh0[idx] = args.dht ? args.dht[idx] : 0.f;
                    }
                } else {  // E after the sequence's first chunk
                    tc_fence_after();
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float hv[32];
                        tmem_load32f(tmem + lane + kColE + 32 * q, hv);
#pragma unroll
                        for (int kk = 0; kk < 32; ++kk) args.dh0[st_base + (32 * q + kk) * kst] = hv[kk];
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ side path
        const int tb = tid - 128;
        int k = 0, gk = 0;
        bool ok = true;
        while (ok) {
            ChainDesc C;
            if (!take(k++, C) || !C.valid) break;
            for (int j = 0; j < C.nc; ++j, ++gk) {
                const int cc = C.s0 + C.nc - 1 - j;
                const int b = gk & 1;
                uint8_t *st = sm + b * kStage;
                const int64_t rem = C.tlen - (int64_t)kChunk * cc;
                const int len = rem < kChunk ? (int)rem : kChunk;
                if (!wait(kBFull + b, gk >> 1)) { ok = false; break; }
                // K~ = diag(e^{G_last - G}) K in place; rows past the sequence
                // end (they belong to the next one) become zero, in dO too
                const float *dec = reinterpret_cast<const float *>(st + kImgDec);
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int c = tb + 128 * r;
                    const int t = c >> 4;
                    const uint32_t off = ((c >> 3) & 1) * 8192 + t * 128 + (c & 7) * 16;
                    uint8_t *ptr = st + kImgK + off;
                    if (t < len) {
                        float x[8];
                        ld_bf16x8(ptr, x);
                        const float d = dec[t];
#pragma unroll
                        for (int u = 0; u < 8; ++u) x[u] *= d;
                        st_bf16x8(ptr, x);
                    } else {
                        st_shared_v4(ptr, 0u, 0u, 0u, 0u);
                        st_shared_v4(st + kImgDo + off, 0u, 0u, 0u, 0u);
                    }
                }
                fence_async_smem();
                mbar_arrive(&bars[kBKready + b]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}


template <int MODE>
cudaError_t launch_scan(const BwdScanArgs &args, dim3 grid, cudaStream_t st) {
    cudaError_t err = cudaFuncSetAttribute(k_tc_bwd_scan<MODE>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemLaunch);
    if (err != cudaSuccess) return err;
    return launch_pdl(k_tc_bwd_scan<MODE>, grid, dim3(kThreads), kSmemLaunch, st, args);
}

}  // namespace

cudaError_t tc_bwd_scan(const Problem &p, const Workspace &ws, int mode, const float *dht,
                        float *dh0, const void *dout, cudaStream_t st) {
    BwdScanArgs args;
    args.p = p;
    args.ws = ws;
    args.lkimg = ws.bwd_lkimg;
    args.dht = dht;
    args.dh0 = dh0;
    const uint64_t rows = (uint64_t)p.B * (uint64_t)p.T;
    const uint64_t H = (uint64_t)p.H;
    if (!make_tmap_bf16_3d(&args.tk, p.k, kD, H, rows, p.sk.h * 2, p.sk.t * 2, 64, 1, 64) ||
        !make_tmap_bf16_3d(&args.tdo, dout, kD, H, rows, kD * 2, H * kD * 2, 64, 1, 64))
        return cudaErrorInvalidValue;
    const int S = mode == 0 ? 1 : ws.n_segments;
    const dim3 grid((unsigned)persistent_grid(p, p.N * S * p.H, 1));
    switch (mode) {
    case 0: return launch_scan<0>(args, grid, st);
    case 1: return launch_scan<1>(args, grid, st);
    case 2: return launch_scan<2>(args, grid, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdr
