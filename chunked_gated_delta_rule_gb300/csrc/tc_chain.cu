// tc_chain.cu -- A6/A7 (and A8/A10 of the segment split) on the tensor-core
// path (BF16, K = V = 128, delta rule): the serial state scan and the output.
//
// Persistent CTAs (one per SM) pull chains -- all chunks of one (sequence,
// head), or of one (sequence, segment, head) -- longest first from an atomic
// counter.  Everything that does not depend on the state was done by
// tc_prep.cu for all chunks in parallel and left in one record per (chunk,
// head); here, per chunk, in order:
//
//   [v_new^T | O] = h^T [W; Q~]^T      (tcgen05, two N = 64 products: W^T
//                                       first, committed on its own; A is
//                                       the BF16 mirror of h^T)
//   v_new^T = U^T - (h^T W^T)
//   h^T <- e^{G_last} h^T + v_new^T K~  (tcgen05 accumulating onto the FP32
//                                       state in TMEM, pre-scaled)
//   O += v_new^T (scale P)^T            (tcgen05 onto the same columns)
//
// with Q~ = scale diag(e^G) Q formed by the prep kernel (so O is the output,
// one rounding to BF16) and K~ = diag(e^{G_last - G}) K formed here, in
// place in the stage.  The formulation is
// the transposed one (value columns are TMEM lanes), so every MMA has M =
// 128.  The A operands (the BF16 mirror of h^T and v_new^T) live in tensor
// memory, so an MMA reads only its B tile from shared memory: shared-memory
// bandwidth, which the stage loads, the K~ pass and the output staging also
// draw on, bounds a chunk's MMAs when A is read from there as well.  The
// warps specialise:
//   warps 0-3  the state path, which is the serial dependency: per chunk the
//              BF16 mirror of h^T (and h^T scaled by e^{G_last} in place),
//              then v_new^T once the first product lands, both written to
//              tensor memory;
//   warps 4-7  the side path: K~ in place once a chunk lands, then the
//              previous chunk's O, staged and stored (a TMA store for whole
//              chunks);
//   warp 8     control: issues every MMA;
//   warp 9     producer: claims chains, decodes them into a small ring that
//              the other roles read, and loads each chunk's record (the byte
//              image of a stage) with bulk copies, and its k tile by TMA,
//              into a two-stage ring;
//              the next chunk, also of the next chain, loads while this one
//              runs.
// Roles hand over through mbarriers; the first product's TMEM buffer is
// double-buffered, so the output of chunk c overlaps chunk c + 1.  Every
// wait is time-bounded: on expiry the CTA records GDR_ERR_TIMEOUT in the
// status word, the other roles leave too, and the CTA exits.
//
// Chunked form: the project statement; the state scan of fla's
// chunk_gated_delta_rule_fwd_kernel_h_blockdim64 (Kev PR #259 intro); the
// BF16 mirror used only as MMA operand with the state canonical in FP32 and
// the segment pre-scan with a K x K transition (cuLA PR #127 "Summary",
// "Root cause and implementation").
#include "gdr_internal.cuh"
#include "gdr_segments.cuh"
#include "tc_chunk.cuh"
#include "tma_host.cuh"

namespace gdr {
namespace {

using namespace tc;

// kModeRecompute: the serial scan of the tensor-core backward's forward
// recompute: no output; per chunk the byte image of the BF16 mirror of the
// state before the chunk, and v_new as a pair of BF16 images (hi + lo), go
// to the workspace for the backward's kernels.  kModeSegRecompute: the same
// per segment, from the composed segment states (the recompute's output
// pass when the sequences are split).
enum TcMode {
    kModeSerial = 0,
    kModePre = 1,
    kModeSegOut = 2,
    kModeRecompute = 3,
    kModeSegRecompute = 4
};

struct TcArgs {
    Problem p;
    Workspace ws;
    CUtensorMap tk;  // k, loaded into the stage for K~
    CUtensorMap to;  // the output o, for TMA stores of whole chunks
};

constexpr int kThreads = 320;  // warps 0-3 state, 4-7 side, 8 control, 9 producer
constexpr int kRing = 3;       // decoded chains handed out ahead (bounds the look-ahead)

// Shared memory (bytes from a 1024-aligned base).  One stage holds one
// record image (layout in tc_chunk.cuh):
//   W^T 16 KB: B operand of h^T W^T (MN-major, N = 64);
//   [Q~b0|Q~b1] 16 KB: B operand of h^T Q~^T (K-major, N = 64)
//   [K~b0|K~b1] 16 KB: B operand of the update (MN-major, N = 128), k as
//                      loaded, scaled in place
//   scale P 8 KB: B operand of O (K-major, N = 64); U^T 16 KB; vectors.
constexpr uint32_t kStage = kRecBytes;
constexpr uint32_t kOffOs = 2 * kStage;        // output staging, 16 KB
constexpr uint32_t kOffRing = kOffOs + 16384;  // decoded chains
enum : int {
    kBFull = 0,     // [2] stage landed (bulk-copy and TMA bytes)
    kBMready = 2,   // mirror written (state path, 128)
    kBAdone = 3,    // h^T W^T done (commit)
    kBVready = 4,   // v_new tile written, state scaled (state path, 128)
    kBHdone = 5,    // state update done (commit)
    kBO2 = 6,       // [2] O complete (commit)
    kBOfree = 8,    // [2] O buffer read (side path, 128)
    kBDrain = 10,   // every issued MMA done (commit, at the end)
    kBFree = 11,    // [2] every product reading the stage done (commit)
    kBKready = 13,  // [2] K~ formed in the stage (side path, 128)
    kBCfull = 15,   // [kRing] chain posted (producer)
    kBCempty = 15 + kRing,  // [kRing] chain read (state, side paths and control: 257)
    kNumBars = 15 + 2 * kRing
};

// One chain of the work list, decoded: (sequence n, segment s, head h[,
// transition]); valid == 0 ends the list; whole: an output-pass chain over
// a whole unsplit sequence (common segment length), from h0 to ht.
struct ChainDesc {
    int64_t n, tstart, tlen;  // the sequence's first token row and length
    int h, s, trans, c_begin, s0, s1, valid, whole;
};
static_assert(sizeof(ChainDesc) == 56, "chain descriptor layout");
constexpr uint32_t kOffBar = kOffRing + 64 * kRing;
constexpr uint32_t kOffMisc = kOffBar + 8 * kNumBars;  // TMEM base, abort flag
constexpr uint32_t kSmemLaunch = kOffMisc + 16 + 1024;

// TMEM columns (512 allocated; one CTA per SM).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColA = 0;    // two buffers of [h^T W^T | O], 128 columns each
constexpr uint32_t kColS = 256;  // FP32 state h^T, 128 columns
constexpr uint32_t kColM = 384;  // BF16 mirror of h^T, two keys a column, 64 columns
constexpr uint32_t kColV = 448;  // BF16 v_new^T, two tokens a column, 32 columns
static_assert(kColV + 32 <= kTmemCols, "TMEM columns");

constexpr uint32_t kIdescW = idesc_bf16(128, 64, 0, 1);   // B = W^T, MN-major
constexpr uint32_t kIdescQ = idesc_bf16(128, 64, 0, 0);   // B = Q~, K-major
constexpr uint32_t kIdescH = idesc_bf16(128, 128, 0, 1);
constexpr uint32_t kIdescO2 = idesc_bf16(128, 64, 0, 0);

// Named barrier of the side path's 128 threads; side_all also ANDs a flag
// across them, so that all of them take the same branch after a wait.
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

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) k_tc_chain(const __grid_constant__ TcArgs args) {
    const Problem &p = args.p;
    const Workspace &ws = args.ws;
    constexpr bool kOut = MODE == kModeSerial || MODE == kModeSegOut;
    constexpr bool kFromH0 = MODE == kModeSerial || MODE == kModeRecompute;
    constexpr bool kFromSeg = MODE == kModeSegOut || MODE == kModeSegRecompute;
    constexpr bool kImages = MODE == kModeRecompute || MODE == kModeSegRecompute;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + kOffMisc);
    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
    ChainDesc *ring = reinterpret_cast<ChainDesc *>(sm + kOffRing);

    const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
    const int row = 32 * (warp & 3) + lane_id;  // TMEM lane = matrix row
    const uint32_t lane = (uint32_t)(32 * (warp & 3)) << 16;
    const int H = (int)p.H;
    const int S = kFromH0 ? 1 : ws.n_segments;

    auto wait = [&](int b, uint32_t parity) -> bool {
        return mbar_wait_or_abort(&bars[b], parity & 1u, p.status, s_abort);
    };
    // Reads chain number k of the ring (all roles but the scheduler).
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
            if (b == kBMready || b == kBVready || b == kBOfree || b == kBOfree + 1 ||
                b == kBKready || b == kBKready + 1)
                cnt = 128;
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
    pdl_wait();  // the workspace and outputs, once the kernels before have finished

    if (warp == 9) {
        // ------------------------------------------------------------ producer
        // Work list: heads fastest, then (transition kind), segment, and the
        // sequences longest first; chains without chunks are skipped.
        if (lane_id == 0) {
            const int kinds = MODE == kModePre ? 2 : 1;
            const int total = (int)(p.N * S * H * kinds);
            int32_t *counter =
                ws.n_chunks + (MODE == kModeSerial || MODE == kModeRecompute ? kCtrSerial
                               : MODE == kModePre                            ? kCtrPre
                               : MODE == kModeSegOut                         ? kCtrSegOut
                                                                             : kCtrSegRecompute);
            int issued = 0;
            for (int posted = 0;; ++posted) {
                ChainDesc c{};
                while (true) {
                    const int id = atomicAdd(counter, 1);
                    if (id >= total) break;
                    int r = id;
                    c.h = r % H;
                    r /= H;
                    c.trans = 0;
                    if (MODE == kModePre) {
                        c.trans = r & 1;
                        r >>= 1;
                    }
                    c.s = r % S;
                    r /= S;
                    c.n = ws.seq_order[r];
                    c.c_begin = ws.seq_chunk0[c.n];
                    const int nc = ws.seq_chunk0[c.n + 1] - c.c_begin;
                    c.s0 = 0;
                    c.s1 = nc;
                    c.whole = 0;
                    if (!kFromH0) {
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
                    atomicMax(counter, (r + 1) * S * kinds * H);
                }
                const int slot = posted % kRing;
                if (posted >= kRing && !wait(kBCempty + slot, (uint32_t)(posted / kRing - 1)))
                    break;
                ring[slot] = c;
                mbar_arrive(&bars[kBCfull + slot]);
                if (!c.valid) break;
                bool ok = true;
                // every chunk's record, into stage issued & 1 once the chunk two
                // before has released it
                for (int cc = c.s0; cc < c.s1; ++cc, ++issued) {
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
                    if (kOut) {  // the image (but K~) and the k tile
                        mbar_arrive_expect_tx(bar, kImgBytes);
                        bulk_load(dst, rec, kImgK, bar);
                        tma_load_3d(dst + kImgK, &args.tk, bar, 0, c.h, tt);
                        tma_load_3d(dst + kImgK + 8192, &args.tk, bar, 64, c.h, tt);
                        bulk_load(dst + kImgP, rec + kImgP, kImgBytes - kImgP, bar);
                    } else {     // W, k, U^T (not for the transition), vectors
                        const uint32_t bytes = 16384u + 16384u + (kImgBytes - kImgVec) +
                                               (c.trans ? 0u : 16384u);
                        mbar_arrive_expect_tx(bar, bytes);
                        bulk_load(dst + kImgW, rec + kImgW, 16384u, bar);
                        tma_load_3d(dst + kImgK, &args.tk, bar, 0, c.h, tt);
                        tma_load_3d(dst + kImgK + 8192, &args.tk, bar, 64, c.h, tt);
                        if (!c.trans) bulk_load(dst + kImgU, rec + kImgU, 16384u, bar);
                        bulk_load(dst + kImgVec, rec + kImgVec, kImgBytes - kImgVec, bar);
                    }
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
                for (int cc = C.s0; cc < C.s1; ++cc, ++gk) {
                    const int b = gk & 1;
                    const uint32_t sta = sb + b * kStage;
                    if (!wait(kBFull + b, gk >> 1) || !wait(kBMready, gk) ||
                        (kOut && gk >= 2 && !wait(kBOfree + b, (gk >> 1) - 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // h^T W^T, then O = h^T Q~^T while v_new is formed (A = the
                    // mirror in TMEM)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_bf16_ts(tmem + kColA + 128 * b, tmem + kColM + 8 * kk,
                                     sdesc_sw128(sta + kImgW + kk * 2048, 16384, 1024), kIdescW,
                                     kk > 0);
                    umma_commit(&bars[kBAdone]);
                    if (kOut) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_bf16_ts(tmem + kColA + 128 * b + 64, tmem + kColM + 8 * kk,
                                         sdesc_sw128(sta + kImgQ + (kk >> 2) * 8192 + (kk & 3) * 32,
                                                     16, 1024),
                                         kIdescQ, kk > 0);
                    }
                    if (!wait(kBVready, gk) || !wait(kBKready + b, gk >> 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16_ts(tmem + kColS, tmem + kColV + 8 * kk,
                                     sdesc_sw128(sta + kImgK + kk * 2048, 8192, 1024), kIdescH, 1u);
                    umma_commit(&bars[kBHdone]);
                    if (kOut) {  // O += v_new^T (scale P)^T
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_bf16_ts(tmem + kColA + 128 * b + 64, tmem + kColV + 8 * kk,
                                         sdesc_sw128(sta + kImgP + kk * 32, 16, 1024), kIdescO2,
                                         1u);
                        umma_commit(&bars[kBO2 + b]);
                    }
                    umma_commit(&bars[kBFree + b]);
                }
            }
            // nothing of this CTA may still run on the tensor cores at exit
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
            const bool trans = C.trans != 0;
            const int64_t seg_base = (C.n * H + h) * (int64_t)S + C.s;
            // h0 / ht column `row` of this (sequence, head): element `key` at
            // st_base + key * (1 or kD) by the state layout
            const int64_t st_base = state_off(p, C.n * H + h, 0, row);
            for (int cc = C.s0; cc < C.s1; ++cc, ++gk) {
                const int b = gk & 1;
                const uint8_t *st = sm + b * kStage;
                if (!wait(kBFull + b, gk >> 1)) { ok = false; break; }
                tc_fence_after();  // the state written by the previous update product
                const float gam_last = reinterpret_cast<const float *>(st + kImgVec)[kImgGamLast];
                // the state before the chunk: column `row` of keys [64 hq, 64 hq + 64)
                auto state_half = [&](int hq, uint32_t (&r0)[32], uint32_t (&r1)[32]) {
                    if (cc == C.s0) {  // the chain's initial state
#pragma unroll
                        for (int kk = 0; kk < 64; ++kk) {
                            const int key = 64 * hq + kk;
                            float v = 0.f;
                            if (kFromH0 || C.whole) {
                                if (p.h0) v = p.h0[st_base + (p.state_vk ? key : key * kD)];
                            } else if (kFromSeg) {
                                v = ws.segH[(seg_base * kD + key) * kD + row];
                            } else if (trans) {
                                v = key == row ? 1.f : 0.f;
                            }
                            if (kk < 32) r0[kk] = __float_as_uint(v);
                            else r1[kk - 32] = __float_as_uint(v);
                        }
                    } else {
                        tmem_ld32(tmem + lane + kColS + 64 * hq, r0);
                        tmem_ld32(tmem + lane + kColS + 64 * hq + 32, r1);
                        tmem_wait_ld();
                        reg_fence(r0);
                        reg_fence(r1);
                    }
                };
                // h_pre -> BF16 mirror in TMEM (two keys a column; the first
                // product's A operand): the chain's critical path, so it goes
                // first.  The recompute also writes the mirror's byte image
                // (128-byte swizzled rows) for the backward's per-chunk
                // gradients.
                uint8_t *limg = kImages
                                    ? ws.bwd_lkimg + ((int64_t)(C.c_begin + cc) * H + h) * kLkImgBytes
                                    : nullptr;
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
                            *reinterpret_cast<uint4 *>(limg + kLkImgH + ox) =
                                make_uint4(m[4 * c8], m[4 * c8 + 1], m[4 * c8 + 2], m[4 * c8 + 3]);
                            *reinterpret_cast<uint4 *>(limg + kLkImgH + oy) =
                                make_uint4(m[16 + 4 * c8], m[16 + 4 * c8 + 1], m[16 + 4 * c8 + 2],
                                           m[16 + 4 * c8 + 3]);
                        }
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars[kBMready]);
                // then the FP32 state scaled by e^{G_last} for the update product,
                // while the first product runs
#pragma unroll 1
                for (int hq = 0; hq < 2; ++hq) {
                    uint32_t r0[32], r1[32];
                    state_half(hq, r0, r1);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        r0[i] = __float_as_uint(__uint_as_float(r0[i]) * gam_last);
                        r1[i] = __float_as_uint(__uint_as_float(r1[i]) * gam_last);
                    }
                    tmem_st32(tmem + lane + kColS + 64 * hq, r0);
                    tmem_st32(tmem + lane + kColS + 64 * hq + 32, r1);
                }
                if (!wait(kBAdone, gk)) { ok = false; break; }
                tc_fence_after();
                {  // v_new^T = U^T - h^T W^T, to TMEM as BF16 (two tokens a column)
                    uint32_t w0[32], w1[32], vv[32];
                    tmem_ld32(tmem + lane + kColA + 128 * b, w0);
                    tmem_ld32(tmem + lane + kColA + 128 * b + 32, w1);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        float u[32];
                        if (!trans) {
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
                        if (kImages) {  // v_new^T as BF16 hi + lo images
                            uint8_t *vimg =
                                ws.bwd_lkimg + ((int64_t)(C.c_begin + cc) * H + h) * kLkImgBytes;
#pragma unroll
                            for (int c8 = 0; c8 < 4; ++c8) {
                                const uint32_t ou = sw128_off(row, 32 * hh + 8 * c8, 128);
                                st_split_bf16x8(vimg + kLkImgVh + ou, vimg + kLkImgVl + ou,
                                                u + 8 * c8);
                            }
                        }
                    }
                    tmem_st32(tmem + lane + kColV, vv);
                }
                tmem_wait_st();  // v_new and the scaled state, before the update product
                tc_fence_before();
                mbar_arrive(&bars[kBVready]);
                if (!wait(kBHdone, gk)) { ok = false; break; }
            }
            if (!ok) break;
            if ((MODE == kModeSerial || C.whole) && C.s0 == C.s1) {  // no tokens: ht = h0 (or 0)
                if (p.ht) {
                    for (int key = 0; key < kD; ++key) {
                        const int64_t idx = st_base + (p.state_vk ? key : key * kD);
                        p.ht[idx] = p.h0 ? p.h0[idx] : 0.f;
                    }
                }
                continue;
            }
            const bool to_ht = (MODE == kModeSerial || (MODE == kModeSegOut && C.whole)) && p.ht;
            if (MODE == kModePre || to_ht) {
                tc_fence_after();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float hv[32];
                    tmem_load32f(tmem + lane + kColS + 32 * q, hv);
                    if (to_ht) {  // compile-time strides in either layout
                        float *dst = p.ht + st_base + (p.state_vk ? 32 * q : 32 * q * kD);
                        if (p.state_vk) {
#pragma unroll
                            for (int kk = 0; kk < 32; ++kk) dst[kk] = hv[kk];
                        } else {
#pragma unroll
                            for (int kk = 0; kk < 32; ++kk) dst[kk * kD] = hv[kk];
                        }
                    } else if (trans) {  // M_s stored transposed: row `row`, as the
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
                            float4 *dst = reinterpret_cast<float4 *>(
                                ws.segM + (seg_base * kD + row) * kD + 32 * q);
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
    } else {
        // ------------------------------------------------------------ side path
        const int tb = tid - 128;
        int k = 0, gk = 0;
        bool ok = true, stores = false, pending = false;
        int64_t p_t0 = 0;
        int p_len = 0, p_h = 0, p_gk = 0;
        uint8_t *os = sm + kOffOs;  // [t][v] as two swizzled 64-column blocks
        // A7 for chunk p_gk: its O tile, BF16, to the output.
        auto out_epilogue = [&]() -> bool {
            const int b = p_gk & 1;
            if (tb == 0 && stores) bulk_wait_read();  // the staging tile is free again
            // all side-path threads agree (and the staging tile's previous
            // contents are stored) before any of them goes on
            if (!side_all(wait(kBO2 + b, p_gk >> 1))) return false;
            tc_fence_after();
            uint32_t r0[32], r1[32];
            tmem_ld32(tmem + lane + kColA + 128 * b + 64, r0);
            tmem_ld32(tmem + lane + kColA + 128 * b + 96, r1);
            tmem_wait_ld();
            reg_fence(r0);
            reg_fence(r1);
            tc_fence_before();
            mbar_arrive(&bars[kBOfree + b]);
            uint8_t *col = os + (row >> 6) * 8192;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                *reinterpret_cast<__nv_bfloat16 *>(col + sw128_off(i, row & 63, 64)) =
                    __float2bfloat16_rn(__uint_as_float(r0[i]));
                *reinterpret_cast<__nv_bfloat16 *>(col + sw128_off(32 + i, row & 63, 64)) =
                    __float2bfloat16_rn(__uint_as_float(r1[i]));
            }
            if (p_len == kChunk) {
                fence_async_smem();
                side_sync();
                if (tb == 0) {
                    tma_store_3d(&args.to, os, 0, p_h, (int)p_t0);
                    tma_store_3d(&args.to, os + 8192, 64, p_h, (int)p_t0);
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
                    if (t < p_len)
                        *reinterpret_cast<uint4 *>(o + tok_at(p.so, p_t0 + t, p_h) + c16 * 8) =
                            *reinterpret_cast<const uint4 *>(os + (c16 >> 3) * 8192 +
                                                             sw128_off(t, (c16 & 7) * 8, 64));
                }
            }
            return true;
        };
        while (ok) {
            ChainDesc C;
            if (!take(k++, C) || !C.valid) break;
            for (int cc = C.s0; cc < C.s1; ++cc, ++gk) {
                const int b = gk & 1;
                uint8_t *st = sm + b * kStage;
                const int64_t rem = C.tlen - (int64_t)kChunk * cc;
                const int len = rem < kChunk ? (int)rem : kChunk;
                if (!wait(kBFull + b, gk >> 1)) { ok = false; break; }
                // K~ = diag(e^{G_last - G}) K in place; rows past the sequence
                // end (they belong to the next one) become zero.
                const float *dec = reinterpret_cast<const float *>(st + kImgDec);
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int c = tb + 128 * r;
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
                mbar_arrive(&bars[kBKready + b]);
                // then the output of the chunk before, whose products are done
                // or close to it
                if (kOut && pending && !out_epilogue()) { ok = false; break; }
                pending = kOut;
                p_t0 = C.tstart + (int64_t)kChunk * cc;
                p_len = len;
                p_h = C.h;
                p_gk = gk;
            }
        }
        if (ok && pending) out_epilogue();
        if (tb == 0 && stores) bulk_wait_read();
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
    return launch_pdl(k_tc_chain<MODE>, grid, dim3(kThreads), kSmemLaunch, st, args);
}

}  // namespace

bool tc_supported(const Problem &p) {
    // TMA and the 16-byte stores of partial chunks: aligned bases and strides
    return p.dtype == GDR_BF16 && p.K == kD && p.V == kD && p.beta != nullptr &&
           rows_aligned16(p.q, p.sq, 2) && rows_aligned16(p.k, p.sk, 2) &&
           rows_aligned16(p.v, p.sv, 2) && rows_aligned16(p.o, p.so, 2);
}

cudaError_t tc_chain(const Problem &p, const Workspace &ws, int mode, cudaStream_t st) {
    TcArgs args;
    args.p = p;
    args.ws = ws;
    const uint64_t rows = (uint64_t)p.B * (uint64_t)p.T;
    const uint64_t H = (uint64_t)p.H;
    if (!make_tmap_bf16_3d(&args.tk, p.k, kD, H, rows, p.sk.h * 2, p.sk.t * 2, 64, 1, 64))
        return cudaErrorInvalidValue;
    if (mode == 3 || mode == 4) {
        args.to = args.tk;  // the recompute writes no output
    } else if (!make_tmap_bf16_3d(&args.to, p.o, kD, H, rows, p.so.h * 2, p.so.t * 2, 64, 1, 64)) {
        return cudaErrorInvalidValue;
    }
    const int S = (mode == 0 || mode == 3) ? 1 : ws.n_segments;
    const int64_t chains = p.N * S * p.H * (mode == 1 ? 2 : 1);
    dim3 grid((unsigned)persistent_grid(p, chains, 1));
    switch (mode) {
    case 0: return launch_chain<kModeSerial>(args, grid, st);
    case 1: return launch_chain<kModePre>(args, grid, st);
    case 2: return launch_chain<kModeSegOut>(args, grid, st);
    case 3: return launch_chain<kModeRecompute>(args, grid, st);
    case 4: return launch_chain<kModeSegRecompute>(args, grid, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdr
