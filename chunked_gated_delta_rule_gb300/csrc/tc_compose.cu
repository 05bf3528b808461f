// tc_compose.cu -- A9 on the tensor cores: the ordered segment composition
// h_{s+1} = M_s h_s + c_s of the delta rule (K = V = 128), the short ordered
// pass that chains the per-segment FP32 transitions (cuLA PR #127 "Root
// cause and implementation").
//
// One CTA carries a whole (sequence, head) -- all 128 value columns -- so a
// batch of many heads needs no more CTAs than it has heads, and a step is one
// 128 x 128 x 128 product on tcgen05 instead of a K x K x (a few columns)
// product on CUDA cores per CTA.  The state X (K x V, FP32) is kept
// transposed in TMEM; a step forms
//
//   D = X_{s+1}^T = c_s^T + X_s^T M_s^T      (D preloaded with c_s^T)
//
// with FP32 operands carried as BF16 pairs (x = hi + lo, about 16
// significant bits): D += Xl Mh^T + Xh Ml^T + Xh Mh^T, the lo x lo term (a
// relative 2^-16 of the product) dropped.  X^T's hi and lo parts are the A
// operands, in TMEM; M_s's B images (hi and lo, MN-major, 128-byte swizzled:
// the pre-scan writes them beside its FP32 summaries) are bulk-copied into
// shared memory one step ahead, and c_s is read into the next-but-one D
// buffer (three of them) while a step runs.
//
// Two-level form (a composition of S segments in about 2 sqrt(S) ordered
// steps): level 1 forms, for every group of G consecutive segments in
// parallel, its transition A_g = M_e ... M_b and offset d_g (the same steps
// from X = M_b with no offset, and from X = c_b); level 2 chains the groups
// from h0 (writing every group's first segment state, and ht); level 3 fills
// in the states inside every group from its first one, in parallel.  Level
// 0 is the single ordered pass over all segments.  Every product has one
// fixed order, whatever the grid.
//
// Warps: 0 issues the MMAs; 1 bulk-loads the B images; 2-9 (twice the four
// TMEM lane quarters, half the keys each) read D, form the next X^T hi / lo
// (keys 0-63 first: the next step's first four K-steps start on them while
// keys 64-127 are formed) and write the states; 10-17 (likewise) preload the
// D buffer two steps ahead with c_s^T (or zeros), from memory.
// Each CTA walks runs blockIdx.x, blockIdx.x + gridDim.x, ...; every role
// counts the same steps, so buffers and barrier phases follow one global
// step counter.  Every wait is time-bounded: on expiry the CTA records
// GDR_ERR_TIMEOUT in the status word and every role leaves.
#include "gdr_internal.cuh"
#include "gdr_segments.cuh"
#include "tc_chunk.cuh"

namespace gdr {
namespace {

using namespace tc;

constexpr int kThreads = 576;
constexpr int kCD = 128;  // K = V
constexpr int kND = 3;    // D buffers: the offsets are read two steps ahead

// Shared memory (1024-aligned base): two buffers of the hi and lo B images,
// barriers.
constexpr uint32_t kOffImg = 0;                    // [2] x (hi 32 KB, lo 32 KB)
constexpr uint32_t kImgLo = 32768;
constexpr uint32_t kOffBar = kOffImg + 2 * 65536;
enum : int {
    kBIready = 0,   // [2] B images landed (bulk-copy bytes)
    kBIfree = 2,    // [2] B images read (commit)
    kBCready = 4,   // [3] D preloaded with c_s^T (c warps, 256)
    kBDdone = 7,    // [3] step's products done (commit)
    kBDfree = 10,   // [3] D read (state warps, 256)
    kBXready = 13,  // [2] X^T hi / lo of keys 0-63, then 64-127, written (state warps, 256)
    kBDrain = 15,   // every issued MMA done (commit, at the end)
    kNumBars = 16
};
constexpr uint32_t kOffMisc = kOffBar + 8 * kNumBars;  // TMEM base, abort flag
constexpr uint32_t kSmemLaunch = kOffMisc + 16 + 1024;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColD = 0;     // [3] D, FP32, 128 columns each
constexpr uint32_t kColXh = 384;  // X^T hi, two BF16 a column
constexpr uint32_t kColXl = 448;  // X^T lo
// D[c][r] += sum_m A[c][m] B[r][m]: A = X^T (K-major, TMEM), B = M with
// B[r][m] at row m of the image (MN-major: r contiguous)
constexpr uint32_t kIdesc = idesc_bf16(128, 128, 0, 1);

struct ComposeArgs {
    Problem p;
    Workspace ws;
    int level;  // 0 single pass; 1 group transitions and offsets; 2 over groups; 3 inside groups
};

// One run of ordered steps of one (sequence, head[, group]).
struct Run {
    int64_t nh;   // sequence * H + head
    int nseg;     // the sequence's segments
    int grp;      // group (levels 1 and 3)
    int kind;     // level 1: 0 the group's transition, 1 its offset
    int b0, e;    // the group's segments [b0, e) (levels 1 and 3)
    int nsteps;   // -1: nothing to do
    int stop;     // nothing to do for this run and every later one
};

__device__ __forceinline__ int64_t n_runs(const Problem &p, const Workspace &ws, int level) {
    const int64_t heads = p.N * p.H;
    const int64_t ngm = ws.grp_size ? (ws.n_segments + ws.grp_size - 1) / ws.grp_size : 1;
    return level == 1 ? heads * ngm * 2 : level == 3 ? heads * ngm : heads;
}

// Runs in order of descending sequence length, heads (and groups) fastest.
__device__ Run decode(const Problem &p, const Workspace &ws, int level, int64_t r) {
    Run u{};
    const int H = (int)p.H, G = ws.grp_size;
    const int ngm = G ? (ws.n_segments + G - 1) / G : 1;
    if (level == 1) {
        u.kind = (int)(r & 1);
        r >>= 1;
    }
    if (level == 1 || level == 3) {
        u.grp = (int)(r % ngm);
        r /= ngm;
    }
    const int h = (int)(r % H);
    const int64_t n = ws.seq_order[r / H];
    u.nh = n * H + h;
    const int nc = ws.seq_chunk0[n + 1] - ws.seq_chunk0[n];
    const int per = seg_per(ws, nc);
    u.nseg = per ? (nc + per - 1) / per : 0;
    const bool ht = p.ht != nullptr;
    // at most one segment under the common length: the output pass runs the
    // sequence whole, from h0 to ht (and, in the exact order, every later one)
    if (seg_len(ws) && u.nseg <= 1) {
        u.nsteps = -1;
        u.stop = whole_from_here(ws, nc, per) ? 1 : 0;
        return u;
    }
    if (level == 0) {
        u.nsteps = u.nseg == 0 ? 0 : u.nseg - 1 + (ht ? 1 : 0);
    } else {
        const int ng = (u.nseg + G - 1) / G;
        if (level == 2) {
            u.nsteps = u.nseg == 0 ? 0 : ng - 1 + (ht ? 1 : 0);
        } else {
            u.b0 = u.grp * G;
            u.e = min(u.nseg, u.b0 + G);
            // level 1: only the groups that level 2 steps over
            const bool used = level == 1 ? u.grp < ng - 1 + (ht ? 1 : 0) : u.grp < ng;
            u.nsteps = used ? u.e - u.b0 - 1 : -1;
        }
    }
    return u;
}

// Transition of step j of a run: its B images (a segment's, or at level 2
// a group's).
__device__ __forceinline__ const uint8_t *trans_img(const Workspace &ws, int level, const Run &u,
                                                   int j) {
    const int64_t S = ws.n_segments;
    if (level == 2) {
        const int64_t ngm = (S + ws.grp_size - 1) / ws.grp_size;
        return ws.grpAimg + (u.nh * ngm + j) * 65536;
    }
    const int s = level == 0 ? j : level == 1 ? u.b0 + 1 + j : u.b0 + j;
    return ws.segMimg + (u.nh * S + s) * 65536;
}

// Offset of step j of a run ([r][c]), or nullptr for none.
__device__ __forceinline__ const float *offset_of(const Workspace &ws, int level, const Run &u,
                                                  int j) {
    const int64_t KV = (int64_t)kCD * kCD, S = ws.n_segments;
    if (level == 2) {
        const int64_t ngm = (S + ws.grp_size - 1) / ws.grp_size;
        return ws.grpD + (u.nh * ngm + j) * KV;
    }
    if (level == 1 && u.kind == 0) return nullptr;
    const int s = level == 0 ? j : level == 1 ? u.b0 + 1 + j : u.b0 + j;
    return ws.segC + (u.nh * S + s) * KV;
}

// 16 TMEM columns of this thread's lane from 16 registers (unwaited).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// x = hi + lo, both BF16 (round to nearest): the pair carries about 16
// significant bits of x.
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
    const float ha = __bfloat162float(__float2bfloat16_rn(a));
    const float hb = __bfloat162float(__float2bfloat16_rn(b));
    hi = pack_bf16x2(ha, hb);
    lo = pack_bf16x2(a - ha, b - hb);
}

__global__ void __launch_bounds__(kThreads, 1) k_tc_compose(const __grid_constant__ ComposeArgs args) {
    const Problem &p = args.p;
    const Workspace &ws = args.ws;
    const int level = args.level;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + kOffMisc);
    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
    const int row = 32 * (warp & 3) + lane_id;  // TMEM lane: value column c of X
    const uint32_t lane = (uint32_t)(32 * (warp & 3)) << 16;
    const int64_t S = ws.n_segments;
    const int64_t KV = (int64_t)kCD * kCD;
    const int64_t ngm = ws.grp_size ? (S + ws.grp_size - 1) / ws.grp_size : 1;

    // Waits on the ordered chain's critical path poll; the roles that run a
    // step ahead sleep between polls, leaving the issue slots to the warps on
    // the chain.
    auto wait = [&](int b, uint32_t parity) -> bool {
        return mbar_wait_or_abort(&bars[b], parity & 1u, p.status, s_abort);
    };
    auto wait_ahead = [&](int b, uint32_t parity) -> bool {
        if (mbar_try_wait(&bars[b], parity & 1u)) return true;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&bars[b], parity & 1u)) {
            if (*s_abort) return false;
            if (globaltimer_ns() - t0 > 2000000000ull) {
                if (p.status) atomicCAS(p.status, 0, (int32_t)GDR_ERR_TIMEOUT);
                *s_abort = 1;
                return false;
            }
            __nanosleep(256);
        }
        return true;
    };

    pdl_trigger();
    if (warp == 0) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) {
            // bulk-copy bytes and commits: one arrival; warp groups: 256
            const bool one = (b >= kBIready && b < kBCready) || (b >= kBDdone && b < kBDfree) ||
                              b == kBDrain;
            const uint32_t cnt = one ? 1u : 256u;
            mbar_init(&bars[b], cnt);
        }
        *s_abort = 0;
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    pdl_wait();  // the summaries, once the kernels before have finished

    const int64_t runs = n_runs(p, ws, level);
    if (warp == 1) {
        // ------------------------------------------------------------ loads
        if (lane_id == 0) {
            uint32_t g = 0;
            bool ok = true;
            for (int64_t r = blockIdx.x; ok && r < runs; r += gridDim.x) {
                const Run u = decode(p, ws, level, r);
                if (u.stop) break;
                for (int j = 0; j < u.nsteps; ++j, ++g) {
                    // the images, straight into a buffer once it is free
                    const uint32_t b = g & 1;
                    if (g >= 2 && !wait_ahead(kBIfree + b, (g >> 1) - 1)) { ok = false; break; }
                    const uint8_t *src = trans_img(ws, level, u, j);
                    mbar_arrive_expect_tx(&bars[kBIready + b], 65536u);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        bulk_load(sm + kOffImg + 65536 * b + 8192 * i, src + 8192 * i, 8192u,
                                  &bars[kBIready + b]);
                }
            }
        }
        __syncwarp();
    } else if (warp == 0) {
        // ------------------------------------------------------------ MMAs
        if (lane_id == 0) {
            uint32_t g = 0;
            bool ok = true;
            for (int64_t r = blockIdx.x; ok && r < runs; r += gridDim.x) {
                const Run u = decode(p, ws, level, r);
                if (u.stop) break;
                for (int j = 0; j < u.nsteps; ++j, ++g) {
                    const uint32_t b = g & 1, bd = g % kND;
                    if (!wait(kBIready + b, g >> 1) || !wait(kBCready + bd, g / kND)) {
                        ok = false;
                        break;
                    }
                    const uint32_t d = tmem + kColD + 128 * bd;
                    const uint32_t img = sb + kOffImg + 65536 * b;
                    // keys 0-63 as soon as X's first half is written, while the
                    // state warps form the second; per half, the small terms
                    // first: Xl Mh^T, Xh Ml^T, then Xh Mh^T
#pragma unroll
                    for (int hk = 0; hk < 2; ++hk) {
                        if (!wait(kBXready + hk, g)) break;
                        tc_fence_after();
#pragma unroll
                        for (int t = 0; t < 3; ++t) {
                            const uint32_t a = tmem + (t == 0 ? kColXl : kColXh);
                            const uint32_t bi = img + (t == 1 ? kImgLo : 0u);
#pragma unroll
                            for (int kk = 4 * hk; kk < 4 * hk + 4; ++kk)
                                umma_bf16_ts(d, a + 8 * kk, sdesc_sw128(bi + kk * 2048, 16384, 1024),
                                             kIdesc, 1u);
                        }
                    }
                    if (*s_abort) {
                        ok = false;
                        break;
                    }
                    umma_commit(&bars[kBDdone + bd]);
                    umma_commit(&bars[kBIfree + b]);
                }
            }
            // nothing of this CTA may still run on the tensor cores at exit
            umma_commit(&bars[kBDrain]);
            mbar_wait(&bars[kBDrain], 0, p.status, 100000000ull);
        }
        __syncwarp();
    } else if (warp >= 10) {
        // ------------------------------------------------------------ D preload
        // Warps 10-17: D^T row `row` = column `row` of c_s, keys [64 ch,
        // 64 ch + 64), read from memory (coalesced: a warp's loads of one key
        // cover 32 consecutive columns) into D two steps ahead.
        const int ch = (warp - 10) >> 2;
        uint32_t g = 0;
        bool ok = true;
        for (int64_t r = blockIdx.x; ok && r < runs; r += gridDim.x) {
            const Run u = decode(p, ws, level, r);
            if (u.stop) break;
            for (int j = 0; j < u.nsteps; ++j, ++g) {
                const uint32_t bd = g % kND;
                const bool got = g < (uint32_t)kND || wait_ahead(kBDfree + bd, g / kND - 1);
                if (!__all_sync(0xffffffffu, got ? 1 : 0)) {
                    ok = false;
                    break;
                }
                const float *c = offset_of(ws, level, u, j);
#pragma unroll 1
                for (int q = 0; q < 2; ++q) {
                    const int r0 = 64 * ch + 32 * q;
                    uint32_t v[32];
                    if (c) {
                        const float *src = c + (int64_t)r0 * kCD + row;
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__ldg(src + i * kCD));
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0u;
                    }
                    tmem_st32(tmem + lane + kColD + 128 * bd + r0, v);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars[kBCready + bd]);
            }
        }
    } else {
        // ------------------------------------------------------------ states
        // Warps 2-9: thread `row` of a lane quarter holds column c = row of
        // X, keys r in [32 eh, 32 eh + 32) and [64 + 32 eh, 96 + 32 eh): the
        // two groups of four warps together write keys 0-63 first.
        const int c = row;
        const int eh = (warp - 2) >> 2;
        auto rq = [&](int q) { return 64 * q + 32 * eh; };
        uint32_t g = 0;
        bool ok = true;
        // X^T row c (32 keys r0 .. r0 + 31) into the A operands
        auto put_x = [&](int r0, const float (&x)[32]) {
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) split2(x[2 * i], x[2 * i + 1], hi[i], lo[i]);
            tmem_st16(tmem + lane + kColXh + r0 / 2, hi);
            tmem_st16(tmem + lane + kColXl + r0 / 2, lo);
        };
        for (int64_t r = blockIdx.x; ok && r < runs; r += gridDim.x) {
            const Run u = decode(p, ws, level, r);
            if (u.stop) break;
            if (u.nsteps < 0) continue;
            const int64_t slot = u.nh * ngm + u.grp;  // level 1: the group's result
            // Where X (element (rr, c) at dst[rr * rstride]) goes after step j
            // (j = -1: X0): rows of segH, the group offset or transition, or ht.
            auto target = [&](int j, int64_t &rstride) -> float * {
                rstride = kCD;
                const bool last = j == u.nsteps - 1;
                if (level == 0 || level == 2) {
                    const int nxt = level == 0 ? j + 1 : (j + 1) * ws.grp_size;
                    if (nxt < u.nseg) return ws.segH + (u.nh * S + nxt) * KV + c;
                    return nullptr;  // ht (when last), below
                }
                if (level == 3) return j < 0 ? nullptr : ws.segH + (u.nh * S + u.b0 + j + 1) * KV + c;
                return last ? ws.grpD + slot * KV + c : nullptr;  // level 1, offsets
            };
            auto put_out = [&](int j, int r0, const float (&x)[32]) {
                if (level == 1 && u.kind == 0) {  // the group transition's B images: row c
                    if (j == u.nsteps - 1) {
                        uint8_t *img = ws.grpAimg + slot * 65536;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t o = sw128_off(c, r0 + 8 * i, 128);
                            st_split_bf16x8(img + o, img + kImgLo + o, x + 8 * i);
                        }
                    }
                    return;
                }
                int64_t rs;
                float *dst = target(j, rs);
                if (dst) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) dst[(int64_t)(r0 + i) * rs] = x[i];
                } else if ((level == 0 || level == 2) && p.ht &&
                           (j == u.nsteps - 1 || (j < 0 && u.nseg == 0))) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) p.ht[state_off(p, u.nh, r0 + i, c)] = x[i];
                }
            };
            // X0: h0 (levels 0, 2), a group's first segment state (3), its
            // first transition or offset (1)
#pragma unroll 1
            for (int q = 0; q < 2; ++q) {
                const int r0 = rq(q);
                float x[32];
                if (level == 0 || level == 2) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        x[i] = p.h0 ? p.h0[state_off(p, u.nh, r0 + i, c)] : 0.f;
                } else if (level == 3) {
                    const float *src = ws.segH + (u.nh * S + u.b0) * KV + (int64_t)r0 * kCD + c;
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[i] = src[i * kCD];
                } else if (u.kind == 0) {  // row c of the images: hi + lo
                    const uint8_t *img = ws.segMimg + (u.nh * S + u.b0) * 65536;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t o = sw128_off(c, r0 + 8 * i, 128);
                        float hi[8], lo[8];
                        ld_bf16x8(img + o, hi);
                        ld_bf16x8(img + kImgLo + o, lo);
#pragma unroll
                        for (int t = 0; t < 8; ++t) x[8 * i + t] = hi[t] + lo[t];
                    }
                } else {
                    const float *src = ws.segC + (u.nh * S + u.b0) * KV + (int64_t)r0 * kCD + c;
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[i] = src[i * kCD];
                }
                // segH of the first segment (levels 0, 2), ht of a sequence
                // without tokens, a one-segment group's result (level 1)
                put_out(-1, r0, x);
                if (u.nsteps > 0) {
                    put_x(r0, x);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&bars[kBXready + q]);
                }
            }
            if (u.nsteps == 0) continue;
            for (int j = 0; j < u.nsteps; ++j, ++g) {
                const uint32_t bd = g % kND;
                if (!__all_sync(0xffffffffu, wait(kBDdone + bd, g / kND) ? 1 : 0)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the next step's operands first (the ordered chain), then the
                // state's copy to memory from a second read of D, while the
                // next step's products run
                if (j + 1 < u.nsteps) {
#pragma unroll 1
                    for (int q = 0; q < 2; ++q) {  // keys 0-63, then 64-127
                        float x[32];
                        tmem_load32f(tmem + lane + kColD + 128 * bd + rq(q), x);
                        put_x(rq(q), x);
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(&bars[kBXready + q]);
                    }
                }
#pragma unroll 1
                for (int q = 0; q < 2; ++q) {
                    float x[32];
                    tmem_load32f(tmem + lane + kColD + 128 * bd + rq(q), x);
                    put_out(j, rq(q), x);
                }
                tc_fence_before();
                mbar_arrive(&bars[kBDfree + bd]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool compose_tc_supported(const Problem &p) {
    return p.beta != nullptr && p.K == kCD && p.V == kCD;
}

cudaError_t compose_tc(const Problem &p, const Workspace &ws, int level, cudaStream_t st) {
    ComposeArgs args;
    args.p = p;
    args.ws = ws;
    args.level = level;
    cudaError_t err = cudaFuncSetAttribute(k_tc_compose, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemLaunch);
    if (err != cudaSuccess) return err;
    const int64_t heads = p.N * p.H;
    const int64_t ngm = ws.grp_size ? (ws.n_segments + ws.grp_size - 1) / ws.grp_size : 1;
    const int64_t runs = level == 1 ? heads * ngm * 2 : level == 3 ? heads * ngm : heads;
    return launch_pdl(k_tc_compose, dim3((unsigned)persistent_grid(p, runs, 1)), dim3(kThreads),
                      kSmemLaunch, st, args);
}

}  // namespace gdr
