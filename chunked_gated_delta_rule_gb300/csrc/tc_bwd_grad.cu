// tc_bwd_grad.cu -- every per-chunk gradient of the backward pass on the
// tensor cores (the tensor-core route: BF16 inputs, K = V = 128, delta rule).
// Per (chunk, head), with h the state before the chunk (forward recompute),
// E the gradient at the chunk's end and dV' the gradient of the chunk's v_new
// V' (reverse scan), T = (I + A)^-1 and the gate factors of the chunked form
// (gamma = e^G, lam = e^{G_last - G}, D_ij = e^{G_i - G_j}):
//
//   dVb = T^T dV'                      dv = diag(beta) dVb
//   dm  = dO V'^T,  Y = dVb V'^T       Z = scale causal(dm) * D,  dA = -strict_lower(Y)
//   S   = diag(beta) dA * D            dKb = -dVb h^T
//   dq  = scale diag(gamma) dO h^T + Z K
//   dk  = diag(lam) V' E^T + Z^T Q + (S + S^T) K + diag(beta gamma) dKb
//   dbeta, dg: row sums of the same terms (below)
//
// Y = T^T (dT T^T) with dT = dV' B'^T the gradient of T in V' = T B'
// (B' = diag(beta)(V - diag(gamma) K h)): dT T^T = dV' (T B')^T = dV' V'^T,
// so neither dT nor B' is formed.
//
// Every product runs on tcgen05 (kind::f16, FP32 accumulators in TMEM).
// The BF16 inputs q, k, dO and the chains' BF16 h and E mirrors enter as
// they are; every FP32 operand (T, dV', V', dVb, Z, S) enters as a
// pair of BF16 tiles hi + lo (lo = x - hi, rounded), so each product carries
// about 16 significant bits of its FP32 operands and the local gradients
// keep FP32-grade accuracy.  Products whose rows are tokens are stacked to
// M = 128: [Q; K] K^T, [dO; dVb] V'^T; the rest are transposed, keys or
// value columns on the TMEM lanes and tokens as N = 64.
//
// Persistent CTAs (one per SM) stride over the (chunk, head) items in three
// MMA groups per item, each followed by an epilogue that reads TMEM; the
// epilogue work the next group does not need runs while that group
// executes, and the next item's tiles load during the last epilogue.  dq,
// dk and dv turn from columns into rows through a small per-warp buffer and
// leave in 16-byte pieces.  Row
// sums over keys or values are warp transposing reductions in a fixed order,
// so results are identical at any grid.  Every wait is time-bounded.
#include "gdr_internal.cuh"
#include "tc_chunk.cuh"
#include "tma_host.cuh"

namespace gdr {
namespace {

using namespace tc;

struct GradArgs {
    Problem p;
    Workspace ws;
    BwdArgs a;
    CUtensorMap tq, tk, tv, tdo;
};

constexpr int kThreads = 256;

// Shared memory.  BF16 tiles are 128-byte swizzled (sw128_off), 64 rows per
// 8 KB block of 64 columns unless noted.
//   H  [0, 32 KB)      h^T image [v][key], two key blocks of 128 rows
//   B  [32, 80 KB)     per value block b (24 KB): dO rows | dVb hi | dVb lo;
//                      the E^T image's key block b sits in the dVb rows until
//                      dVb is written
//   C  [80, 112 KB)    per key block b (16 KB): q rows | k rows
//   D  [112, 144 KB)   V'^T hi | V'^T lo ([v][t], 128 rows)
//   F  [144, 192 KB)   dV'^T hi | dV'^T lo ([v][i], 128 rows) | T hi | T lo
//                      ([i][j]); after the first group: Z hi | Z lo | S hi
//                      | S lo ([i][j])
//   V  [192, 208 KB)   v rows
//   G, beta of the item (FP32, 512 B); per warp 1 KB where a 16-token x
//   32-column block of dq, dk or dv turns from columns into rows; the FP32
//   scalars
// The images arrive by bulk copies, dO, q, k and v by TMA, in two groups:
// H, B, D, V and the vectors once the item before has finished its second
// group of products, C and F once it has finished its last.
constexpr uint32_t kOffH = 0;
constexpr uint32_t kOffB = 32768;
constexpr uint32_t kBlkB = 24576;
constexpr uint32_t kOffC = kOffB + 2 * kBlkB;
constexpr uint32_t kBlkC = 16384;
constexpr uint32_t kOffD = kOffC + 2 * kBlkC;
constexpr uint32_t kOffF = kOffD + 32768;
constexpr uint32_t kFdvHi = 0, kFdvLo = 16384, kFtHi = 32768, kFtLo = 40960;
constexpr uint32_t kFzHi = 0, kFzLo = 8192, kFsHi = 16384, kFsLo = 24576;
constexpr uint32_t kOffV = kOffF + 49152;
constexpr uint32_t kOffVec = kOffV + 16384;
constexpr uint32_t kOffOut = kOffVec + kLkImgVecBytes;  // per warp 1 KB: output rows in transit
constexpr uint32_t kOffMisc = kOffOut + 8 * 1024;
// FP32 scalars in the misc area: gate vectors, per-warp partial row sums
constexpr int kVG = 0, kVGam = 64, kVLam = 128, kVB = 192, kVEp = 256;
constexpr int kR1 = 320, kR2 = kR1 + 256, kR3 = kR2 + 256, kR4 = kR3 + 256;  // [4 lane quarters][64]
constexpr int kRowR = kR4 + 256, kColR = kRowR + 128, kRdA = kColR + 128, kColRA = kRdA + 128;  // [2][64]
constexpr int kR3f = kColRA + 128, kDg = kR3f + 64, kEh = kDg + 64;
constexpr int kMiscFloats = kEh + 8;
constexpr uint32_t kOffBar = kOffMisc + kMiscFloats * 4;
constexpr int kNumBars = 5;  // first load group landed, groups 1-3 done, second load group landed
constexpr uint32_t kSmemLaunch = kOffBar + 8 * kNumBars + 16 + 1024;
static_assert(kOffBar % 8 == 0, "barrier alignment");
static_assert(kSmemLaunch <= 232448, "shared memory per CTA");
constexpr uint32_t kLoadA = 3 * 32768 + 2 * 16384 + kLkImgVecBytes;  // h, E, V'; dO, v; G, beta
constexpr uint32_t kLoadB = 2 * 16384 + 32768 + 16384;                // q, k; dV', T

// TMEM columns (128 lanes each, FP32).  Products of an FP32 operand's hi and
// lo halves run as one N = 128 MMA into two 64-column halves, summed when
// read; a region is reused once its readers are done:
//   group 1: P1 [0, 64)  P3 [64, 192)  [Q K^T; K K^T] [192, 256)  dVb^T [256, 384)
//   group 2: [dm; Y] [256, 384)  dVb lo V' hi^T (rows 64-127) [384, 448)  dVb h^T [448, 512)
//   group 3: (Z K)^T [192, 320)  (Z^T Q + S^T K + S K)^T [320, 448)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kCP1 = 0;     // (dO h^T)^T            [key][t]
constexpr uint32_t kCP3 = 64;    // (V' E^T)^T            [key][t], hi | lo halves
constexpr uint32_t kCQK = 192;   // [Q K^T; K K^T]        [t | 64 + t][j]
constexpr uint32_t kCDvb = 256;  // dVb^T [v][j]: T hi | T lo halves (dV' lo T hi in the first)
constexpr uint32_t kCDmY = 256;  // [dO V'^T; dVb V'^T]  [i | 64 + i][j], V' hi | lo halves
constexpr uint32_t kCD2 = 384;   // rows 64-127: dVb lo V' hi^T
constexpr uint32_t kCKb = 448;   // (dVb h^T)^T           [key][i]
constexpr uint32_t kCXq = 192;   // (Z K)^T               [key][i], Z hi | lo halves
constexpr uint32_t kCXk = 320;   // (Z^T Q + S^T K + S K)^T, hi | lo halves

constexpr uint32_t kIdMnK = idesc_bf16(128, 64, 1, 0);    // A MN-major, B K-major
constexpr uint32_t kIdKK = idesc_bf16(128, 64, 0, 0);     // both K-major
constexpr uint32_t kIdKMn = idesc_bf16(128, 64, 0, 1);    // A K-major, B MN-major
constexpr uint32_t kIdMnMn2 = idesc_bf16(128, 128, 1, 1);  // N = 128 (hi | lo)
constexpr uint32_t kIdKMn2 = idesc_bf16(128, 128, 0, 1);
constexpr uint32_t kIdMnK2 = idesc_bf16(128, 128, 1, 0);

// Column sums of a warp's 32 x 32 block: on entry lane l holds x[c] = entry
// (l, c); on return x[0] of lane l is the sum over the 32 lanes of column l.
// Five exchange rounds halve the columns each lane keeps; the order of the
// additions is fixed.
__device__ __forceinline__ float warp_colsum32(float (&x)[32], int lane_id) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool up = (lane_id & s) != 0;
#pragma unroll
        for (int c = 0; c < s; ++c) {
            const float send = up ? x[c] : x[c + s];
            const float keep = up ? x[c + s] : x[c];
            x[c] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return x[0];
}

__device__ __forceinline__ float bf16_at(const uint8_t *p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
}

__device__ __forceinline__ void st_bf16_at(uint8_t *p, float x) {
    *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(x);
}

// Two / three 32-column TMEM loads under one wait.
__device__ __forceinline__ void tmem_load2(uint32_t a0, uint32_t a1, float (&f0)[32],
                                           float (&f1)[32]) {
    uint32_t r0[32], r1[32];
    tmem_ld32(a0, r0);
    tmem_ld32(a1, r1);
    tmem_wait_ld();
    reg_fence(r0);
    reg_fence(r1);
#pragma unroll
    for (int u = 0; u < 32; ++u) {
        f0[u] = __uint_as_float(r0[u]);
        f1[u] = __uint_as_float(r1[u]);
    }
}
__device__ __forceinline__ void tmem_load3(uint32_t a0, uint32_t a1, uint32_t a2, float (&f0)[32],
                                           float (&f1)[32], float (&f2)[32]) {
    uint32_t r0[32], r1[32], r2[32];
    tmem_ld32(a0, r0);
    tmem_ld32(a1, r1);
    tmem_ld32(a2, r2);
    tmem_wait_ld();
    reg_fence(r0);
    reg_fence(r1);
    reg_fence(r2);
#pragma unroll
    for (int u = 0; u < 32; ++u) {
        f0[u] = __uint_as_float(r0[u]);
        f1[u] = __uint_as_float(r1[u]);
        f2[u] = __uint_as_float(r2[u]);
    }
}

__global__ void __launch_bounds__(kThreads, 1) k_tc_bwd_grad(const __grid_constant__ GradArgs args) {
    const Problem &p = args.p;
    const Workspace &ws = args.ws;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    float *mf = reinterpret_cast<float *>(sm + kOffMisc);
    const float *vecs = reinterpret_cast<const float *>(sm + kOffVec);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + kOffBar + 8 * kNumBars);
    const int4 *tab = reinterpret_cast<const int4 *>(ws.chunk_tab);
    const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
    const int q4 = warp & 3, hf = warp >> 2;
    const int r = 32 * q4 + lane_id;              // TMEM lane of this thread
    const uint32_t lane = (uint32_t)(32 * q4) << 16;
    const int j0 = 32 * hf;                       // this thread's 32 columns
    const int H = (int)p.H;
    const float scale = p.scale;

    pdl_trigger();
    if (warp == 0) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) mbar_init(&bars[b], 1);
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t tl = tmem + lane;
    pdl_wait();  // the images from the kernels before
    const int n_items = *ws.n_chunks * H;

    auto issue_a = [&](int it_) {  // h, E, V', dO, v, G and beta
        const int4 e = tab[it_ / H];
        const int hh = it_ % H;
        const uint8_t *img = ws.bwd_lkimg + (int64_t)it_ * kLkImgBytes;
        mbar_arrive_expect_tx(&bars[0], kLoadA);
        bulk_load(sm + kOffH, img + kLkImgH, 16384u, &bars[0]);
        bulk_load(sm + kOffH + 16384, img + kLkImgH + 16384, 16384u, &bars[0]);
        bulk_load(sm + kOffD, img + kLkImgVh, 16384u, &bars[0]);
        bulk_load(sm + kOffD + 16384, img + kLkImgVl, 16384u, &bars[0]);
        bulk_load(sm + kOffVec, img + kLkImgVec, kLkImgVecBytes, &bars[0]);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            bulk_load(sm + kOffB + b * kBlkB + 8192, img + kLkImgE + b * 16384, 16384u, &bars[0]);
            tma_load_3d(sm + kOffB + b * kBlkB, &args.tdo, &bars[0], 64 * b, hh, e.y);
            tma_load_3d(sm + kOffV + b * 8192, &args.tv, &bars[0], 64 * b, hh, e.y);
        }
    };
    auto issue_b = [&](int it_) {  // q, k, dV', T
        const int4 e = tab[it_ / H];
        const int hh = it_ % H;
        const uint8_t *img = ws.bwd_lkimg + (int64_t)it_ * kLkImgBytes;
        mbar_arrive_expect_tx(&bars[4], kLoadB);
        bulk_load(sm + kOffF + kFdvHi, img + kLkImgDh, 16384u, &bars[4]);
        bulk_load(sm + kOffF + kFdvLo, img + kLkImgDl, 16384u, &bars[4]);
        bulk_load(sm + kOffF + kFtHi, img + kLkImgTh, 8192u, &bars[4]);
        bulk_load(sm + kOffF + kFtLo, img + kLkImgTl, 8192u, &bars[4]);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            tma_load_3d(sm + kOffC + b * kBlkC, &args.tq, &bars[4], 64 * b, hh, e.y);
            tma_load_3d(sm + kOffC + b * kBlkC + 8192, &args.tk, &bars[4], 64 * b, hh, e.y);
        }
    };
    // Descriptor bases: a descriptor of the tile at byte offset o from the
    // base is base + o / 16 (the start address field; o stays below 256 KB).
    const uint64_t dK = sdesc_sw128(sb, 16, 1024);        // K-major
    const uint64_t dM8 = sdesc_sw128(sb, 8192, 1024);     // MN-major, atoms 8 KB apart
    const uint64_t dM16 = sdesc_sw128(sb, 16384, 1024);   // MN-major, atoms 16 KB apart
    const uint64_t dM24 = sdesc_sw128(sb, kBlkB, 1024);   // MN-major, atoms 24 KB apart
    auto at = [](uint64_t base, uint32_t off) { return base + (uint64_t)(off >> 4); };
    // Values v[u] of column r for tokens j0 + u -> rows t0 + j0 + u of a
    // [tokens][H][128] BF16 output, rows past len skipped.  The warp's 32
    // columns x 32 tokens turn into rows through its 1 KB of shared memory,
    // 16 tokens at a time, and leave in 16-byte pieces.
    uint8_t *wout = sm + kOffOut + warp * 1024;
    auto store_cols = [&](__nv_bfloat16 *out, const float (&v)[32], int64_t t0, int hh, int len) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 16; ++u) st_bf16_at(wout + u * 64 + lane_id * 2, v[16 * half + u]);
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int c = lane_id + 32 * k, row = c >> 2, piece = c & 3;
                const int tok = j0 + 16 * half + row;
                if (tok < len)
                    *reinterpret_cast<uint4 *>(out + ((t0 + tok) * H + hh) * kD + 32 * q4 + piece * 8) =
                        *reinterpret_cast<const uint4 *>(wout + row * 64 + piece * 16);
            }
        }
    };

    int item = blockIdx.x;
    if (tid == 0 && item < n_items) {
        issue_a(item);
        issue_b(item);
    }
    for (uint32_t it = 0; item < n_items; ++it) {
        const uint32_t ph = it & 1u;
        const int4 e = tab[item / H];
        const int hh = item % H;
        const int64_t t0 = e.y;
        const int len = e.z;
        const int next = item + (int)gridDim.x;

        bool ok = mbar_wait(&bars[0], ph, p.status) && mbar_wait(&bars[4], ph, p.status);
        if (__syncthreads_or(!ok)) break;
        if (len < kChunk) {  // dO, q, k rows past the sequence end belong to the next one
            for (int idx = tid; idx < 6 * (kChunk - len) * 8; idx += kThreads) {
                const int tile = idx / ((kChunk - len) * 8), rem = idx % ((kChunk - len) * 8);
                const int t = len + (rem >> 3), c = rem & 7;
                const uint32_t base = tile < 2 ? kOffB + tile * kBlkB
                                               : kOffC + ((tile - 2) >> 1) * kBlkC + ((tile - 2) & 1) * 8192;
                st_shared_v4(sm + base + (t >> 3) * 1024 + (t & 7) * 128 + c * 16, 0u, 0u, 0u, 0u);
            }
        }
        fence_async_smem();
        // gate vectors; e^{G_i - G_j} = e^{G_i - G_last} e^{G_last - G_j} unless
        // the chunk's log gates spread over 80 (then one exponential each)
        bool wide = false;
        if (tid < 64) {
            const bool in = tid < len;
            const float G = vecs[tid], Gl = vecs[len - 1];
            mf[kVG + tid] = G;
            mf[kVGam + tid] = in ? expf(G) : 0.f;
            mf[kVLam + tid] = in ? expf(Gl - G) : 0.f;
            mf[kVEp + tid] = in ? expf(G - Gl) : 0.f;
            mf[kVB + tid] = in ? vecs[64 + tid] : 0.f;
            wide = in && fabsf(G - Gl) >= 80.f;
        }
        tc_fence_before();
        wide = __syncthreads_or(wide);
        // ---- group 1: P1^T, P3^T, [Q K^T; K K^T], dVb^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // over v
                umma_bf16(tmem + kCP1, at(dM16, kOffH + kk * 2048),
                          at(dK, kOffB + (kk >> 2) * kBlkB + (kk & 3) * 32), kIdMnK, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // over v; B = [V' hi | V' lo]
                umma_bf16(tmem + kCP3, at(dM24, kOffB + 8192 + kk * 2048),
                          at(dM16, kOffD + kk * 2048), kIdMnMn2, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // over keys
                umma_bf16(tmem + kCQK, at(dK, kOffC + (kk >> 2) * kBlkC + (kk & 3) * 32),
                          at(dK, kOffC + 8192 + (kk >> 2) * kBlkC + (kk & 3) * 32), kIdKK, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // over tokens i: dV' hi [T hi | T lo]
                umma_bf16(tmem + kCDvb, at(dK, kOffF + kFdvHi + kk * 32),
                          at(dM8, kOffF + kFtHi + kk * 2048), kIdKMn2, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // dV' lo T hi, into the first half
                umma_bf16(tmem + kCDvb, at(dK, kOffF + kFdvLo + kk * 32),
                          at(dM8, kOffF + kFtHi + kk * 2048), kIdKMn, 1u);
            umma_commit(&bars[1]);
        }
        {  // <E, h> over the two images (the same layout), meanwhile
            float eh = 0.f;
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const int c = tid + kThreads * rr;  // 16-byte chunk of a 32 KB image
                float ev[8], hv[8];
                ld_bf16x8(sm + kOffB + (c >> 10) * kBlkB + 8192 + (c & 1023) * 16, ev);
                ld_bf16x8(sm + kOffH + c * 16, hv);
#pragma unroll
                for (int u = 0; u < 8; ++u) eh = fmaf(ev[u], hv[u], eh);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) eh += __shfl_xor_sync(0xffffffffu, eh, off);
            if (lane_id == 0) mf[kEh + warp] = eh;
        }
        ok = mbar_wait(&bars[1], ph, p.status);
        if (__syncthreads_or(!ok)) break;  // also: every thread is done with the E image
        tc_fence_after();
        // ---- epilogue 1 (lanes = value columns, columns = tokens): dVb -> its
        // hi / lo tiles (group 2's operand), dv, rowdot(dVb, V)
        {
            float f[32], x[32];
            tmem_load2(tl + kCDvb + j0, tl + kCDvb + 64 + j0, f, x);  // dVb[j][v = r]
#pragma unroll
            for (int u = 0; u < 32; ++u) f[u] += x[u];
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int j = j0 + u;
                x[u] = j < len
                           ? f[u] * bf16_at(sm + kOffV + (r >> 6) * 8192 + sw128_off(j, r & 63, 64))
                           : 0.f;
                const __nv_bfloat16 hi = __float2bfloat16_rn(f[u]);
                const uint32_t o = kOffB + (r >> 6) * kBlkB + sw128_off(j, r & 63, 64);
                *reinterpret_cast<__nv_bfloat16 *>(sm + o + 8192) = hi;
                st_bf16_at(sm + o + 16384, f[u] - __bfloat162float(hi));
            }
            mf[kR4 + 64 * q4 + j0 + lane_id] = warp_colsum32(x, lane_id);
#pragma unroll
            for (int u = 0; u < 32; ++u) x[u] = mf[kVB + j0 + u] * f[u];
            store_cols(static_cast<__nv_bfloat16 *>(args.a.dv), x, t0, hh, len);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- group 2: [dm; Y], the dVb lo part of Y, (dVb h^T)^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // over v; B = [V' hi | V' lo]
                umma_bf16(tmem + kCDmY, at(dK, kOffB + (kk >> 2) * kBlkB + (kk & 3) * 32),
                          at(dM16, kOffD + kk * 2048), kIdKMn2, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // [dVb hi; dVb lo] V' hi^T: rows 64-127 used
                umma_bf16(tmem + kCD2, at(dK, kOffB + 8192 + (kk >> 2) * kBlkB + (kk & 3) * 32),
                          at(dM8, kOffD + kk * 2048), kIdKMn, kk > 0);
#pragma unroll
            for (int pz = 0; pz < 2; ++pz)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // over v; dVb hi, then lo
                    umma_bf16(tmem + kCKb, at(dM16, kOffH + kk * 2048),
                              at(dK, kOffB + 8192 + pz * 8192 + (kk >> 2) * kBlkB + (kk & 3) * 32),
                              kIdMnK, (pz | kk) != 0);
            umma_commit(&bars[2]);
        }
        // while group 2 runs: rowdot(P1, Q), rowdot(P3, K)
        {
            float f[32], g[32], x[32];
            const uint32_t oq = kOffC + (r >> 6) * kBlkC;
            tmem_load3(tl + kCP1 + j0, tl + kCP3 + j0, tl + kCP3 + 64 + j0, f, g, x);  // P1, P3
#pragma unroll
            for (int u = 0; u < 32; ++u) g[u] += x[u];
#pragma unroll
            for (int u = 0; u < 32; ++u) x[u] = f[u] * bf16_at(sm + oq + sw128_off(j0 + u, r & 63, 64));
            mf[kR1 + 64 * q4 + j0 + lane_id] = warp_colsum32(x, lane_id);
#pragma unroll
            for (int u = 0; u < 32; ++u)
                x[u] = g[u] * bf16_at(sm + oq + 8192 + sw128_off(j0 + u, r & 63, 64));
            mf[kR3 + 64 * q4 + j0 + lane_id] = warp_colsum32(x, lane_id);
        }
        ok = mbar_wait(&bars[2], ph, p.status);
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        if (tid == 0 && next < n_items) issue_a(next);  // H, B, D, V and the vectors are free
        // ---- epilogue 2 (stacked rows: lanes 0-63 row i of dm, 64-127 of Y)
        {
            float f[32], g[32], srow[32];
            if (q4 < 2) {
                const int i = r;
                float f2[32];
                tmem_load3(tl + kCDmY + j0, tl + kCDmY + 64 + j0, tl + kCQK + j0, f, f2, g);
#pragma unroll
                for (int u = 0; u < 32; ++u) f[u] += f2[u];  // dm[i][j]; g: (Q K^T)[i][j]
                const float Gi = mf[kVG + i], epi = mf[kVEp + i];
                float z[32], rowR = 0.f;
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int j = j0 + u;
                    const bool c = i < len && j <= i;
                    const float d = c ? (wide ? expf(Gi - mf[kVG + j]) : epi * mf[kVLam + j]) : 0.f;
                    z[u] = scale * f[u] * d;
                    g[u] = z[u] * g[u];  // R = Z * (Q K^T)
                    rowR += g[u];
                }
                mf[kRowR + 64 * hf + i] = rowR;
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    const uint32_t o = sw128_chunk(i, (j0 >> 3) + c8, 64);
                    st_split_bf16x8(sm + kOffF + kFzHi + o, sm + kOffF + kFzLo + o, z + 8 * c8);
                }
                mf[kColR + 64 * q4 + j0 + lane_id] = warp_colsum32(g, lane_id);
            } else {
                const int i = r - 64;
                float y2[32];
                tmem_load3(tl + kCDmY + j0, tl + kCDmY + 64 + j0, tl + kCD2 + j0, f, y2, g);
#pragma unroll
                for (int u = 0; u < 32; ++u) f[u] += y2[u] + g[u];  // Y[i][j]: its three parts
                tmem_load32f(tl + kCQK + j0, g);                   // (K K^T)[i][j]
                const float Gi = mf[kVG + i], bi = mf[kVB + i], epi = mf[kVEp + i];
                float rdA = 0.f;
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int j = j0 + u;
                    const bool sl = i < len && j < i;
                    const float d = sl ? (wide ? expf(Gi - mf[kVG + j]) : epi * mf[kVLam + j]) : 0.f;
                    const float dA = sl ? -f[u] : 0.f;
                    const float kd = g[u] * d;
                    rdA = fmaf(dA, kd, rdA);
                    g[u] = bi * dA * kd;
                    srow[u] = bi * dA * d;
                }
                mf[kRdA + 64 * hf + i] = rdA;
                // row i of S (zero on and above the diagonal)
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    const uint32_t o = sw128_chunk(i, (j0 >> 3) + c8, 64);
                    st_split_bf16x8(sm + kOffF + kFsHi + o, sm + kOffF + kFsLo + o, srow + 8 * c8);
                }
                mf[kColRA + 64 * (q4 - 2) + j0 + lane_id] = warp_colsum32(g, lane_id);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- group 3: (Z K)^T, (Z^T Q + S^T K + S K)^T, each over [hi | lo]
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // over tokens j; B = [Z hi; Z lo] rows
                umma_bf16(tmem + kCXq, at(dM16, kOffC + 8192 + kk * 2048),
                          at(dK, kOffF + kFzHi + kk * 32), kIdMnK2, kk > 0);
#pragma unroll
            for (int t3 = 0; t3 < 2; ++t3) {  // Q^T [Z hi | Z lo], K^T [S hi | S lo]
                const uint32_t oa = kOffC + (t3 ? 8192u : 0u);
                const uint32_t ob = kOffF + (t3 ? kFsHi : kFzHi);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(tmem + kCXk, at(dM16, oa + kk * 2048), at(dM8, ob + kk * 2048),
                              kIdMnMn2, (t3 | kk) != 0);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // K^T S^T: [S hi; S lo] rows as the K-major operand
                umma_bf16(tmem + kCXk, at(dM16, kOffC + 8192 + kk * 2048),
                          at(dK, kOffF + kFsHi + kk * 32), kIdMnK2, 1u);
            umma_commit(&bars[3]);
        }
        {  // while group 3 runs: r2 = rowdot(dKb, K), dKb = -dVb h^T
            float f[32];
            tmem_load32f(tl + kCKb + j0, f);
            const uint32_t ok_ = kOffC + (r >> 6) * kBlkC + 8192;
#pragma unroll
            for (int u = 0; u < 32; ++u) f[u] = -f[u] * bf16_at(sm + ok_ + sw128_off(j0 + u, r & 63, 64));
            mf[kR2 + 64 * q4 + j0 + lane_id] = warp_colsum32(f, lane_id);
        }
        ok = mbar_wait(&bars[3], ph, p.status);
        if (__syncthreads_or(!ok)) break;  // every MMA of the item done: C and F free
        tc_fence_after();
        if (tid == 0 && next < n_items) issue_b(next);
        // ---- epilogue 3: dq, dk (lanes = keys)
        {
            float f[32], x[32], y[32];
            tmem_load3(tl + kCP1 + j0, tl + kCXq + j0, tl + kCXq + 64 + j0, f, x, y);
#pragma unroll
            for (int u = 0; u < 32; ++u) x[u] = fmaf(scale * mf[kVGam + j0 + u], f[u], x[u] + y[u]);
            store_cols(static_cast<__nv_bfloat16 *>(args.a.dq), x, t0, hh, len);
            tmem_load3(tl + kCP3 + j0, tl + kCP3 + 64 + j0, tl + kCKb + j0, f, y, x);
#pragma unroll
            for (int u = 0; u < 32; ++u) {  // x: -beta gamma dKb + lam P3
                const int i = j0 + u;
                x[u] = fmaf(-mf[kVB + i] * mf[kVGam + i], x[u], mf[kVLam + i] * (f[u] + y[u]));
            }
            tmem_load2(tl + kCXk + j0, tl + kCXk + 64 + j0, f, y);
#pragma unroll
            for (int u = 0; u < 32; ++u) x[u] += f[u] + y[u];
            store_cols(static_cast<__nv_bfloat16 *>(args.a.dk), x, t0, hh, len);
        }
        // ---- dbeta and the gate gradient
        if (tid < 64) {
            const int i = tid;
            float r1 = 0.f, r2 = 0.f, r3 = 0.f, r4 = 0.f;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                r1 += mf[kR1 + 64 * qq + i];
                r2 += mf[kR2 + 64 * qq + i];
                r3 += mf[kR3 + 64 * qq + i];
                r4 += mf[kR4 + 64 * qq + i];
            }
            const float rowR = mf[kRowR + i] + mf[kRowR + 64 + i];
            const float colR = mf[kColR + i] + mf[kColR + 64 + i];
            const float rdA = mf[kRdA + i] + mf[kRdA + 64 + i];
            const float colRA = mf[kColRA + i] + mf[kColRA + 64 + i];
            const float gam = mf[kVGam + i], lam = mf[kVLam + i], bi = mf[kVB + i];
            float dG = 0.f;
            if (i < len) {
                dG = scale * gam * r1 + (rowR - colR) - lam * r3 + bi * rdA - colRA + bi * gam * r2;
                args.a.dbeta[(t0 + i) * H + hh] = r4 + gam * r2 + rdA;
            }
            mf[kDg + i] = dG;
            mf[kR3f + i] = r3;
        }
        __syncthreads();
        if (warp == 0) {
            // the chunk's last token also carries the state terms: e^{G_last}
            // <E, h> and sum_j lam_j rowdot(P3, K)_j (lam is zero past len);
            // then dg = the suffix sums of dG, in a fixed order: lane l holds
            // tokens 2l and 2l + 1
            float lam3 = fmaf(mf[kVLam + lane_id], mf[kR3f + lane_id],
                              mf[kVLam + 32 + lane_id] * mf[kR3f + 32 + lane_id]);
            float eh = lane_id < kThreads / 32 ? mf[kEh + lane_id] : 0.f;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                lam3 += __shfl_xor_sync(0xffffffffu, lam3, off);
                eh += __shfl_xor_sync(0xffffffffu, eh, off);
            }
            float d0 = mf[kDg + 2 * lane_id], d1 = mf[kDg + 2 * lane_id + 1];
            const float extra = fmaf(mf[kVGam + len - 1], eh, lam3);
            if (2 * lane_id == len - 1) d0 += extra;
            if (2 * lane_id + 1 == len - 1) d1 += extra;
            float suf = d0 + d1;  // inclusive suffix sum over the lanes' pairs
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_down_sync(0xffffffffu, suf, off);
                if (lane_id + off < 32) suf += y;
            }
            float above = __shfl_down_sync(0xffffffffu, suf, 1);
            if (lane_id == 31) above = 0.f;
            const float run1 = above + d1, run0 = run1 + d0;
            if (2 * lane_id < len) args.a.dg[(t0 + 2 * lane_id) * H + hh] = run0;
            if (2 * lane_id + 1 < len) args.a.dg[(t0 + 2 * lane_id + 1) * H + hh] = run1;
        }
        tc_fence_before();
        __syncthreads();  // TMEM and the scalars are reused
        item = next;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t tc_bwd_grad(const Problem &p, const Workspace &ws, const BwdArgs &a,
                        cudaStream_t st) {
    if (ws.max_chunks == 0) return cudaSuccess;
    GradArgs args;
    args.p = p;
    args.ws = ws;
    args.a = a;
    const uint64_t rows = (uint64_t)p.B * (uint64_t)p.T;
    const uint64_t H = (uint64_t)p.H;
    if (!make_tmap_bf16_3d(&args.tq, p.q, kD, H, rows, p.sq.h * 2, p.sq.t * 2, 64, 1, 64) ||
        !make_tmap_bf16_3d(&args.tk, p.k, kD, H, rows, p.sk.h * 2, p.sk.t * 2, 64, 1, 64) ||
        !make_tmap_bf16_3d(&args.tv, p.v, kD, H, rows, p.sv.h * 2, p.sv.t * 2, 64, 1, 64) ||
        !make_tmap_bf16_3d(&args.tdo, a.dout, kD, H, rows, kD * 2, H * kD * 2, 64, 1, 64))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(k_tc_bwd_grad,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemLaunch);
    if (err != cudaSuccess) return err;
    const int64_t items = ws.max_chunks * p.H;  // an upper bound; the kernel reads the count
    const dim3 grid((unsigned)persistent_grid(p, items, 1));
    return launch_pdl(k_tc_bwd_grad, grid, dim3(kThreads), kSmemLaunch, st, args);
}

}  // namespace gdr
