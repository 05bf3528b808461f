// tc_prep.cu -- A2-A5 on the tensor-core path (BF16, K = V = 128, delta rule):
// everything of the chunked form that does not depend on the state, for
// every (chunk, head) in parallel.  Persistent CTAs (three per SM) walk the
// (chunk, head) items; per item:
//
//   G (gate cumsum), D1 = [K; Q] K^T on tcgen05 (rows 0-63 K K^T, rows 64-127
//   Q K^T), A_ij = beta_i e^{G_i - G_j} (k_i . k_j) for i > j, T = (I + A)^-1
//   (tc_inverse.cuh), W^T = K^T (T diag(beta e^G))^T and U^T = V^T
//   (T diag(beta))^T on tcgen05, P = (Q K^T) * e^{G_i - G_j} for j <= i.
//
// The results, with Q~ = scale diag(e^G) Q, go to one record per (chunk,
// head): the byte image of the scan kernel's shared-memory stage (layout in
// tc_chunk.cuh), assembled here in shared memory and written by bulk async
// copies, which the scan kernel (tc_chain.cu) loads back, so the serial chain
// only does the state-dependent products.  The next item's table row and
// gates are loaded early, and its K and Q tiles start loading as soon as the
// current item's last product has consumed them, while the current item's
// results are still being staged and written; V, which only the last
// product reads, loads while the inverse runs.  Chunked form: the project
// statement; the WY/UT preparation ahead of fla's state-scan kernel
// chunk_gated_delta_rule_fwd_kernel_h_blockdim64 (Kev PR #259 intro).
#include "gdr_internal.cuh"
#include "tc_chunk.cuh"
#include "tc_inverse.cuh"
#include "tma_host.cuh"

namespace gdr {
namespace {

using namespace tc;

struct PrepArgs {
    Problem p;
    Workspace ws;
    CUtensorMap tq, tk, tv;
};

constexpr int kThreads = 256;

// Shared memory (bytes from a 1024-aligned base), 74 KB so that three CTAs
// fit an SM.  Each region serves several tiles in turn:
//   [Kb0|Qb0|Kb1|Qb1]  K and Q (the A operand [K; Q] of D1); Q~ is formed in
//                      place once D1 is done and, once its copies have read
//                      it, B_W and B_U take the two Q blocks;
//   kOffV (16 KB)      the previous item's W staging, this item's scale P
//                      staging, then this item's V (loaded once the P copy
//                      has read the slot; only the last product needs it);
//   kOffAT             A, then T in place (FP32, ld kInvLd); U^T staging
//                      after the last product.
constexpr uint32_t kOffBW = 8192, kOffBU = 24576;       // over Qb0, Qb1
constexpr uint32_t kOffV = 32768;                       // [Vb0|Vb1]
constexpr uint32_t kOffStP = kOffV;                     // scale P staging, 8 KB
constexpr uint32_t kOffStW = kOffV;                     // W staging, 16 KB
constexpr uint32_t kOffAT = 49152;                      // A / T
constexpr uint32_t kOffStU = kOffAT;                    // U^T staging, 16 KB
constexpr uint32_t kOffX = kOffAT + 64 * kInvLd * 4;    // inverse scratch
constexpr uint32_t kOffVec = kOffX + 4 * kInvScratchFloats;  // gate vectors, two items'
constexpr uint32_t kOffBar = kOffVec + 2 * 1600;        // K/Q tiles, products, V tile
constexpr uint32_t kSmemLaunch = kOffBar + 64 + 1024;
static_assert(kOffStU % 1024 == 0 && kOffStP % 1024 == 0, "staging tiles are 1 KB aligned");
static_assert(kSmemLaunch <= 76800, "three CTAs per SM");

// TMEM: D1, then W^T over it (D1 is consumed before the last product), U^T.
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kColD1 = 0, kColW = 0, kColU = 64;

constexpr uint32_t kIdescKK64 = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t kIdescMK64 = idesc_bf16(128, 64, 1, 0);

// Rows of two 8 KB tiles at `a` and `a + 16384` scaled in place by c f[row]
// (64 rows of 128 bytes each, in 16-byte pieces; thread t of n threads).
__device__ __forceinline__ void scale_rows_in_place(uint8_t *a, const float *f, float c, int t,
                                                    int n) {
    for (int idx = t; idx < 1024; idx += n) {
        const int row = (idx >> 3) & 63;
        uint8_t *ptr = a + (idx >> 9) * 16384 + row * 128 + (idx & 7) * 16;
        float x[8];
        ld_bf16x8(ptr, x);
        const float m = c * f[row];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] *= m;
        st_bf16x8(ptr, x);
    }
}

// kBwd: the backward's recompute also stores the T images, G and beta (a separate
// instantiation, so that the forward's kernel carries none of it).
template <bool kBwd>
__global__ void __launch_bounds__(kThreads, 3) k_tc_prep(const __grid_constant__ PrepArgs args) {
    const Problem &p = args.p;
    const Workspace &ws = args.ws;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);  // K/Q tma, mma, V tma
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + kOffBar + 24);
    float *sAT = reinterpret_cast<float *>(sm + kOffAT);
    float *sX = reinterpret_cast<float *>(sm + kOffX);
    const int4 *tab = reinterpret_cast<const int4 *>(ws.chunk_tab);

    const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int row = 32 * quad + lane_id;  // TMEM lane = matrix row
    const int H = (int)p.H;
    pdl_trigger();
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    pdl_wait();  // the chunk table, once the kernel before has finished
    const int n_items = *ws.n_chunks * H;  // below 2^31 (checked by the host)
    int item = blockIdx.x;

    // The gates of a chunk-head (padded tokens: g = beta = 0), loaded by warp 0.
    auto load_gates = [&](const int4 &e, int h, float (&g2)[2], float (&b2)[2]) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int tok = 2 * lane_id + u;
            g2[u] = tok < e.z ? p.g[((int64_t)e.y + tok) * H + h] : 0.f;
            b2[u] = tok < e.z ? p.beta[((int64_t)e.y + tok) * H + h] : 0.f;
        }
    };
    auto issue_inputs = [&](const int4 &e, int h) {
        mbar_arrive_expect_tx(&bars[0], 32768u);
        tma_load_3d(sm + 0, &args.tk, &bars[0], 0, h, e.y);
        tma_load_3d(sm + 16384, &args.tk, &bars[0], 64, h, e.y);
        tma_load_3d(sm + 8192, &args.tq, &bars[0], 0, h, e.y);
        tma_load_3d(sm + 24576, &args.tq, &bars[0], 64, h, e.y);
    };

    int4 e = make_int4(0, 0, 0, 0);
    int h = 0;
    float g2[2] = {0.f, 0.f}, b2[2] = {0.f, 0.f};
    if (item < n_items) {
        e = tab[item / H];
        h = item % H;
        if (warp == 0) load_gates(e, h, g2, b2);
        if (tid == 0) issue_inputs(e, h);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    if (item >= n_items) {  // more CTAs than items
        if (warp == 0) tmem_dealloc(tmem, kTmemCols);
        return;
    }
    const uint32_t lane = (uint32_t)(32 * quad) << 16;

    for (uint32_t it = 0;; ++it) {
        const int len = e.z;
        uint8_t *img = ws.rec + (int64_t)item * kRecBytes;
        const int nxt = item + (int)gridDim.x;
        const bool more = nxt < n_items;
        int4 en = e;
        int hn = h;
        float g2n[2] = {0.f, 0.f}, b2n[2] = {0.f, 0.f};

        // The gate vectors of this item, in the buffer its predecessor's
        // copies no longer read (they waited for that before it began).
        float *vec = reinterpret_cast<float *>(sm + kOffVec + (it & 1) * 1600);
        const float *sG = vec, *sBeta = vec + 64, *sBG = vec + 128, *sDec = vec + 192,
                    *sGam = vec + 256, *sEP = vec + 320, *sScal = vec + 384;
        if (warp == 0) {
            gate_vectors(vec, g2, b2, len, lane_id);
            if (kBwd) {  // G and beta for the backward's per-chunk gradients
                float *gv = reinterpret_cast<float *>(ws.bwd_lkimg + (int64_t)item * kLkImgBytes +
                                                      kLkImgVec);
#pragma unroll
                for (int c = 0; c < 4; ++c) gv[32 * c + lane_id] = vec[32 * c + lane_id];
            }
        }
        bool ok = mbar_wait(&bars[0], it & 1u, p.status);
        if (__syncthreads_or(!ok)) break;
        if (len < 64) {  // rows past the sequence end belong to the next one: zero them
            const int rows = 64 - len;
            for (int idx = tid; idx < rows * 4 * 8; idx += kThreads) {
                const int r = len + idx / 32, blk = (idx / 8) & 3, c16 = idx & 7;
                st_shared_v4(sm + blk * 8192 + r * 128 + c16 * 16, 0u, 0u, 0u, 0u);
            }
            fence_async_smem();
        }
        __syncthreads();

        // A3 (+ Q K^T): D1 = [K; Q] K^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a = sb + (kk >> 2) * 16384 + (kk & 3) * 32;
                umma_bf16(tmem + kColD1, sdesc_sw128(a, 16, 1024), sdesc_sw128(a, 16, 1024),
                          kIdescKK64, kk > 0);
            }
            umma_commit(&bars[1]);
        }
        if (more) {  // the next item's table row and gates, in flight early
            en = tab[nxt / H];
            hn = (int)(nxt % H);
            if (warp == 0) load_gates(en, hn, g2n, b2n);
        }
        ok = mbar_wait(&bars[1], 0, p.status);
        // the previous item's copies have read their staging tiles (W, U^T,
        // its gate vectors) before they are written again
        if (lane_id == 0) bulk_wait_read();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        {
            float f[32];
            tmem_load32f(tmem + lane + kColD1 + 32 * half, f);
            const int i = row & 63;
            const int j0 = 32 * half;
            // A rows keep j < i (beta_i folded in); P rows keep j <= i.
            const int jlim = quad < 2 ? i : i + 1;
            const float rowf = quad < 2 ? sBeta[i] : p.scale;
            if (sScal[2] != 0.f) {  // e^{G_i - G_j} = e^{G_i - G_last} e^{G_last - G_j}
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
                    *reinterpret_cast<float4 *>(sAT + i * kInvLd + j0 + 4 * c4) =
                        make_float4(f[4 * c4], f[4 * c4 + 1], f[4 * c4 + 2], f[4 * c4 + 3]);
            } else {  // row i of scale P
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8)
                    st_bf16x8(sm + kOffStP + sw128_off(i, j0 + 8 * c8, 64), f + 8 * c8);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 224) {  // scale P out, so that V can take its slot
            bulk_store(img + kImgP, sm + kOffStP, 8192u);
            bulk_commit();
        }

        // A4: T = (I + A)^-1.  The diagonal blocks on warps 0-1 while warps 2-7
        // form Q~ = scale diag(e^G) Q in place (no product reads Q any more).
        if (tid < 64)
            invert_diag16(sAT, tid);
        else
            scale_rows_in_place(sm + 8192, sGam, p.scale, tid - 64, kThreads - 64);
        fence_async_smem();
        __syncthreads();
        if (lane_id == 0 && (warp == 5 || warp == 6)) {  // Q~ blocks, one copy per warp
            bulk_store(img + kImgQ + (warp - 5) * 8192, sm + 8192 + (warp - 5) * 16384, 8192u);
            bulk_commit();
            bulk_wait_read();  // B_W, B_U take these blocks (warps 4-7 idle in the first merge step)
        } else if (tid == 224) {  // V into the slot P has left
            bulk_wait_read();
            mbar_arrive_expect_tx(&bars[2], 16384u);
            tma_load_3d(sm + kOffV, &args.tv, &bars[2], 0, h, e.y);
            tma_load_3d(sm + kOffV + 8192, &args.tv, &bars[2], 64, h, e.y);
        }
        invert_merge(sAT, sX, tid);

        // A5 operands: rows of T diag(beta e^G) (rows 0-63) and T diag(beta)
        // (rows 64-127), BF16, columns [32 half, 32 half + 32).
        {
            const int i = row & 63;
            const float *scale_vec = quad < 2 ? sBG : sBeta;
            uint8_t *dst = sm + (quad < 2 ? kOffBW : kOffBU);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                const int j0 = 32 * half + 8 * c8;
                const float4 a0 = *reinterpret_cast<const float4 *>(sAT + i * kInvLd + j0);
                const float4 a1 = *reinterpret_cast<const float4 *>(sAT + i * kInvLd + j0 + 4);
                const float tv[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                if (kBwd && quad < 2) {  // T for the backward as BF16 hi + lo images:
                    // zero above the diagonal and in rows past the sequence end
                    float tz[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) tz[u] = (j0 + u <= i && i < len) ? tv[u] : 0.f;
                    uint8_t *timg = ws.bwd_lkimg + (int64_t)item * kLkImgBytes;
                    const uint32_t ot = sw128_off(i, j0, 64);
                    st_split_bf16x8(timg + kLkImgTh + ot, timg + kLkImgTl + ot, tz);
                }
                float x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) x[u] = j0 + u <= i ? tv[u] * scale_vec[j0 + u] : 0.f;
                st_bf16x8(dst + sw128_off(i, j0, 64), x);
            }
        }
        ok = true;
        if (len < 64) {  // V's rows past the sequence end, once V has landed
            ok = mbar_wait(&bars[2], it & 1u, p.status);
            const int rows = 64 - len;
            for (int idx = tid; ok && idx < rows * 2 * 8; idx += kThreads) {
                const int r = len + idx / 16, blk = (idx / 8) & 1, c16 = idx & 7;
                st_shared_v4(sm + kOffV + blk * 8192 + r * 128 + c16 * 16, 0u, 0u, 0u, 0u);
            }
        }
        fence_async_smem();
        if (__syncthreads_or(!ok)) break;
        if (tid == 0 && mbar_wait(&bars[2], it & 1u, p.status)) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                umma_bf16(tmem + kColW, sdesc_sw128(sb + kk * 2048, 16384, 1024),
                          sdesc_sw128(sb + kOffBW + kk * 32, 16, 1024), kIdescMK64, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                umma_bf16(tmem + kColU, sdesc_sw128(sb + kOffV + kk * 2048, 8192, 1024),
                          sdesc_sw128(sb + kOffBU + kk * 32, 16, 1024), kIdescMK64, kk > 0);
            umma_commit(&bars[1]);
        }
        ok = mbar_wait(&bars[1], 1, p.status);
        // K and the Q blocks are free once the products have read them: the
        // next item's K and Q start loading now.
        if (lane_id == 0) bulk_wait_read();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        if (tid == 0 && more) issue_inputs(en, hn);
        {  // W^T (row k) and U^T (row v), t in [32 half, 32 half + 32), staged
            float f[32];
            tmem_load32f(tmem + lane + kColW + 32 * half, f);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8)
                st_bf16x8(sm + kOffStW + sw128_off(row, 32 * half + 8 * c8, 128), f + 8 * c8);
            tmem_load32f(tmem + lane + kColU + 32 * half, f);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8)
                st_bf16x8(sm + kOffStU + sw128_off(row, 32 * half + 8 * c8, 128), f + 8 * c8);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // one copy per warp (lane 0), so they are issued side by side
        if (lane_id == 0 && warp < 5) {
            switch (warp) {
            case 0: bulk_store(img + kImgW, sm + kOffStW, 8192u); break;
            case 1: bulk_store(img + kImgW + 8192, sm + kOffStW + 8192, 8192u); break;
            case 2: bulk_store(img + kImgU, sm + kOffStU, 16384u); break;
            case 3: bulk_store(img + kImgVec, vec + 384, 16u); break;  // G_last, e^{G_last}
            default: bulk_store(img + kImgDec, sDec, 256u); break;     // e^{G_last - G}
            }
            bulk_commit();
        }
        if (!more) break;
        item = nxt;
        e = en;
        h = hn;
        g2[0] = g2n[0];
        g2[1] = g2n[1];
        b2[0] = b2n[0];
        b2[1] = b2n[1];
    }
    if (lane_id == 0) bulk_wait_read();  // every issuing thread, its own copies
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t tc_prep(const Problem &p, const Workspace &ws, cudaStream_t st) {
    if (ws.max_chunks == 0) return cudaSuccess;
    PrepArgs args;
    args.p = p;
    args.ws = ws;
    const uint64_t rows = (uint64_t)p.B * (uint64_t)p.T;
    const uint64_t H = (uint64_t)p.H;
    if (!make_tmap_bf16_3d(&args.tq, p.q, kD, H, rows, p.sq.h * 2, p.sq.t * 2, 64, 1, 64) ||
        !make_tmap_bf16_3d(&args.tk, p.k, kD, H, rows, p.sk.h * 2, p.sk.t * 2, 64, 1, 64) ||
        !make_tmap_bf16_3d(&args.tv, p.v, kD, H, rows, p.sv.h * 2, p.sv.t * 2, 64, 1, 64))
        return cudaErrorInvalidValue;
    auto kernel = ws.bwd_tc ? k_tc_prep<true> : k_tc_prep<false>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemLaunch);
    if (err != cudaSuccess) return err;
    const int64_t items = ws.max_chunks * p.H;  // an upper bound; the kernel reads the count
    if (items > INT32_MAX - 4 * (int64_t)device_sms()) return cudaErrorInvalidValue;
    const int64_t grid = persistent_grid(p, items, 3);  // three CTAs per SM
    return launch_pdl(kernel, dim3((unsigned)grid), dim3(kThreads), kSmemLaunch, st, args);
}

}  // namespace gdr
