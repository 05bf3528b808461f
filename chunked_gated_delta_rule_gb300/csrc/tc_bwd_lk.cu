// tc_bwd_lk.cu -- the L x K products of the backward pass on the tensor
// cores (the tensor-core route: BF16, K = V = 128, delta rule).  Per (chunk,
// head), over the value dimension:
//
//   P1 = dO h^T     P2 = dV' h^T     P3 = V' E^T      (64 tokens x K keys)
//   <E, h> over each 64-key slice
//
// with h the state before the chunk (forward recompute), E the gradient at
// the chunk's end and V', dV' the chunk's v_new and its gradient (reverse
// scan).  h^T, V'^T, E^T and -dV'^T arrive as BF16 byte images of the
// chains' own MMA operands (128-byte swizzled, [v][key] / [v][t]), so they
// load with bulk copies and feed tcgen05 as MN-major operands: in the
// transposed form P^T = X Y^T with the keys on the TMEM lanes (M = 128),
// tokens as N = 64 and the value dimension as the reduction; dO loads by
// TMA as the K-major operand.  <E, h> is the elementwise product of the two
// images (same layout), summed in a fixed order.
//
// Persistent CTAs (one per SM) stride over the (chunk, head) items; the
// next item's loads overlap this item's TMEM read-back (two TMEM buffers).
// Every wait is time-bounded.
#include "gdr_internal.cuh"
#include "tc_chunk.cuh"
#include "tma_host.cuh"

namespace gdr {
namespace {

using namespace tc;

struct LkArgs {
    Problem p;
    Workspace ws;
    float *P1, *P2, *P3, *ehp;
    CUtensorMap tdo;
};

constexpr int kThreads = 256;
constexpr uint32_t kOffImg = 0;                       // the item's images, kLkImgBytes
constexpr uint32_t kOffDo = kLkImgBytes;              // dO [t][v], two 64-column blocks
constexpr uint32_t kOffRed = kOffDo + 16384;          // <E, h> partial sums [2][256]
constexpr uint32_t kOffBar = kOffRed + 2 * kThreads * 4;
constexpr uint32_t kSmemLaunch = kOffBar + 32 + 1024;
constexpr uint32_t kTmemCols = 512;                   // two buffers of [P1 | P2 | P3]

constexpr uint32_t kIdescP1 = idesc_bf16(128, 64, 1, 0);  // A h^T (MN-major), B dO (K-major)
constexpr uint32_t kIdescPx = idesc_bf16(128, 64, 1, 1);  // both MN-major

__global__ void __launch_bounds__(kThreads, 1) k_tc_bwd_lk(const __grid_constant__ LkArgs args) {
    const Problem &p = args.p;
    const Workspace &ws = args.ws;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);  // [0] loads, [1] products
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + kOffBar + 16);
    float *sRed = reinterpret_cast<float *>(sm + kOffRed);
    const int4 *tab = reinterpret_cast<const int4 *>(ws.chunk_tab);
    const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
    const int key = 32 * (warp & 3) + lane_id;  // TMEM lane
    const uint32_t lane = (uint32_t)(32 * (warp & 3)) << 16;
    const int H = (int)p.H;

    pdl_trigger();
    if (warp == 0) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    pdl_wait();  // the images and dV', once the reverse scan has finished
    const int n_items = *ws.n_chunks * H;

    auto issue = [&](int item) {  // the item's images and its dO tile
        const int4 e = tab[item / H];
        const int h = item % H;
        mbar_arrive_expect_tx(&bars[0], kLkImgBytes + 16384u);
        const uint8_t *src = ws.bwd_lkimg + (int64_t)item * kLkImgBytes;
        for (int c = 0; c < 6; ++c)  // six 16 KB pieces
            bulk_load(sm + kOffImg + c * 16384, src + c * 16384, 16384u, &bars[0]);
        tma_load_3d(sm + kOffDo, &args.tdo, &bars[0], 0, h, e.y);
        tma_load_3d(sm + kOffDo + 8192, &args.tdo, &bars[0], 64, h, e.y);
    };
    int item = blockIdx.x;
    if (tid == 0 && item < n_items) issue(item);
    bool ok = true;
    for (uint32_t it = 0; item < n_items && ok; ++it) {
        const int len = tab[item / H].z;
        const uint32_t b = it & 1u;
        ok = mbar_wait(&bars[0], it & 1u, p.status);
        if (__syncthreads_or(!ok)) break;
        if (len < kChunk) {  // dO rows past the sequence end belong to the next one
            for (int idx = tid; idx < (kChunk - len) * 16; idx += kThreads) {
                const int t = len + (idx >> 4), c = idx & 15;
                st_shared_v4(sm + kOffDo + (c >> 3) * 8192 + t * 128 + (c & 7) * 16, 0u, 0u, 0u,
                             0u);
            }
            fence_async_smem();
        }
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t d = tmem + 256 * b;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // over v, 16 a step
                const uint64_t ah = sdesc_sw128(sb + kOffImg + kLkImgH + kk * 2048, 16384, 1024);
                umma_bf16(d, ah,
                          sdesc_sw128(sb + kOffDo + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024),
                          kIdescP1, kk > 0);
                umma_bf16(d + 64, ah, sdesc_sw128(sb + kOffImg + kLkImgDv + kk * 2048, 8192, 1024),
                          kIdescPx, kk > 0);
                umma_bf16(d + 128, sdesc_sw128(sb + kOffImg + kLkImgE + kk * 2048, 16384, 1024),
                          sdesc_sw128(sb + kOffImg + kLkImgV + kk * 2048, 8192, 1024), kIdescPx,
                          kk > 0);
            }
            umma_commit(&bars[1]);
        }
        {  // <E, h>: the two images share a layout; block 0 holds keys 0-63
            float part[2] = {0.f, 0.f};
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int c = tid + kThreads * r;  // 16-byte chunk of the 32 KB images
                float e[8], hv[8];
                ld_bf16x8(sm + kOffImg + kLkImgE + c * 16, e);
                ld_bf16x8(sm + kOffImg + kLkImgH + c * 16, hv);
                float s = 0.f;
#pragma unroll
                for (int u = 0; u < 8; ++u) s = fmaf(e[u], hv[u], s);
                part[c >= 1024] += s;
            }
            sRed[tid] = part[0];
            sRed[kThreads + tid] = part[1];
        }
        ok = mbar_wait(&bars[1], it & 1u, p.status);
        if (__syncthreads_or(!ok)) break;  // products done, images read: smem free
        tc_fence_after();
        const int next = item + (int)gridDim.x;
        if (tid == 0 && next < n_items) issue(next);
        if (tid < 2) {  // fixed-order sums of the slice's partials
            float s = 0.f;
            for (int t = 0; t < kThreads; ++t) s += sRed[tid * kThreads + t];
            args.ehp[(int64_t)item * 2 + tid] = s;
        }
        // P^T rows (lanes = keys) to P[t][key]: warps 0-3 P1 and P3 columns
        // 0-31, warps 4-7 P2 (negated: the image holds -dV') and P3 columns
        // 32-63
        {
            const uint32_t d = tmem + 256 * b + lane;
            const int64_t base = ((int64_t)item * kChunk) * kD + key;
            const bool lo = warp < 4;
            float *P = lo ? args.P1 : args.P2;
            const float sgn = lo ? 1.f : -1.f;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float f[32];
                tmem_load32f(d + (lo ? 0 : 64) + 32 * hh, f);
#pragma unroll
                for (int u = 0; u < 32; ++u) P[base + (int64_t)(32 * hh + u) * kD] = sgn * f[u];
            }
            float f[32];
            tmem_load32f(d + 128 + (lo ? 0 : 32), f);
#pragma unroll
            for (int u = 0; u < 32; ++u)
                args.P3[base + (int64_t)((lo ? 0 : 32) + u) * kD] = f[u];
        }
        tc_fence_before();
        __syncthreads();  // sRed and the TMEM buffer are reused
        item = next;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t tc_bwd_lk(const Problem &p, const Workspace &ws, const void *dout, float *P1,
                      float *P2, float *P3, float *ehp, cudaStream_t st) {
    if (ws.max_chunks == 0) return cudaSuccess;
    LkArgs args;
    args.p = p;
    args.ws = ws;
    args.P1 = P1;
    args.P2 = P2;
    args.P3 = P3;
    args.ehp = ehp;
    const uint64_t rows = (uint64_t)p.B * (uint64_t)p.T;
    const uint64_t H = (uint64_t)p.H;
    if (!make_tmap_bf16_3d(&args.tdo, dout, kD, H, rows, kD * 2, H * kD * 2, 64, 1, 64))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(k_tc_bwd_lk,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemLaunch);
    if (err != cudaSuccess) return err;
    const int64_t items = ws.max_chunks * p.H;  // an upper bound; the kernel reads the count
    const dim3 grid((unsigned)persistent_grid(p, items, 1));
    return launch_pdl(k_tc_bwd_lk, grid, dim3(kThreads), kSmemLaunch, st, args);
}

}  // namespace gdr
