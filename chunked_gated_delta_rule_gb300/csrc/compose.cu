// compose.cu -- A9, the ordered segment composition h_{s+1} = M_s h_s + c_s
// (cuLA PR #127 "Root cause and implementation": the per-segment FP32
// transition chained by a short ordered pass), FP32 on CUDA cores.
//
// Delta rule: one CTA (512 threads, one per SM) owns CC = 4, 8 or 16 value
// columns of one (sequence, head) and walks its segments in order.  Each
// segment's K x K transition (stored transposed, [m][r] = M_s[r][m]) is
// streamed into shared memory by a 1-D bulk async copy, double-buffered so
// the next one loads while this one is applied.  A thread owns two state
// rows x four columns over one slice of the reduction index m; the slices'
// partial sums are added in a fixed order, so every output element has one
// fixed summation order.
#include "gdr_internal.cuh"
#include "gdr_segments.cuh"
#include "tc_common.cuh"

namespace gdr {
namespace {

using namespace tc;

constexpr int kComposeThreads = 512;

template <int CC>
__global__ void __launch_bounds__(kComposeThreads, 1) k_compose_mt(Problem p, Workspace ws) {
    constexpr int NCG = CC / 4;                         // four-column groups
    constexpr int NMS = kComposeThreads / (64 * NCG);   // slices of m
    const int K = (int)p.K, V = (int)p.V, H = (int)p.H, S = ws.n_segments;
    const int col0 = blockIdx.x * CC;
    const int64_t n = blockIdx.y;
    const int h = blockIdx.z;
    extern __shared__ uint8_t smem_raw[];
    float *sM0 = reinterpret_cast<float *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    float *sM1 = sM0 + K * K;
    float *sH0 = sM1 + K * K;      // [K][CC], current / next by parity
    float *sH1 = sH0 + K * CC;
    float *sPart = sH1 + K * CC;   // [NMS - 1][K][CC] partial sums
    __shared__ uint64_t bars[2];
    const int tid = threadIdx.x;
    const int cg = tid % NCG, rp = (tid / NCG) % 64, ms = tid / (NCG * 64);
    const int r0 = 2 * rp, c0 = 4 * cg;
    const bool active = r0 < K;
    const int mlen = K / NMS, m0 = ms * mlen;
    pdl_trigger();
    pdl_wait();

    const int nc = ws.seq_chunk0[n + 1] - ws.seq_chunk0[n];
    const int per = seg_per(ws, nc);
    const int nseg = per ? (nc + per - 1) / per : 0;
    // at most one segment under the common length: the output pass runs it
    // whole, from h0 to ht
    if (seg_len(ws) && nseg <= 1) return;
    const int64_t sbase = (n * H + h) * (int64_t)S;
    for (int idx = tid; idx < K * CC; idx += kComposeThreads) {
        const int key = idx / CC, c = idx - key * CC;
        sH0[idx] = p.h0 ? p.h0[state_off(p, n * H + h, key, col0 + c)] : 0.f;
    }
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init_fence();
    }
    __syncthreads();
    // A transition arrives as 8 bulk copies issued by 8 warps side by side
    // (one request per SM is far slower than the L2 can serve); the byte
    // count is announced on the barrier before any copy is issued.
    const uint32_t mbytes = (uint32_t)(K * K * 4), piece = mbytes / 8;
    auto load_m = [&](float *buf, int64_t seg, uint64_t *bar) {
        if ((tid & 31) == 0 && tid < 256) {
            const int w = tid >> 5;
            bulk_load(reinterpret_cast<uint8_t *>(buf) + w * piece,
                      reinterpret_cast<const uint8_t *>(ws.segM + seg * K * K) + w * piece, piece,
                      bar);
        }
    };
    if (tid == 0 && nseg > 0) mbar_arrive_expect_tx(&bars[0], mbytes);
    __syncthreads();
    if (nseg > 0) load_m(sM0, sbase, &bars[0]);
    if (tid == 0 && nseg > 1) mbar_arrive_expect_tx(&bars[1], mbytes);
    __syncthreads();
    // c_s is loaded one step ahead (a global load's latency would otherwise
    // sit on every step's critical path)
    auto load_c = [&](int s, float4 (&cv)[2]) {
        cv[0] = cv[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (ms == 0 && active && s < nseg) {
            const int64_t hrow = (sbase + s) * K;
#pragma unroll
            for (int i = 0; i < 2; ++i)
                cv[i] = __ldg(reinterpret_cast<const float4 *>(ws.segC + (hrow + r0 + i) * V +
                                                               col0 + c0));
        }
    };
    float4 cnext[2];
    load_c(0, cnext);
    for (int s = 0; s < nseg; ++s) {
        const float *sM = (s & 1) ? sM1 : sM0;
        const float *cur = (s & 1) ? sH1 : sH0;
        float *nxt = (s & 1) ? sH0 : sH1;
        if (s + 1 < nseg) load_m((s & 1) ? sM0 : sM1, sbase + s + 1, &bars[(s + 1) & 1]);
        const int64_t hrow = (sbase + s) * K;
        if (ms == 0 && active) {  // h_s, the segment's initial state
#pragma unroll
            for (int i = 0; i < 2; ++i)
                *reinterpret_cast<float4 *>(ws.segH + (hrow + r0 + i) * V + col0 + c0) =
                    *reinterpret_cast<const float4 *>(cur + (r0 + i) * CC + c0);
        }
        const float4 cv[2] = {cnext[0], cnext[1]};  // c_s
        load_c(s + 1, cnext);
        // every thread waits for the transition itself; whether all of them
        // got it is agreed at the barrier after the partial sums
        const bool ok = mbar_wait(&bars[s & 1], (uint32_t)(s >> 1) & 1u, p.status);
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if (active && ok) {
#pragma unroll 8
            for (int m = m0; m < m0 + mlen; ++m) {
                const float2 a = *reinterpret_cast<const float2 *>(sM + m * K + r0);
                const float4 hv = *reinterpret_cast<const float4 *>(cur + m * CC + c0);
                const float b[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[0][j] = fmaf(a.x, b[j], acc[0][j]);
                    acc[1][j] = fmaf(a.y, b[j], acc[1][j]);
                }
            }
            if (ms > 0) {
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    *reinterpret_cast<float4 *>(sPart + ((ms - 1) * K + r0 + i) * CC + c0) =
                        make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            }
        }
        if (__syncthreads_or(!ok)) return;
        if (ms == 0 && active) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                float y[4] = {acc[i][0], acc[i][1], acc[i][2], acc[i][3]};
#pragma unroll
                for (int q = 0; q < NMS - 1; ++q) {
                    const float4 pv =
                        *reinterpret_cast<const float4 *>(sPart + (q * K + r0 + i) * CC + c0);
                    y[0] += pv.x;
                    y[1] += pv.y;
                    y[2] += pv.z;
                    y[3] += pv.w;
                }
                *reinterpret_cast<float4 *>(nxt + (r0 + i) * CC + c0) = make_float4(
                    y[0] + cv[i].x, y[1] + cv[i].y, y[2] + cv[i].z, y[3] + cv[i].w);
            }
        }
        fence_async_smem();  // the transition buffer is refilled by the async proxy next
        // the barrier of the step after next expects its bytes before any copy
        if (tid == 0 && s + 2 < nseg) mbar_arrive_expect_tx(&bars[s & 1], mbytes);
        __syncthreads();
    }
    if (p.ht) {
        const float *fin = (nseg & 1) ? sH1 : sH0;
        for (int idx = tid; idx < K * CC; idx += kComposeThreads) {
            const int key = idx / CC, c = idx - key * CC;
            p.ht[state_off(p, n * H + h, key, col0 + c)] = fin[idx];
        }
    }
}

template <int CC>
cudaError_t launch_compose(const Problem &p, const Workspace &ws, cudaStream_t st) {
    constexpr int NMS = kComposeThreads / (64 * (CC / 4));
    const size_t smem = 128 + sizeof(float) * (2 * (size_t)p.K * p.K + (1 + NMS) * (size_t)p.K * CC);
    cudaError_t err = cudaFuncSetAttribute(k_compose_mt<CC>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid((unsigned)(p.V / CC), (unsigned)p.N, (unsigned)p.H);
    return launch_pdl(k_compose_mt<CC>, grid, dim3(kComposeThreads), smem, st, p, ws);
}

// Beta-free composition (scaled-identity transitions, cuLA PR #127 "Scope":
// the diagonal affine maps of the gated-linear-attention form): every state
// element evolves on its own, h_{s+1} = d_s h_s + c_s, so one thread owns one
// element of one (sequence, head) and walks the segments in order; a warp
// touches 128 contiguous bytes per access.  Bandwidth-bound: c_s read once,
// h_s written once.
__global__ void __launch_bounds__(256) k_compose_scalar(Problem p, Workspace ws) {
    const int64_t kv = p.K * p.V;
    const int64_t idx = (int64_t)blockIdx.x * 256 + threadIdx.x;
    pdl_trigger();
    pdl_wait();
    if (idx >= p.N * p.H * kv) return;
    const int64_t nh = idx / kv, e = idx - nh * kv;
    const int64_t n = nh / p.H;
    const int S = ws.n_segments;
    const int nc = ws.seq_chunk0[n + 1] - ws.seq_chunk0[n];
    const int per = seg_per(ws, nc);
    const int nseg = per ? (nc + per - 1) / per : 0;
    // at most one segment under the common length: the output pass runs it
    // whole, from h0 to ht
    if (seg_len(ws) && nseg <= 1) return;
    const float *__restrict__ C = ws.segC + nh * S * kv + e;
    float *__restrict__ Hs = ws.segH + nh * S * kv + e;
    const float *__restrict__ D = ws.segD + nh * S;
    // this element in h0 / ht: idx itself in the default layout
    const int64_t sidx = p.state_vk ? state_off(p, nh, e / p.V, e % p.V) : idx;
    float h = p.h0 ? p.h0[sidx] : 0.f;
    for (int s = 0; s < nseg; ++s) {
        const float c = C[s * kv];
        Hs[s * kv] = h;
        h = fmaf(D[s], h, c);
    }
    if (p.ht) p.ht[sidx] = h;
}

}  // namespace

cudaError_t compose_scalar(const Problem &p, const Workspace &ws, cudaStream_t st) {
    const int64_t total = p.N * p.H * p.K * p.V;
    if (total == 0) return cudaSuccess;
    return launch_pdl(k_compose_scalar, dim3((unsigned)((total + 255) / 256)), dim3(256), 0, st,
                      p, ws);
}

bool compose_mt_supported(const Problem &p) {
    // K a multiple of 32 keeps every slice of m the same length
    return p.beta != nullptr && p.K <= 128 && p.K % 32 == 0 && p.V % 8 == 0;
}

// The narrowest value tile (4, 8, 16 columns) whose CTAs still fit one wave:
// a step's time is one CTA's share of the K x K x CC products.
cudaError_t compose_mt(const Problem &p, const Workspace &ws, cudaStream_t st) {
    const int64_t sms = device_sms();
    const int64_t heads = p.N * p.H;
    if ((p.V / 4) * heads <= sms) return launch_compose<4>(p, ws, st);
    if (p.V % 16 == 0 && (p.V / 8) * heads > sms) return launch_compose<16>(p, ws, st);
    return launch_compose<8>(p, ws, st);
}

}  // namespace gdr
