// compose.cu -- A9, the ordered segment composition h_{s+1} = M_s h_s + c_s
// for the delta rule (cuLA PR #127 "Root cause and implementation": the
// per-segment FP32 transition chained by a short ordered pass), FP32 on CUDA
// cores.  One CTA owns 32 value columns of one (sequence, head) and walks its
// segments in order; each segment's K x K transition (stored transposed, so
// the 4 output rows a thread needs are one 16-byte load) is streamed into
// shared memory by a 1-D bulk async copy, double-buffered so the next
// transition loads while this one is applied.  Every output element is
// accumulated by one thread in a fixed order.
#include "gdr_internal.cuh"
#include "tc_common.cuh"

namespace gdr {
namespace {

using namespace tc;

constexpr int kCC = 32;  // value columns per CTA

__global__ void __launch_bounds__(256) k_compose_mt(Problem p, Workspace ws) {
    const int K = (int)p.K, V = (int)p.V, H = (int)p.H, S = ws.n_segments;
    const int tile = blockIdx.x;
    const int64_t n = blockIdx.y;
    const int h = blockIdx.z;
    const int col0 = tile * kCC;
    extern __shared__ uint8_t smem_raw[];
    float *sM0 = reinterpret_cast<float *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    float *sM1 = sM0 + K * K;
    float *sH = sM1 + K * K;  // [K][kCC]
    __shared__ uint64_t bars[2];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cg = lane & 7;                  // columns 4cg .. 4cg+3
    const int rg = warp * 4 + (lane >> 3);    // rows 4rg .. 4rg+3
    const bool active = rg < K / 4;

    const int nc = ws.seq_chunk0[n + 1] - ws.seq_chunk0[n];
    const int per = (nc + S - 1) / S;
    const int nseg = per ? (nc + per - 1) / per : 0;
    const int64_t sbase = (n * H + h) * (int64_t)S;
    for (int idx = tid; idx < K * kCC; idx += 256) {
        const int key = idx / kCC, c = idx - key * kCC;
        sH[idx] = p.h0 ? p.h0[((n * H + h) * K + key) * (int64_t)V + col0 + c] : 0.f;
    }
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init_fence();
    }
    __syncthreads();
    const uint32_t mbytes = (uint32_t)(K * K * 4);
    if (tid == 0 && nseg > 0) {
        mbar_arrive_expect_tx(&bars[0], mbytes);
        bulk_load(sM0, ws.segM + sbase * K * K, mbytes, &bars[0]);
    }
    for (int s = 0; s < nseg; ++s) {
        const float *sM = (s & 1) ? sM1 : sM0;
        if (tid == 0 && s + 1 < nseg) {
            float *nxt = (s & 1) ? sM0 : sM1;
            mbar_arrive_expect_tx(&bars[(s + 1) & 1], mbytes);
            bulk_load(nxt, ws.segM + (sbase + s + 1) * K * K, mbytes, &bars[(s + 1) & 1]);
        }
        float *hs_out = ws.segH + (sbase + s) * K * V;
        for (int idx = tid; idx < K * kCC; idx += 256) {
            const int key = idx / kCC, c = idx - key * kCC;
            hs_out[(int64_t)key * V + col0 + c] = sH[idx];
        }
        const bool ok = mbar_wait(&bars[s & 1], (uint32_t)(s >> 1) & 1u, p.status);
        if (__syncthreads_or(!ok)) return;
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
        if (active) {
            for (int m = 0; m < K; ++m) {
                const float4 mt = *reinterpret_cast<const float4 *>(sM + m * K + 4 * rg);
                const float4 hv = *reinterpret_cast<const float4 *>(sH + m * kCC + 4 * cg);
                const float a[4] = {mt.x, mt.y, mt.z, mt.w};
                const float b[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
        }
        fence_async_smem();
        __syncthreads();
        if (active) {
            const float *C = ws.segC + (sbase + s) * K * V;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = 4 * rg + i, c = 4 * cg + j;
                    sH[r * kCC + c] = acc[i][j] + C[(int64_t)r * V + col0 + c];
                }
        }
        __syncthreads();
    }
    if (p.ht) {
        for (int idx = tid; idx < K * kCC; idx += 256) {
            const int key = idx / kCC, c = idx - key * kCC;
            p.ht[((n * H + h) * K + key) * (int64_t)V + col0 + c] = sH[idx];
        }
    }
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
    if (idx >= p.N * p.H * kv) return;
    const int64_t nh = idx / kv, e = idx - nh * kv;
    const int64_t n = nh / p.H;
    const int S = ws.n_segments;
    const int nc = ws.seq_chunk0[n + 1] - ws.seq_chunk0[n];
    const int per = (nc + S - 1) / S;
    const int nseg = per ? (nc + per - 1) / per : 0;
    const float *__restrict__ C = ws.segC + nh * S * kv + e;
    float *__restrict__ Hs = ws.segH + nh * S * kv + e;
    const float *__restrict__ D = ws.segD + nh * S;
    float h = p.h0 ? p.h0[idx] : 0.f;
    for (int s = 0; s < nseg; ++s) {
        const float c = C[s * kv];
        Hs[s * kv] = h;
        h = fmaf(D[s], h, c);
    }
    if (p.ht) p.ht[idx] = h;
}

}  // namespace

cudaError_t compose_scalar(const Problem &p, const Workspace &ws, cudaStream_t st) {
    const int64_t total = p.N * p.H * p.K * p.V;
    if (total == 0) return cudaSuccess;
    k_compose_scalar<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(p, ws);
    return cudaGetLastError();
}

bool compose_mt_supported(const Problem &p) {
    return p.beta != nullptr && p.K <= 128 && p.K % 16 == 0 && p.V % kCC == 0;
}

cudaError_t compose_mt(const Problem &p, const Workspace &ws, cudaStream_t st) {
    const size_t smem = 128 + sizeof(float) * (2 * (size_t)p.K * p.K + (size_t)p.K * kCC);
    cudaError_t err = cudaFuncSetAttribute(k_compose_mt,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid((unsigned)(p.V / kCC), (unsigned)p.N, (unsigned)p.H);
    k_compose_mt<<<grid, 256, smem, st>>>(p, ws);
    return cudaGetLastError();
}

}  // namespace gdr
