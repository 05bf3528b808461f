// recurrent.cu -- the per-token recurrence itself, for serving (a decode step
// or a few tokens a sequence): every sequence starts from a state row of a
// caller-owned pool, runs its tokens in order and writes the final state back
// into the same row.  Where a 64-token chunk would be mostly padding, this is
// the operator to call (the "question rows" with their own states of Kev PR
// #259 "Not covered", the indexed-state idea).  Per token, with h = S^T:
//
//   h <- e^{g_t} h;   u = beta_t (v_t - h^T k_t);   h <- h + k_t u^T
//   (beta-free: h <- h + k_t v_t^T);   o_t = scale h^T q_t
//
// which is the delta rule S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) +
// beta_t v_t k_t^T, o_t = scale S_t q_t of the project statement.  FP32
// arithmetic; q, k, v are widened from BF16 on load.
//
// One CTA per (sequence, head, 32-column value tile): warp w holds rows
// [w K/8, (w+1) K/8) of the tile in registers (lane = column), so the state
// is read once and written once per call; h^T k and h^T q are reduced
// across the eight warps through shared memory in a fixed order.
#include <type_traits>

#include "gdr_internal.cuh"

namespace gdr {
namespace {

constexpr int kRThreads = 256;  // eight warps
constexpr int kRCols = 32;      // value columns per CTA (one per lane)
constexpr int kRMaxRows = kMaxK / 8;

template <typename Tin>
__device__ __forceinline__ float ld_in(const void *p, int64_t i) {
    const Tin x = reinterpret_cast<const Tin *>(p)[i];
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) return __bfloat162float(x);
    else if constexpr (std::is_same<Tin, __half>::value) return __half2float(x);
    else return x;
}
template <typename Tin>
__device__ __forceinline__ void st_out(void *p, int64_t i, float x) {
    Tin *q = reinterpret_cast<Tin *>(p);
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) q[i] = __float2bfloat16_rn(x);
    else if constexpr (std::is_same<Tin, __half>::value) q[i] = __float2half_rn(x);
    else q[i] = x;
}

// Four CTAs an SM (at most 64 registers a thread, no spills) up to K = 128:
// the state loads of four tiles in flight per SM (decode step of 256
// sequences x 16 heads: 161 us against 201 us with three).
template <typename Tin, int RPW>
__global__ void __launch_bounds__(kRThreads, RPW <= 16 ? 4 : 2)
    k_recurrent(Problem p, float *state, int64_t n_states, const int32_t *state_idx) {
    const int K = (int)p.K, V = (int)p.V, H = (int)p.H;
    const int64_t n = blockIdx.y;
    const int h = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int col = blockIdx.x * kRCols + lane;
    const bool live = col < V;
    const int r0 = warp * RPW;  // this warp's first row
    __shared__ float sk[kMaxK], sq[kMaxK], sv[kRCols], sg[2];
    __shared__ float sred[2][8][kRCols];

    const int64_t t0 = seq_start(p, n);
    const int64_t t1 = seq_end(p, n);
    if (t1 < t0) {  // malformed cu_seqlens: nothing for this sequence
        if (tid == 0 && blockIdx.x == 0 && h == 0 && p.status)
            atomicCAS(p.status, 0, (int32_t)GDR_ERR_SEQLENS);
        return;
    }
    const int64_t row_id = state_idx ? (int64_t)state_idx[n] : n;
    if (row_id < 0 || row_id >= n_states) {
        if (tid == 0 && blockIdx.x == 0 && h == 0 && p.status)
            atomicCAS(p.status, 0, (int32_t)GDR_ERR_INDEX);
        return;
    }
    // element (key, col) of the pool row's state for head h (either layout)
    auto at = [&](int key) -> int64_t { return state_off(p, row_id * H + h, key, col); };
    float hr[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) hr[r] = (live && r0 + r < K) ? state[at(r0 + r)] : 0.f;

    const bool delta = p.beta != nullptr;
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t th = t * H + h;
        for (int i = tid; i < K; i += kRThreads) {
            sk[i] = ld_in<Tin>(p.k, tok_at(p.sk, t, h) + i);
            sq[i] = ld_in<Tin>(p.q, tok_at(p.sq, t, h) + i);
        }
        if (tid < kRCols) {
            const int c = blockIdx.x * kRCols + tid;
            sv[tid] = c < V ? ld_in<Tin>(p.v, tok_at(p.sv, t, h) + c) : 0.f;
        }
        if (tid == 0) {
            sg[0] = __expf(p.g[th]);
            sg[1] = delta ? p.beta[th] : 0.f;
        }
        __syncthreads();
        const float a = sg[0];
        float part = 0.f;
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            hr[r] *= a;
            if (r0 + r < K) part = fmaf(hr[r], sk[r0 + r], part);
        }
        float u;
        if (delta) {  // u = beta (v - h^T k), the eight warps' partial sums in order
            sred[0][warp][lane] = part;
            __syncthreads();
            float hk = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) hk += sred[0][w][lane];
            u = sg[1] * (sv[lane] - hk);
        } else {
            u = sv[lane];
        }
        float po = 0.f;
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            if (r0 + r < K) {
                hr[r] = fmaf(sk[r0 + r], u, hr[r]);
                po = fmaf(hr[r], sq[r0 + r], po);
            }
        }
        sred[1][warp][lane] = po;
        __syncthreads();
        if (warp == 0 && live) {
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) o += sred[1][w][lane];
            st_out<Tin>(p.o, tok_at(p.so, t, h) + col, p.scale * o);
        }
        __syncthreads();  // sk, sq, sv, sred are refilled for the next token
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r)
        if (live && r0 + r < K) state[at(r0 + r)] = hr[r];
}

template <typename Tin>
cudaError_t launch_rec(const Problem &p, float *state, int64_t n_states, const int32_t *idx,
                       cudaStream_t st) {
    dim3 grid((unsigned)((p.V + kRCols - 1) / kRCols), (unsigned)p.N, (unsigned)p.H);
    const int rpw = (int)((p.K + 7) / 8);
    if (rpw <= 8) k_recurrent<Tin, 8><<<grid, kRThreads, 0, st>>>(p, state, n_states, idx);
    else if (rpw <= 16) k_recurrent<Tin, 16><<<grid, kRThreads, 0, st>>>(p, state, n_states, idx);
    else k_recurrent<Tin, kRMaxRows><<<grid, kRThreads, 0, st>>>(p, state, n_states, idx);
    return cudaGetLastError();
}

}  // namespace

cudaError_t recurrent_fwd(const Problem &p, float *state, int64_t n_states,
                          const int32_t *state_idx, cudaStream_t st) {
    if (p.N == 0) return cudaSuccess;
    if (p.dtype == GDR_BF16) return launch_rec<__nv_bfloat16>(p, state, n_states, state_idx, st);
    if (p.dtype == GDR_F16) return launch_rec<__half>(p, state, n_states, state_idx, st);
    return launch_rec<float>(p, state, n_states, state_idx, st);
}

}  // namespace gdr
