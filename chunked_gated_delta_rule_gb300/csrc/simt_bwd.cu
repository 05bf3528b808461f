// simt_bwd.cu -- backward pass of the chunked gated delta rule on CUDA cores,
// FP32 arithmetic for every input type.  The gradient of
// L = <do, o> + <dht, ht> with respect to q, k, v, g, beta and h0.
//
// The pages run the state-gradient recurrence in reverse, chunk by chunk
// (flash-linear-attention ABC issue #23, "Problem": the reverse dH kernel
// loops serially over every 64-token chunk; "Proposed Dataflow" step 4), and
// ask for dQ/dK/dV and state gradients ("Fixture-First Correctness
// Contract").  This file differentiates the chunked form of the forward pass
// (the UT / WY form of the project statement), per chunk of length L with
// chunk-local gate cumsum G, gamma = e^G, Gam = e^{G_last},
// lam_j = e^{G_last - G_j}, D_ij = e^{G_i - G_j}:
//
//   forward:   A = strict_lower(diag(beta) (K K^T * D)),  T = (I + A)^-1
//              W = T diag(beta gamma) K,  U = T diag(beta) V,  V' = U - W h
//              O = scale [diag(gamma) Q h + M V'],  M = causal(Q K^T * D)
//              h_out = Gam h + (diag(lam) K)^T V'
//   backward, with E = dL/dh_out (dht after the last chunk):
//              dV'    = scale M^T dO + diag(lam) K E
//              dh     = Gam E + scale (diag(gamma) Q)^T dO - W^T dV'
//              Z      = scale causal(dO V'^T) * D            (dL/d(Q K^T))
//              dQ     = scale diag(gamma) dO h^T + Z K
//              dKb    = -T^T dV' h^T,   dVb = T^T dV'
//              dT     = dV' (diag(beta) V)^T - dV' h^T (diag(beta gamma) K)^T
//              dA     = -strict_lower(T^T dT T^T),   S = diag(beta) dA * D
//              dK     = Z^T Q + diag(lam) V' E^T + diag(beta gamma) dKb + S K + S^T K
//              dV     = diag(beta) dVb
//              dbeta  = rowdot(dVb, V) + gamma rowdot(dKb, K) + rowsum(dA * K K^T * D)
//              dG     = gate terms of every e^G factor;  dg = reverse cumsum of dG
// Beta-free mode: V' = V, W = 0, no A / T terms; dv = dV'.
//
// Kernels, after the forward recompute of the CUDA-core path (chunk table,
// prep, serial scan: G, W, U, the state before each chunk and V'):
//   k_bwd_gram   per (chunk, head): M, K K^T * D (strictly lower), T
//   k_bwd_dscan  per (sequence, head, value tile): the reverse scan over the
//                chunks, storing E at each chunk's end and dV' (dv if
//                beta-free); dh0 at the end
//   k_bwd_lk     per (chunk, head, 64-key slice): dO h^T, dV' h^T, V' E^T and
//                the partial <E, h>
//   k_bwd_local  per (chunk, head): dq, dk, dv, dbeta, dg
// Every output element is summed by one thread in a fixed order, so results
// are bit-identical from run to run.
#include "gdr_internal.cuh"
#include "gdr_launch.cuh"
#include "simt_tile.cuh"

namespace gdr {
namespace {

constexpr int kBT = 256;      // threads per CTA
constexpr int kSl = 64;       // slice width of the key / value loops
constexpr int kLd = kSl + 1;  // padded row of a 64 x 64 tile

__device__ __forceinline__ float ldx(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ldx(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ float ldx(const __half *p, int64_t i) { return __half2float(p[i]); }
__device__ __forceinline__ void stx(float *p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void stx(__nv_bfloat16 *p, int64_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}
__device__ __forceinline__ void stx(__half *p, int64_t i, float x) { p[i] = __float2half_rn(x); }

struct ChunkInfo {
    int64_t t0;  // first flat token (row-major over [B, T])
    int len;     // tokens in the chunk (1..64)
};

__device__ __forceinline__ ChunkInfo chunk_info(const Workspace &ws, int64_t gc) {
    const int4 e = reinterpret_cast<const int4 *>(ws.chunk_tab)[gc];
    return ChunkInfo{(int64_t)e.y, e.z};
}

// True when every caller tensor the backward kernels read by rows (q, k, v
// with their strides, dout contiguous) has 16-byte aligned rows (K and V are
// multiples of 16): the tiles then load in 16-byte pieces.
template <typename T>
__device__ __forceinline__ bool inputs_vec16(const Problem &p, const BwdArgs &a) {
    const int es = (int)sizeof(T);
    return rows_aligned16(p.q, p.sq, es) && rows_aligned16(p.k, p.sk, es) &&
           rows_aligned16(p.v, p.sv, es) && rows_aligned16(a.dout, dense_stride(p.H, p.V), es);
}

// Rows [0, 64) x columns [c0, c0 + 64) of a token-major input [tokens][H][D]
// (rows beyond len and columns beyond D read as 0) into a 64 x 65 tile, in
// 16-byte pieces when `vec` (D is a multiple of 16, so a piece is entirely
// inside or outside the row).
template <typename T>
__device__ __forceinline__ void load_tok_tile(float *dst, const T *src, int64_t t0, int len,
                                              const TokStride &st, int h, int D, int c0, int tid,
                                              bool vec = false) {
    if (vec) {
        constexpr int E = 16 / (int)sizeof(T);
        constexpr int PR = kSl / E;  // pieces per row
        for (int idx = tid; idx < kChunk * PR; idx += kBT) {
            const int i = idx / PR, c = (idx - i * PR) * E;
            float x[E];
            if (i < len && c0 + c < D) {
                const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(
                    src + tok_at(st, t0 + i, h) + c0 + c));
                unpack16(raw, src, x);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) x[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < E; ++e) dst[i * kLd + c + e] = x[e];
        }
        return;
    }
    for (int idx = tid; idx < kChunk * kSl; idx += kBT) {
        const int i = idx >> 6, c = idx & 63;
        float x = 0.f;
        if (i < len && c0 + c < D) x = ldx(src, tok_at(st, t0 + i, h) + c0 + c);
        dst[i * kLd + c] = x;
    }
}

// Rows [r0, r0 + 64) x columns [c0, c0 + 64) of a row-major FP32 workspace
// matrix with `rows` rows and row stride `ld` (columns beyond `cols` read as
// 0), in float4 pieces: workspace matrices start on 256-byte boundaries and
// ld, cols and c0 are multiples of 16.
__device__ __forceinline__ void load_mat_tile(float *dst, const float *src, int r0, int rows,
                                              int c0, int cols, int64_t ld, int tid) {
    for (int idx = tid; idx < kSl * (kSl / 4); idx += kBT) {
        const int i = idx >> 4, c = (idx & 15) * 4;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r0 + i < rows && c0 + c < cols)
            x = __ldg(reinterpret_cast<const float4 *>(src + (int64_t)(r0 + i) * ld + c0 + c));
        float *d = dst + i * kLd + c;
        d[0] = x.x;
        d[1] = x.y;
        d[2] = x.z;
        d[3] = x.w;
    }
}

// ---------------------------------------------------------------------------
// k_bwd_gram: M = causal(Q K^T * D) (diagonal included), Kd = strictly lower
// (K K^T * D) and, in delta mode, T = (I + diag(beta) Kd)^-1.
template <typename Tin>
__global__ void __launch_bounds__(kBT) k_bwd_gram(Problem p, Workspace ws, BwdWs bw) {
    const int64_t gc = blockIdx.x;
    const int h = blockIdx.y;
    if (gc >= *ws.n_chunks) return;
    const ChunkInfo ci = chunk_info(ws, gc);
    const int H = (int)p.H, K = (int)p.K, tid = threadIdx.x;
    const bool delta = p.beta != nullptr;
    extern __shared__ float sm[];
    float *sQ = sm, *sK = sQ + kChunk * kLd, *sA = sK + kChunk * kLd;
    float *sG = sA + kChunk * kLd, *sB = sG + kChunk;
    if (tid < kChunk) {
        sG[tid] = ws.G[(gc * H + h) * kChunk + tid];
        sB[tid] = (delta && tid < ci.len) ? p.beta[(ci.t0 + tid) * H + h] : 0.f;
    }
    const bool vec = rows_aligned16(p.q, p.sq, sizeof(Tin)) && rows_aligned16(p.k, p.sk, sizeof(Tin));
    float qk[4][4], kk[4][4];
    acc_zero(qk);
    acc_zero(kk);
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    for (int c0 = 0; c0 < K; c0 += kSl) {
        __syncthreads();
        load_tok_tile(sQ, q, ci.t0, ci.len, p.sq, h, K, c0, tid, vec);
        load_tok_tile(sK, k, ci.t0, ci.len, p.sk, h, K, c0, tid, vec);
        __syncthreads();
        const int kn = min(kSl, K - c0);
        mm_abT<4>(qk, sQ, kLd, sK, kLd, kn, tid);
        if (delta) mm_abT<4>(kk, sK, kLd, sK, kLd, kn, tid);
    }
    float *Mg = bw.Mq + (gc * H + h) * (int64_t)kChunk * kChunk;
    float *Kdg = bw.Kd + (gc * H + h) * (int64_t)kChunk * kChunk;
    const int i0 = 4 * (tid >> 4), j0 = tid & 15;
    FOR_TILE(4) {
        const int i = i0 + r, j = j0 + 16 * s;
        const bool in = i < ci.len;
        const float d = (in && j <= i) ? expf(sG[i] - sG[j]) : 0.f;
        Mg[i * kChunk + j] = (in && j <= i) ? qk[r][s] * d : 0.f;
        if (delta) {
            const float kd = (in && j < i) ? kk[r][s] * d : 0.f;
            Kdg[i * kChunk + j] = kd;
            sA[i * kLd + j] = sB[i] * kd;
        }
    }
    if (!delta) return;
    __syncthreads();
    // T = (I + A)^-1 by forward substitution, one column per thread, into sQ
    if (tid < kChunk) {
        const int m = tid;
        for (int i = 0; i < kChunk; ++i) {
            float x;
            if (i < m) {
                x = 0.f;
            } else if (i == m) {
                x = 1.f;
            } else {
                float sum = 0.f;
                for (int jj = m; jj < i; ++jj) sum = fmaf(sA[i * kLd + jj], sQ[jj * kLd + m], sum);
                x = -sum;
            }
            sQ[i * kLd + m] = x;
        }
    }
    __syncthreads();
    float *Tg = bw.Tm + (gc * H + h) * (int64_t)kChunk * kChunk;
    for (int idx = tid; idx < kChunk * kChunk; idx += kBT)
        Tg[idx] = sQ[(idx >> 6) * kLd + (idx & 63)];
}

// ---------------------------------------------------------------------------
// k_bwd_dscan: the reverse scan of one (sequence, head, value tile), chunks
// from last to first.  E is dL/d(state at the chunk's end).  Each step is
// affine in E: E_start = (Gam I - W^T diag(lam) K) E_end + C, C collecting
// the dO terms, so the scan splits into segments like the forward one (the
// pages' "Proposed Dataflow" step 4: the reverse recurrence mirrors the
// split).  mode 0: whole sequence from dht, writes dh0; mode 1: segment
// pre-scan from E = 0 (-> the segment's offset c; its K x K map is the
// transpose of the forward map, see k_bwd_maps); mode 2: segment output pass
// from the composed E at the segment's end.  Modes 0 and 2 store E and dV'
// per chunk.
// Segment s of a sequence's nseg segments keeps its summaries in slot
// nseg - 1 - s, so the ordered composition runs from the last segment to the
// first: it starts from dht and ends at dh0.
template <typename Tin, int BV>
__global__ void __launch_bounds__(kBT) k_bwd_dscan(Problem p, Workspace ws, BwdArgs a,
                                                   BwdWs bw, int mode) {
    constexpr int LDE = BV + 1;
    constexpr int NS = BV / 16;  // column groups of the 64 x BV tiles
    const int H = (int)p.H, K = (int)p.K, V = (int)p.V;
    const bool delta_mode = p.beta != nullptr;
    const int S = mode == 0 ? 1 : ws.n_segments;
    const int n_vtiles = V / BV;
    const int ntiles = n_vtiles;
    int64_t bid = blockIdx.x;
    const int tile = (int)(bid % ntiles);
    bid /= ntiles;
    const int seg = (int)(bid % S);
    const int64_t n = bid / S;
    const int col0 = tile * BV;
    const int h = blockIdx.y, tid = threadIdx.x;
    const int i0 = 4 * (tid >> 4), j0 = tid & 15;
    const bool delta = p.beta != nullptr;
    extern __shared__ float sm[];
    float *sE = sm;                       // [K][BV+1]
    float *sM = sE + K * LDE;             // [64][65]
    float *sDo = sM + kChunk * kLd;       // [64][BV+1]
    float *sDv = sDo + kChunk * LDE;      // [64][BV+1]
    float *sX = sDv + kChunk * LDE;       // [64][65] key slice of K, or of diag(gamma) Q
    float *sY = sX + kChunk * kLd;        // [64][65] key slice of W
    float *sGam = sY + kChunk * kLd, *sLam = sGam + kChunk;

    const int64_t nh = n * H + h;
    const int c_begin = ws.seq_chunk0[n];
    const int nc = ws.seq_chunk0[n + 1] - c_begin;
    int s0 = 0, s1 = nc, slot = 0;
    if (mode != 0) {
        const int per = (nc + S - 1) / S;
        const int nseg = per ? (nc + per - 1) / per : 0;
        s0 = seg * per;
        s1 = min(nc, s0 + per);
        if (s0 >= s1) return;
        slot = nseg - 1 - seg;
    }
    const int64_t seg_base = nh * (int64_t)S + slot;
    for (int idx = tid; idx < K * BV; idx += kBT) {
        const int key = idx / BV, c = idx - key * BV;
        float x = 0.f;
        if (mode == 0)
            x = a.dht ? a.dht[state_off(p, nh, key, col0 + c)] : 0.f;
        else if (mode == 2)
            x = ws.segH[(seg_base * K + key) * V + col0 + c];
        sE[key * LDE + c] = x;
    }
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *dout = static_cast<const Tin *>(a.dout);
    const bool vec = inputs_vec16<Tin>(p, a);
    float dprod = 1.f;
    for (int cc = s1 - 1; cc >= s0; --cc) {
        const int64_t gc = c_begin + cc;
        const ChunkInfo ci = chunk_info(ws, gc);
        const int64_t item = gc * H + h;
        __syncthreads();
        if (mode != 1) {
            float *Eg = bw.dhend + item * (int64_t)K * V;
            for (int idx = tid; idx < K * BV; idx += kBT) {
                const int key = idx / BV, c = idx - key * BV;
                Eg[(int64_t)key * V + col0 + c] = sE[key * LDE + c];
            }
        }
        if (tid < kChunk) {
            const float *G = ws.G + item * kChunk;
            const bool in = tid < ci.len;
            sGam[tid] = in ? expf(G[tid]) : 0.f;
            sLam[tid] = in ? expf(G[ci.len - 1] - G[tid]) : 0.f;
        }
        for (int idx = tid; idx < kChunk * kChunk; idx += kBT)
            sM[(idx >> 6) * kLd + (idx & 63)] = bw.Mq[item * kChunk * kChunk + idx];
        for (int idx = tid; idx < kChunk * BV; idx += kBT) {
            const int i = idx / BV, c = idx - i * BV;
            sDo[i * LDE + c] =
                i < ci.len ? ldx(dout, ((ci.t0 + i) * H + h) * (int64_t)V + col0 + c) : 0.f;
        }
        // dV' = scale M^T dO + diag(lam) K E
        float acc[4][NS];
        acc_zero(acc);
        for (int k0 = 0; k0 < K; k0 += kSl) {
            __syncthreads();
            load_tok_tile(sX, k, ci.t0, ci.len, p.sk, h, K, k0, tid, vec);
            __syncthreads();
            mm_ab<NS>(acc, sX, kLd, sE + k0 * LDE, LDE, min(kSl, K - k0), tid);
        }
        float mt[4][NS];
        acc_zero(mt);
        mm_atb<NS>(mt, sM, kLd, sDo, LDE, kChunk, tid);
        const float gam_last = expf(ws.G[item * kChunk + ci.len - 1]);
        FOR_TILE(NS) {
            const int i = i0 + r, c = j0 + 16 * s;
            const float dvn = i < ci.len ? fmaf(p.scale, mt[r][s], sLam[i] * acc[r][s]) : 0.f;
            sDv[i * LDE + c] = dvn;
            if (i < ci.len && mode != 1) {
                if (delta)
                    bw.dvn[(item * kChunk + i) * (int64_t)V + col0 + c] = dvn;
                else
                    stx(static_cast<Tin *>(a.dv), ((ci.t0 + i) * H + h) * (int64_t)V + col0 + c,
                        dvn);
            }
        }
        // E <- Gam E + scale (diag(gamma) Q)^T dO - W^T dV'
        for (int k0 = 0; k0 < K; k0 += kSl) {
            __syncthreads();
            for (int idx = tid; idx < kChunk * kSl; idx += kBT) {
                const int i = idx >> 6, c = idx & 63;
                float x = 0.f;
                if (i < ci.len && k0 + c < K)
                    x = sGam[i] * ldx(q, tok_at(p.sq, ci.t0 + i, h) + k0 + c);
                sX[i * kLd + c] = x;
            }
            if (delta)
                load_mat_tile(sY, ws.W + item * (int64_t)kChunk * K, 0, kChunk, k0, K, K, tid);
            __syncthreads();
            float e1[4][NS], e2[4][NS];
            acc_zero(e1);
            acc_zero(e2);
            mm_atb<NS>(e1, sX, kLd, sDo, LDE, kChunk, tid);
            if (delta) mm_atb<NS>(e2, sY, kLd, sDv, LDE, kChunk, tid);
            const int kn = min(kSl, K - k0);
            FOR_TILE(NS) {
                const int kk = i0 + r, c = j0 + 16 * s;
                if (kk < kn) {
                    float *e = &sE[(k0 + kk) * LDE + c];
                    *e = fmaf(gam_last, *e, fmaf(p.scale, e1[r][s], -e2[r][s]));
                }
            }
        }
        dprod *= gam_last;
    }
    __syncthreads();
    if (mode == 0) {
        if (a.dh0) {
            for (int idx = tid; idx < K * BV; idx += kBT) {
                const int key = idx / BV, c = idx - key * BV;
                a.dh0[state_off(p, nh, key, col0 + c)] = sE[key * LDE + c];
            }
        }
    } else if (mode == 1) {
        for (int idx = tid; idx < K * BV; idx += kBT) {
            const int key = idx / BV, c = idx - key * BV;
            ws.segC[(seg_base * K + key) * V + col0 + c] = sE[key * LDE + c];
        }
        if (!delta_mode && tile == 0 && tid == 0) ws.segD[seg_base] = dprod;
    }
}

// ---------------------------------------------------------------------------
// k_bwd_maps: the K x K maps of the reverse scan's segments, from the forward
// recompute's.  The reverse step is the transpose of the forward step
// (Gam I - W^T diag(lam) K = (Gam I - K^T diag(lam) W)^T), so a segment's
// reverse map is the transpose of its forward map.  The forward pre-scan
// stores map M_s of segment s transposed; the composition of the reverse
// scan reads its maps transposed too, in reversed slots, so block s is
// copied untransposed (M_s^T transposed back) into slot nseg - 1 - s of
// segMb.  One CTA per (sequence, head, segment), 32 x 32 tiles through
// shared memory.
__global__ void __launch_bounds__(kBT) k_bwd_maps(Problem p, Workspace ws, float *segMb) {
    const int K = (int)p.K, H = (int)p.H, S = ws.n_segments, tid = threadIdx.x;
    const int s = (int)(blockIdx.x % S);
    const int64_t nh = blockIdx.x / S, n = nh / H;
    const int nc = ws.seq_chunk0[n + 1] - ws.seq_chunk0[n];
    const int per = (nc + S - 1) / S;
    const int nseg = per ? (nc + per - 1) / per : 0;
    if (s >= nseg) return;
    const float *src = ws.segM + (nh * S + s) * (int64_t)K * K;
    float *dst = segMb + (nh * S + (nseg - 1 - s)) * (int64_t)K * K;
    __shared__ float tile[32][33];
    for (int r0 = 0; r0 < K; r0 += 32) {
        for (int c0 = 0; c0 < K; c0 += 32) {
            __syncthreads();
            for (int idx = tid; idx < 32 * 32; idx += kBT) {
                const int y = idx >> 5, x = idx & 31;
                if (r0 + y < K && c0 + x < K) tile[y][x] = src[(int64_t)(r0 + y) * K + c0 + x];
            }
            __syncthreads();
            for (int idx = tid; idx < 32 * 32; idx += kBT) {
                const int y = idx >> 5, x = idx & 31;
                if (c0 + y < K && r0 + x < K) dst[(int64_t)(c0 + y) * K + r0 + x] = tile[x][y];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// k_bwd_lk: for one (chunk, head, 64-key slice) the L x K products over the
// value dimension P1 = dO h^T, P2 = dV' h^T (delta), P3 = V' E^T, and the
// slice's share of <E, h>.
template <typename Tin>
__global__ void __launch_bounds__(kBT) k_bwd_lk(Problem p, Workspace ws, BwdArgs a, BwdWs bw) {
    const int64_t gc = blockIdx.x;
    const int h = blockIdx.y, ks = blockIdx.z, k0 = ks * kSl;
    if (gc >= *ws.n_chunks) return;
    const ChunkInfo ci = chunk_info(ws, gc);
    const int H = (int)p.H, K = (int)p.K, V = (int)p.V, tid = threadIdx.x;
    const bool delta = p.beta != nullptr;
    const int64_t item = gc * H + h;
    extern __shared__ float sm[];
    float *sDo = sm, *sDv = sDo + kChunk * kLd, *sVn = sDv + kChunk * kLd;
    float *sH = sVn + kChunk * kLd, *sE = sH + kChunk * kLd, *sRed = sE + kChunk * kLd;
    const Tin *dout = static_cast<const Tin *>(a.dout);
    const Tin *v = static_cast<const Tin *>(p.v);
    const float *hg = ws.hpre + item * (int64_t)K * V;
    const float *eg = bw.dhend + item * (int64_t)K * V;
    const bool vec = inputs_vec16<Tin>(p, a);
    float p1[4][4], p2[4][4], p3[4][4];
    acc_zero(p1);
    acc_zero(p2);
    acc_zero(p3);
    float eh = 0.f;
    for (int c0 = 0; c0 < V; c0 += kSl) {
        __syncthreads();
        load_tok_tile(sDo, dout, ci.t0, ci.len, dense_stride(H, V), h, V, c0, tid, vec);
        if (delta) {
            load_mat_tile(sDv, bw.dvn + item * (int64_t)kChunk * V, 0, ci.len, c0, V, V, tid);
            load_mat_tile(sVn, ws.vnew + item * (int64_t)kChunk * V, 0, ci.len, c0, V, V, tid);
        } else {
            load_tok_tile(sVn, v, ci.t0, ci.len, p.sv, h, V, c0, tid, vec);
        }
        load_mat_tile(sH, hg, k0, K, c0, V, V, tid);
        load_mat_tile(sE, eg, k0, K, c0, V, V, tid);
        __syncthreads();
        const int cn = min(kSl, V - c0);
        mm_abT<4>(p1, sDo, kLd, sH, kLd, cn, tid);
        if (delta) mm_abT<4>(p2, sDv, kLd, sH, kLd, cn, tid);
        mm_abT<4>(p3, sVn, kLd, sE, kLd, cn, tid);
        // <E, h> over this key slice: thread tid owns key tid & 63 and a
        // quarter of the slice's columns
        {
            const int key = tid & 63, part = tid >> 6;
            for (int c = part; c < cn; c += 4) eh = fmaf(sE[key * kLd + c], sH[key * kLd + c], eh);
        }
    }
    const int i0 = 4 * (tid >> 4), j0 = tid & 15;
    FOR_TILE(4) {
        const int i = i0 + r, kk = j0 + 16 * s;
        if (k0 + kk < K) {
            const int64_t o = (item * kChunk + i) * (int64_t)K + k0 + kk;
            bw.P1[o] = p1[r][s];
            if (delta) bw.P2[o] = p2[r][s];
            bw.P3[o] = p3[r][s];
        }
    }
    sRed[tid] = eh;
    __syncthreads();
    if (tid == 0) {
        float sum = 0.f;
        for (int t = 0; t < kBT; ++t) sum += sRed[t];
        bw.ehp[item * ((K + kSl - 1) / kSl) + ks] = sum;
    }
}

// ---------------------------------------------------------------------------
// k_bwd_local: every local gradient of one (chunk, head).  Matrices are
// stored with exact zeros outside their support (causal, strictly lower,
// rows past the chunk's length), so full 64-wide products give the masked
// sums.
template <typename Tin>
__global__ void __launch_bounds__(kBT) k_bwd_local(Problem p, Workspace ws, BwdArgs a,
                                                   BwdWs bw) {
    const int64_t gc = blockIdx.x;
    const int h = blockIdx.y;
    if (gc >= *ws.n_chunks) return;
    const ChunkInfo ci = chunk_info(ws, gc);
    const int H = (int)p.H, K = (int)p.K, V = (int)p.V, tid = threadIdx.x, len = ci.len;
    const int i0 = 4 * (tid >> 4), j0 = tid & 15;
    const bool delta = p.beta != nullptr;
    const int64_t item = gc * H + h;
    const float scale = p.scale;
    extern __shared__ float sm[];
    constexpr int T64 = kChunk * kLd;
    float *sM = sm;             // M = causal(Q K^T * D)
    float *sZ = sM + T64;       // Z = scale causal(dO V'^T) * D
    float *sR = sZ + T64;       // R = Z * (Q K^T), then S = diag(beta) dA * D
    float *s1 = sR + T64;       // slices
    float *s2 = s1 + T64;
    float *s3 = s2 + T64;
    float *s4 = s3 + T64;
    float *s5 = s4 + T64;
    float *s6 = s5 + T64;       // dKb / dVb slice
    float *sKd = s6 + T64;      // delta only from here
    float *sT = sKd + T64;
    float *sdT = sT + T64;      // dT, then dA
    float *sX = sdT + T64;      // dT T^T
    float *vec = delta ? sX + T64 : sKd;  // 13 tiles (delta) or 9, then 13 vectors
    float *sG = vec, *sGam = sG + kChunk, *sLam = sGam + kChunk, *sB = sLam + kChunk;
    float *r1 = sB + kChunk, *r2 = r1 + kChunk, *r3 = r2 + kChunk, *r4 = r3 + kChunk;
    float *rdA = r4 + kChunk, *rowR = rdA + kChunk, *colR = rowR + kChunk;
    float *colRA = colR + kChunk, *sdG = colRA + kChunk;

    if (tid < kChunk) {
        const bool in = tid < len;
        const float G = ws.G[item * kChunk + tid];
        sG[tid] = G;
        sGam[tid] = in ? expf(G) : 0.f;
        sLam[tid] = in ? expf(ws.G[item * kChunk + len - 1] - G) : 0.f;
        sB[tid] = (delta && in) ? p.beta[(ci.t0 + tid) * H + h] : 0.f;
        r1[tid] = r2[tid] = r3[tid] = r4[tid] = 0.f;
    }
    for (int idx = tid; idx < kChunk * kChunk; idx += kBT) {
        const int i = idx >> 6, j = idx & 63;
        sM[i * kLd + j] = bw.Mq[item * kChunk * kChunk + idx];
        if (delta) {
            sKd[i * kLd + j] = bw.Kd[item * kChunk * kChunk + idx];
            sT[i * kLd + j] = bw.Tm[item * kChunk * kChunk + idx];
        }
    }
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    const Tin *dout = static_cast<const Tin *>(a.dout);
    const bool v16 = inputs_vec16<Tin>(p, a);

    // value loop: dMraw = dO V'^T; delta: dTa = dV' V^T (times beta_j below)
    {
        float dm[4][4], dt[4][4];
        acc_zero(dm);
        acc_zero(dt);
        for (int c0 = 0; c0 < V; c0 += kSl) {
            __syncthreads();
            load_tok_tile(s1, dout, ci.t0, len, dense_stride(H, V), h, V, c0, tid, v16);
            if (delta) {
                load_mat_tile(s2, ws.vnew + item * (int64_t)kChunk * V, 0, len, c0, V, V, tid);
                load_mat_tile(s3, bw.dvn + item * (int64_t)kChunk * V, 0, len, c0, V, V, tid);
                load_tok_tile(s4, v, ci.t0, len, p.sv, h, V, c0, tid, v16);
            } else {
                load_tok_tile(s2, v, ci.t0, len, p.sv, h, V, c0, tid, v16);
            }
            __syncthreads();
            const int cn = min(kSl, V - c0);
            mm_abT<4>(dm, s1, kLd, s2, kLd, cn, tid);
            if (delta) mm_abT<4>(dt, s3, kLd, s4, kLd, cn, tid);
        }
        FOR_TILE(4) {
            const int i = i0 + r, j = j0 + 16 * s;
            const bool causal = i < len && j <= i;
            const float d = causal ? expf(sG[i] - sG[j]) : 0.f;
            sZ[i * kLd + j] = causal ? scale * dm[r][s] * d : 0.f;
            sR[i * kLd + j] = causal ? scale * dm[r][s] * sM[i * kLd + j] : 0.f;
            if (delta) sdT[i * kLd + j] = dt[r][s] * sB[j];
        }
    }
    __syncthreads();
    // gate terms of M: row sums minus column sums of R
    if (tid < kChunk) {
        float sum = 0.f;
        for (int j = 0; j < kChunk; ++j) sum += sR[tid * kLd + j];
        rowR[tid] = sum;
    } else if (tid < 2 * kChunk) {
        const int j = tid - kChunk;
        float sum = 0.f;
        for (int i = 0; i < kChunk; ++i) sum += sR[i * kLd + j];
        colR[j] = sum;
    }

    if (delta) {
        // dTb = -(dV' h^T) (diag(beta gamma) K)^T over the keys; dT = dTa + dTb
        float tb[4][4];
        acc_zero(tb);
        for (int k0 = 0; k0 < K; k0 += kSl) {
            __syncthreads();
            load_mat_tile(s1, bw.P2 + item * (int64_t)kChunk * K, 0, kChunk, k0, K, K, tid);
            load_tok_tile(s2, k, ci.t0, len, p.sk, h, K, k0, tid, v16);
            __syncthreads();
            mm_abT<4>(tb, s1, kLd, s2, kLd, min(kSl, K - k0), tid);
        }
        FOR_TILE(4) {
            const int i = i0 + r, j = j0 + 16 * s;
            sdT[i * kLd + j] = fmaf(-sB[j] * sGam[j], tb[r][s], sdT[i * kLd + j]);
        }
        __syncthreads();
        // X = dT T^T
        {
            float x[4][4];
            acc_zero(x);
            mm_abT<4>(x, sdT, kLd, sT, kLd, kChunk, tid);
            FOR_TILE(4) sX[(i0 + r) * kLd + j0 + 16 * s] = x[r][s];
        }
        __syncthreads();
        // dA = -strict_lower(T^T X);  S = diag(beta) dA * D  (into sR)
        {
            float y[4][4];
            acc_zero(y);
            mm_atb<4>(y, sT, kLd, sX, kLd, kChunk, tid);
            FOR_TILE(4) {
                const int i = i0 + r, j = j0 + 16 * s;
                const bool sl = j < i && i < len;
                const float yv = sl ? -y[r][s] : 0.f;
                sdT[i * kLd + j] = yv;
                sR[i * kLd + j] = sl ? sB[i] * yv * expf(sG[i] - sG[j]) : 0.f;
            }
        }
        __syncthreads();
        // dbeta from A: rowdot(dA, Kd); the gate terms of A: rows minus columns
        // of dA * A = diag(beta) dA * Kd
        if (tid < kChunk) {
            float sum = 0.f;
            for (int j = 0; j < kChunk; ++j) sum = fmaf(sdT[tid * kLd + j], sKd[tid * kLd + j], sum);
            rdA[tid] = sum;
        } else if (tid < 2 * kChunk) {
            const int j = tid - kChunk;
            float sum = 0.f;
            for (int i = 0; i < kChunk; ++i)
                sum = fmaf(sB[i] * sdT[i * kLd + j], sKd[i * kLd + j], sum);
            colRA[j] = sum;
        }
    }

    // key loop: dq, dk and the row sums r1 = rowdot(P1, Q), r2 = rowdot(dKb, K),
    // r3 = rowdot(P3, K)
    Tin *dq = static_cast<Tin *>(a.dq);
    Tin *dk = static_cast<Tin *>(a.dk);
    for (int k0 = 0; k0 < K; k0 += kSl) {
        __syncthreads();
        load_tok_tile(s1, q, ci.t0, len, p.sq, h, K, k0, tid, v16);
        load_tok_tile(s2, k, ci.t0, len, p.sk, h, K, k0, tid, v16);
        load_mat_tile(s3, bw.P1 + item * (int64_t)kChunk * K, 0, kChunk, k0, K, K, tid);
        load_mat_tile(s4, bw.P3 + item * (int64_t)kChunk * K, 0, kChunk, k0, K, K, tid);
        if (delta) load_mat_tile(s5, bw.P2 + item * (int64_t)kChunk * K, 0, kChunk, k0, K, K, tid);
        __syncthreads();
        const int kn = min(kSl, K - k0);
        if (delta) {  // dKb = -T^T P2
            float kb[4][4];
            acc_zero(kb);
            mm_atb<4>(kb, sT, kLd, s5, kLd, kChunk, tid);
            FOR_TILE(4) s6[(i0 + r) * kLd + j0 + 16 * s] = -kb[r][s];
            __syncthreads();
        }
        float xq[4][4], xk[4][4];
        acc_zero(xq);
        acc_zero(xk);
        mm_ab<4>(xq, sZ, kLd, s2, kLd, kChunk, tid);       // sum_j Z_ij k_j
        mm_atb<4>(xk, sZ, kLd, s1, kLd, kChunk, tid);      // sum_m Z_mi q_m
        if (delta) {
            mm_ab<4>(xk, sR, kLd, s2, kLd, kChunk, tid);   // sum_m S_im k_m
            mm_atb<4>(xk, sR, kLd, s2, kLd, kChunk, tid);  // sum_m S_mi k_m
        }
        FOR_TILE(4) {
            const int i = i0 + r, kk = j0 + 16 * s;
            if (i < len && kk < kn) {
                const float yq = fmaf(scale * sGam[i], s3[i * kLd + kk], xq[r][s]);
                float yk = fmaf(sLam[i], s4[i * kLd + kk], xk[r][s]);
                if (delta) yk = fmaf(sB[i] * sGam[i], s6[i * kLd + kk], yk);
                const int64_t o = ((ci.t0 + i) * H + h) * (int64_t)K + k0 + kk;
                stx(dq, o, yq);
                stx(dk, o, yk);
            }
        }
        if (tid < kChunk) {
            const int i = tid;
            float x1 = r1[i], x2 = r2[i], x3 = r3[i];
            for (int c = 0; c < kn; ++c) {
                x1 = fmaf(s3[i * kLd + c], s1[i * kLd + c], x1);
                if (delta) x2 = fmaf(s6[i * kLd + c], s2[i * kLd + c], x2);
                x3 = fmaf(s4[i * kLd + c], s2[i * kLd + c], x3);
            }
            r1[i] = x1;
            r2[i] = x2;
            r3[i] = x3;
        }
    }

    if (delta) {
        // value loop: dVb = T^T dV';  dv = diag(beta) dVb;  r4 = rowdot(dVb, V)
        Tin *dv = static_cast<Tin *>(a.dv);
        for (int c0 = 0; c0 < V; c0 += kSl) {
            __syncthreads();
            load_mat_tile(s3, bw.dvn + item * (int64_t)kChunk * V, 0, len, c0, V, V, tid);
            load_tok_tile(s4, v, ci.t0, len, p.sv, h, V, c0, tid, v16);
            __syncthreads();
            const int cn = min(kSl, V - c0);
            float vb[4][4];
            acc_zero(vb);
            mm_atb<4>(vb, sT, kLd, s3, kLd, kChunk, tid);
            FOR_TILE(4) {
                const int i = i0 + r, c = j0 + 16 * s;
                s6[i * kLd + c] = vb[r][s];
                if (i < len && c < cn)
                    stx(dv, ((ci.t0 + i) * H + h) * (int64_t)V + c0 + c, sB[i] * vb[r][s]);
            }
            __syncthreads();
            if (tid < kChunk) {
                float x = r4[tid];
                for (int cc = 0; cc < cn; ++cc) x = fmaf(s6[tid * kLd + cc], s4[tid * kLd + cc], x);
                r4[tid] = x;
            }
        }
    }
    __syncthreads();
    if (tid < kChunk) {
        const int i = tid;
        float dG = 0.f;
        if (i < len) {
            dG = scale * sGam[i] * r1[i] + (rowR[i] - colR[i]) - sLam[i] * r3[i];
            if (delta) {
                dG += sB[i] * rdA[i] - colRA[i] + sB[i] * sGam[i] * r2[i];
                a.dbeta[(ci.t0 + i) * H + h] = r4[i] + sGam[i] * r2[i] + rdA[i];
            }
        }
        sdG[i] = dG;
    }
    __syncthreads();
    if (tid == 0) {
        // the chunk's last token also carries the state terms: Gam <E, h> and
        // sum_j lam_j rowdot(P3, K)_j
        const int nks = (K + kSl - 1) / kSl;
        float eh = 0.f;
        for (int sl = 0; sl < nks; ++sl) eh += bw.ehp[item * nks + sl];
        float lam3 = 0.f;
        for (int j = 0; j < len; ++j) lam3 = fmaf(sLam[j], r3[j], lam3);
        sdG[len - 1] += fmaf(sGam[len - 1], eh, lam3);
        float run = 0.f;
        for (int i = len - 1; i >= 0; --i) {
            run += sdG[i];
            a.dg[(ci.t0 + i) * H + h] = run;
        }
    }
}

template <typename F>
cudaError_t set_smem_bwd(F *f, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(f),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename Tin>
cudaError_t launch_bwd(const Problem &p, const Workspace &ws, const BwdArgs &a, const BwdWs &bw,
                       cudaStream_t st, LaunchRecorder &rec) {
    const bool delta = p.beta != nullptr;
    const unsigned mc = (unsigned)ws.max_chunks, H = (unsigned)p.H;
    const int K = (int)p.K, V = (int)p.V;
    cudaError_t e;
    // gram
    {
        const size_t smem = sizeof(float) * (3 * kChunk * kLd + 2 * kChunk);
        if ((e = set_smem_bwd(k_bwd_gram<Tin>, smem)) != cudaSuccess) return e;
        if ((e = rec.begin(kKBwdGram)) != cudaSuccess) return e;
        k_bwd_gram<Tin><<<dim3(mc, H), kBT, smem, st>>>(p, ws, bw);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = rec.end()) != cudaSuccess) return e;
    }
    // reverse scan: serial, or segment pre-scan + ordered composition from the
    // last segment to the first + segment output pass
    {
        const int S = ws.n_segments;
        const int bv = V % 32 == 0 ? 32 : 16;
        const size_t smem = sizeof(float) * ((size_t)K * (bv + 1) + 3 * kChunk * kLd +
                                             2 * kChunk * (bv + 1) + 2 * kChunk);
        auto launch = [&](int mode) -> cudaError_t {
            const int ntiles = V / bv;
            const dim3 grid((unsigned)(p.N * (mode == 0 ? 1 : S) * ntiles), H);
            cudaError_t r;
            if (bv == 32) {
                if ((r = set_smem_bwd(k_bwd_dscan<Tin, 32>, smem)) != cudaSuccess) return r;
                k_bwd_dscan<Tin, 32><<<grid, kBT, smem, st>>>(p, ws, a, bw, mode);
            } else {
                if ((r = set_smem_bwd(k_bwd_dscan<Tin, 16>, smem)) != cudaSuccess) return r;
                k_bwd_dscan<Tin, 16><<<grid, kBT, smem, st>>>(p, ws, a, bw, mode);
            }
            return cudaGetLastError();
        };
        if (S <= 1) {
            if ((e = rec.begin(kKBwdScan)) != cudaSuccess) return e;
            if ((e = launch(0)) != cudaSuccess) return e;
            if ((e = rec.end()) != cudaSuccess) return e;
        } else {
            if ((e = rec.begin(kKBwdPre)) != cudaSuccess) return e;
            if ((e = launch(1)) != cudaSuccess) return e;
            if ((e = rec.end()) != cudaSuccess) return e;
            // the composition starts from dht and ends at dh0, with the
            // transposed forward maps in reversed slots
            Problem pr = p;
            pr.h0 = a.dht;
            pr.ht = a.dh0;
            Workspace wr = ws;
            if (delta) {
                if ((e = rec.begin(kKBwdMaps)) != cudaSuccess) return e;
                k_bwd_maps<<<(unsigned)(p.N * H * S), kBT, 0, st>>>(p, ws, bw.segMb);
                if ((e = cudaGetLastError()) != cudaSuccess) return e;
                if ((e = rec.end()) != cudaSuccess) return e;
                wr.segM = bw.segMb;
            }
            if ((e = rec.begin(delta ? kKCompose : kKComposeScalar)) != cudaSuccess) return e;
            if (!delta) e = compose_scalar(pr, wr, st);
            else if (compose_mt_supported(pr)) e = compose_mt(pr, wr, st);
            else e = simt_compose(pr, wr, bv, st);
            if (e != cudaSuccess) return e;
            if ((e = rec.end()) != cudaSuccess) return e;
            if ((e = rec.begin(kKBwdSegOut)) != cudaSuccess) return e;
            if ((e = launch(2)) != cudaSuccess) return e;
            if ((e = rec.end()) != cudaSuccess) return e;
        }
    }
    // L x K products
    {
        const size_t smem = sizeof(float) * (5 * kChunk * kLd + kBT);
        if ((e = set_smem_bwd(k_bwd_lk<Tin>, smem)) != cudaSuccess) return e;
        if ((e = rec.begin(kKBwdLk)) != cudaSuccess) return e;
        k_bwd_lk<Tin><<<dim3(mc, H, (unsigned)((K + kSl - 1) / kSl)), kBT, smem, st>>>(p, ws, a, bw);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = rec.end()) != cudaSuccess) return e;
    }
    // local gradients
    {
        const size_t smem = sizeof(float) * ((delta ? 13 : 9) * kChunk * kLd + 13 * kChunk);
        if ((e = set_smem_bwd(k_bwd_local<Tin>, smem)) != cudaSuccess) return e;
        if ((e = rec.begin(kKBwdLocal)) != cudaSuccess) return e;
        k_bwd_local<Tin><<<dim3(mc, H), kBT, smem, st>>>(p, ws, a, bw);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = rec.end()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t bwd_maps(const Problem &p, const Workspace &ws, float *segMb, cudaStream_t st) {
    k_bwd_maps<<<(unsigned)(p.N * p.H * ws.n_segments), kBT, 0, st>>>(p, ws, segMb);
    return cudaGetLastError();
}

cudaError_t simt_bwd(const Problem &p, const Workspace &ws, const BwdArgs &a, const BwdWs &bw,
                     cudaStream_t st, LaunchRecorder &rec) {
    if (p.dtype == GDR_BF16) return launch_bwd<__nv_bfloat16>(p, ws, a, bw, st, rec);
    if (p.dtype == GDR_F16) return launch_bwd<__half>(p, ws, a, bw, st, rec);
    return launch_bwd<float>(p, ws, a, bw, st, rec);
}

}  // namespace gdr
