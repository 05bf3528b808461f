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

// Rows [0, 64) x columns [c0, c0 + 64) of a token-major input [tokens][H][D]
// (rows beyond len and columns beyond D read as 0) into a 64 x 65 tile.
template <typename T>
__device__ __forceinline__ void load_tok_tile(float *dst, const T *src, int64_t t0, int len,
                                              int H, int h, int D, int c0, int tid) {
    for (int idx = tid; idx < kChunk * kSl; idx += kBT) {
        const int i = idx >> 6, c = idx & 63;
        float x = 0.f;
        if (i < len && c0 + c < D) x = ldx(src, ((t0 + i) * H + h) * (int64_t)D + c0 + c);
        dst[i * kLd + c] = x;
    }
}

// Rows [r0, r0 + 64) x columns [c0, c0 + 64) of a row-major FP32 matrix with
// `rows` rows and row stride `ld` (columns beyond `cols` read as 0).
__device__ __forceinline__ void load_mat_tile(float *dst, const float *src, int r0, int rows,
                                              int c0, int cols, int64_t ld, int tid) {
    for (int idx = tid; idx < kSl * kSl; idx += kBT) {
        const int i = idx >> 6, c = idx & 63;
        float x = 0.f;
        if (r0 + i < rows && c0 + c < cols) x = src[(int64_t)(r0 + i) * ld + c0 + c];
        dst[i * kLd + c] = x;
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
    float qk[16], kk[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) qk[r] = kk[r] = 0.f;
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    for (int c0 = 0; c0 < K; c0 += kSl) {
        __syncthreads();
        load_tok_tile(sQ, q, ci.t0, ci.len, H, h, K, c0, tid);
        load_tok_tile(sK, k, ci.t0, ci.len, H, h, K, c0, tid);
        __syncthreads();
        const int j = tid & 63;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int i = (tid >> 6) + 4 * r;
            float a = qk[r], b = kk[r];
            for (int c = 0; c < kSl; ++c) {
                a = fmaf(sQ[i * kLd + c], sK[j * kLd + c], a);
                b = fmaf(sK[i * kLd + c], sK[j * kLd + c], b);
            }
            qk[r] = a;
            kk[r] = b;
        }
    }
    float *Mg = bw.Mq + (gc * H + h) * (int64_t)kChunk * kChunk;
    float *Kdg = bw.Kd + (gc * H + h) * (int64_t)kChunk * kChunk;
    const int j = tid & 63;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const int i = (tid >> 6) + 4 * r;
        const bool in = i < ci.len;
        const float d = (in && j <= i) ? expf(sG[i] - sG[j]) : 0.f;
        Mg[i * kChunk + j] = (in && j <= i) ? qk[r] * d : 0.f;
        if (delta) {
            const float kd = (in && j < i) ? kk[r] * d : 0.f;
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
                float s = 0.f;
                for (int jj = m; jj < i; ++jj) s = fmaf(sA[i * kLd + jj], sQ[jj * kLd + m], s);
                x = -s;
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
// from last to first.  E is dL/d(state at the chunk's end).
template <typename Tin, int BV>
__global__ void __launch_bounds__(kBT) k_bwd_dscan(Problem p, Workspace ws, BwdArgs a,
                                                   BwdWs bw) {
    constexpr int LDE = BV + 1;
    constexpr int NR = kChunk * BV / kBT;  // (i, c) outputs per thread
    const int H = (int)p.H, K = (int)p.K, V = (int)p.V;
    const int ntiles = V / BV;
    const int64_t n = blockIdx.x / ntiles;
    const int tile = (int)(blockIdx.x % ntiles), col0 = tile * BV;
    const int h = blockIdx.y, tid = threadIdx.x;
    const bool delta = p.beta != nullptr;
    extern __shared__ float sm[];
    float *sE = sm;                       // [K][BV+1]
    float *sM = sE + K * LDE;             // [64][65]
    float *sDo = sM + kChunk * kLd;       // [64][BV+1]
    float *sDv = sDo + kChunk * LDE;      // [64][BV+1]
    float *sX = sDv + kChunk * LDE;       // [64][65] key slice of K / Q
    float *sY = sX + kChunk * kLd;        // [64][65] key slice of W
    float *sGam = sY + kChunk * kLd, *sLam = sGam + kChunk;

    const int64_t nh = n * H + h;
    for (int idx = tid; idx < K * BV; idx += kBT) {
        const int key = idx / BV, c = idx - key * BV;
        sE[key * LDE + c] = a.dht ? a.dht[state_off(p, nh, key, col0 + c)] : 0.f;
    }
    const int c_begin = ws.seq_chunk0[n];
    const int nc = ws.seq_chunk0[n + 1] - c_begin;
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *dout = static_cast<const Tin *>(a.dout);
    for (int cc = nc - 1; cc >= 0; --cc) {
        const int64_t gc = c_begin + cc;
        const ChunkInfo ci = chunk_info(ws, gc);
        const int64_t item = gc * H + h;
        __syncthreads();
        float *Eg = bw.dhend + item * (int64_t)K * V;
        for (int idx = tid; idx < K * BV; idx += kBT) {
            const int key = idx / BV, c = idx - key * BV;
            Eg[(int64_t)key * V + col0 + c] = sE[key * LDE + c];
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
        __syncthreads();
        // dV' = scale M^T dO + diag(lam) K E
        float acc[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[r] = 0.f;
        for (int k0 = 0; k0 < K; k0 += kSl) {
            __syncthreads();
            load_tok_tile(sX, k, ci.t0, ci.len, H, h, K, k0, tid);
            __syncthreads();
            const int kn = min(kSl, K - k0);
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const int idx = tid + r * kBT, i = idx / BV, c = idx - i * BV;
                float s = acc[r];
                for (int kk = 0; kk < kn; ++kk)
                    s = fmaf(sX[i * kLd + kk], sE[(k0 + kk) * LDE + c], s);
                acc[r] = s;
            }
        }
        const float gam_last = expf(ws.G[item * kChunk + ci.len - 1]);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const int idx = tid + r * kBT, i = idx / BV, c = idx - i * BV;
            float mt = 0.f;
            for (int j = i; j < ci.len; ++j) mt = fmaf(sM[j * kLd + i], sDo[j * LDE + c], mt);
            const float dvn = i < ci.len ? fmaf(p.scale, mt, sLam[i] * acc[r]) : 0.f;
            sDv[i * LDE + c] = dvn;
            if (i < ci.len) {
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
            load_tok_tile(sX, q, ci.t0, ci.len, H, h, K, k0, tid);
            if (delta)
                load_mat_tile(sY, ws.W + item * (int64_t)kChunk * K, 0, kChunk, k0, K, K, tid);
            __syncthreads();
            const int kn = min(kSl, K - k0);
            for (int idx = tid; idx < kn * BV; idx += kBT) {
                const int kk = idx / BV, c = idx - kk * BV;
                float s1 = 0.f, s2 = 0.f;
                for (int i = 0; i < ci.len; ++i) {
                    s1 = fmaf(sGam[i] * sX[i * kLd + kk], sDo[i * LDE + c], s1);
                    if (delta) s2 = fmaf(sY[i * kLd + kk], sDv[i * LDE + c], s2);
                }
                float *e = &sE[(k0 + kk) * LDE + c];
                *e = fmaf(gam_last, *e, fmaf(p.scale, s1, -s2));
            }
        }
    }
    __syncthreads();
    if (a.dh0) {
        for (int idx = tid; idx < K * BV; idx += kBT) {
            const int key = idx / BV, c = idx - key * BV;
            a.dh0[state_off(p, nh, key, col0 + c)] = sE[key * LDE + c];
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
    float p1[16], p2[16], p3[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) p1[r] = p2[r] = p3[r] = 0.f;
    float eh = 0.f;
    for (int c0 = 0; c0 < V; c0 += kSl) {
        __syncthreads();
        load_tok_tile(sDo, dout, ci.t0, ci.len, H, h, V, c0, tid);
        if (delta) {
            load_mat_tile(sDv, bw.dvn + item * (int64_t)kChunk * V, 0, ci.len, c0, V, V, tid);
            load_mat_tile(sVn, ws.vnew + item * (int64_t)kChunk * V, 0, ci.len, c0, V, V, tid);
        } else {
            load_tok_tile(sVn, v, ci.t0, ci.len, H, h, V, c0, tid);
        }
        load_mat_tile(sH, hg, k0, K, c0, V, V, tid);
        load_mat_tile(sE, eg, k0, K, c0, V, V, tid);
        __syncthreads();
        const int cn = min(kSl, V - c0);
        const int kk = tid & 63;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int i = (tid >> 6) + 4 * r;
            float s1 = p1[r], s2 = p2[r], s3 = p3[r];
            for (int c = 0; c < cn; ++c) {
                const float hv = sH[kk * kLd + c];
                s1 = fmaf(sDo[i * kLd + c], hv, s1);
                if (delta) s2 = fmaf(sDv[i * kLd + c], hv, s2);
                s3 = fmaf(sVn[i * kLd + c], sE[kk * kLd + c], s3);
            }
            p1[r] = s1;
            p2[r] = s2;
            p3[r] = s3;
        }
        // <E, h> over this key slice: thread tid owns key tid & 63 and a
        // quarter of the slice's columns
        {
            const int key = tid & 63, part = tid >> 6;
            for (int c = part; c < cn; c += 4) eh = fmaf(sE[key * kLd + c], sH[key * kLd + c], eh);
        }
    }
    const int kk = tid & 63;
    if (k0 + kk < K) {
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int i = (tid >> 6) + 4 * r;
            const int64_t o = (item * kChunk + i) * (int64_t)K + k0 + kk;
            bw.P1[o] = p1[r];
            if (delta) bw.P2[o] = p2[r];
            bw.P3[o] = p3[r];
        }
    }
    sRed[tid] = eh;
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int t = 0; t < kBT; ++t) s += sRed[t];
        bw.ehp[item * ((K + kSl - 1) / kSl) + ks] = s;
    }
}

// ---------------------------------------------------------------------------
// k_bwd_local: every local gradient of one (chunk, head).
template <typename Tin>
__global__ void __launch_bounds__(kBT) k_bwd_local(Problem p, Workspace ws, BwdArgs a,
                                                   BwdWs bw) {
    const int64_t gc = blockIdx.x;
    const int h = blockIdx.y;
    if (gc >= *ws.n_chunks) return;
    const ChunkInfo ci = chunk_info(ws, gc);
    const int H = (int)p.H, K = (int)p.K, V = (int)p.V, tid = threadIdx.x, len = ci.len;
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
    const int jj = tid & 63;

    // value loop: dMraw = dO V'^T; delta: dTa = dV' (diag(beta) V)^T
    float dm[16], dt[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) dm[r] = dt[r] = 0.f;
    for (int c0 = 0; c0 < V; c0 += kSl) {
        __syncthreads();
        load_tok_tile(s1, dout, ci.t0, len, H, h, V, c0, tid);
        if (delta) {
            load_mat_tile(s2, ws.vnew + item * (int64_t)kChunk * V, 0, len, c0, V, V, tid);
            load_mat_tile(s3, bw.dvn + item * (int64_t)kChunk * V, 0, len, c0, V, V, tid);
            load_tok_tile(s4, v, ci.t0, len, H, h, V, c0, tid);
        } else {
            load_tok_tile(s2, v, ci.t0, len, H, h, V, c0, tid);
        }
        __syncthreads();
        const int cn = min(kSl, V - c0);
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int i = (tid >> 6) + 4 * r;
            float x = dm[r], y = dt[r];
            for (int c = 0; c < cn; ++c) {
                x = fmaf(s1[i * kLd + c], s2[jj * kLd + c], x);
                if (delta) y = fmaf(s3[i * kLd + c], s4[jj * kLd + c], y);
            }
            dm[r] = x;
            dt[r] = y;
        }
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const int i = (tid >> 6) + 4 * r;
        const bool causal = i < len && jj <= i;
        const float d = causal ? expf(sG[i] - sG[jj]) : 0.f;
        const float z = causal ? scale * dm[r] * d : 0.f;
        sZ[i * kLd + jj] = z;
        sR[i * kLd + jj] = causal ? scale * dm[r] * sM[i * kLd + jj] : 0.f;
        if (delta) sdT[i * kLd + jj] = dt[r] * sB[jj];
    }
    __syncthreads();
    // gate terms of M: row sums minus column sums of R
    if (tid < kChunk) {
        float s = 0.f;
        for (int j = 0; j < kChunk; ++j) s += sR[tid * kLd + j];
        rowR[tid] = s;
    } else if (tid < 2 * kChunk) {
        const int j = tid - kChunk;
        float s = 0.f;
        for (int i = 0; i < kChunk; ++i) s += sR[i * kLd + j];
        colR[j] = s;
    }

    if (delta) {
        // dTb = -(dV' h^T) (diag(beta gamma) K)^T over the keys; dT = dTa + dTb
        float tb[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) tb[r] = 0.f;
        for (int k0 = 0; k0 < K; k0 += kSl) {
            __syncthreads();
            load_mat_tile(s1, bw.P2 + item * (int64_t)kChunk * K, 0, kChunk, k0, K, K, tid);
            load_tok_tile(s2, k, ci.t0, len, H, h, K, k0, tid);
            __syncthreads();
            const int kn = min(kSl, K - k0);
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int i = (tid >> 6) + 4 * r;
                float x = tb[r];
                for (int c = 0; c < kn; ++c) x = fmaf(s1[i * kLd + c], s2[jj * kLd + c], x);
                tb[r] = x;
            }
        }
        __syncthreads();
        const float bg = sB[jj] * sGam[jj];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int i = (tid >> 6) + 4 * r;
            sdT[i * kLd + jj] = fmaf(-bg, tb[r], sdT[i * kLd + jj]);
        }
        __syncthreads();
        // X = dT T^T  (T lower triangular: T_jm = 0 for m > j)
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int i = (tid >> 6) + 4 * r;
            float x = 0.f;
            for (int m = 0; m <= jj; ++m) x = fmaf(sdT[i * kLd + m], sT[jj * kLd + m], x);
            sX[i * kLd + jj] = x;
        }
        __syncthreads();
        // dA = -strict_lower(T^T X);  S = diag(beta) dA * D  (into sR)
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int i = (tid >> 6) + 4 * r;
            float y = 0.f;
            if (jj < i && i < len) {
                for (int m = i; m < kChunk; ++m) y = fmaf(sT[m * kLd + i], sX[m * kLd + jj], y);
                y = -y;
            }
            sdT[i * kLd + jj] = y;
            sR[i * kLd + jj] = (jj < i && i < len) ? sB[i] * y * expf(sG[i] - sG[jj]) : 0.f;
        }
        __syncthreads();
        // dbeta from A: rowdot(dA, Kd); the gate terms of A: rows minus columns
        // of dA * A = diag(beta) dA * Kd
        if (tid < kChunk) {
            float s = 0.f;
            for (int j = 0; j < kChunk; ++j) s = fmaf(sdT[tid * kLd + j], sKd[tid * kLd + j], s);
            rdA[tid] = s;
        } else if (tid < 2 * kChunk) {
            const int j = tid - kChunk;
            float s = 0.f;
            for (int i = 0; i < kChunk; ++i)
                s = fmaf(sB[i] * sdT[i * kLd + j], sKd[i * kLd + j], s);
            colRA[j] = s;
        }
    }

    // key loop: dq, dk and the row sums r1 = rowdot(P1, Q), r2 = rowdot(dKb, K),
    // r3 = rowdot(P3, K)
    Tin *dq = static_cast<Tin *>(a.dq);
    Tin *dk = static_cast<Tin *>(a.dk);
    for (int k0 = 0; k0 < K; k0 += kSl) {
        __syncthreads();
        load_tok_tile(s1, q, ci.t0, len, H, h, K, k0, tid);
        load_tok_tile(s2, k, ci.t0, len, H, h, K, k0, tid);
        load_mat_tile(s3, bw.P1 + item * (int64_t)kChunk * K, 0, kChunk, k0, K, K, tid);
        load_mat_tile(s4, bw.P3 + item * (int64_t)kChunk * K, 0, kChunk, k0, K, K, tid);
        if (delta) load_mat_tile(s5, bw.P2 + item * (int64_t)kChunk * K, 0, kChunk, k0, K, K, tid);
        __syncthreads();
        const int kn = min(kSl, K - k0);
        const int kk = tid & 63;
        // dKb = -T^T P2
        if (delta) {
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int i = (tid >> 6) + 4 * r;
                float x = 0.f;
                for (int m = i; m < len; ++m) x = fmaf(sT[m * kLd + i], s5[m * kLd + kk], x);
                s6[i * kLd + kk] = -x;
            }
            __syncthreads();
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int i = (tid >> 6) + 4 * r;
            if (i >= len || kk >= kn) continue;
            // dq_i = scale gamma_i P1_i + sum_{j <= i} Z_ij k_j
            float xq = 0.f;
            for (int j = 0; j <= i; ++j) xq = fmaf(sZ[i * kLd + j], s2[j * kLd + kk], xq);
            xq = fmaf(scale * sGam[i], s3[i * kLd + kk], xq);
            // dk_i = sum_{m >= i} Z_mi q_m + lam_i P3_i (+ beta_i gamma_i dKb_i
            //        + sum_{m < i} S_im k_m + sum_{m > i} S_mi k_m)
            float xk = 0.f;
            for (int m = i; m < len; ++m) xk = fmaf(sZ[m * kLd + i], s1[m * kLd + kk], xk);
            xk = fmaf(sLam[i], s4[i * kLd + kk], xk);
            if (delta) {
                xk = fmaf(sB[i] * sGam[i], s6[i * kLd + kk], xk);
                for (int m = 0; m < i; ++m) xk = fmaf(sR[i * kLd + m], s2[m * kLd + kk], xk);
                for (int m = i + 1; m < len; ++m) xk = fmaf(sR[m * kLd + i], s2[m * kLd + kk], xk);
            }
            const int64_t o = ((ci.t0 + i) * H + h) * (int64_t)K + k0 + kk;
            stx(dq, o, xq);
            stx(dk, o, xk);
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
            load_tok_tile(s4, v, ci.t0, len, H, h, V, c0, tid);
            __syncthreads();
            const int cn = min(kSl, V - c0);
            const int c = tid & 63;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int i = (tid >> 6) + 4 * r;
                float x = 0.f;
                for (int m = i; m < len; ++m) x = fmaf(sT[m * kLd + i], s3[m * kLd + c], x);
                s6[i * kLd + c] = x;
                if (i < len && c < cn)
                    stx(dv, ((ci.t0 + i) * H + h) * (int64_t)V + c0 + c, sB[i] * x);
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
        for (int s = 0; s < nks; ++s) eh += bw.ehp[item * nks + s];
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
    // reverse scan
    {
        const bool wide = V % 32 == 0;
        const int bv = wide ? 32 : 16;
        const size_t smem = sizeof(float) * ((size_t)K * (bv + 1) + 3 * kChunk * kLd +
                                             2 * kChunk * (bv + 1) + 2 * kChunk);
        const dim3 grid((unsigned)(p.N * (V / bv)), H);
        if ((e = rec.begin(kKBwdScan)) != cudaSuccess) return e;
        if (wide) {
            if ((e = set_smem_bwd(k_bwd_dscan<Tin, 32>, smem)) != cudaSuccess) return e;
            k_bwd_dscan<Tin, 32><<<grid, kBT, smem, st>>>(p, ws, a, bw);
        } else {
            if ((e = set_smem_bwd(k_bwd_dscan<Tin, 16>, smem)) != cudaSuccess) return e;
            k_bwd_dscan<Tin, 16><<<grid, kBT, smem, st>>>(p, ws, a, bw);
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = rec.end()) != cudaSuccess) return e;
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

cudaError_t simt_bwd(const Problem &p, const Workspace &ws, const BwdArgs &a, const BwdWs &bw,
                     cudaStream_t st, LaunchRecorder &rec) {
    if (p.dtype == GDR_BF16) return launch_bwd<__nv_bfloat16>(p, ws, a, bw, st, rec);
    if (p.dtype == GDR_F16) return launch_bwd<__half>(p, ws, a, bw, st, rec);
    return launch_bwd<float>(p, ws, a, bw, st, rec);
}

}  // namespace gdr
