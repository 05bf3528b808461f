// simt_path.cu -- CUDA-core FP32 path of the chunked gated-delta-rule forward
// pass.  Used for FP32 inputs (where the 1e-5 accuracy bound rules out
// BF16/TF32 tensor-core operands) and for any shape the tensor-core path does
// not cover.  BF16 inputs are widened to FP32 on load; all arithmetic and
// the state are FP32.
//
// Every output element is produced by one thread with a fixed, sequential
// accumulation order, so results do not depend on the value-tile width or on
// the grid: all launch plans give bit-identical results.
//
// Chunked form (project statement; the state scan of fla's
// chunk_gated_delta_rule_fwd_kernel_h_blockdim64, Kev PR #259 intro):
//   G = chunk-local inclusive cumsum of the log gate g
//   A_ij = beta_i e^{G_i - G_j} (k_i . k_j)  for i > j, else 0
//   T = (I + A)^-1;  W = T diag(beta e^G) K;  U = T diag(beta) V
//   v_new = U - W h;  h <- e^{G_last} h + K^T (v_new e^{G_last - G})
//   o = scale [(Q e^G) h + (Q K^T * e^{G_i - G_j}, j <= i) v_new]
// Segment split (cuLA PR #127 "Root cause and implementation"): per segment
// a local state c_s (scan from 0) and a K x K transition M_s (the same scan
// on identity columns with U = 0), then h_{s+1} = M_s h_s + c_s.
#include "gdr_internal.cuh"
#include "gdr_segments.cuh"
#include "simt_tile.cuh"

namespace gdr {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float ld_in(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_out(float *p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, int64_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}
__device__ __forceinline__ float ld_in(const __half *p, int64_t i) { return __half2float(p[i]); }
__device__ __forceinline__ void st_out(__half *p, int64_t i, float x) { p[i] = __float2half_rn(x); }

__device__ __forceinline__ void report(int32_t *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// A1: chunk indexing.  One block.  Builds the (sequence, first token, length,
// chunk-in-sequence) table for every 64-token chunk and the first global
// chunk of every sequence.  Malformed cu_seqlens (not non-decreasing, not
// starting at 0, not ending at T, or more chunks than the table holds) make
// the call compute nothing and set GDR_ERR_SEQLENS in the status word.
// Also writes the sequences in descending order of chunk count (a counting
// sort; counts above 127 share the top bucket, and the order inside a bucket
// is whatever the shared-memory atomics give: it only decides which CTA
// takes which chain) for the persistent tensor-core kernels, which take the
// longest chains first, and zeroes their chain counters.  Every pass is
// block-parallel: each thread owns a contiguous run of sequences, and the
// chunk offsets come from a block-wide scan.  Up to kSmemSeqs sequences the
// counts and offsets live in shared memory; beyond that in global memory.
constexpr int kSmemSeqs = 8192;
constexpr int kBuckets = kOrderBuckets;

__device__ __forceinline__ int chunk_bucket(int c) { return c < kBuckets - 1 ? c : kBuckets - 1; }

__global__ void __launch_bounds__(kThreads) k_chunk_table(const Problem p, int64_t N, int64_t T,
                                                          int64_t max_chunks,
                                                          int32_t *__restrict__ tab,
                                                          int32_t *__restrict__ seq_chunk0,
                                                          int32_t *__restrict__ n_chunks,
                                                          int32_t *__restrict__ seq_order,
                                                          int common_S, int32_t *status) {
    __shared__ int s_bad, s_longest;
    __shared__ int s_hist[kBuckets];
    __shared__ long long s_part[kThreads / 32];
    __shared__ int s_c0[kSmemSeqs + 1];
    const bool in_smem = N <= kSmemSeqs;
    int32_t *c0 = in_smem ? s_c0 : seq_chunk0;  // chunk counts, then prefix offsets
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();  // the first kernel of a call: launched in stream order, it waits for nothing
    for (int b = tid; b < kBuckets; b += kThreads) s_hist[b] = 0;
    if (tid < kNumCtr - 1) n_chunks[1 + tid] = 0;
    if (tid == 0) s_longest = 0;
    if (tid == 0) s_bad = (is_varlen_p(p) && (seq_bound(p, 0) != 0 || seq_bound(p, N) != T)) ? 1 : 0;
    __syncthreads();
    // this thread's run of sequences, their chunk counts and the histogram
    const int64_t per = (N + kThreads - 1) / kThreads;
    const int64_t lo = min(N, (int64_t)tid * per), hi = min(N, lo + per);
    long long local = 0;
    for (int64_t n = lo; n < hi; ++n) {
        const int64_t a = seq_start(p, n);
        const int64_t len = seq_end(p, n) - a;
        if (len < 0) s_bad = 1;
        const int64_t c = len < 0 ? 0 : (len + kChunk - 1) / kChunk;
        const int32_t cc = (int32_t)(c <= max_chunks ? c : max_chunks + 1);
        c0[n] = cc;
        local += cc;
        atomicAdd(&s_hist[chunk_bucket(cc)], 1);
        atomicMax(&s_longest, cc);
    }
    // block-wide exclusive scan of the runs' chunk totals
    long long incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) s_part[warp] = incl;
    __syncthreads();
    long long before = 0, total = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
        if (w < warp) before += s_part[w];
        total += s_part[w];
    }
    const bool bad = s_bad || total > max_chunks;
    if (!bad) {
        int32_t run = (int32_t)(before + incl - local);
        for (int64_t n = lo; n < hi; ++n) {
            const int32_t c = c0[n];
            c0[n] = run;
            run += c;
        }
        if (tid == 0) c0[N] = (int32_t)total;
    }
    if (tid == 0) {
        *n_chunks = bad ? 0 : (int32_t)total;
        // the common segment length (at least 1), or 0 for the own-length rule
        n_chunks[kCtrSegLen] =
            bad || !common_S ? 0 : max(1, (s_longest + common_S - 1) / common_S);
        if (bad) report(status, GDR_ERR_SEQLENS);
    }
    if (bad) {
        for (int64_t n = tid; n <= N; n += kThreads) seq_chunk0[n] = 0;
        for (int64_t n = tid; n < N; n += kThreads) seq_order[n] = (int32_t)n;
        return;
    }
    // bucket b starts after every longer bucket: a reverse exclusive scan of
    // the histogram by warp 0, four buckets a lane from the top
    if (warp == 0) {
        int h4[4], sum = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            h4[u] = s_hist[kBuckets - 1 - (4 * lane + u)];
            sum += h4[u];
        }
        int inc = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += y;
        }
        int run = inc - sum;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            s_hist[kBuckets - 1 - (4 * lane + u)] = run;
            run += h4[u];
        }
    }
    __syncthreads();
    for (int64_t n = lo; n < hi; ++n)
        seq_order[atomicAdd(&s_hist[chunk_bucket(c0[n + 1] - c0[n])], 1)] = (int32_t)n;
    if (in_smem)
        for (int64_t n = tid; n <= N; n += kThreads) seq_chunk0[n] = c0[n];
    // one warp per sequence, its lanes over the sequence's chunks
    const int nwarps = kThreads >> 5;
    for (int64_t n = warp; n < N; n += nwarps) {
        const int64_t a = seq_start(p, n);
        const int64_t len = seq_end(p, n) - a;
        const int32_t first = c0[n];
        const int32_t cnt = c0[n + 1] - first;
        for (int32_t c = lane; c < cnt; c += 32) {
            const int64_t rem = len - (int64_t)c * kChunk;
            *reinterpret_cast<int4 *>(tab + 4 * (int64_t)(first + c)) =
                make_int4((int32_t)n, (int32_t)(a + (int64_t)c * kChunk),
                          (int32_t)(rem < kChunk ? rem : kChunk), c);
        }
    }
}

// A2-A5: per (chunk, head) gate cumsum; in delta mode also the Gram matrix
// A, the unit-lower-triangular inverse T = (I + A)^-1 and the WY factors W, U.
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
k_prep(Problem p, Workspace ws) {
    const int64_t chunk = blockIdx.x;
    const int h = blockIdx.y;
    if (chunk >= *ws.n_chunks) return;
    const int4 e = reinterpret_cast<const int4 *>(ws.chunk_tab)[chunk];
    const int64_t t0 = e.y;
    const int len = e.z;
    const int H = (int)p.H, K = (int)p.K, V = (int)p.V;
    const int tid = threadIdx.x;
    const int i0 = 4 * (tid >> 4), j0 = tid & 15;
    const int Kp = (K + 63) & ~63;  // keys padded with zero columns to whole 64-column tiles
    const int ldk = Kp + 1;

    extern __shared__ float sm[];
    float *sG = sm;
    float *sB = sG + kChunk;
    float *sBG = sB + kChunk;
    float *sK = sBG + kChunk;          // [64][Kp+1]
    float *sA = sK + kChunk * ldk;     // [64][65]
    float *sT = sA + kChunk * 65;      // [64][65]
    float *sV = sT + kChunk * 65;      // [64][65] value block

    const bool delta = p.beta != nullptr;
    if (tid < kChunk) {
        sG[tid] = tid < len ? p.g[(t0 + tid) * H + h] : 0.f;
        sB[tid] = (delta && tid < len) ? p.beta[(t0 + tid) * H + h] : 0.f;
    }
    __syncthreads();
    if (tid == 0) {  // fixed left-to-right order
        float acc = 0.f;
        for (int i = 0; i < kChunk; ++i) {
            acc += sG[i];
            sG[i] = acc;
        }
    }
    __syncthreads();
    if (tid < kChunk) ws.G[(chunk * H + h) * kChunk + tid] = sG[tid];
    if (!delta) return;
    if (tid < kChunk) sBG[tid] = sB[tid] * expf(sG[tid]);

    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    const bool vin = rows_aligned16(p.k, p.sk, sizeof(Tin)) && rows_aligned16(p.v, p.sv, sizeof(Tin));
    constexpr int E = 16 / (int)sizeof(Tin);  // elements per 16-byte piece
    if (vin) {
        const int pr = Kp / E;
        for (int idx = tid; idx < kChunk * pr; idx += kThreads) {
            const int i = idx / pr, c = (idx - i * pr) * E;
            float x[E];
            if (i < len && c < K) {
                const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(
                    k + tok_at(p.sk, t0 + i, h) + c));
                unpack16(raw, k, x);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) x[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < E; ++e) sK[i * ldk + c + e] = x[e];
        }
    } else {
        for (int idx = tid; idx < kChunk * Kp; idx += kThreads) {
            const int i = idx / Kp, c = idx - i * Kp;
            sK[i * ldk + c] =
                (i < len && c < K) ? ld_in(k, tok_at(p.sk, t0 + i, h) + c) : 0.f;
        }
    }
    __syncthreads();
    // A3: A_ij = beta_i e^{G_i - G_j} (k_i . k_j), strictly lower (the mask is
    // applied before exp, so e^{G_i - G_j} is only formed for i > j).
    {
        float d[4][4];
        acc_zero(d);
        mm_abT<4>(d, sK, ldk, sK, ldk, Kp, tid);
        FOR_TILE(4) {
            const int i = i0 + r, jj = j0 + 16 * s;
            sA[i * 65 + jj] = (jj < i && i < len) ? sB[i] * expf(sG[i] - sG[jj]) * d[r][s] : 0.f;
        }
    }
    __syncthreads();
    // A4: T = (I + A)^-1.  Column m solves (I + A) x = e_m by forward
    // substitution; columns are independent, one thread each.
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
                for (int jj = m; jj < i; ++jj) sum = fmaf(sA[i * 65 + jj], sT[jj * 65 + m], sum);
                x = -sum;
            }
            sT[i * 65 + m] = x;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < kChunk * Kp; idx += kThreads) {
        const int i = idx / Kp, c = idx - i * Kp;
        sK[i * ldk + c] *= sBG[i];
    }
    __syncthreads();
    // A5: W = T diag(beta e^G) K, in 64-column blocks (T is zero above its
    // diagonal, so the full product is the triangular one)
    float *Wg = ws.W + (chunk * H + h) * (int64_t)kChunk * K;
    for (int kb = 0; kb < Kp; kb += 64) {
        float w[4][4];
        acc_zero(w);
        mm_ab<4>(w, sT, 65, sK + kb, ldk, kChunk, tid);
        FOR_TILE(4) {
            const int i = i0 + r, c = kb + j0 + 16 * s;
            if (c < K) Wg[(int64_t)i * K + c] = w[r][s];
        }
    }
    // A5: U = T diag(beta) V, in 64-column blocks
    float *Ug = ws.U + (chunk * H + h) * (int64_t)kChunk * V;
    for (int v0 = 0; v0 < V; v0 += 64) {
        __syncthreads();
        if (vin) {
            for (int idx = tid; idx < kChunk * (64 / E); idx += kThreads) {
                const int i = idx / (64 / E), c = (idx - i * (64 / E)) * E;
                float x[E];
                if (i < len && v0 + c < V) {
                    const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(
                        v + tok_at(p.sv, t0 + i, h) + v0 + c));
                    unpack16(raw, v, x);
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) x[e] = 0.f;
                }
#pragma unroll
                for (int e = 0; e < E; ++e) sV[i * 65 + c + e] = sB[i] * x[e];
            }
        } else {
            for (int idx = tid; idx < kChunk * 64; idx += kThreads) {
                const int i = idx >> 6, c = idx & 63;
                sV[i * 65 + c] = (i < len && v0 + c < V)
                    ? sB[i] * ld_in(v, tok_at(p.sv, t0 + i, h) + v0 + c) : 0.f;
            }
        }
        __syncthreads();
        float u[4][4];
        acc_zero(u);
        mm_ab<4>(u, sT, 65, sV, 65, kChunk, tid);
        FOR_TILE(4) {
            const int i = i0 + r, c = v0 + j0 + 16 * s;
            if (c < V) Ug[(int64_t)i * V + c] = u[r][s];
        }
    }
}

// A6 / A8 / A10: the serial state scan over the chunks of one (sequence,
// segment, head, column tile).  mode 0: whole sequence from h0, writes ht;
// mode 1: segment pre-scan from zero (value columns -> c_s) or identity
// (transition columns, U = 0 -> M_s); mode 2: segment output pass from the
// composed segment state.  Modes 0 and 2 store h_pre and v_new for the
// output kernel.
template <typename Tin, int BV>
__global__ void __launch_bounds__(kThreads)
k_scan(Problem p, Workspace ws, int mode) {
    const int H = (int)p.H, K = (int)p.K, V = (int)p.V;
    const int S = mode == 0 ? 1 : ws.n_segments;
    const bool delta = p.beta != nullptr;
    const int n_vtiles = V / BV;
    const int ntiles = (mode == 1 && delta) ? (V + K) / BV : n_vtiles;
    int64_t bid = blockIdx.x;
    const int tile = (int)(bid % ntiles);
    bid /= ntiles;
    const int s = (int)(bid % S);
    const int64_t n = bid / S;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;

    const int c_begin = ws.seq_chunk0[n];
    const int nc = ws.seq_chunk0[n + 1] - c_begin;
    int s0 = 0, s1 = nc;
    if (mode != 0) {
        const int per = (nc + S - 1) / S;
        s0 = s * per;
        s1 = min(nc, s0 + per);
        if (s0 >= s1) return;
    }
    const bool trans = tile >= n_vtiles;
    const int col0 = trans ? (tile - n_vtiles) * BV : tile * BV;
    constexpr int NS = BV / 16;
    const int i0 = 4 * (tid >> 4), j0 = tid & 15;
    const int Kp = (K + 63) & ~63;  // keys padded with zeros to whole 64-row tiles
    const int ldk = Kp + 1;
    constexpr int ldh = BV + 1;

    extern __shared__ float sm[];
    float *hs = sm;                   // [Kp][BV+1] state tile (rows >= K stay 0)
    float *sK = hs + Kp * ldh;        // [64][Kp+1]
    float *sW = sK + kChunk * ldk;    // [64][Kp+1] (delta)
    float *vn = sW + (delta ? kChunk * ldk : 0);  // [64][BV+1]
    float *sG = vn + kChunk * ldh;    // [64]

    const int64_t seg_base = ((n * H + h) * (int64_t)S + s);
    for (int idx = tid; idx < Kp * BV; idx += kThreads) {
        const int key = idx / BV, c = idx - key * BV;
        float x = 0.f;
        if (key >= K) {
            x = 0.f;
        } else if (mode == 0) {
            if (p.h0) x = p.h0[state_off(p, n * H + h, key, col0 + c)];
        } else if (mode == 2) {
            x = ws.segH[(seg_base * K + key) * V + col0 + c];
        } else if (trans) {
            x = (key == col0 + c) ? 1.f : 0.f;
        }
        hs[key * ldh + c] = x;
    }
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    const bool vk = rows_aligned16(p.k, p.sk, sizeof(Tin));
    float dprod = 1.f;

    for (int cc = s0; cc < s1; ++cc) {
        const int64_t gc = c_begin + cc;
        const int4 e = reinterpret_cast<const int4 *>(ws.chunk_tab)[gc];
        const int64_t t0 = e.y;
        const int len = e.z;
        __syncthreads();
        if (tid < kChunk) sG[tid] = ws.G[(gc * H + h) * kChunk + tid];
        if (vk) {  // 16-byte pieces (K is a multiple of 16)
            constexpr int E = 16 / (int)sizeof(Tin);
            const int pr = Kp / E;
            for (int idx = tid; idx < kChunk * pr; idx += kThreads) {
                const int i = idx / pr, c = (idx - i * pr) * E;
                float x[E];
                if (i < len && c < K) {
                    const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(
                        k + tok_at(p.sk, t0 + i, h) + c));
                    unpack16(raw, k, x);
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) x[e] = 0.f;
                }
#pragma unroll
                for (int e = 0; e < E; ++e) sK[i * ldk + c + e] = x[e];
            }
        } else {
            for (int idx = tid; idx < kChunk * Kp; idx += kThreads) {
                const int i = idx / Kp, c = idx - i * Kp;
                sK[i * ldk + c] =
                    (i < len && c < K) ? ld_in(k, tok_at(p.sk, t0 + i, h) + c) : 0.f;
            }
        }
        if (delta) {  // W rows: float4 pieces of the workspace
            const float *Wg = ws.W + (gc * H + h) * (int64_t)kChunk * K;
            for (int idx = tid; idx < kChunk * (Kp / 4); idx += kThreads) {
                const int i = idx / (Kp / 4), c = (idx - i * (Kp / 4)) * 4;
                float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
                if (c < K) w = __ldg(reinterpret_cast<const float4 *>(Wg + (int64_t)i * K + c));
                float *d = sW + i * ldk + c;
                d[0] = w.x;
                d[1] = w.y;
                d[2] = w.z;
                d[3] = w.w;
            }
        }
        if (mode != 1) {
            float *hp = ws.hpre + (gc * H + h) * (int64_t)K * V;
            for (int idx = tid; idx < K * BV; idx += kThreads) {
                const int key = idx / BV, c = idx - key * BV;
                hp[(int64_t)key * V + col0 + c] = hs[key * ldh + c];
            }
        }
        __syncthreads();
        const float gl = sG[len - 1];
        const float gam = expf(gl);
        // v_new = U - W h (delta) or V (beta-free), then scaled by e^{G_last - G}
        {
            float acc[4][NS];
            acc_zero(acc);
            if (delta) mm_ab<NS>(acc, sW, ldk, hs, ldh, Kp, tid);
            FOR_TILE(NS) {
                const int i = i0 + r, c = j0 + 16 * s;
                float x = 0.f;
                if (i < len) {
                    if (delta) {
                        const float u = trans ? 0.f
                            : ws.U[((gc * H + h) * kChunk + i) * (int64_t)V + col0 + c];
                        x = u - acc[r][s];
                        if (mode != 1)
                            ws.vnew[((gc * H + h) * kChunk + i) * (int64_t)V + col0 + c] = x;
                    } else {
                        x = ld_in(v, tok_at(p.sv, t0 + i, h) + col0 + c);
                    }
                    x *= expf(gl - sG[i]);
                }
                vn[i * ldh + c] = x;
            }
        }
        __syncthreads();
        // h <- e^{G_last} h + K^T (v_new e^{G_last - G}), in 64-key blocks
        for (int kb = 0; kb < Kp; kb += 64) {
            float acc[4][NS];
            acc_zero(acc);
            mm_atb<NS>(acc, sK + kb, ldk, vn, ldh, len, tid);
            FOR_TILE(NS) {
                const int key = kb + i0 + r, c = j0 + 16 * s;
                if (key < K) hs[key * ldh + c] = fmaf(gam, hs[key * ldh + c], acc[r][s]);
            }
        }
        dprod *= gam;
    }
    __syncthreads();
    if (mode == 0) {
        if (p.ht) {
            for (int idx = tid; idx < K * BV; idx += kThreads) {
                const int key = idx / BV, c = idx - key * BV;
                p.ht[state_off(p, n * H + h, key, col0 + c)] = hs[key * ldh + c];
            }
        }
    } else if (mode == 1) {
        for (int idx = tid; idx < K * BV; idx += kThreads) {
            const int key = idx / BV, c = idx - key * BV;
            if (trans)  // stored transposed: row m of M^T is column m of M
                ws.segM[(seg_base * K + col0 + c) * K + key] = hs[key * ldh + c];
            else
                ws.segC[(seg_base * K + key) * V + col0 + c] = hs[key * ldh + c];
        }
        if (!delta && tile == 0 && tid == 0) ws.segD[seg_base] = dprod;
    }
}

// A9: ordered composition over the segments of one (sequence, head, value
// tile): records each segment's initial state and h_{s+1} = M_s h_s + c_s
// (beta-free: d_s h_s + c_s); the last state is ht.  M_s is stored
// transposed.  Used for the beta-free mode and for K > 128 (the delta rule
// with K <= 128 uses k_compose_mt in compose.cu).
template <int BV>
__global__ void __launch_bounds__(kThreads)
k_compose(Problem p, Workspace ws) {
    const int H = (int)p.H, K = (int)p.K, V = (int)p.V;
    const int S = ws.n_segments;
    const int n_vtiles = V / BV;
    const int tile = blockIdx.x % n_vtiles;
    const int64_t n = blockIdx.x / n_vtiles;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int col0 = tile * BV;
    const bool delta = p.beta != nullptr;
    constexpr int ldh = BV + 1;
    extern __shared__ float sm[];
    float *hs = sm;
    float *hn = sm + K * ldh;

    const int nc = ws.seq_chunk0[n + 1] - ws.seq_chunk0[n];
    const int per = (nc + S - 1) / S;
    const int nseg = per ? (nc + per - 1) / per : 0;
    for (int idx = tid; idx < K * BV; idx += kThreads) {
        const int key = idx / BV, c = idx - key * BV;
        hs[key * ldh + c] = p.h0 ? p.h0[state_off(p, n * H + h, key, col0 + c)] : 0.f;
    }
    __syncthreads();
    for (int s = 0; s < nseg; ++s) {
        const int64_t seg_base = ((n * H + h) * (int64_t)S + s);
        const float *M = ws.segM + seg_base * K * K;
        const float *C = ws.segC + seg_base * K * V;
        const float d = delta ? 0.f : ws.segD[seg_base];
        for (int idx = tid; idx < K * BV; idx += kThreads) {
            const int key = idx / BV, c = idx - key * BV;
            ws.segH[(seg_base * K + key) * V + col0 + c] = hs[key * ldh + c];
            float acc;
            if (delta) {
                acc = 0.f;
                for (int m = 0; m < K; ++m) acc = fmaf(M[(int64_t)m * K + key], hs[m * ldh + c], acc);
                acc += C[(int64_t)key * V + col0 + c];
            } else {
                acc = fmaf(d, hs[key * ldh + c], C[(int64_t)key * V + col0 + c]);
            }
            hn[key * ldh + c] = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < K * BV; idx += kThreads) {
            const int key = idx / BV, c = idx - key * BV;
            hs[key * ldh + c] = hn[key * ldh + c];
        }
        __syncthreads();
    }
    if (p.ht) {
        for (int idx = tid; idx < K * BV; idx += kThreads) {
            const int key = idx / BV, c = idx - key * BV;
            p.ht[state_off(p, n * H + h, key, col0 + c)] = hs[key * ldh + c];
        }
    }
}

// A7: o = scale [(Q e^G) h_pre + (Q K^T * e^{G_i - G_j}, j <= i) v_new]
// per (chunk, head, value block).  The causal mask includes the diagonal:
// o_t reads the state after token t's own write.
template <typename Tin, int BVO>
__global__ void __launch_bounds__(kThreads)
k_output(Problem p, Workspace ws) {
    constexpr int NS = BVO / 16;
    constexpr int ldo = BVO + 1;
    const int64_t chunk = blockIdx.x;
    const int h = blockIdx.y;
    if (chunk >= *ws.n_chunks) return;
    const int4 e = reinterpret_cast<const int4 *>(ws.chunk_tab)[chunk];
    const int64_t t0 = e.y;
    const int len = e.z;
    const int H = (int)p.H, K = (int)p.K, V = (int)p.V;
    const int col0 = blockIdx.z * BVO;
    const int tid = threadIdx.x;
    const int i0 = 4 * (tid >> 4), j0 = tid & 15;
    const int Kp = (K + 63) & ~63;  // keys padded with zeros to whole 64-column tiles
    const int ldk = Kp + 1;
    const bool delta = p.beta != nullptr;

    extern __shared__ float sm[];
    float *sQ = sm;                  // [64][Kp+1]
    float *sK = sQ + kChunk * ldk;   // [64][Kp+1]
    float *sP = sK + kChunk * ldk;   // [64][65]
    float *sHp = sP + kChunk * 65;   // [Kp][BVO+1]
    float *sVn = sHp + Kp * ldo;     // [64][BVO+1]
    float *sG = sVn + kChunk * ldo;

    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    if (tid < kChunk) sG[tid] = ws.G[(chunk * H + h) * kChunk + tid];
    const bool vin = rows_aligned16(p.q, p.sq, sizeof(Tin)) && rows_aligned16(p.k, p.sk, sizeof(Tin));
    if (vin) {  // 16-byte pieces (K is a multiple of 16)
        constexpr int E = 16 / (int)sizeof(Tin);
        const int pr = Kp / E;
        for (int idx = tid; idx < kChunk * pr; idx += kThreads) {
            const int i = idx / pr, c = (idx - i * pr) * E;
            float xq[E], xk[E];
            if (i < len && c < K) {
                unpack16(__ldg(reinterpret_cast<const uint4 *>(q + tok_at(p.sq, t0 + i, h) + c)),
                         q, xq);
                unpack16(__ldg(reinterpret_cast<const uint4 *>(k + tok_at(p.sk, t0 + i, h) + c)),
                         k, xk);
            } else {
#pragma unroll
                for (int e2 = 0; e2 < E; ++e2) xq[e2] = xk[e2] = 0.f;
            }
#pragma unroll
            for (int e2 = 0; e2 < E; ++e2) {
                sQ[i * ldk + c + e2] = xq[e2];
                sK[i * ldk + c + e2] = xk[e2];
            }
        }
    } else {
        for (int idx = tid; idx < kChunk * Kp; idx += kThreads) {
            const int i = idx / Kp, c = idx - i * Kp;
            const bool in = i < len && c < K;
            sQ[i * ldk + c] = in ? ld_in(q, tok_at(p.sq, t0 + i, h) + c) : 0.f;
            sK[i * ldk + c] = in ? ld_in(k, tok_at(p.sk, t0 + i, h) + c) : 0.f;
        }
    }
    const float *hp = ws.hpre + (chunk * H + h) * (int64_t)K * V;
    for (int idx = tid; idx < Kp * BVO; idx += kThreads) {
        const int key = idx / BVO, c = idx - key * BVO;
        sHp[key * ldo + c] = key < K ? hp[(int64_t)key * V + col0 + c] : 0.f;
    }
    for (int idx = tid; idx < kChunk * BVO; idx += kThreads) {
        const int i = idx / BVO, c = idx - i * BVO;
        float x = 0.f;
        if (i < len) {
            x = delta ? ws.vnew[((chunk * H + h) * kChunk + i) * (int64_t)V + col0 + c]
                      : ld_in(v, tok_at(p.sv, t0 + i, h) + col0 + c);
        }
        sVn[i * ldo + c] = x;
    }
    __syncthreads();
    {  // P = Q K^T * e^{G_i - G_j}, causal with the diagonal
        float d[4][4];
        acc_zero(d);
        mm_abT<4>(d, sQ, ldk, sK, ldk, Kp, tid);
        FOR_TILE(4) {
            const int i = i0 + r, jj = j0 + 16 * s;
            sP[i * 65 + jj] = (jj <= i && i < len) ? d[r][s] * expf(sG[i] - sG[jj]) : 0.f;
        }
    }
    __syncthreads();
    Tin *o = static_cast<Tin *>(p.o);
    float a1[4][NS], a2[4][NS];
    acc_zero(a1);
    acc_zero(a2);
    mm_ab<NS>(a1, sQ, ldk, sHp, ldo, Kp, tid);
    mm_ab<NS>(a2, sP, 65, sVn, ldo, kChunk, tid);
    FOR_TILE(NS) {
        const int i = i0 + r, c = j0 + 16 * s;
        if (i < len) {
            const float y = p.scale * fmaf(expf(sG[i]), a1[r][s], a2[r][s]);
            st_out(o, tok_at(p.so, t0 + i, h) + col0 + c, y);
        }
    }
}

template <typename F>
cudaError_t set_smem(F *f, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(f),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t simt_chunk_table(const Problem &p, const Workspace &ws, bool common,
                             cudaStream_t st) {
    k_chunk_table<<<1, kThreads, 0, st>>>(p, p.N, p.T, ws.max_chunks, ws.chunk_tab,
                                          ws.seq_chunk0, ws.n_chunks, ws.seq_order,
                                          common ? ws.n_segments : 0, p.status);
    return cudaGetLastError();
}

cudaError_t simt_prep(const Problem &p, const Workspace &ws, cudaStream_t st) {
    if (ws.max_chunks == 0) return cudaSuccess;
    const int Kp = ((int)p.K + 63) & ~63;
    const size_t smem = sizeof(float) * (3 * kChunk + kChunk * (Kp + 1) + 3 * kChunk * 65);
    dim3 grid((unsigned)ws.max_chunks, (unsigned)p.H);
    cudaError_t err;
    if (p.dtype == GDR_BF16) {
        if ((err = set_smem(k_prep<__nv_bfloat16>, smem)) != cudaSuccess) return err;
        k_prep<__nv_bfloat16><<<grid, kThreads, smem, st>>>(p, ws);
    } else if (p.dtype == GDR_F16) {
        if ((err = set_smem(k_prep<__half>, smem)) != cudaSuccess) return err;
        k_prep<__half><<<grid, kThreads, smem, st>>>(p, ws);
    } else {
        if ((err = set_smem(k_prep<float>, smem)) != cudaSuccess) return err;
        k_prep<float><<<grid, kThreads, smem, st>>>(p, ws);
    }
    return cudaGetLastError();
}

template <typename Tin, int BV>
static cudaError_t launch_scan(const Problem &p, const Workspace &ws, int mode,
                               cudaStream_t st) {
    const int K = (int)p.K, V = (int)p.V;
    const bool delta = p.beta != nullptr;
    const int S = mode == 0 ? 1 : ws.n_segments;
    const int ntiles = (mode == 1 && delta) ? (V + K) / BV : V / BV;
    const int Kp = (K + 63) & ~63;
    const size_t smem = sizeof(float) *
        ((size_t)Kp * (BV + 1) + (size_t)kChunk * (Kp + 1) * (delta ? 2 : 1) +
         (size_t)kChunk * (BV + 1) + kChunk);
    cudaError_t err = set_smem(k_scan<Tin, BV>, smem);
    if (err != cudaSuccess) return err;
    dim3 grid((unsigned)((int64_t)ntiles * p.N * S), (unsigned)p.H);
    k_scan<Tin, BV><<<grid, kThreads, smem, st>>>(p, ws, mode);
    return cudaGetLastError();
}

cudaError_t simt_scan(const Problem &p, const Workspace &ws, int mode, int bv,
                      cudaStream_t st) {
    if (p.dtype == GDR_BF16) {
        switch (bv) {
        case 16: return launch_scan<__nv_bfloat16, 16>(p, ws, mode, st);
        case 32: return launch_scan<__nv_bfloat16, 32>(p, ws, mode, st);
        case 64: return launch_scan<__nv_bfloat16, 64>(p, ws, mode, st);
        }
    } else if (p.dtype == GDR_F16) {
        switch (bv) {
        case 16: return launch_scan<__half, 16>(p, ws, mode, st);
        case 32: return launch_scan<__half, 32>(p, ws, mode, st);
        case 64: return launch_scan<__half, 64>(p, ws, mode, st);
        }
    } else {
        switch (bv) {
        case 16: return launch_scan<float, 16>(p, ws, mode, st);
        case 32: return launch_scan<float, 32>(p, ws, mode, st);
        case 64: return launch_scan<float, 64>(p, ws, mode, st);
        }
    }
    return cudaErrorInvalidValue;
}

template <int BV>
static cudaError_t launch_compose(const Problem &p, const Workspace &ws, cudaStream_t st) {
    const size_t smem = sizeof(float) * 2 * (size_t)p.K * (BV + 1);
    cudaError_t err = set_smem(k_compose<BV>, smem);
    if (err != cudaSuccess) return err;
    dim3 grid((unsigned)((p.V / BV) * p.N), (unsigned)p.H);
    k_compose<BV><<<grid, kThreads, smem, st>>>(p, ws);
    return cudaGetLastError();
}

cudaError_t simt_compose(const Problem &p, const Workspace &ws, int bv, cudaStream_t st) {
    switch (bv) {
    case 16: return launch_compose<16>(p, ws, st);
    case 32: return launch_compose<32>(p, ws, st);
    case 64: return launch_compose<64>(p, ws, st);
    }
    return cudaErrorInvalidValue;
}

template <typename Tin, int BVO>
static cudaError_t launch_output(const Problem &p, const Workspace &ws, cudaStream_t st) {
    const int Kp = ((int)p.K + 63) & ~63;
    const size_t smem = sizeof(float) *
        (2 * (size_t)kChunk * (Kp + 1) + kChunk * 65 + (size_t)Kp * (BVO + 1) +
         (size_t)kChunk * (BVO + 1) + kChunk);
    cudaError_t err = set_smem(k_output<Tin, BVO>, smem);
    if (err != cudaSuccess) return err;
    dim3 grid((unsigned)ws.max_chunks, (unsigned)p.H, (unsigned)(p.V / BVO));
    k_output<Tin, BVO><<<grid, kThreads, smem, st>>>(p, ws);
    return cudaGetLastError();
}

template <typename Tin>
static cudaError_t output_for(const Problem &p, const Workspace &ws, cudaStream_t st) {
    int bvo = p.K <= 128 ? 64 : 32;
    while (p.V % bvo) bvo >>= 1;
    if (bvo == 64) return launch_output<Tin, 64>(p, ws, st);
    if (bvo == 32) return launch_output<Tin, 32>(p, ws, st);
    return launch_output<Tin, 16>(p, ws, st);
}

cudaError_t simt_output(const Problem &p, const Workspace &ws, cudaStream_t st) {
    if (ws.max_chunks == 0) return cudaSuccess;
    if (p.dtype == GDR_BF16) return output_for<__nv_bfloat16>(p, ws, st);
    if (p.dtype == GDR_F16) return output_for<__half>(p, ws, st);
    return output_for<float>(p, ws, st);
}

}  // namespace gdr
