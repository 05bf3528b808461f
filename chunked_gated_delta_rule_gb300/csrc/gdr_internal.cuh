// gdr_internal.cuh -- structures shared by the host runtime and the kernels
// of the chunked gated-delta-rule forward pass (not part of the public ABI).
#pragma once

#include <cstdint>
#include <cstddef>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gdr.h"

namespace gdr {

// Programmatic dependent launch.  Every kernel of a call after the first is
// launched with launch_pdl, so it may be scheduled while the kernels before
// it in the stream still run: it sets up (TMEM, barriers) and then calls
// pdl_wait(), which returns once every earlier kernel of the call has
// finished and its writes are visible; nothing of the workspace or the
// outputs is read or written before that.  Kernels call pdl_trigger() early
// so that the next launch is not held back until they exit.  A grid's
// dependents are scheduled only after all of its CTAs have started, so a
// waiting CTA never keeps one of them from running.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args &&...args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kChunk = 64;       // tokens per chunk
constexpr int kMaxK = 256;       // largest key dim supported
constexpr int kMaxV = 1024;      // largest value dim supported
constexpr int kMaxSegments = 64; // largest segment count (delta rule, backward)
// Largest segment count of the beta-free forward pass.  A count at or above
// a sequence's chunk count gives every chunk its own segment: the
// chunk-parallel producer dataflow of the ABC issue's "Proposed Dataflow"
// (per-chunk FP32 contributions, an ordered scalar-decay scan, an output
// pass from each chunk's boundary state).
constexpr int kMaxSegmentsBetaFree = 4096;

// Element strides of the token and head dimensions of a [tokens, H, D]
// tensor whose last dimension is contiguous (tokens flatten B and T).
struct TokStride {
    int64_t t, h;
};
__host__ __device__ __forceinline__ int64_t tok_at(const TokStride &s, int64_t t, int64_t h) {
    return t * s.t + h * s.h;
}

// Everything a kernel needs to address the caller's tensors.
struct Problem {
    const void *q, *k, *v;      // [B,T,H,K] / [B,T,H,V], dtype (strides sq, sk, sv)
    const float *g, *beta;      // [B,T,H]; beta == nullptr => beta-free
    const int32_t *cu;          // [N+1] or nullptr (dense); int32 offsets
    const int64_t *cu64;        // the same table as int64 (GDR_SEQLENS_I64), or nullptr
    const float *h0;            // [N,H,K,V] or nullptr
    void *o;                    // [B,T,H,V], dtype
    float *ht;                  // [N,H,K,V] or nullptr
    int64_t B, T, H, K, V, N;   // N = B when dense
    int dtype;                  // GDR_F32 | GDR_BF16
    float scale;
    int32_t *status;            // device status word or nullptr
    int state_vk;               // h0 / ht laid out [N,H,V,K] (S) instead of [N,H,K,V]
    int grid_limit;             // > 0: at most this many CTAs per persistent kernel
    TokStride sq, sk, sv, so;   // strides of q, k, v, o (contiguous: H*K, K / H*V, V)
};

// 16-byte vector loads of a [tokens, H, D] tensor: an aligned base and
// strides that keep every row start aligned (es = element size in bytes).
__host__ __device__ __forceinline__ bool rows_aligned16(const void *ptr, const TokStride &s,
                                                        int es) {
    return ((reinterpret_cast<uintptr_t>(ptr) | (uintptr_t)(s.t * es) | (uintptr_t)(s.h * es)) &
            15u) == 0;
}

// Contiguous [tokens, H, D] strides.
__host__ __device__ __forceinline__ TokStride dense_stride(int64_t H, int64_t D) {
    return TokStride{H * D, D};
}

// Streaming multiprocessors of the current device (152 on GB300 when no
// device can be queried: host-only plan lookups).
inline int device_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0) {
        cudaGetLastError();  // clear the sticky error of a failed query
        return 152;
    }
    return sms;
}

// CTAs of a persistent kernel that pulls `items` work units: per_sm CTAs on
// every SM, fewer when there are fewer units, and at most p.grid_limit when
// that is set.  Results never depend on the grid: every unit is computed by
// one CTA in a fixed order whichever CTA takes it.
inline int64_t persistent_grid(const Problem &p, int64_t items, int per_sm) {
    int64_t g = (int64_t)device_sms() * per_sm;
    if (items < g) g = items;
    if (p.grid_limit > 0 && g > p.grid_limit) g = p.grid_limit;
    return g < 1 ? 1 : g;
}

// cu_seqlens[i] in either width; a sequence's first token and end.
__host__ __device__ __forceinline__ int64_t seq_bound(const Problem &p, int64_t i) {
    return p.cu64 ? p.cu64[i] : (int64_t)p.cu[i];
}
__host__ __device__ __forceinline__ bool is_varlen_p(const Problem &p) {
    return p.cu != nullptr || p.cu64 != nullptr;
}
__host__ __device__ __forceinline__ int64_t seq_start(const Problem &p, int64_t n) {
    return is_varlen_p(p) ? seq_bound(p, n) : n * p.T;
}
__host__ __device__ __forceinline__ int64_t seq_end(const Problem &p, int64_t n) {
    return is_varlen_p(p) ? seq_bound(p, n + 1) : (n + 1) * p.T;
}
// Offset of element (key, v) of the state of (sequence, head) nh = n H + h
// in h0 / ht (and the recurrent pool): h = S^T [K][V], or S [V][K].
__host__ __device__ __forceinline__ int64_t state_off(const Problem &p, int64_t nh, int64_t key,
                                                      int64_t v) {
    return p.state_vk ? (nh * p.V + v) * p.K + key : (nh * p.K + key) * p.V + v;
}

// Scratch carved out of one device allocation (offsets fixed by the host).
struct Workspace {
    int32_t *chunk_tab;   // [max_chunks][4]: seq, first flat token, len, chunk-in-seq
    int32_t *seq_chunk0;  // [N+1]: first global chunk of each sequence
    int32_t *n_chunks;    // [8]: total chunks, then the chain counters of the
                          // persistent tensor-core kernels (zeroed per call;
                          // indices kCtr*)
    int32_t *seq_order;   // [N]: sequences by descending chunk count
    float *G;             // [max_chunks][H][64]: chunk-local gate cumsum
    float *W;             // [max_chunks][H][64][K]   (delta mode)
    float *U;             // [max_chunks][H][64][V]   (delta mode)
    float *hpre;          // [max_chunks][H][K][V]: state before each chunk
    float *vnew;          // [max_chunks][H][64][V]   (delta mode)
    float *segM;          // [N][H][S][K][K] transition per segment (delta), transposed
                          // (the tensor-core pre-scans write it for the backward only)
    float *segC;          // [N][H][S][K][V] local state per segment
    float *segH;          // [N][H][S][K][V] composed initial state per segment
    float *segD;          // [N][H][S] scalar transition (beta-free)
    uint8_t *rec;         // [max_chunks][H] per-chunk records of the
                          // tensor-core path (tc_chunk.cuh)
    // Transitions as the tensor-core composition's B operands: per
    // transition 64 KB, the BF16 hi image then the lo image (x = hi + lo) of
    // its transposed FP32 rows [m][r], each row m 128-byte swizzled in two
    // 64-column blocks of 16 KB (sw128_off(m, r, 128)).
    uint8_t *segMimg;     // [N][H][S] the segment transitions (tensor-core pre-scans)
    uint8_t *grpAimg;     // [N][H][ceil(S/G)] the group transitions (two-level composition)
    float *grpD;          // [N][H][ceil(S/G)][K][V] group offsets
    int64_t max_chunks;
    int n_segments;       // S (1 = serial)
    int grp_size;         // G, segments a group of the two-level composition (0: one level)
    int bwd_tc;           // the tensor-core backward's forward recompute: tc_prep
                          // also stores the T images, G and beta, the chain
                          // the h mirror and v_new images (bwd_lkimg)
    // [chunks][H][kLkImgBytes] (bwd_tc): the MMA operands of the backward's
    // per-chunk gradients as byte images of BF16 tiles (128-byte swizzled
    // rows, sw128_off): the chains' state mirrors h^T (the state before the
    // chunk, from the recompute) and E^T (the gradient at the chunk's end,
    // from the reverse scan), [v][key] in two 16 KB key blocks; and the FP32
    // operands as hi + lo pairs: v_new^T (recompute) and dV'^T (reverse
    // scan), [v][t] with 128 rows; T (prep), [i][j] with 64 rows; and the
    // chunk's gate cumsum G and beta (prep, FP32)
    uint8_t *bwd_lkimg;
};

// Chain counters in Workspace::n_chunks, one per persistent pass of a call.
constexpr int kCtrSerial = 1, kCtrPre = 2, kCtrSegOut = 3, kCtrSegRecompute = 4,
              kCtrBwdSerial = 5, kCtrBwdPre = 6, kCtrBwdSegOut = 7, kNumCtr = 8;

constexpr uint32_t kLkImgH = 0, kLkImgE = 32768;
constexpr uint32_t kLkImgVh = 65536, kLkImgVl = 81920;    // v_new^T hi, lo
constexpr uint32_t kLkImgDh = 98304, kLkImgDl = 114688;   // dV'^T hi, lo
constexpr uint32_t kLkImgTh = 131072, kLkImgTl = 139264;  // T hi, lo
constexpr uint32_t kLkImgVec = 147456;                    // FP32 G[64], beta[64] (prep)
constexpr uint32_t kLkImgVecBytes = 512;
constexpr uint32_t kLkImgBytes = kLkImgVec + kLkImgVecBytes;

// Backward pass: the caller's gradient tensors (dq, dk, dv in the input
// dtype; dg, dbeta, dh0 FP32; dht / dh0 in the state layout of h0).
struct BwdArgs {
    const void *dout;   // [B,T,H,V] dL/do
    const float *dht;   // [N,H,K,V] dL/dht or nullptr
    void *dq, *dk, *dv; // [B,T,H,K] / [B,T,H,V]
    float *dg, *dbeta;  // [B,T,H]; dbeta nullptr in the beta-free mode
    float *dh0;         // [N,H,K,V] or nullptr
};

// Backward scratch, per (chunk, head) item.
struct BwdWs {
    float *Mq;     // [items][64][64] causal(Q K^T * D), diagonal included
    float *Kd;     // [items][64][64] strictly lower K K^T * D (delta)
    float *Tm;     // [items][64][64] T = (I + A)^-1 (delta)
    float *dhend;  // [items][K][V] dL/d(state at the chunk's end)
    float *dvn;    // [items][64][V] dL/dV' (delta)
    float *P1;     // [items][64][K] dO h^T
    float *P2;     // [items][64][K] dV' h^T (delta)
    float *P3;     // [items][64][K] V' E^T
    float *ehp;    // [items][ceil(K/64)] <E, h> per 64-key slice
    float *segMb;  // [N][H][S][K][K] the reverse scan's segment maps (delta, split)
};

}  // namespace gdr
