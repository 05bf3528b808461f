// gdr_api.cu -- host runtime behind include/gdr.h: argument validation, launch
// plan (A13), workspace layout, and the launch sequence of the forward pass.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "gdr_internal.cuh"
#include "gdr_segments.cuh"
#include "gdr_launch.cuh"

namespace gdr {

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Device memory the library allocates during a call comes from a
// stream-ordered pool of its own, one per device, whose release threshold
// keeps freed blocks mapped.  The default pool returns its memory to the
// driver at every synchronisation, and mapping a call's few hundred MB again
// costs as much as a host call's copies.  gdr_release_cached() trims these
// pools.  While the stream is being captured into a graph the allocation
// stays on the default pool, as graph-owned memory.
constexpr int kMaxDevices = 64;
std::mutex g_pool_mu;
cudaMemPool_t g_pools[kMaxDevices] = {};

cudaError_t lib_pool(int dev, cudaMemPool_t *out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_pool_mu);
    if (!g_pools[dev]) {
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        cudaError_t e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess) return e;
        uint64_t keep = UINT64_MAX;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return e;
        }
        g_pools[dev] = pool;
    }
    *out = g_pools[dev];
    return cudaSuccess;
}

cudaError_t lib_malloc(void **ptr, size_t bytes, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return e;
    if (cs != cudaStreamCaptureStatusNone) return cudaMallocAsync(ptr, bytes, st);
    int dev = 0;
    e = cudaStreamGetDevice(st, &dev);
    if (e != cudaSuccess) return e;
    cudaMemPool_t pool = nullptr;
    e = lib_pool(dev, &pool);
    if (e != cudaSuccess) return e;
    return cudaMallocFromPoolAsync(ptr, bytes, pool, st);
}

// The host entry's copy streams (inputs in, outputs out), one pair per
// device, created on first use.  The caller's stream must belong to the
// current device.
struct CopyStreams {
    cudaStream_t in = nullptr, out = nullptr;
};
CopyStreams g_copy[kMaxDevices];

cudaError_t copy_streams(cudaStream_t st, CopyStreams *out) {
    int dev = 0, cur = 0;
    cudaError_t e = cudaStreamGetDevice(st, &dev);
    if (e == cudaSuccess) e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return e;
    if (dev != cur || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_pool_mu);
    CopyStreams &c = g_copy[dev];
    if (!c.in) {
        cudaStream_t a = nullptr, b = nullptr;
        e = cudaStreamCreateWithFlags(&a, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&b, cudaStreamNonBlocking);
        if (e != cudaSuccess) {
            if (a) cudaStreamDestroy(a);
            return e;
        }
        c.in = a;
        c.out = b;
    }
    *out = c;
    return cudaSuccess;
}

// Groups of whole sequences (batch rows when dense) for the host entry's
// overlap of copies and passes: about 32 MB of input a group, at most 4 (a
// small group's passes cost about 50 us whatever its size).  The first and
// last groups take half a share of the tokens: the outputs start leaving
// sooner and the pass and copy out after the last input are shorter.  Group
// i holds sequences [n[i], n[i + 1]).
struct HostGroups {
    std::vector<int64_t> n;
    int count() const { return (int)n.size() - 1; }
};

HostGroups host_groups(const std::vector<int64_t> &cu, size_t tok_bytes, size_t seq_bytes) {
    const int64_t ns = (int64_t)cu.size() - 1, T = cu[ns];
    const double total = (double)T * (double)tok_bytes + (double)ns * (double)seq_bytes;
    const int64_t want =
        std::max<int64_t>(1, std::min<int64_t>({std::llround(total / (32.0 * (1 << 20))), 4, ns}));
    HostGroups G;
    G.n.push_back(0);
    for (int64_t i = 1; i < want; ++i) {  // cut i at (2i - 1) / (2 (want - 1)) of the tokens
        const int64_t target = T * (2 * i - 1) / (2 * (want - 1));
        int64_t n = G.n.back() + 1;
        while (n < ns && cu[n] < target) ++n;
        if (n >= ns) break;
        G.n.push_back(n);
    }
    G.n.push_back(ns);
    return G;
}

bool is_varlen(const gdr_dims &d) { return d.N > 0; }
int64_t n_seqs(const gdr_dims &d) { return is_varlen(d) ? d.N : d.B; }

// Upper bound on the number of 64-token chunks: the chunk table is sized on
// the host, before cu_seqlens (device data) is read.  Each sequence adds at
// most one partial chunk.
int64_t max_chunks_of(const gdr_dims &d) {
    if (is_varlen(d)) return d.T / kChunk + d.N + 1;
    return d.B * ((d.T + kChunk - 1) / kChunk);
}

// The token / head strides of a tensor whose last dimension has D elements:
// the caller's pair, or the contiguous one for {0, 0}.
TokStride stride_of(const int64_t (&s)[2], int64_t H, int64_t D) {
    if (s[0] == 0 && s[1] == 0) return dense_stride(H, D);
    return TokStride{s[0], s[1]};
}

bool has_strides(const gdr_dims &d) {
    for (const int64_t *s : {d.q_stride, d.k_stride, d.v_stride, d.o_stride})
        if (s[0] || s[1]) return true;
    return false;
}

// Both entries zero or both positive; o's rows must not overlap: the inner
// of its two dimensions spaces rows at least V apart and the outer spans it.
int validate_strides(const gdr_dims &d) {
    for (const int64_t *s : {d.q_stride, d.k_stride, d.v_stride, d.o_stride})
        if ((s[0] == 0) != (s[1] == 0) || s[0] < 0 || s[1] < 0) return GDR_ERR_INVALID;
    const TokStride o = stride_of(d.o_stride, d.H, d.V);
    const int64_t tokens = d.B * d.T;
    bool ok;
    if (d.H == 1) ok = tokens <= 1 || o.t >= d.V;
    else if (tokens <= 1) ok = o.h >= d.V;
    else if (o.h <= o.t) ok = o.h >= d.V && o.t >= d.H * o.h;  // heads inside tokens
    else ok = o.t >= d.V && o.h >= tokens * o.t;                // tokens inside heads
    return ok ? GDR_OK : GDR_ERR_INVALID;
}

// Fills the tensor strides of a problem from its dims.
void set_strides(Problem &p, const gdr_dims &d) {
    p.sq = stride_of(d.q_stride, d.H, d.K);
    p.sk = stride_of(d.k_stride, d.H, d.K);
    p.sv = stride_of(d.v_stride, d.H, d.V);
    p.so = stride_of(d.o_stride, d.H, d.V);
}

int validate_dims(const gdr_dims *d) {
    if (!d) return GDR_ERR_INVALID;
    if (d->B < 1 || d->T < 0 || d->H < 1 || d->K < 1 || d->V < 1 || d->N < 0)
        return GDR_ERR_INVALID;
    if (d->dtype != GDR_F32 && d->dtype != GDR_BF16 && d->dtype != GDR_F16) return GDR_ERR_INVALID;
    if (d->flags & ~(GDR_SEQLENS_I64 | GDR_STATE_VK)) return GDR_ERR_INVALID;
    if (d->max_len < 0) return GDR_ERR_INVALID;
    if (validate_strides(*d) != GDR_OK) return GDR_ERR_INVALID;
    if (is_varlen(*d) && d->B != 1) return GDR_ERR_INVALID;
    if (d->K % 16 || d->V % 16) return GDR_ERR_UNSUPPORTED;
    if (d->K > kMaxK || d->V > kMaxV) return GDR_ERR_UNSUPPORTED;
    if (d->H > 65535) return GDR_ERR_UNSUPPORTED;
    if (d->B * d->T >= (int64_t)INT32_MAX) return GDR_ERR_UNSUPPORTED;
    return GDR_OK;
}

// Chunks of the longest sequence and the mean chunks per sequence.  Varlen:
// the longest from the caller's max_len hint (clamped to T), else the mean;
// dense: every sequence has T tokens.
struct ChunkStats {
    int64_t longest, mean, total;  // total = chunks of all sequences
};

ChunkStats chunk_stats(const gdr_dims &d) {
    ChunkStats c{};
    if (!is_varlen(d)) {
        c.longest = c.mean = (d.T + kChunk - 1) / kChunk;
        c.total = c.mean * d.B;
        return c;
    }
    c.mean = d.N ? (d.T / d.N + kChunk - 1) / kChunk : 0;
    const int64_t L = d.max_len > 0 ? std::min<int64_t>(d.max_len, d.T) : 0;
    c.longest = L > 0 ? std::max<int64_t>(c.mean, (L + kChunk - 1) / kChunk) : c.mean;
    // every sequence adds at most one partial chunk
    c.total = std::max<int64_t>(c.longest, d.T / kChunk + (d.N + 1) / 2);
    return c;
}

// Value columns per scan CTA, among the widths that divide both V and K (the
// transition tiles of the segment pre-scan cover K columns) and keep the
// scan's shared memory within 227 KB: 32 columns, measured fastest on GB300
// (wide varlen batch 2.29 ms against 2.53 at 64 and 2.64 at 16; beta-free
// K = 256, V = 512: 5.51 against 5.66 and 6.92); 16 when 32-column tiles
// leave SMs without a chain and the sequences are too short for a segment
// split to add chains (tiny dense FP32: 0.102 ms against 0.110 and 0.129);
// 64 only when neither divides.
int pick_bv(const gdr_dims &d) {
    const size_t Kp = ((size_t)d.K + 63) & ~(size_t)63;  // keys padded to 64-row tiles
    auto fits = [&](int bv) {
        if (d.V % bv || d.K % bv) return false;
        const size_t smem = sizeof(float) * (Kp * (bv + 1) + 2 * (size_t)kChunk * (Kp + 1) +
                                             (size_t)kChunk * (bv + 1) + kChunk);
        return smem <= 227 * 1024;
    };
    if (fits(32)) {
        const int64_t chains = n_seqs(d) * d.H * (d.V / 32);
        const int64_t cps = chunk_stats(d).longest;
        return (chains < device_sms() && cps < 32 && fits(16)) ? 16 : 32;  // a split needs 32 chunks
    }
    for (int bv : {16, 64})
        if (fits(bv)) return bv;
    return 16;
}

// Segment count when the caller passes 0.
// Tensor-core path: a cost model fitted to GB300 timings of its kernels.  A
// chain pass costs t microseconds per chunk; its chains run one per SM,
// longest first, so a pass lasts about t times the larger of the longest
// chain and the chunk steps each SM takes (all chains' chunks over the SMs,
// in whole waves when the chains are alike).  A split runs a pre-scan pass
// (two summaries per segment for the delta rule: local state and
// transition), an ordered composition costing t_step per segment, and an
// output pass; every sequence is cut into at most S runs of whole chunks, so
// the longest chain shrinks to ceil(longest / S) chunks while the work stays
// the same.  The model reproduces the measured best counts (16K x 16 heads:
// 8; 64K x 8 heads: 16; 64K x 1 head: 64; beta-free K = 256, V = 512,
// 2 x 8K x 4 heads: 4; the wide varlen batch: 1), and splits a batch whose
// longest sequence (the max_len hint) dwarfs the rest.
// CUDA-core path: split until about two CTAs per SM, at most 64 segments,
// while every segment of the longest sequence keeps at least 8 chunks (one
// 64K-token head's backward: 8.2 ms at 16 segments, 5.1 at 32, 3.8 at 64).
// The delta pre-scan of `segs` (sequence, segment, head) chains runs each of
// their two summaries as its own chain while all of them fit one wave.
bool prescan_split_kinds(int64_t segs) { return 2 * segs <= device_sms(); }

}  // namespace

int64_t split_seqs(const gdr_dims &d, int S) {
    const int64_t nseq = n_seqs(d);
    if (S <= 1 || nseq <= 1) return S <= 1 ? 0 : nseq;
    const ChunkStats cs = chunk_stats(d);
    const int64_t per = (cs.longest + S - 1) / S;
    const int64_t rest = (cs.total - cs.longest) / (nseq - 1);  // the others' mean, in chunks
    return rest > per ? nseq : 1;
}

namespace {

int auto_segments(const gdr_dims &d, bool beta_free, int path, int bv) {
    const int64_t nseq = n_seqs(d);
    const ChunkStats cs = chunk_stats(d);
    const int64_t cps = cs.longest;
    const int64_t sms = device_sms();
    if (path != 2) {
        const int64_t chains = nseq * d.H * (d.V / bv);
        int S = 1;
        while (S < kMaxSegments && chains * S < 2 * sms && cps / (2 * S) >= 8) S *= 2;
        return S;
    }
    const int64_t tiles = beta_free ? d.V / 128 : 1;  // chains per (sequence, head)
    const int64_t chains = nseq * d.H * tiles;
    const double steps = (double)cs.total * (double)(d.H * tiles);  // chunk steps of a pass
    auto waves = [&](int64_t c) { return (double)((c + sms - 1) / sms); };
    // chunk steps one SM runs in a pass whose longest chain has `per` chunks
    // and whose `n` chains are as long as their work allows
    auto pass = [&](double per, int64_t n) {
        const double uniform = per * waves(n);          // alike chains, in whole waves
        const double spread = steps / (double)sms;      // a mix, packed longest first
        return std::max(per, cs.longest == cs.mean ? uniform : std::max(spread, per));
    };
    const double t_serial = beta_free ? 3.3 : 2.4, t_pre = beta_free ? 2.0 : 2.4,
                 t_out = beta_free ? 3.7 : 2.4;
    const double state_mb = (double)(nseq * d.H) * (double)(d.K * d.V) * 4.0 / (1 << 20);
    const int64_t heads = nseq * d.H;  // composition tile: 4, 8 or 16 value columns
    // a delta composition step per wave of its CTAs (one value tile of one
    // (sequence, head) each, one CTA per SM): a batch of many sequences pays
    // it many times over (101 x 16 heads: 85 waves, 1.1 ms at 3 segments)
    const int64_t cc = heads * (d.V / 4) <= sms ? 4 : heads * (d.V / 8) <= sms ? 8 : 16;
    const double t_step = beta_free ? (0.65 * state_mb > 0.5 ? 0.65 * state_mb : 0.5)
                          : (cc == 4 ? 1.8 : cc == 8 ? 2.6 : 4.4) * waves(heads * (d.V / cc));
    double best = t_serial * pass((double)cps, chains);
    int best_s = 1;
    for (int S = 2; S <= kMaxSegments && S <= cps; ++S) {
        const int64_t per = (cps + S - 1) / S;
        if (S > 2 && (cps + S - 2) / (S - 1) == per) continue;  // same runs as S - 1
        // the tensor-core forward keeps one segment length for all sequences:
        // when the others fit one segment, only the longest is pre-scanned and
        // composed, and the output pass runs the others whole
        if (split_seqs(d, S) < nseq) {
            // the pre-scan: the long sequence's H x S chains, in waves when
            // both summaries share a CTA; the output pass: the longest chain,
            // or the spread of all chunk steps plus one whole short chain at
            // its tail (measured, 16K + 31 short x 4 heads, S = 12 / 16 / 24
            // / 32: output pass 53 / 43 / 45 / 53 us)
            const int64_t segs = d.H * tiles * (int64_t)S;
            const double pre = beta_free                  ? t_pre * (double)per * waves(segs)
                               : prescan_split_kinds(segs) ? t_pre * (double)per
                                                           : 8.0 + t_pre * (double)per * waves(segs);
            const double rest = (double)(cs.total - cps) / (double)(nseq - 1);
            const double out = t_out * std::max((double)per, steps / (double)sms + rest);
            // the beta-free composition walks the split sequences' states only
            // (the others' threads leave at once)
            const double split_mb = state_mb * (double)split_seqs(d, S) / (double)nseq;
            const double comp = beta_free ? std::max(0.5, 0.65 * split_mb) * S
                                          : compose_plan(d, S, true).cost_us;
            const double est = pre + out + comp;
            if (est < best) {
                best = est;
                best_s = S;
            }
            continue;
        }
        // segment chains: the longest sequence's S, the mean one's as many
        // as its chunks allow
        const int64_t segs = nseq * d.H * tiles * std::min<int64_t>(S, std::max<int64_t>(cs.mean, 1));
        double pre;
        if (beta_free) pre = t_pre * pass((double)per, segs);
        else if (prescan_split_kinds(segs)) pre = t_pre * (double)per;
        else pre = 2.9 * pass((double)per, segs);
        // the composition at its CUDA-core cost: a batch of many short
        // sequences splits each of them too, and the tensor-core pass's
        // lower cost there does not make up for the extra segment chains
        const double est = pre + t_out * pass((double)per, segs) + t_step * S;
        if (est < best) {
            best = est;
            best_s = S;
        }
    }
    return best_s;
}

// Shapes the tensor-core path covers (pointer alignment is checked per call):
// the delta rule at K = V = 128; the beta-free mode at K in {128, 256} with
// V a multiple of 128.
bool tc_shape_any_dtype(const gdr_dims &d, bool beta_free) {
    if (!beta_free) return d.K == 128 && d.V == 128;
    return (d.K == 128 || d.K == 256) && d.V % 128 == 0;
}

bool tc_shape(const gdr_dims &d, bool beta_free) {
    return d.dtype == GDR_BF16 && tc_shape_any_dtype(d, beta_free);
}

// gdr_plan::compose: 0 for the CUDA-core composition (or none), 1 for the
// tensor-core pass, G >= 2 for its two-level form in groups of G segments.
int compose_of(const gdr_dims &d, bool beta_free, int path, int S) {
    if (path != 2 || beta_free || S <= 1) return 0;
    const ComposePlan c = compose_plan(d, S, true);
    return c.kind == 0 ? 0 : c.kind == 1 ? 1 : c.grp_size;
}

int make_plan(const gdr_dims &d, bool beta_free, int n_segments, const gdr_options *opt,
              gdr_plan *plan) {
    gdr_plan p{};
    p.path = tc_shape(d, beta_free) ? 2 : 1;
    p.bv = p.path == 2 ? 128 : pick_bv(d);
    if (opt && opt->force_path) {
        if (opt->force_path != 1 && opt->force_path != 2) return GDR_ERR_INVALID;
        // FP16 inputs run the tensor-core kernels on BF16 copies, when forced
        const bool tc_ok = tc_shape(d, beta_free) ||
                           (d.dtype == GDR_F16 && tc_shape_any_dtype(d, beta_free));
        if (opt->force_path == 2 && !tc_ok) return GDR_ERR_UNSUPPORTED;
        p.path = opt->force_path;
        p.bv = p.path == 2 ? 128 : pick_bv(d);
    }
    if (opt && opt->force_bv) {
        const int bv = opt->force_bv;
        if (bv != 16 && bv != 32 && bv != 64 && bv != 128) return GDR_ERR_INVALID;
        if (p.path == 1 && (bv == 128 || d.V % bv || d.K % bv)) return GDR_ERR_UNSUPPORTED;
        if (p.path == 2 && bv != 128) return GDR_ERR_UNSUPPORTED;
        p.bv = bv;
    }
    if (n_segments < 0) return GDR_ERR_INVALID;
    if (n_segments > (beta_free ? kMaxSegmentsBetaFree : kMaxSegments))
        return GDR_ERR_UNSUPPORTED;
    p.n_segments = n_segments == 0 ? auto_segments(d, beta_free, p.path, p.bv) : n_segments;
    p.compose = compose_of(d, beta_free, p.path, p.n_segments);
    *plan = p;
    return GDR_OK;
}

}  // namespace

// The plan a forward call runs and the scratch it needs: the shape's plan,
// moved to the CUDA-core path when the tensor-core kernels cannot take the
// pointers (16-byte aligned q, k, v, o), with that path's own value tile and
// (for n_segments = 0) segment count.  Every forward entry point plans
// through here, so a caller that sizes scratch in advance
// (gdr_chunk_fwd_noalloc) sizes it for the path that will run.  FP16 inputs
// forced onto the tensor cores run on aligned BF16 copies.
int plan_for_call(const gdr_dims &d, bool beta_free, int n_segments, const gdr_options *opt,
                  const void *q, const void *k, const void *v, const void *o, gdr_plan *plan,
                  size_t *ws_bytes) {
    gdr_plan p{};
    int rc = validate_dims(&d);
    if (rc != GDR_OK) return rc;
    rc = make_plan(d, beta_free, n_segments, opt, &p);
    if (rc != GDR_OK) return rc;
    const bool copies = p.path == 2 && d.dtype == GDR_F16;
    if (copies && has_strides(d)) return GDR_ERR_UNSUPPORTED;  // the copies are contiguous
    const int es = d.dtype == GDR_F32 ? 4 : 2;
    if (p.path == 2 && !copies &&
        !(rows_aligned16(q, stride_of(d.q_stride, d.H, d.K), es) &&
          rows_aligned16(k, stride_of(d.k_stride, d.H, d.K), es) &&
          rows_aligned16(v, stride_of(d.v_stride, d.H, d.V), es) &&
          rows_aligned16(o, stride_of(d.o_stride, d.H, d.V), es))) {
        if (opt && opt->force_path == 2) return GDR_ERR_INVALID;  // misaligned pointers
        p.path = 1;
        p.bv = pick_bv(d);
        if (n_segments == 0) p.n_segments = auto_segments(d, beta_free, 1, p.bv);
        p.compose = 0;
    }
    *plan = p;
    if (ws_bytes) *ws_bytes = workspace_layout(d, beta_free, p.n_segments, p.path).total;
    return GDR_OK;
}

WorkspaceLayout workspace_layout(const gdr_dims &d, bool beta_free, int S, int path) {
    const bool delta = !beta_free;
    const bool simt = path == 1;
    const int64_t mc = max_chunks_of(d);
    const int64_t ns = n_seqs(d);
    const size_t H = (size_t)d.H, K = (size_t)d.K, V = (size_t)d.V;
    WorkspaceLayout L{};
    L.max_chunks = mc;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes);
        return at;
    };
    L.off_tab = take(sizeof(int32_t) * 4 * (size_t)mc);
    L.off_seq0 = take(sizeof(int32_t) * (size_t)(ns + 1));
    L.off_nchunks = take(sizeof(int32_t) * kNumCtrSlots);
    L.off_order = take(sizeof(int32_t) * (size_t)ns);
    L.off_G = take(simt ? sizeof(float) * (size_t)mc * H * kChunk : 0);
    L.off_W = take(simt && delta ? sizeof(float) * (size_t)mc * H * kChunk * K : 0);
    L.off_U = take(simt && delta ? sizeof(float) * (size_t)mc * H * kChunk * V : 0);
    L.off_hpre = take(simt ? sizeof(float) * (size_t)mc * H * K * V : 0);
    L.off_vnew = take(simt && delta ? sizeof(float) * (size_t)mc * H * kChunk * V : 0);
    const size_t segs = S > 1 ? (size_t)ns * H * (size_t)S : 0;
    L.off_segM = take(delta ? sizeof(float) * segs * K * K : 0);
    L.off_segC = take(sizeof(float) * segs * K * V);
    L.off_segH = take(sizeof(float) * segs * K * V);
    L.off_segD = take(delta ? 0 : sizeof(float) * segs);
    L.off_rec = take(simt || !delta ? 0 : (size_t)mc * H * 74752u);  // paths 2 and 3
    // the tensor-core composition's transition images, and the two-level
    // form's group transitions and offsets (tensor-core paths, delta rule)
    const ComposePlan cp =
        (!simt && delta && S > 1) ? compose_plan(d, S, path == 2) : ComposePlan{0, 0, 0.0};
    L.seg_images = cp.kind != 0;
    L.off_segMimg = take(L.seg_images ? segs * 65536u : 0);
    L.grp_size = cp.grp_size;
    const size_t grps = L.grp_size ? (size_t)ns * H * (size_t)((S + L.grp_size - 1) / L.grp_size) : 0;
    L.off_grpA = take(grps * 65536u);
    L.off_grpD = take(sizeof(float) * grps * K * V);
    L.total = off;
    return L;
}

// Fitted to GB300 (microseconds): the CUDA-core composition costs t_step
// per segment and wave of its CTAs (4, 8 or 16 value columns of one
// (sequence, head) each); the tensor-core pass about 11.6 + 1.87 per segment
// and wave of (sequence, head) runs; its two-level form about 33.5 for its
// three launches and 1.59 per step of each level (G - 1, ceil(S / G),
// G - 1 steps, in waves of their runs).  Measured, CUDA cores / single pass
// / two levels: 64K tokens x 8 heads at S = 19: 51 / 47 / 51; 64K x 1 head
// at S = 54: 92 / 113 / 65; 16K x 16 heads at S = 9: 41 / 29 / 45; a
// 16K-token sequence among 31 short ones x 4 heads at S = 7: 154 / 33 / 107.
// With one common segment length the tensor-core passes' runs of unsplit
// sequences end at once: their waves count the split sequences' heads.
ComposePlan compose_plan(const gdr_dims &d, int S, bool common) {
    const int64_t all = n_seqs(d) * d.H, sms = device_sms();
    const int64_t heads = common ? split_seqs(d, S) * d.H : all;
    auto waves = [&](int64_t n) { return (double)((n + sms - 1) / sms); };
    const int64_t cc = all * (d.V / 4) <= sms ? 4 : all * (d.V / 8) <= sms ? 8 : 16;
    ComposePlan c{0, 0, (cc == 4 ? 1.8 : cc == 8 ? 2.6 : 4.4) * waves(all * (d.V / cc)) * S};
    if (d.K != 128 || d.V != 128) return c;
    const double one = 11.6 + 1.87 * S * waves(heads);
    if (one < c.cost_us) c = ComposePlan{1, 0, one};
    if (S >= 4) {
        int G = 2;
        while ((G + 1) * (G + 1) <= S) ++G;  // floor(sqrt(S))
        const int64_t ng = (S + G - 1) / G;
        const double two = 33.5 + 1.59 * ((G - 1) * waves(2 * heads * ng) + ng * waves(heads) +
                                           (G - 1) * waves(heads * ng));
        if (two < c.cost_us) c = ComposePlan{2, G, two};
    }
    return c;
}

Workspace carve_workspace(void *base, const WorkspaceLayout &L, int S) {
    char *b = static_cast<char *>(base);
    Workspace w{};
    w.chunk_tab = reinterpret_cast<int32_t *>(b + L.off_tab);
    w.seq_chunk0 = reinterpret_cast<int32_t *>(b + L.off_seq0);
    w.n_chunks = reinterpret_cast<int32_t *>(b + L.off_nchunks);
    w.seq_order = reinterpret_cast<int32_t *>(b + L.off_order);
    w.G = reinterpret_cast<float *>(b + L.off_G);
    w.W = reinterpret_cast<float *>(b + L.off_W);
    w.U = reinterpret_cast<float *>(b + L.off_U);
    w.hpre = reinterpret_cast<float *>(b + L.off_hpre);
    w.vnew = reinterpret_cast<float *>(b + L.off_vnew);
    w.segM = reinterpret_cast<float *>(b + L.off_segM);
    w.segC = reinterpret_cast<float *>(b + L.off_segC);
    w.segH = reinterpret_cast<float *>(b + L.off_segH);
    w.segD = reinterpret_cast<float *>(b + L.off_segD);
    w.rec = reinterpret_cast<uint8_t *>(b + L.off_rec);
    w.segMimg = L.seg_images ? reinterpret_cast<uint8_t *>(b + L.off_segMimg) : nullptr;
    w.grpAimg = reinterpret_cast<uint8_t *>(b + L.off_grpA);
    w.grpD = reinterpret_cast<float *>(b + L.off_grpD);
    w.max_chunks = L.max_chunks;
    w.n_segments = S;
    w.grp_size = L.grp_size;
    return w;
}

// Backward scratch: the CUDA-core forward workspace (serial plan) followed by
// the per-(chunk, head) buffers of BwdWs.
struct BwdLayout {
    WorkspaceLayout fwd;
    size_t off_Mq, off_Kd, off_Tm, off_dhend, off_dvn, off_P1, off_P2, off_P3, off_ehp,
        off_segMb, off_lkimg, total;
};

BwdLayout bwd_layout(const gdr_dims &d, bool beta_free, int n_segments, bool tc_route) {
    BwdLayout B{};
    B.fwd = workspace_layout(d, beta_free, n_segments, tc_route ? 3 : 1);
    size_t off = B.fwd.total;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes);
        return at;
    };
    const bool delta = !beta_free;
    const size_t items = (size_t)B.fwd.max_chunks * (size_t)d.H;
    const size_t K = (size_t)d.K, V = (size_t)d.V, sq = (size_t)kChunk * kChunk;
    // the tensor-core route keeps its operands in the images; the CUDA-core
    // route every buffer of BwdWs
    const bool cc = !tc_route;
    B.off_Mq = take(cc ? sizeof(float) * items * sq : 0);
    B.off_Kd = take(cc && delta ? sizeof(float) * items * sq : 0);
    B.off_Tm = take(cc && delta ? sizeof(float) * items * sq : 0);
    B.off_dhend = take(cc ? sizeof(float) * items * K * V : 0);
    B.off_dvn = take(cc && delta ? sizeof(float) * items * kChunk * V : 0);
    B.off_P1 = take(cc ? sizeof(float) * items * kChunk * K : 0);
    B.off_P2 = take(cc && delta ? sizeof(float) * items * kChunk * K : 0);
    B.off_P3 = take(cc ? sizeof(float) * items * kChunk * K : 0);
    B.off_ehp = take(cc ? sizeof(float) * items * ((K + 63) / 64) : 0);
    const size_t segs = n_segments > 1 ? (size_t)n_seqs(d) * d.H * (size_t)n_segments : 0;
    B.off_segMb = take(delta ? sizeof(float) * segs * K * K : 0);
    B.off_lkimg = take(tc_route ? items * (size_t)kLkImgBytes : 0);
    B.total = off;
    return B;
}

BwdWs carve_bwd(void *base, const BwdLayout &B) {
    char *b = static_cast<char *>(base);
    auto f = [&](size_t at) { return reinterpret_cast<float *>(b + at); };
    BwdWs w{};
    w.Mq = f(B.off_Mq);
    w.Kd = f(B.off_Kd);
    w.Tm = f(B.off_Tm);
    w.dhend = f(B.off_dhend);
    w.dvn = f(B.off_dvn);
    w.P1 = f(B.off_P1);
    w.P2 = f(B.off_P2);
    w.P3 = f(B.off_P3);
    w.ehp = f(B.off_ehp);
    w.segMb = f(B.off_segMb);
    return w;
}

namespace {

#define GDR_TRY(expr)                                                  \
    do {                                                               \
        cudaError_t e_ = (expr);                                       \
        if (e_ != cudaSuccess) return GDR_ERR_CUDA;                    \
    } while (0)

#define GDR_LAUNCH(rec, id, expr)                                      \
    do {                                                               \
        GDR_TRY((rec).begin(id));                                      \
        GDR_TRY(expr);                                                 \
        GDR_TRY((rec).end());                                          \
    } while (0)

// The delta rule's segment composition on the tensor-core paths, as the
// workspace was planned (compose_plan): on CUDA cores when the pre-scan left
// no transition images, else the tensor-core pass or its two-level form.
int run_compose_tc(const Problem &p, const Workspace &ws, cudaStream_t st, LaunchRecorder &rec) {
    if (!ws.segMimg) {
        GDR_LAUNCH(rec, kKCompose, compose_mt(p, ws, st));
    } else if (ws.grp_size == 0) {
        GDR_LAUNCH(rec, kKTcCompose, compose_tc(p, ws, 0, st));
    } else {
        GDR_LAUNCH(rec, kKTcComposeGroups, compose_tc(p, ws, 1, st));
        GDR_LAUNCH(rec, kKTcComposeTop, compose_tc(p, ws, 2, st));
        GDR_LAUNCH(rec, kKTcComposeFill, compose_tc(p, ws, 3, st));
    }
    return GDR_OK;
}

int run_simt(const Problem &p, const Workspace &ws, const gdr_plan &plan, cudaStream_t st,
             LaunchRecorder &rec) {
    GDR_LAUNCH(rec, kKChunkTable, simt_chunk_table(p, ws, false, st));
    GDR_LAUNCH(rec, kKPrep, simt_prep(p, ws, st));
    if (plan.n_segments <= 1) {
        GDR_LAUNCH(rec, kKScanSerial, simt_scan(p, ws, 0, plan.bv, st));
    } else {
        GDR_LAUNCH(rec, kKScanPre, simt_scan(p, ws, 1, plan.bv, st));
        if (p.beta == nullptr)
            GDR_LAUNCH(rec, kKComposeScalar, compose_scalar(p, ws, st));
        else if (compose_mt_supported(p))
            GDR_LAUNCH(rec, kKCompose, compose_mt(p, ws, st));
        else
            GDR_LAUNCH(rec, kKCompose, simt_compose(p, ws, plan.bv, st));
        GDR_LAUNCH(rec, kKScanSegOut, simt_scan(p, ws, 2, plan.bv, st));
    }
    GDR_LAUNCH(rec, kKOutput, simt_output(p, ws, st));
    return GDR_OK;
}

// A split cuts every sequence into runs of one common length (the chunk
// table fixes it), so shorter sequences run whole in the output pass;
// split: the sequences that rule cuts (split_seqs), for the pre-scan's form.
int run_tc(const Problem &p, const Workspace &ws, const gdr_plan &plan, int64_t split,
           cudaStream_t st, LaunchRecorder &rec) {
    GDR_LAUNCH(rec, kKChunkTable, simt_chunk_table(p, ws, plan.n_segments > 1, st));
    if (p.beta == nullptr) {
        if (plan.n_segments <= 1) {
            GDR_LAUNCH(rec, kKTcGlaSerial, tc_gla(p, ws, 0, st));
        } else {
            GDR_LAUNCH(rec, kKTcGlaPre, tc_gla(p, ws, 1, st));
            GDR_LAUNCH(rec, kKComposeScalar, compose_scalar(p, ws, st));
            GDR_LAUNCH(rec, kKTcGlaSegOut, tc_gla(p, ws, 2, st));
        }
        return GDR_OK;
    }
    GDR_LAUNCH(rec, kKTcPrep, tc_prep(p, ws, st));
    if (plan.n_segments <= 1) {
        GDR_LAUNCH(rec, kKTcSerial, tc_chain(p, ws, 0, st));
    } else {
        if (prescan_split_kinds(split * plan.n_segments * p.H))
            GDR_LAUNCH(rec, kKTcPre, tc_chain(p, ws, 1, st));
        else
            GDR_LAUNCH(rec, kKTcPreDual, tc_prescan(p, ws, st));
        if (int rc = run_compose_tc(p, ws, st, rec)) return rc;
        GDR_LAUNCH(rec, kKTcSegOut, tc_chain(p, ws, 2, st));
    }
    return GDR_OK;
}

// Backward: the forward recompute (the state before each chunk and V'),
// then the backward kernels.  Route 2, all on the tensor cores: the
// preparation (records, and the T, G and beta images), the serial chain in
// its recompute mode (the h and v_new images), the
// reverse scan and the per-chunk gradients; route 1: the CUDA-core forward
// and backward kernels.
int run_bwd(const Problem &p, const Workspace &ws, const BwdArgs &a, const BwdWs &bw, int bv,
            int route, cudaStream_t st, LaunchRecorder &rec) {
    GDR_LAUNCH(rec, kKChunkTable, simt_chunk_table(p, ws, false, st));
    if (route == 2) {
        GDR_LAUNCH(rec, kKTcPrep, tc_prep(p, ws, st));
        if (ws.n_segments <= 1) {
            GDR_LAUNCH(rec, kKTcRecompute, tc_chain(p, ws, 3, st));
            GDR_LAUNCH(rec, kKTcBwdScan, tc_bwd_scan(p, ws, 0, a.dht, a.dh0, a.dout, st));
        } else {
            // the forward's split, its output pass keeping the images; then
            // the reverse scan's: offsets from E = 0, the composition from
            // dht to dh0 over the transposed forward maps in reversed slots,
            // and the output pass from each segment's composed end
            Problem pf = p;
            pf.ht = nullptr;
            if (prescan_split_kinds(p.N * ws.n_segments * p.H))
                GDR_LAUNCH(rec, kKTcPre, tc_chain(pf, ws, 1, st));
            else
                GDR_LAUNCH(rec, kKTcPreDual, tc_prescan(pf, ws, st));
            if (int rc = run_compose_tc(pf, ws, st, rec)) return rc;
            GDR_LAUNCH(rec, kKTcSegRecompute, tc_chain(pf, ws, 4, st));
            GDR_LAUNCH(rec, kKBwdMaps, bwd_maps(p, ws, bw.segMb, st));
            GDR_LAUNCH(rec, kKTcBwdPre, tc_bwd_scan(p, ws, 1, nullptr, nullptr, a.dout, st));
            Problem pr = p;
            pr.h0 = a.dht;
            pr.ht = a.dh0;
            Workspace wr = ws;
            wr.segM = bw.segMb;
            wr.segMimg = nullptr;  // the reverse maps exist as FP32 rows only: CUDA cores
            if (int rc = run_compose_tc(pr, wr, st, rec)) return rc;
            GDR_LAUNCH(rec, kKTcBwdSegOut, tc_bwd_scan(p, ws, 2, nullptr, nullptr, a.dout, st));
        }
        GDR_LAUNCH(rec, kKTcBwdGrad, tc_bwd_grad(p, ws, a, st));
        return GDR_OK;
    }
    GDR_LAUNCH(rec, kKPrep, simt_prep(p, ws, st));
    if (ws.n_segments <= 1) {
        GDR_LAUNCH(rec, kKScanSerial, simt_scan(p, ws, 0, bv, st));
    } else {
        GDR_LAUNCH(rec, kKScanPre, simt_scan(p, ws, 1, bv, st));
        if (p.beta == nullptr)
            GDR_LAUNCH(rec, kKComposeScalar, compose_scalar(p, ws, st));
        else if (compose_mt_supported(p))
            GDR_LAUNCH(rec, kKCompose, compose_mt(p, ws, st));
        else
            GDR_LAUNCH(rec, kKCompose, simt_compose(p, ws, bv, st));
        GDR_LAUNCH(rec, kKScanSegOut, simt_scan(p, ws, 2, bv, st));
    }
    GDR_TRY(simt_bwd(p, ws, a, bw, st, rec));
    return GDR_OK;
}

}  // namespace
}  // namespace gdr

using namespace gdr;

extern "C" {

int gdr_version(void) { return 100; }

int gdr_release_cached(void) {
    int rc = GDR_OK;
    std::lock_guard<std::mutex> lock(g_pool_mu);
    for (cudaMemPool_t pool : g_pools)
        if (pool && cudaMemPoolTrimTo(pool, 0) != cudaSuccess) rc = GDR_ERR_CUDA;
    return rc;
}

const char *gdr_kernel_name(int id) {
    switch (id) {
    case kKChunkTable: return "simt_chunk_table";
    case kKPrep: return "simt_prep";
    case kKScanSerial: return "simt_scan_serial";
    case kKScanPre: return "simt_scan_prescan";
    case kKCompose: return "compose_delta";
    case kKTcCompose: return "tc_compose";
    case kKTcComposeGroups: return "tc_compose_groups";
    case kKTcComposeTop: return "tc_compose_top";
    case kKTcComposeFill: return "tc_compose_fill";
    case kKScanSegOut: return "simt_scan_segment_out";
    case kKOutput: return "simt_output";
    case kKTcSerial: return "tc_chain_serial";
    case kKTcPre: return "tc_chain_prescan";
    case kKTcSegOut: return "tc_chain_segment_out";
    case kKTcPrep: return "tc_prep";
    case kKTcGlaSerial: return "tc_gla_serial";
    case kKTcGlaPre: return "tc_gla_prescan";
    case kKTcGlaSegOut: return "tc_gla_segment_out";
    case kKComposeScalar: return "compose_scalar";
    case kKTcPreDual: return "tc_prescan_dual";
    case kKBwdGram: return "bwd_gram";
    case kKBwdScan: return "bwd_dscan";
    case kKBwdLk: return "bwd_lk";
    case kKBwdLocal: return "bwd_local";
    case kKBwdPre: return "bwd_dscan_prescan";
    case kKBwdSegOut: return "bwd_dscan_segment_out";
    case kKBwdMaps: return "bwd_maps";
    case kKConvertIn: return "convert_f16_to_bf16";
    case kKConvertOut: return "convert_bf16_to_f16";
    case kKTcRecompute: return "tc_chain_recompute";
    case kKTcBwdScan: return "tc_bwd_scan";
    case kKTcBwdGrad: return "tc_bwd_grad";
    case kKTcSegRecompute: return "tc_chain_segment_recompute";
    case kKTcBwdPre: return "tc_bwd_scan_prescan";
    case kKTcBwdSegOut: return "tc_bwd_scan_segment_out";
    default: return "?";
    }
}

const char *gdr_error_string(int code) {
    switch (code) {
    case GDR_OK: return "ok";
    case GDR_ERR_INVALID: return "invalid argument";
    case GDR_ERR_UNSUPPORTED: return "unsupported shape or option";
    case GDR_ERR_CUDA: return "CUDA runtime or launch error";
    case GDR_ERR_TIMEOUT: return "device-side bounded wait expired";
    case GDR_ERR_SEQLENS: return "malformed cu_seqlens";
    case GDR_ERR_WORKSPACE: return "workspace too small";
    case GDR_ERR_INDEX: return "state index out of range";
    default: return "unknown error code";
    }
}

int gdr_recurrent_fwd(const gdr_dims *dims, const void *q, const void *k, const void *v,
                      const float *g, const float *beta, const int32_t *cu_seqlens, float *state,
                      int64_t n_states, const int32_t *state_indices, void *o, int32_t *status,
                      gdr_stream_t stream) {
    int rc = validate_dims(dims);
    if (rc != GDR_OK) return rc;
    if (!q || !k || !v || !g || !o || !state || n_states < 1) return GDR_ERR_INVALID;
    if ((cu_seqlens != nullptr) != is_varlen(*dims)) return GDR_ERR_INVALID;
    if (!state_indices && n_states < n_seqs(*dims)) return GDR_ERR_INVALID;
    if (n_seqs(*dims) > 65535) return GDR_ERR_UNSUPPORTED;  // one grid row per sequence
    Problem p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
    if (dims->flags & GDR_SEQLENS_I64) p.cu64 = reinterpret_cast<const int64_t *>(cu_seqlens);
    else p.cu = cu_seqlens;
    p.state_vk = (dims->flags & GDR_STATE_VK) != 0;
    p.o = o;
    p.B = dims->B; p.T = dims->T; p.H = dims->H; p.K = dims->K; p.V = dims->V;
    set_strides(p, *dims);
    p.N = n_seqs(*dims);
    p.dtype = dims->dtype;
    p.scale = 1.0f / std::sqrt((float)dims->K);
    p.status = status;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return recurrent_fwd(p, state, n_states, state_indices, st) == cudaSuccess ? GDR_OK
                                                                                 : GDR_ERR_CUDA;
}

int gdr_plan_query(const gdr_dims *dims, int beta_free, int n_segments, gdr_plan *out) {
    int rc = validate_dims(dims);
    if (rc != GDR_OK) return rc;
    if (!out) return GDR_ERR_INVALID;
    return make_plan(*dims, beta_free != 0, n_segments, nullptr, out);
}

size_t gdr_workspace_size(const gdr_dims *dims, int beta_free, int n_segments) {
    if (validate_dims(dims) != GDR_OK) return 0;
    gdr_plan plan;
    if (make_plan(*dims, beta_free != 0, n_segments, nullptr, &plan) != GDR_OK) return 0;
    return workspace_layout(*dims, beta_free != 0, plan.n_segments, plan.path).total;
}


int gdr_chunk_fwd_ex(const gdr_dims *dims, const void *q, const void *k, const void *v,
                     const float *g, const float *beta, const int32_t *cu_seqlens,
                     const float *h0, void *o, float *ht, int n_segments,
                     const gdr_options *opt, gdr_stream_t stream) {
    int rc = validate_dims(dims);
    if (rc != GDR_OK) return rc;
    if (!q || !k || !v || !g || !o) return GDR_ERR_INVALID;
    if ((cu_seqlens != nullptr) != is_varlen(*dims)) return GDR_ERR_INVALID;
    const bool beta_free = beta == nullptr;
    if (opt && !(opt->scale >= 0.f)) return GDR_ERR_INVALID;  // rejects NaN too
    if (opt && opt->grid_limit < 0) return GDR_ERR_INVALID;
    gdr_plan plan;
    size_t ws_need = 0;
    rc = plan_for_call(*dims, beta_free, n_segments, opt, q, k, v, o, &plan, &ws_need);
    if (rc != GDR_OK) return rc;
    if (opt && opt->workspace && opt->workspace_bytes < ws_need) return GDR_ERR_WORKSPACE;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Problem p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
    if (dims->flags & GDR_SEQLENS_I64) p.cu64 = reinterpret_cast<const int64_t *>(cu_seqlens);
    else p.cu = cu_seqlens;
    p.state_vk = (dims->flags & GDR_STATE_VK) != 0;
    p.h0 = h0; p.o = o; p.ht = ht;
    p.B = dims->B; p.T = dims->T; p.H = dims->H; p.K = dims->K; p.V = dims->V;
    set_strides(p, *dims);
    p.N = n_seqs(*dims);
    p.dtype = dims->dtype;
    p.scale = (opt && opt->scale > 0.f) ? opt->scale : 1.0f / std::sqrt((float)dims->K);
    p.status = opt ? opt->status : nullptr;
    p.grid_limit = opt ? opt->grid_limit : 0;
    if (p.N == 0) return GDR_OK;
    // FP16 inputs on the tensor-core path: the kernels read BF16 copies of q,
    // k, v and write o in BF16, converted back to FP16 after the pass
    void *conv = nullptr;
    void *o_f16 = nullptr;
    const int64_t nqk = dims->B * dims->T * dims->H * dims->K;
    const int64_t nvo = dims->B * dims->T * dims->H * dims->V;
    LaunchRecorder rec;
    rec.st = st;
    if (opt) {
        rec.events = reinterpret_cast<cudaEvent_t *>(opt->events);
        rec.max_launches = opt->events ? opt->max_launches : 0;
        rec.ids = opt->launch_ids;
        if (!opt->events && opt->launch_ids) rec.max_launches = opt->max_launches;
    }
    if (plan.path == 2 && p.dtype == GDR_F16) {
        const size_t bqk = align_up(sizeof(uint16_t) * (size_t)nqk);
        const size_t bvo = align_up(sizeof(uint16_t) * (size_t)nvo);
        if (lib_malloc(&conv, 2 * bqk + 2 * bvo + kAlign, st) != cudaSuccess) return GDR_ERR_CUDA;
        char *c = static_cast<char *>(conv);
        void *qb = c, *kb = c + bqk, *vb = c + 2 * bqk, *ob = c + 2 * bqk + bvo;
        const void *src[3] = {q, k, v};
        void *dst[3] = {qb, kb, vb};
        const int64_t cnt[3] = {nqk, nqk, nvo};
        for (int i = 0; i < 3; ++i) {
            if (rec.begin(kKConvertIn) != cudaSuccess ||
                convert_f16_to_bf16(src[i], dst[i], cnt[i], st) != cudaSuccess ||
                rec.end() != cudaSuccess) {
                cudaFreeAsync(conv, st);
                return GDR_ERR_CUDA;
            }
        }
        p.q = qb; p.k = kb; p.v = vb;
        o_f16 = p.o;
        p.o = ob;
        p.dtype = GDR_BF16;
    }
    // every return from here on releases the conversion scratch
    auto fail = [&](int code) {
        if (conv) cudaFreeAsync(conv, st);
        return code;
    };
    // plan_for_call moved misaligned calls to the CUDA-core path already
    if (plan.path == 2 && !(beta_free ? tc_gla_supported(p) : tc_supported(p)))
        return fail(GDR_ERR_INVALID);

    const WorkspaceLayout L = workspace_layout(*dims, beta_free, plan.n_segments, plan.path);
    void *base = nullptr;
    bool owned = false;
    if (opt && opt->workspace) {
        if (opt->workspace_bytes < L.total) return fail(GDR_ERR_WORKSPACE);
        if (reinterpret_cast<uintptr_t>(opt->workspace) % kAlign) return fail(GDR_ERR_INVALID);
        base = opt->workspace;
    } else {
        if (lib_malloc(&base, L.total, st) != cudaSuccess) return fail(GDR_ERR_CUDA);
        owned = true;
    }
    const Workspace ws = carve_workspace(base, L, plan.n_segments);
    rc = plan.path == 2 ? run_tc(p, ws, plan, split_seqs(*dims, plan.n_segments), st, rec)
                        : run_simt(p, ws, plan, st, rec);
    if (conv) {
        if (rc == GDR_OK && (rec.begin(kKConvertOut) != cudaSuccess ||
                             convert_bf16_to_f16(p.o, o_f16, nvo, st) != cudaSuccess ||
                             rec.end() != cudaSuccess))
            rc = GDR_ERR_CUDA;
        if (cudaFreeAsync(conv, st) != cudaSuccess && rc == GDR_OK) rc = GDR_ERR_CUDA;
    }
    if (opt && opt->n_launches) *opt->n_launches = rec.count;
    if (owned) {
        if (cudaFreeAsync(base, st) != cudaSuccess && rc == GDR_OK) rc = GDR_ERR_CUDA;
    }
    return rc;
}

int gdr_chunk_fwd(const gdr_dims *dims, const void *q, const void *k, const void *v,
                  const float *g, const float *beta, const int32_t *cu_seqlens,
                  const float *h0, void *o, float *ht, int n_segments,
                  gdr_stream_t stream) {
    return gdr_chunk_fwd_ex(dims, q, k, v, g, beta, cu_seqlens, h0, o, ht, n_segments,
                            nullptr, stream);
}

// The backward's plan.  Route 2, the tensor-core route (the tensor-core
// forward recompute, reverse scan and per-chunk gradients; BF16 operands,
// see gdr.h), for BF16 inputs with K = V = 128 and the delta rule, split
// into segments by the tensor-core forward's rule unless the caller fixes
// the count (its scans cost about 1.5 times the forward's per chunk, its
// compositions the same, so the forward's cost model picks close to the
// backward's best; 64K tokens: 8 heads 1.85 ms at 19 segments against 8.5
// serial, 1 head 0.64 ms at 54).  Route 1, the CUDA-core route (FP32
// arithmetic), otherwise, with the CUDA-core path's value tile (32 columns
// on the wide varlen batch: its scan 0.98 ms at 64, 0.74 ms at 32) and
// segment rule unless the caller fixes the count.  force_path 1 or 2 picks
// a route.
int bwd_plan(const gdr_dims &d, bool beta_free, int n_segments, const gdr_options *opt,
             int *route, int *bv, int *S) {
    if (n_segments < 0) return GDR_ERR_INVALID;
    if (n_segments > kMaxSegments) return GDR_ERR_UNSUPPORTED;
    const int force = opt ? opt->force_path : 0;
    if (force < 0 || force > 2) return GDR_ERR_INVALID;
    const bool tc_ok = d.dtype == GDR_BF16 && d.K == 128 && d.V == 128 && !beta_free;
    if (force == 2 && !tc_ok) return GDR_ERR_UNSUPPORTED;
    *route = force ? force : (tc_ok ? 2 : 1);
    *bv = pick_bv(d);
    *S = n_segments > 0 ? n_segments : auto_segments(d, beta_free, *route == 2 ? 2 : 1, *bv);
    return GDR_OK;
}

size_t gdr_bwd_workspace_size(const gdr_dims *dims, int beta_free, int n_segments) {
    if (validate_dims(dims) != GDR_OK) return 0;
    int route = 1, bv = 0, S = 1;
    if (bwd_plan(*dims, beta_free != 0, n_segments, nullptr, &route, &bv, &S) != GDR_OK) return 0;
    // enough for either route (force_path may pick the other one, and a
    // misaligned call moves to the CUDA-core route)
    gdr_options o{};
    o.force_path = 1;
    int r1 = 1, S1 = 1;
    if (bwd_plan(*dims, beta_free != 0, n_segments, &o, &r1, &bv, &S1) != GDR_OK) return 0;
    size_t bytes = bwd_layout(*dims, beta_free != 0, S1, false).total;
    o.force_path = 2;
    int r2 = 2, S2 = 1;
    if (bwd_plan(*dims, beta_free != 0, n_segments, &o, &r2, &bv, &S2) == GDR_OK)
        bytes = std::max(bytes, bwd_layout(*dims, beta_free != 0, S2, true).total);
    return bytes;
}

int gdr_chunk_bwd(const gdr_dims *dims, const void *q, const void *k, const void *v,
                  const float *g, const float *beta, const int32_t *cu_seqlens,
                  const float *h0, const void *dout, const float *dht, void *dq, void *dk,
                  void *dv, float *dg, float *dbeta, float *dh0, int n_segments,
                  const gdr_options *opt, gdr_stream_t stream) {
    int rc = validate_dims(dims);
    if (rc != GDR_OK) return rc;
    if (!q || !k || !v || !g || !dout || !dq || !dk || !dv || !dg) return GDR_ERR_INVALID;
    if ((beta != nullptr) != (dbeta != nullptr)) return GDR_ERR_INVALID;
    if ((cu_seqlens != nullptr) != is_varlen(*dims)) return GDR_ERR_INVALID;
    if (opt && !(opt->scale >= 0.f)) return GDR_ERR_INVALID;  // rejects NaN too
    if (opt && (opt->force_bv != 0 || opt->grid_limit < 0)) return GDR_ERR_INVALID;
    const bool beta_free = beta == nullptr;
    int route = 1, bv_rec = 0, S = 1;
    rc = bwd_plan(*dims, beta_free, n_segments, opt, &route, &bv_rec, &S);
    if (rc != GDR_OK) return rc;
    if (route == 2) {  // TMA reads q, k, v and dO: aligned rows
        const bool aligned = rows_aligned16(q, stride_of(dims->q_stride, dims->H, dims->K), 2) &&
                             rows_aligned16(k, stride_of(dims->k_stride, dims->H, dims->K), 2) &&
                             rows_aligned16(v, stride_of(dims->v_stride, dims->H, dims->V), 2) &&
                             rows_aligned16(dout, dense_stride(dims->H, dims->V), 2);
        if (!aligned) {
            if (opt && opt->force_path == 2) return GDR_ERR_INVALID;
            route = 1;
            S = n_segments > 0 ? n_segments : auto_segments(*dims, beta_free, 1, bv_rec);
        }
    }

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Problem p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
    if (dims->flags & GDR_SEQLENS_I64) p.cu64 = reinterpret_cast<const int64_t *>(cu_seqlens);
    else p.cu = cu_seqlens;
    p.state_vk = (dims->flags & GDR_STATE_VK) != 0;
    p.h0 = h0;
    p.B = dims->B; p.T = dims->T; p.H = dims->H; p.K = dims->K; p.V = dims->V;
    set_strides(p, *dims);
    p.N = n_seqs(*dims);
    p.dtype = dims->dtype;
    p.scale = (opt && opt->scale > 0.f) ? opt->scale : 1.0f / std::sqrt((float)dims->K);
    p.status = opt ? opt->status : nullptr;
    p.grid_limit = opt ? opt->grid_limit : 0;
    if (p.N == 0) return GDR_OK;

    const BwdLayout B = bwd_layout(*dims, beta_free, S, route == 2);
    void *base = nullptr;
    bool owned = false;
    if (opt && opt->workspace) {
        if (opt->workspace_bytes < B.total) return GDR_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(opt->workspace) % kAlign) return GDR_ERR_INVALID;
        base = opt->workspace;
    } else {
        if (lib_malloc(&base, B.total, st) != cudaSuccess) return GDR_ERR_CUDA;
        owned = true;
    }
    Workspace ws = carve_workspace(base, B.fwd, S);
    const BwdWs bw = carve_bwd(base, B);
    ws.bwd_tc = route == 2;
    if (ws.bwd_tc) {
        ws.bwd_lkimg = static_cast<uint8_t *>(base) + B.off_lkimg;
    }
    BwdArgs a{};
    a.dout = dout; a.dht = dht; a.dq = dq; a.dk = dk; a.dv = dv;
    a.dg = dg; a.dbeta = dbeta; a.dh0 = dh0;
    LaunchRecorder rec;
    rec.st = st;
    if (opt) {
        rec.events = reinterpret_cast<cudaEvent_t *>(opt->events);
        rec.max_launches = opt->events ? opt->max_launches : 0;
        rec.ids = opt->launch_ids;
        if (!opt->events && opt->launch_ids) rec.max_launches = opt->max_launches;
    }
    rc = run_bwd(p, ws, a, bw, bv_rec, route, st, rec);
    if (opt && opt->n_launches) *opt->n_launches = rec.count;
    if (owned) {
        if (cudaFreeAsync(base, st) != cudaSuccess && rc == GDR_OK) rc = GDR_ERR_CUDA;
    }
    return rc;
}

}  // extern "C"

namespace gdr {
namespace {

// The host entry for one long sequence (dense with B == 1, or varlen with one
// sequence), which cannot be cut into groups of whole sequences: it is cut
// into `want` pieces of whole chunks (the first and last half a share), run
// as consecutive passes, each starting from the state the previous one
// ended with (kept on the device), while the next piece's inputs arrive and
// the previous piece's outputs leave.  The state carries exactly across any
// split point, so the result is the sequence's up to rounding.
int host_fwd_pieces(const gdr_dims &D, int64_t T, int want, const void *q, const void *k,
                    const void *v, const float *g, const float *beta, const float *h0, void *o,
                    float *ht, int n_segments, cudaStream_t st) {
    const size_t es = D.dtype == GDR_F32 ? 4 : 2;
    const size_t rq = (size_t)D.H * D.K * es, rv = (size_t)D.H * D.V * es, rg = (size_t)D.H * 4;
    const size_t rh = (size_t)D.H * D.K * D.V * 4;
    const int64_t chunks = (T + kChunk - 1) / kChunk;
    std::vector<int64_t> cut{0};  // token offsets of the pieces
    for (int i = 1; i < want; ++i) {
        const int64_t c = chunks * (2 * i - 1) / (2 * (want - 1)) * kChunk;
        if (c > cut.back() && c < T) cut.push_back(c);
    }
    cut.push_back(T);
    const int P = (int)cut.size() - 1;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t at = off; off = align_up(off + bytes); return at; };
    const size_t oq = take(T * rq), ok = take(T * rq), ov = take(T * rv), og = take(T * rg);
    const size_t ob = take(beta ? T * rg : 0), oo = take(T * rv);
    const size_t oh0 = take(h0 ? rh : 0), os0 = take(rh), os1 = take(rh);  // states in flight
    const size_t ocu = take(D.N > 0 ? 2 * P * sizeof(int32_t) : 0);
    char *d = nullptr;
    if (lib_malloc(reinterpret_cast<void **>(&d), off, st) != cudaSuccess) return GDR_ERR_CUDA;
    CopyStreams cs{};
    const bool piped = copy_streams(st, &cs) == cudaSuccess;
    cudaStream_t s_in = piped ? cs.in : st, s_out = piped ? cs.out : st;
    std::vector<cudaEvent_t> ev;
    auto order = [&](cudaStream_t from, cudaStream_t to) {
        if (!piped || from == to) return cudaSuccess;
        cudaEvent_t e = nullptr;
        cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
        if (r != cudaSuccess) return r;
        ev.push_back(e);
        r = cudaEventRecord(e, from);
        return r == cudaSuccess ? cudaStreamWaitEvent(to, e, 0) : r;
    };
    auto h2d = [&](size_t at, const void *src, size_t bytes) {
        return bytes ? cudaMemcpyAsync(d + at, src, bytes, cudaMemcpyHostToDevice, s_in)
                     : cudaSuccess;
    };
    const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k),
               *hv = static_cast<const char *>(v), *hg = reinterpret_cast<const char *>(g),
               *hb = reinterpret_cast<const char *>(beta);
    char *ho = static_cast<char *>(o);
    // every piece's cu_seqlens (varlen: one sequence of the piece's length)
    std::vector<int32_t> pcu;
    for (int i = 0; i < P; ++i) {
        pcu.push_back(0);
        pcu.push_back((int32_t)(cut[i + 1] - cut[i]));
    }
    int rc = GDR_OK;
    if (order(st, s_in) != cudaSuccess || order(st, s_out) != cudaSuccess ||
        (D.N > 0 && h2d(ocu, pcu.data(), pcu.size() * sizeof(int32_t)) != cudaSuccess) ||
        (h0 && h2d(oh0, h0, rh) != cudaSuccess))
        rc = GDR_ERR_CUDA;
    std::vector<cudaEvent_t> arrived((size_t)P, nullptr);
    for (int i = 0; i < P && rc == GDR_OK; ++i) {  // every piece's inputs queued first
        const size_t t0 = (size_t)cut[i], nt = (size_t)(cut[i + 1] - cut[i]);
        if (h2d(oq + t0 * rq, hq + t0 * rq, nt * rq) != cudaSuccess ||
            h2d(ok + t0 * rq, hk + t0 * rq, nt * rq) != cudaSuccess ||
            h2d(ov + t0 * rv, hv + t0 * rv, nt * rv) != cudaSuccess ||
            h2d(og + t0 * rg, hg + t0 * rg, nt * rg) != cudaSuccess ||
            (beta && h2d(ob + t0 * rg, hb + t0 * rg, nt * rg) != cudaSuccess)) {
            rc = GDR_ERR_CUDA;
            break;
        }
        if (piped) {
            if (cudaEventCreateWithFlags(&arrived[i], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventRecord(arrived[i], s_in) != cudaSuccess) {
                rc = GDR_ERR_CUDA;
                break;
            }
            ev.push_back(arrived[i]);
        }
    }
    for (int i = 0; i < P && rc == GDR_OK; ++i) {
        const size_t t0 = (size_t)cut[i], nt = (size_t)(cut[i + 1] - cut[i]);
        if (piped && cudaStreamWaitEvent(st, arrived[i], 0) != cudaSuccess) {
            rc = GDR_ERR_CUDA;
            break;
        }
        gdr_dims gd = D;
        gd.flags &= ~GDR_SEQLENS_I64;
        if (D.N > 0) {
            gd.T = (int64_t)nt;
            gd.max_len = (int64_t)nt;
        } else {
            gd.T = (int64_t)nt;
        }
        const float *pin = i == 0 ? (h0 ? reinterpret_cast<float *>(d + oh0) : nullptr)
                                  : reinterpret_cast<float *>(d + ((i - 1) & 1 ? os1 : os0));
        float *pout = reinterpret_cast<float *>(d + (i & 1 ? os1 : os0));
        const int32_t *gc =
            D.N > 0 ? reinterpret_cast<const int32_t *>(d + ocu + 2 * i * sizeof(int32_t)) : nullptr;
        rc = gdr_chunk_fwd(&gd, d + oq + t0 * rq, d + ok + t0 * rq, d + ov + t0 * rv,
                           reinterpret_cast<float *>(d + og + t0 * rg),
                           beta ? reinterpret_cast<float *>(d + ob + t0 * rg) : nullptr, gc, pin,
                           d + oo + t0 * rv, pout, n_segments,
                           reinterpret_cast<gdr_stream_t>(st));
        if (rc != GDR_OK) break;
        if (order(st, s_out) != cudaSuccess ||
            cudaMemcpyAsync(ho + t0 * rv, d + oo + t0 * rv, nt * rv, cudaMemcpyDeviceToHost,
                            s_out) != cudaSuccess ||
            (ht && i == P - 1 &&
             cudaMemcpyAsync(ht, pout, rh, cudaMemcpyDeviceToHost, s_out) != cudaSuccess))
            rc = GDR_ERR_CUDA;
    }
    if (order(s_in, st) != cudaSuccess || order(s_out, st) != cudaSuccess) {
        cudaStreamSynchronize(s_in);
        cudaStreamSynchronize(s_out);
        if (rc == GDR_OK) rc = GDR_ERR_CUDA;
    }
    if (cudaFreeAsync(d, st) != cudaSuccess && rc == GDR_OK) rc = GDR_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess && rc == GDR_OK) rc = GDR_ERR_CUDA;
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
    return rc;
}

}  // namespace
}  // namespace gdr

extern "C" {

int gdr_chunk_fwd_host(const gdr_dims *dims, const void *q, const void *k, const void *v,
                       const float *g, const float *beta, const int32_t *cu_seqlens,
                       const float *h0, void *o, float *ht, int n_segments,
                       gdr_stream_t stream) {
    int rc = validate_dims(dims);
    if (rc != GDR_OK) return rc;
    if (has_strides(*dims)) return GDR_ERR_UNSUPPORTED;  // host buffers are copied whole
    if (!q || !k || !v || !g || !o) return GDR_ERR_INVALID;
    if ((cu_seqlens != nullptr) != is_varlen(*dims)) return GDR_ERR_INVALID;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const gdr_dims &D = *dims;
    const bool varlen = is_varlen(D);
    const int64_t ns = n_seqs(D);
    // token offsets of the sequences (host data here, so checked on the host)
    std::vector<int64_t> cu((size_t)ns + 1);
    for (int64_t n = 0; n <= ns; ++n) {
        if (!varlen) cu[n] = n * D.T;
        else if (D.flags & GDR_SEQLENS_I64) cu[n] = reinterpret_cast<const int64_t *>(cu_seqlens)[n];
        else cu[n] = cu_seqlens[n];
        if (n > 0 && cu[n] < cu[n - 1]) return GDR_ERR_SEQLENS;
    }
    if (cu[0] != 0 || cu[ns] != D.B * D.T) return GDR_ERR_SEQLENS;

    const size_t es = D.dtype == GDR_F32 ? 4 : 2;
    const size_t rq = (size_t)D.H * D.K * es, rv = (size_t)D.H * D.V * es, rg = (size_t)D.H * 4;
    const size_t rh = (size_t)D.H * D.K * D.V * 4;  // one sequence's state
    const size_t ntok = (size_t)cu[ns];
    const HostGroups G = host_groups(cu, 2 * rq + rv + rg * (beta ? 2 : 1), rh * (h0 ? 1 : 0));
    if (ns == 1 && ntok >= 2 * (size_t)kChunk) {  // one long sequence: pieces of it
        const double total = (double)ntok * (double)(2 * rq + rv + rg * (beta ? 2 : 1));
        const int want = (int)std::min<int64_t>(4, std::llround(total / (32.0 * (1 << 20))));
        if (want >= 2)
            return host_fwd_pieces(D, (int64_t)ntok, want, q, k, v, g, beta, h0, o, ht,
                                   n_segments, st);
    }
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t at = off; off = align_up(off + bytes); return at; };
    const size_t oq = take(ntok * rq), ok = take(ntok * rq), ov = take(ntok * rv);
    const size_t og = take(ntok * rg), ob = take(beta ? ntok * rg : 0);
    const size_t oh0 = take(h0 ? ns * rh : 0), oo = take(ntok * rv), oht = take(ht ? ns * rh : 0);
    const size_t ocu = take(varlen ? (ns + G.count()) * sizeof(int32_t) : 0);
    // each group's cu_seqlens, rebased to its first token (int32: T < 2^31)
    std::vector<int32_t> gcu;
    if (varlen) {
        gcu.reserve((size_t)(ns + G.count()));
        for (int i = 0; i < G.count(); ++i)
            for (int64_t n = G.n[i]; n <= G.n[i + 1]; ++n)
                gcu.push_back((int32_t)(cu[n] - cu[G.n[i]]));
    }
    char *d = nullptr;
    if (lib_malloc(reinterpret_cast<void **>(&d), off ? off : kAlign, st) != cudaSuccess)
        return GDR_ERR_CUDA;

    // Copies in on one stream, the passes on `stream`, copies out on a third:
    // group i + 1 arrives while group i runs and group i - 1 leaves.
    CopyStreams cs{};
    const bool piped = G.count() > 1 && copy_streams(st, &cs) == cudaSuccess;
    cudaStream_t s_in = piped ? cs.in : st, s_out = piped ? cs.out : st;
    std::vector<cudaEvent_t> ev;
    auto new_event = [&](cudaEvent_t *e) {
        if (!piped) return cudaSuccess;
        const cudaError_t r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
        if (r == cudaSuccess) ev.push_back(*e);
        return r;
    };
    auto order = [&](cudaStream_t from, cudaStream_t to) {  // `to` waits for `from`'s work so far
        if (!piped || from == to) return cudaSuccess;
        cudaEvent_t e = nullptr;
        cudaError_t r = new_event(&e);
        if (r == cudaSuccess) r = cudaEventRecord(e, from);
        if (r == cudaSuccess) r = cudaStreamWaitEvent(to, e, 0);
        return r;
    };
    auto h2d = [&](size_t at, const void *src, size_t bytes) {
        return bytes ? cudaMemcpyAsync(d + at, src, bytes, cudaMemcpyHostToDevice, s_in)
                     : cudaSuccess;
    };
    auto d2h = [&](void *dst, size_t at, size_t bytes) {
        return bytes ? cudaMemcpyAsync(dst, d + at, bytes, cudaMemcpyDeviceToHost, s_out)
                     : cudaSuccess;
    };
    const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k),
               *hv = static_cast<const char *>(v), *hg = reinterpret_cast<const char *>(g),
               *hb = reinterpret_cast<const char *>(beta), *hh0 = reinterpret_cast<const char *>(h0);
    char *ho = static_cast<char *>(o), *hht = reinterpret_cast<char *>(ht);
    rc = GDR_OK;
    if (order(st, s_in) != cudaSuccess || order(st, s_out) != cudaSuccess ||
        (varlen && h2d(ocu, gcu.data(), gcu.size() * sizeof(int32_t)) != cudaSuccess))
        rc = GDR_ERR_CUDA;
    // every group's inputs are queued first, so the copies in never wait for
    // the host to launch a pass
    std::vector<cudaEvent_t> arrived((size_t)G.count(), nullptr);
    for (int i = 0; i < G.count() && rc == GDR_OK; ++i) {
        const size_t t0 = (size_t)cu[G.n[i]], nt = (size_t)cu[G.n[i + 1]] - t0;
        const size_t n0 = (size_t)G.n[i], nn = (size_t)(G.n[i + 1] - G.n[i]);
        if (h2d(oq + t0 * rq, hq + t0 * rq, nt * rq) != cudaSuccess ||
            h2d(ok + t0 * rq, hk + t0 * rq, nt * rq) != cudaSuccess ||
            h2d(ov + t0 * rv, hv + t0 * rv, nt * rv) != cudaSuccess ||
            h2d(og + t0 * rg, hg + t0 * rg, nt * rg) != cudaSuccess ||
            (beta && h2d(ob + t0 * rg, hb + t0 * rg, nt * rg) != cudaSuccess) ||
            (h0 && h2d(oh0 + n0 * rh, hh0 + n0 * rh, nn * rh) != cudaSuccess) ||
            new_event(&arrived[i]) != cudaSuccess ||
            (piped && cudaEventRecord(arrived[i], s_in) != cudaSuccess))
            rc = GDR_ERR_CUDA;
    }
    for (int i = 0; i < G.count() && rc == GDR_OK; ++i) {
        const size_t t0 = (size_t)cu[G.n[i]], nt = (size_t)cu[G.n[i + 1]] - t0;
        const size_t n0 = (size_t)G.n[i], nn = (size_t)(G.n[i + 1] - G.n[i]);
        if (piped && cudaStreamWaitEvent(st, arrived[i], 0) != cudaSuccess) {
            rc = GDR_ERR_CUDA;
            break;
        }
        gdr_dims gd = D;
        if (varlen) {
            gd.N = (int32_t)nn;
            gd.T = (int64_t)nt;
            gd.flags &= ~GDR_SEQLENS_I64;
            gd.max_len = 0;  // the group's longest sequence, read from the host table
            for (size_t n = n0; n < n0 + nn; ++n) gd.max_len = std::max(gd.max_len, cu[n + 1] - cu[n]);
        } else {
            gd.B = (int64_t)nn;
        }
        const int32_t *gc = varlen ? reinterpret_cast<const int32_t *>(
                                         d + ocu + (size_t)(G.n[i] + i) * sizeof(int32_t))
                                   : nullptr;
        rc = gdr_chunk_fwd(&gd, d + oq + t0 * rq, d + ok + t0 * rq, d + ov + t0 * rv,
                           reinterpret_cast<float *>(d + og + t0 * rg),
                           beta ? reinterpret_cast<float *>(d + ob + t0 * rg) : nullptr, gc,
                           h0 ? reinterpret_cast<float *>(d + oh0 + n0 * rh) : nullptr,
                           d + oo + t0 * rv,
                           ht ? reinterpret_cast<float *>(d + oht + n0 * rh) : nullptr,
                           n_segments, stream);
        if (rc != GDR_OK) break;
        if (order(st, s_out) != cudaSuccess || d2h(ho + t0 * rv, oo + t0 * rv, nt * rv) != cudaSuccess ||
            (ht && d2h(hht + n0 * rh, oht + n0 * rh, nn * rh) != cudaSuccess))
            rc = GDR_ERR_CUDA;
    }
    // `stream` waits for the copy streams before the block is freed; should
    // that ordering fail, the host waits for them instead
    if (order(s_in, st) != cudaSuccess || order(s_out, st) != cudaSuccess) {
        cudaStreamSynchronize(s_in);
        cudaStreamSynchronize(s_out);
        if (rc == GDR_OK) rc = GDR_ERR_CUDA;
    }
    if (cudaFreeAsync(d, st) != cudaSuccess && rc == GDR_OK) rc = GDR_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess && rc == GDR_OK) rc = GDR_ERR_CUDA;
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
    return rc;
}

}  // extern "C"
