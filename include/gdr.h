/*
 * gdr.h -- C ABI of the GB300 chunked gated-delta-rule forward pass.
 *
 * One call computes, for every sequence n and head h, the forward pass of
 * gated delta-rule linear attention over 64-token chunks:
 *
 *   per token   S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *               o_t = scale * S_t q_t,   alpha_t = exp(g_t),  scale = 1/sqrt(K)
 *
 *   per chunk   (the state scan of fla's chunk_gated_delta_rule_fwd_kernel_h,
 *               Kev PR #259 intro; the serial recurrence of cuLA PR #127
 *               "Summary"): chunk-local cumsum G of the log gate g;
 *               A = strictly-lower(diag(beta) * decay-masked K K^T);
 *               T = (I + A)^-1;  W = T diag(beta e^G) K;  U = T diag(beta) V;
 *               then serially over chunks, with h = S^T (K x V, FP32):
 *               v_new = U - W h;   o = scale [(Q e^G) h + causal(Q K^T * decay) v_new]
 *               h <- e^{G_last} h + K^T (v_new * e^{G_last - G}).
 *
 *   segment split (cuLA PR #127 "Summary", "Root cause and implementation":
 *               intra-card context parallelism): each run of whole chunks
 *               emits a local state c_s and a K x K affine transition M_s in
 *               FP32; an ordered pass h_{s+1} = M_s h_s + c_s chains them;
 *               then every segment produces its outputs in parallel.
 *
 *   beta-free   (beta == NULL; the diagonal affine chunk transform of
 *               flash-linear-attention issue #23 "Proposed Dataflow"):
 *               S_t = alpha_t S_{t-1} + v_t k_t^T, the transition is a scalar.
 *
 * Layouts (row-major; q, k, v and o may carry token and head strides,
 * see gdr_dims, everything else is contiguous):
 *   q, k        [B, T, H, K]   dtype GDR_BF16, GDR_F16 or GDR_F32 (same for
 *                              q, k, v, o)
 *   v, o        [B, T, H, V]
 *   g, beta     [B, T, H]      float32; g is the per-token LOG gate (<= 0)
 *   cu_seqlens  [N + 1]        int32 (int64 with GDR_SEQLENS_I64) prefix
 *                              offsets of N packed sequences (varlen:
 *                              dims.N = N > 0, B == 1, T = total)
 *   h0, ht      [Nseq, H, K, V] float32 state h = S^T, Nseq = N (varlen)
 *                              or B (dense); [Nseq, H, V, K] (S itself)
 *                              with GDR_STATE_VK
 *
 * Ownership: every pointer is caller-owned.  gdr_chunk_fwd* take DEVICE
 * pointers, enqueue work on `stream` and return without synchronising; the
 * library keeps no pointer after the call returns.  Scratch is taken
 * stream-ordered on `stream` unless the caller passes a workspace through
 * gdr_chunk_fwd_ex: from a pool per device that the library owns and that
 * keeps freed memory mapped for the next call (gdr_release_cached hands it
 * back), or, while `stream` is being captured into a graph, from the
 * device's default pool (cudaMallocAsync / cudaFreeAsync).
 *
 * Errors: every entry point returns 0 on success or a negative GDR_ERR_*
 * code; arguments are checked before any work is enqueued, so a rejected
 * call leaves the outputs untouched.  cu_seqlens is device data and is not
 * read on the host: it must be non-decreasing with cu[0] = 0 and cu[N] = T.
 * The device checks this before any other work; a malformed table makes the
 * call compute nothing and, if a status word is given (gdr_chunk_fwd_ex),
 * sets it to GDR_ERR_SEQLENS.
 */
#ifndef GDR_H_
#define GDR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st *gdr_stream_t;

/* Element type of q, k, v and o.  GDR_F16 runs on the CUDA-core path (the
 * tensor-core kernels take BF16). */
enum gdr_dtype { GDR_F32 = 0, GDR_BF16 = 1, GDR_F16 = 2 };

/* Return codes. */
enum gdr_status {
    GDR_OK = 0,
    GDR_ERR_INVALID = -1,      /* null pointer, bad size, misaligned row   */
    GDR_ERR_UNSUPPORTED = -2,  /* valid but not implemented (e.g. K > 256) */
    GDR_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed      */
    GDR_ERR_TIMEOUT = -4,      /* device status: a bounded wait expired     */
    GDR_ERR_SEQLENS = -5,      /* device status: cu_seqlens malformed       */
    GDR_ERR_WORKSPACE = -6,    /* caller workspace too small                */
    GDR_ERR_INDEX = -7         /* device status: a state index out of range */
};

/* Layout flags of gdr_dims.flags (bitwise OR; 0 = the defaults above). */
enum gdr_flags {
    GDR_SEQLENS_I64 = 1, /* cu_seqlens holds int64 offsets (pass the pointer
                            through the int32_t * parameter)                */
    GDR_STATE_VK = 2     /* h0, ht and the recurrent state pool are S, laid
                            out [.., H, V, K], instead of h = S^T           */
};

/* Problem size.  Dense layout: N = 0 (there are B sequences of T tokens).
 * Varlen layout: N > 0 sequences packed along T (the total length), B == 1,
 * cu_seqlens required.
 * max_len is a planning hint for the varlen layout, like the max_seqlen
 * argument of varlen attention kernels: the number of tokens of the longest
 * sequence, or 0 when the caller does not know it (the plan then assumes the
 * mean length T / N).  cu_seqlens is device data that the host never reads,
 * so without the hint a batch with one long sequence among many short ones
 * looks uniform and the plan keeps the serial scan, whose time is set by the
 * longest sequence.  The hint only steers the automatic segment count
 * (n_segments = 0); a wrong value costs time, never correctness.  Ignored
 * for the dense layout (every sequence has T tokens). */
typedef struct gdr_dims {
    int64_t B, T, H, K, V, N;
    int32_t dtype;   /* enum gdr_dtype */
    int32_t flags;   /* enum gdr_flags */
    int64_t max_len; /* longest sequence (varlen), 0 = unknown */
    /* Element strides of q, k, v and o: [0] from one token to the next, [1]
     * from one head to the next; {0, 0} means contiguous ({H*K, K} for q and
     * k, {H*V, V} for v and o).  The key / value dimension is always
     * contiguous, and tokens flatten B and T (a dense batch row starts T
     * token strides after the previous one).  So q, k and v may be views of
     * one fused projection, e.g. of a [B, T, 3, H, K] tensor: token stride
     * 3*H*K, head stride K, base pointers K*H elements apart.  Both entries
     * of a pair are zero or both positive; o's two strides must not let two
     * elements share an address (its rows are at least V apart and one of
     * its dimensions spans the other).  The tensor-core kernels read through
     * TMA, which wants 16-byte multiples: a stride of a BF16 tensor that is
     * not a multiple of 8 elements, like a misaligned base, moves the call
     * to the CUDA-core path.  gdr_chunk_fwd_host takes contiguous tensors
     * only (GDR_ERR_UNSUPPORTED otherwise); gdr_chunk_bwd reads q, k, v
     * through their strides and ignores o_stride (its dout and gradients
     * are contiguous). */
    int64_t q_stride[2], k_stride[2], v_stride[2], o_stride[2];
} gdr_dims;

/* Launch plan (A13): chosen per shape from measured timings; every plan of
 * one path gives bit-identical results for a fixed segment count. */
typedef struct gdr_plan {
    int32_t path;       /* 1 = CUDA-core FP32 path, 2 = tensor-core path    */
    int32_t bv;         /* value columns per scan CTA                      */
    int32_t n_segments; /* 1 = serial scan, S > 1 = segment split           */
    int32_t compose;    /* the split's ordered composition (delta rule):
                           0 on CUDA cores (or no split), 1 one pass on the
                           tensor cores, G >= 2 the tensor cores' two-level
                           form in groups of G segments                     */
} gdr_plan;

/* Options of gdr_chunk_fwd_ex.  Zero-initialise, then set what you need. */
typedef struct gdr_options {
    float scale;            /* readout scale; 0 => 1/sqrt(K)                */
    int32_t force_path;     /* 0 => plan; 1 CUDA-core path; 2 tensor cores
                               (FP16 inputs: the kernels read BF16 copies of
                               q, k, v and o is converted back to FP16, in
                               one extra stream-ordered allocation)         */
    int32_t force_bv;       /* 0 => plan; else value columns per scan CTA   */
    void *workspace;        /* device scratch, NULL => stream-ordered alloc */
    size_t workspace_bytes; /* size of `workspace`                          */
    int32_t *status;        /* device int32 status word or NULL; kernels
                               write a GDR_ERR_* code there on a device-side
                               failure (never trap); caller zeroes it        */
    /* Per-launch timing for benchmarks.  If `events` is non-NULL it holds
     * 2 * max_launches cudaEvent_t handles created by the caller; the
     * library records events[2i] just before and events[2i+1] just after its
     * i-th kernel launch on `stream` (launches past max_launches are not
     * recorded), stores the kernel id of launch i in launch_ids[i] (host
     * array, may be NULL; see gdr_kernel_name) and the number of kernel
     * launches of the call in *n_launches (host, may be NULL). */
    void **events;
    int32_t max_launches;
    int32_t *launch_ids;
    int32_t *n_launches;
    /* 0 => the plan's grids.  > 0: the persistent tensor-core kernels (which
     * pull their work items from a counter) run with at most this many
     * CTAs.  Results are identical for every value: each chain or chunk is
     * computed by one CTA in a fixed order whichever CTA takes it (tests of
     * bit-identity across launch configurations). */
    int32_t grid_limit;
} gdr_options;

/*
 * gdr_chunk_fwd -- the forward pass on device buffers (see top of file).
 *   beta        NULL selects the beta-free mode.
 *   cu_seqlens  NULL selects the dense layout.
 *   h0          NULL: zero initial state.   ht  NULL: final state not written.
 *   n_segments  0: plan chooses; 1: serial scan; S > 1: split every sequence
 *               into runs of whole chunks: ceil(longest sequence's chunks /
 *               S) a run on the tensor-core path (a sequence no longer than
 *               that stays one run, taken whole from h0 to ht), ceil(own
 *               chunks / S) on the CUDA-core path.  At most 64 for
 *               the delta rule; at most 4096 in the beta-free mode, where a
 *               count at or above the chunk count gives every chunk its own
 *               segment: the chunk-parallel producer dataflow of
 *               flash-linear-attention issue #23 "Proposed Dataflow" (each
 *               chunk's FP32 contribution computed in parallel, an ordered
 *               scan applying the scalar decays, the output of every chunk
 *               from its boundary state).
 * Returns GDR_OK or GDR_ERR_*.
 */
int gdr_chunk_fwd(const gdr_dims *dims, const void *q, const void *k,
                  const void *v, const float *g, const float *beta,
                  const int32_t *cu_seqlens, const float *h0, void *o,
                  float *ht, int n_segments, gdr_stream_t stream);

/* As gdr_chunk_fwd, with options (scale override, forced plan for tests,
 * caller workspace, device status word).  opt == NULL equals gdr_chunk_fwd. */
int gdr_chunk_fwd_ex(const gdr_dims *dims, const void *q, const void *k,
                     const void *v, const float *g, const float *beta,
                     const int32_t *cu_seqlens, const float *h0, void *o,
                     float *ht, int n_segments, const gdr_options *opt,
                     gdr_stream_t stream);

/*
 * gdr_chunk_fwd_host -- the same pass on HOST buffers (same layouts).  The
 * call copies the inputs to the device, runs gdr_chunk_fwd on `stream`,
 * copies o (and ht) back and synchronises `stream` before returning.
 *   - Batches of 48 MB of input and more are cut into 2 to 4 groups of
 *     whole sequences (batch rows when dense), each run as its own
 *     gdr_chunk_fwd: group i + 1's inputs arrive and group i - 1's outputs
 *     leave while group i runs, on two copy streams of the library ordered
 *     against `stream` with events.  Each sequence's result is the one
 *     gdr_chunk_fwd gives it (plans may differ with the group's size).
 *     One long sequence is cut into pieces of whole chunks instead, run as
 *     consecutive passes, each starting from the state the previous one
 *     ended with (kept on the device): the same result up to rounding
 *     (identical bits with n_segments = 1).
 *   - cu_seqlens is host data here and is checked on the host: a table
 *     that is not non-decreasing from 0 to T returns GDR_ERR_SEQLENS before
 *     any work is enqueued.
 *   - Pinned host memory gives asynchronous copies; pageable memory works
 *     but copies synchronously.  Device buffers are stream-ordered
 *     allocations from the library's pool (see Ownership above).
 */
int gdr_chunk_fwd_host(const gdr_dims *dims, const void *q, const void *k,
                       const void *v, const float *g, const float *beta,
                       const int32_t *cu_seqlens, const float *h0, void *o,
                       float *ht, int n_segments, gdr_stream_t stream);

/*
 * gdr_chunk_fwd_noalloc -- gdr_chunk_fwd that allocates nothing.  The pages
 * describe no counterpart; this entry point exists for callers that cannot
 * let a library allocate device memory while they run (engines that reserve
 * nearly all HBM up front and treat a later allocation as a failure,
 * frameworks that own the allocator, code where an allocation call is not
 * allowed or would block).  Its scratch is a 64 MiB array inside the library,
 * held on every GPU that loads the library until the process exits.
 *   - Same arguments, layouts and results as gdr_chunk_fwd; device buffers,
 *     work enqueued on `stream`, no synchronisation.
 *   - Returns GDR_ERR_WORKSPACE, computing nothing, when the problem needs
 *     more than 64 MiB of scratch (gdr_workspace_size tells in advance).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call outside stream capture.
 *   - All calls share the one array: calls that overlap on the GPU (several
 *     streams or host threads) race on it; order them.  No part of the
 *     scratch has to start at zero.
 */
int gdr_chunk_fwd_noalloc(const gdr_dims *dims, const void *q, const void *k,
                          const void *v, const float *g, const float *beta,
                          const int32_t *cu_seqlens, const float *h0, void *o,
                          float *ht, int n_segments, gdr_stream_t stream);

/*
 * gdr_recurrent_fwd -- the per-token recurrence itself (the formula at the
 * top of the file, token by token), for serving: a decode step or a few
 * tokens a sequence, where a 64-token chunk would be mostly padding (the
 * "question rows" with states of their own, Kev PR #259 "Not covered").
 * Every sequence takes its initial state from a row of a caller-owned pool,
 * runs its tokens in order and writes its final state back into that row.
 *   dims, q, k, v, g, beta, cu_seqlens, o   as for gdr_chunk_fwd (device
 *                 pointers; beta NULL selects the beta-free mode).
 *   state         [n_states, H, K, V] float32 pool of states h = S^T, read
 *                 and written in place (device).
 *   state_indices [Nseq] int32 pool row of each sequence (device), or NULL
 *                 for row n.  The rows of one call must be distinct.
 *   status        device int32 word or NULL: an index outside [0, n_states)
 *                 skips its sequence and sets GDR_ERR_INDEX there (malformed
 *                 cu_seqlens: GDR_ERR_SEQLENS); the caller zeroes it.
 * FP32 arithmetic for both input types; scale = 1/sqrt(K).  Work is enqueued
 * on `stream`; no allocation, no synchronisation.
 */
int gdr_recurrent_fwd(const gdr_dims *dims, const void *q, const void *k,
                      const void *v, const float *g, const float *beta,
                      const int32_t *cu_seqlens, float *state, int64_t n_states,
                      const int32_t *state_indices, void *o, int32_t *status,
                      gdr_stream_t stream);

/*
 * gdr_chunk_bwd -- the backward pass: the gradients of
 * L = <do, o> + <dht, ht> with respect to q, k, v, g, beta and h0, where o
 * and ht are what gdr_chunk_fwd computes from the same inputs.  The state
 * gradient runs backward over the chunks (the reverse dH recurrence of the
 * flash-linear-attention ABC issue #23 pages, "Problem" and "Proposed
 * Dataflow" step 4; gradients dQ/dK/dV and of the states, its
 * "Fixture-First Correctness Contract"), through the chunked form's WY
 * factors.  Two routes:
 *   - tensor-core route (BF16 inputs, K = V = 128, delta rule): the
 *     forward recompute is the tensor-core forward's (per-chunk records,
 *     the chain keeping the BF16 state mirror and v_new of each chunk),
 *     then the reverse scan and every per-chunk gradient, all on tcgen05
 *     with FP32 accumulation: BF16 operands in the scans (the forward's own
 *     rounding), FP32 operands of the per-chunk products as BF16 hi + lo
 *     pairs; every gradient lies within 1e-2 (relative L2) of the exact
 *     one.  Long sequences split into segments like the forward pass (the
 *     reverse scan composed from dht to dh0 over the transposed forward
 *     maps), at the forward's segment rule unless n_segments says;
 *   - CUDA-core route (every input type): FP32 arithmetic throughout, with
 *     a segment split of long sequences.
 *   The plan takes the tensor-core route where it applies;
 *   opt->force_path 1 or 2 picks the route.
 *   dims, q, k, v, g, beta, cu_seqlens, h0   as for gdr_chunk_fwd (device).
 *   dout    [B,T,H,V] dL/do, the input dtype.
 *   dht     [Nseq,H,K,V] FP32 dL/dht (state layout of h0), or NULL for 0.
 *   dq, dk  [B,T,H,K], dv [B,T,H,V] outputs in the input dtype.
 *   dg      [B,T,H] FP32 output;  dbeta [B,T,H] FP32 output, required
 *           exactly when beta is given (NULL in the beta-free mode).
 *   dh0     [Nseq,H,K,V] FP32 output (state layout of h0), or NULL.
 *   n_segments  0 = automatic; S > 1 splits every sequence into S runs of
 *           whole chunks for both the forward recompute and the reverse
 *           scan: each step of the reverse recurrence is affine in the
 *           state gradient, so per segment a pre-scan produces its offset
 *           and K x K map, an ordered composition runs from the last segment
 *           to the first (from dht to dh0), and an output pass rebuilds the
 *           per-chunk gradients (the pages' "Proposed Dataflow" step 4).
 *   opt     NULL, or gdr_options with scale, status, workspace (at least
 *           gdr_bwd_workspace_size bytes), the launch events, force_path
 *           (0 plan, 1 CUDA-core route, 2 tensor-core route) and
 *           grid_limit; force_bv must be 0.
 * The pass recomputes the forward states and then runs the backward
 * kernels; work is enqueued on `stream`, not synchronised.  Every gradient is written for every token of every
 * sequence; results are bit-identical from run to run.
 */
int gdr_chunk_bwd(const gdr_dims *dims, const void *q, const void *k,
                  const void *v, const float *g, const float *beta,
                  const int32_t *cu_seqlens, const float *h0,
                  const void *dout, const float *dht, void *dq, void *dk,
                  void *dv, float *dg, float *dbeta, float *dh0,
                  int n_segments, const gdr_options *opt, gdr_stream_t stream);

/* Bytes of device scratch gdr_chunk_bwd needs for this problem (beta_free
 * != 0 for the beta-free mode; n_segments as passed to gdr_chunk_bwd),
 * enough for either route (force_path 0, 1 or 2).  0 on invalid arguments. */
size_t gdr_bwd_workspace_size(const gdr_dims *dims, int beta_free, int n_segments);

/* Bytes of device scratch gdr_chunk_fwd_ex needs for this problem
 * (beta_free != 0 for the beta-free mode).  0 on invalid arguments. */
size_t gdr_workspace_size(const gdr_dims *dims, int beta_free,
                          int n_segments);

/* The plan gdr_chunk_fwd would use (host-only lookup, no GPU needed). */
int gdr_plan_query(const gdr_dims *dims, int beta_free, int n_segments,
                   gdr_plan *out);

/* Name of a kernel id reported through gdr_options.launch_ids ("?" if
 * unknown). */
const char *gdr_kernel_name(int id);

/* Static description of a return code. */
const char *gdr_error_string(int code);

/* Hands the device memory that the library's pools keep between calls back
 * to the driver, on every device the library has allocated on.  Memory that
 * enqueued work still uses is kept.  Returns GDR_OK or GDR_ERR_CUDA. */
int gdr_release_cached(void);

/* Library version as major*10000 + minor*100 + patch. */
int gdr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H_ */
