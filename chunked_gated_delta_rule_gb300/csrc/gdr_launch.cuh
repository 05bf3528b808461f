// gdr_launch.cuh -- host-side declarations shared by the runtime's
// translation units: workspace layout, kernel ids, the launch recorder and
// the launch functions of every kernel family (each defined in its own .cu
// file).  Device code does not include this header, so editing it leaves
// the kernels' sources untouched.
#pragma once

#include "gdr_internal.cuh"

namespace gdr {

// Byte layout of the workspace for one problem.
struct WorkspaceLayout {
    size_t off_tab, off_seq0, off_nchunks, off_order, off_G, off_W, off_U, off_hpre,
        off_vnew, off_segM, off_segC, off_segH, off_segD, off_rec, off_segMimg, off_grpA, off_grpD,
        total;
    int64_t max_chunks;
    int grp_size;     // G of the two-level tensor-core composition (0: one level)
    bool seg_images;  // transition images: the composition runs on the tensor cores
};

// How the delta rule's segment composition runs on the tensor-core paths:
// kind 0 on CUDA cores (compose_mt), 1 the single ordered tensor-core pass,
// 2 its two-level form with groups of grp_size segments; cost_us the
// estimate of the cheapest (a model of GB300 timings, from the shape and
// the device's SM count, never from a launch's grid).
struct ComposePlan {
    int kind, grp_size;
    double cost_us;
};
// common: one segment length for every sequence (the tensor-core forward),
// so only the sequences longer than it take part (split_seqs).
ComposePlan compose_plan(const gdr_dims &d, int S, bool common);
// Sequences a split into S segments of one common length (ceil(longest / S)
// chunks) cuts, from the host's length statistics: the longest alone when
// the others' mean fits one segment, else all of them.
int64_t split_seqs(const gdr_dims &d, int S);

// path 1: CUDA-core path (chunk table, G, W, U, h_pre, v_new, segments);
// path 2: tensor-core path (chunk table, records and segment summaries);
// path 3: the tensor-core backward's forward recompute (chunk table and
// records; its images are in the backward's own scratch).
WorkspaceLayout workspace_layout(const gdr_dims &d, bool beta_free, int n_segments, int path);
Workspace carve_workspace(void *base, const WorkspaceLayout &L, int n_segments);

// The plan a forward call runs (the shape's plan, on the CUDA-core path when
// the tensor-core kernels cannot take the pointers) and its scratch bytes;
// GDR_OK or the code the call itself would return for these arguments.
int plan_for_call(const gdr_dims &d, bool beta_free, int n_segments, const gdr_options *opt,
                  const void *q, const void *k, const void *v, const void *o, gdr_plan *plan,
                  size_t *ws_bytes);

// Kernel ids reported through gdr_options.launch_ids.
enum KernelId {
    kKChunkTable = 0,
    kKPrep = 1,
    kKScanSerial = 2,
    kKScanPre = 3,
    kKCompose = 4,
    kKScanSegOut = 5,
    kKOutput = 6,
    kKTcSerial = 7,
    kKTcPre = 8,
    kKTcSegOut = 9,
    kKTcPrep = 10,
    kKTcGlaSerial = 11,
    kKTcGlaPre = 12,
    kKTcGlaSegOut = 13,
    kKComposeScalar = 14,
    kKTcPreDual = 15,
    kKBwdGram = 16,
    kKBwdScan = 17,
    kKBwdLk = 18,
    kKBwdLocal = 19,
    kKBwdPre = 20,
    kKBwdSegOut = 21,
    kKBwdMaps = 22,
    kKConvertIn = 23,
    kKConvertOut = 24,
    kKTcRecompute = 25,
    kKTcBwdScan = 26,
    kKTcBwdGrad = 27,
    kKTcSegRecompute = 28,
    kKTcBwdPre = 29,
    kKTcBwdSegOut = 30,
    kKTcCompose = 31,
    kKTcComposeGroups = 32,
    kKTcComposeTop = 33,
    kKTcComposeFill = 34,
    kKNumIds
};

// Records caller-provided events around each launch (benchmark hook).
struct LaunchRecorder {
    cudaEvent_t *events = nullptr;
    int max_launches = 0;
    int32_t *ids = nullptr;
    int count = 0;
    cudaStream_t st = nullptr;
    cudaError_t begin(int id) {
        if (ids && count < max_launches) ids[count] = id;
        if (events && count < max_launches) return cudaEventRecord(events[2 * count], st);
        return cudaSuccess;
    }
    cudaError_t end() {
        cudaError_t e = cudaSuccess;
        if (events && count < max_launches) e = cudaEventRecord(events[2 * count + 1], st);
        ++count;
        return e;
    }
};

// ---- CUDA-core FP32 path (any supported shape; arithmetic in FP32) --------
// common: fix one segment length for the call, ceil(longest / S) chunks
// (gdr_segments.cuh), else every sequence is cut by its own length.
cudaError_t simt_chunk_table(const Problem &p, const Workspace &ws, bool common,
                             cudaStream_t st);
cudaError_t simt_prep(const Problem &p, const Workspace &ws, cudaStream_t st);
// mode 0: serial scan (h0 -> ht), stores hpre / vnew
// mode 1: segment pre-scan (zero / identity start), stores segC / segM / segD
// mode 2: segment output pass (start from segH), stores hpre / vnew
cudaError_t simt_scan(const Problem &p, const Workspace &ws, int mode, int bv,
                      cudaStream_t st);
cudaError_t simt_compose(const Problem &p, const Workspace &ws, int bv,
                         cudaStream_t st);
cudaError_t simt_output(const Problem &p, const Workspace &ws, cudaStream_t st);
// FP16 <-> BF16 element copies (n elements), for FP16 inputs on the
// tensor-core path.
cudaError_t convert_f16_to_bf16(const void *src, void *dst, int64_t n, cudaStream_t st);
cudaError_t convert_bf16_to_f16(const void *src, void *dst, int64_t n, cudaStream_t st);
// Backward pass on CUDA cores after the CUDA-core forward recompute (G,
// W, hpre, vnew in ws).
cudaError_t simt_bwd(const Problem &p, const Workspace &ws, const BwdArgs &a, const BwdWs &bw,
                     cudaStream_t st, LaunchRecorder &rec);
// The reverse state-gradient scan on the tensor cores (BF16, K = V = 128,
// delta rule).  mode 0: serial from dht to dh0, the E^T and dV'^T images
// into ws.bwd_lkimg; 1: segment pre-scan from E = 0, each segment's offset
// into ws.segC (segment s of nseg non-empty ones in slot nseg - 1 - s); 2:
// segment output pass from the composed ends in ws.segH (the same slots),
// the images.
cudaError_t tc_bwd_scan(const Problem &p, const Workspace &ws, int mode, const float *dht,
                        float *dh0, const void *dout, cudaStream_t st);
// The reverse scan's segment maps from the forward recompute's (ws.segM):
// the transposes, in reversed slots, for the composition from the last
// segment to the first.
cudaError_t bwd_maps(const Problem &p, const Workspace &ws, float *segMb, cudaStream_t st);
// Every per-chunk gradient of the backward on the tensor cores (dq, dk, dv,
// dbeta, dg), from the images in ws.bwd_lkimg (h, E, v_new, dV', T), dO, q,
// k, v and G (ws.G).
cudaError_t tc_bwd_grad(const Problem &p, const Workspace &ws, const BwdArgs &a,
                        cudaStream_t st);
// Composition for the delta rule with K <= 128 and V % 32 == 0 (both paths):
// bulk-copied transposed transitions, 32 value columns per CTA.
bool compose_mt_supported(const Problem &p);
cudaError_t compose_mt(const Problem &p, const Workspace &ws, cudaStream_t st);
// Composition for the delta rule at K = V = 128 on the tensor cores
// (tc_compose.cu): level 0 the single ordered pass over every segment; with
// ws.grp_size = G > 0, level 1 the group transitions and offsets, level 2
// the pass over the groups, level 3 the states inside every group.
bool compose_tc_supported(const Problem &p);
cudaError_t compose_tc(const Problem &p, const Workspace &ws, int level, cudaStream_t st);
// A9 for the beta-free form (scalar transitions d_s).
cudaError_t compose_scalar(const Problem &p, const Workspace &ws, cudaStream_t st);

// ---- tensor-core path (BF16, K = V = 128, delta rule) ---------------------
// Shapes and pointer alignment the tensor-core kernels take.
bool tc_supported(const Problem &p);
// Beta-free mode on tensor cores (BF16, K in {128, 256}, V % 128 == 0).
bool tc_gla_supported(const Problem &p);
cudaError_t tc_gla(const Problem &p, const Workspace &ws, int mode, cudaStream_t st);
// A2-A5 for every (chunk, head) in parallel -> per-chunk records.
cudaError_t tc_prep(const Problem &p, const Workspace &ws, cudaStream_t st);
// mode 0: serial scan + output (h0 -> ht); 1: segment pre-scan (c_s and M_s
// chains); 2: segment output pass from the composed segment states; 3: the
// backward's recompute (serial from h0, the h mirror and v_new images
// stored, no output); 4: the same per segment from the composed states.
cudaError_t tc_chain(const Problem &p, const Workspace &ws, int mode, cudaStream_t st);
// The per-token recurrence from (and back into) rows of a state pool.
cudaError_t recurrent_fwd(const Problem &p, float *state, int64_t n_states,
                          const int32_t *state_idx, cudaStream_t st);
// Segment pre-scan with both summaries (c_s and M_s) of a chain in one CTA.
// tc_chain's mode 1 runs them as separate chains, which is faster while both
// kinds fit one wave (prescan_split_kinds).
cudaError_t tc_prescan(const Problem &p, const Workspace &ws, cudaStream_t st);

}  // namespace gdr
