// Segment bounds of a split scan: how a sequence of nc chunks is cut into
// runs of whole chunks, shared by the chunk table (which fixes the length
// for the call), the chain and pre-scan kernels and the compositions.
//
// Two rules.  Own length: every sequence is cut into S runs of
// ceil(nc / S) chunks (the last one shorter).  Common length (the
// tensor-core delta forward): every sequence is cut into runs of
// L = ceil(longest / S) chunks, so a sequence of at most L chunks is one
// run, taken whole by the output pass from h0 to ht with no pre-scan and no
// composition, and a batch whose longest sequence dwarfs the rest splits
// that one alone.
#pragma once

#include "gdr_internal.cuh"

namespace gdr {

// Workspace::n_chunks slot after the chain counters: L under the common
// rule (at least 1), 0 under the own-length rule; written by the chunk
// table, read by every kernel after it.
constexpr int kCtrSegLen = kNumCtr;
constexpr int kNumCtrSlots = kNumCtr + 1;

// seq_order sorts sequences by chunk count in kOrderBuckets buckets, the top
// one holding every sequence of kOrderBuckets - 1 chunks or more: below that
// count the order is exactly descending.
constexpr int kOrderBuckets = 128;

__device__ __forceinline__ int seg_len(const Workspace &ws) { return ws.n_chunks[kCtrSegLen]; }

// Chunks per run of a sequence of nc chunks.
__device__ __forceinline__ int seg_per(const Workspace &ws, int nc) {
    const int L = seg_len(ws);
    return L ? L : (nc + ws.n_segments - 1) / ws.n_segments;
}

// Under the common rule: whether a sequence of nc chunks (per a run) runs
// whole, and every sequence after it in seq_order does too.
__device__ __forceinline__ bool whole_from_here(const Workspace &ws, int nc, int per) {
    return seg_len(ws) != 0 && nc <= per && nc < kOrderBuckets - 1;
}

}  // namespace gdr
