// noalloc.cu -- gdr_chunk_fwd_noalloc: the forward pass with its scratch in a
// fixed device array that the library owns, for callers that must not
// allocate device memory.
//
// Who needs this.  Some callers cannot let a library allocate GPU memory at
// call time: serving engines that reserve nearly all HBM for caches at start
// and treat any later allocation as a failure; code inside frameworks that
// own the allocator and forbid side allocations; and code that runs where a
// CUDA allocation call is not allowed or would block.  gdr_chunk_fwd takes
// its scratch with cudaMallocAsync, and gdr_chunk_fwd_ex needs the caller to
// supply scratch, which such callers may not be able to do either.  This
// entry point needs neither: its scratch is a file-scope __device__ array of
// kNoAllocScratchBytes that every GPU loading the library holds until the
// process exits.
//
// The device address of that array is taken once per device, on the first
// call made with that device current (cudaGetSymbolAddress; the host-side
// name of a __device__ array is not a device address).  Make that first call
// outside any stream capture.  Every call shares the one array: calls whose
// work overlaps on the GPU (other streams, other host threads) race on it
// and must be ordered by the caller.  No word of the scratch has to start at
// zero: every word a call reads is written earlier by the same call.
#include <mutex>

#include "gdr_internal.cuh"
#include "gdr_launch.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on
// first use per device).  Returns nullptr on a CUDA error.
void *scratch_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int gdr_chunk_fwd_noalloc(const gdr_dims *dims, const void *q, const void *k,
                                     const void *v, const float *g, const float *beta,
                                     const int32_t *cu_seqlens, const float *h0, void *o,
                                     float *ht, int n_segments, gdr_stream_t stream) {
    if (!dims || !q || !k || !v || !g || !o) return GDR_ERR_INVALID;
    if ((cu_seqlens != nullptr) != (dims->N > 0)) return GDR_ERR_INVALID;
    // the scratch of the path this call will run (misaligned pointers move a
    // tensor-core shape to the CUDA-core path, which needs more); invalid or
    // unsupported arguments return the code gdr_chunk_fwd would
    gdr_plan plan;
    size_t need = 0;
    const int rc = gdr::plan_for_call(*dims, beta == nullptr, n_segments, nullptr, q, k, v, o,
                                      &plan, &need);
    if (rc != GDR_OK) return rc;
    if (need > kNoAllocScratchBytes) return GDR_ERR_WORKSPACE;  // problem too large
    void *scratch = scratch_for_current_device();
    if (!scratch) return GDR_ERR_CUDA;
    gdr_options opt{};
    opt.workspace = scratch;
    opt.workspace_bytes = kNoAllocScratchBytes;
    return gdr_chunk_fwd_ex(dims, q, k, v, g, beta, cu_seqlens, h0, o, ht, n_segments, &opt,
                            stream);
}
