// gdn_noalloc.cu -- inference forward that allocates nothing.
//
// Some callers cannot allocate device memory at the point where they run the
// op: plugin hosts and inference runtimes that forbid allocation while a
// request is being enqueued, code running inside a CUDA stream capture (where
// cudaMalloc is not a legal call), or embedded / real-time hosts whose device
// memory is fixed up front.  For them this file keeps the forward's scratch
// in a file-scope device array that exists for as long as the library is
// loaded, so the entry point needs nothing from the caller beyond its inputs
// and outputs.
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_internal.cuh"

namespace {

// Scratch for the intermediates of the chunked forward (gate sums, norms,
// per-chunk T, W, U, P, Delta and state checkpoints).  Every GPU that loads
// the library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, resolved once per
// device with that device current.  Returns nullptr on failure.
void* scratch_on_current_device(cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        *err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (*err != cudaSuccess) return nullptr;
        g_noalloc_ptr[dev] = ptr;
    }
    return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" size_t gdn_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" gdn_status gdn_forward_noalloc(const gdn_shape* shape, const void* q, const void* k,
                                          const void* v, const void* a, const void* b,
                                          const float* A_log, const float* dt_bias,
                                          const float* state0, const uint8_t* mask, void* o,
                                          float* state_T, void* stream) {
    size_t need = 0, seg = 0;
    gdn_status st = gdn_workspace_bytes(shape, 2, &need);
    if (st == GDN_OK) st = gdn_segment_bytes(shape, 0, &seg);
    if (st != GDN_OK) return st;
    // the automatic segment count's buffers are part of `need`; when only the
    // single-pass scan fits, that runs instead
    const bool fits = need <= kNoAllocScratchBytes;
    if (!fits && need - seg > kNoAllocScratchBytes) return GDN_ERR_WORKSPACE_TOO_SMALL;
    cudaError_t err = cudaSuccess;
    void* scratch = scratch_on_current_device(&err);
    if (scratch == nullptr) return GDN_ERR_CUDA;
    // Nothing in the scratch has to start at zero: every intermediate is
    // written before it is read.  The previous call's contents are simply
    // overwritten.
    if (fits)
        return gdn_forward(shape, q, k, v, a, b, A_log, dt_bias, state0, mask, o, state_T, nullptr,
                           0, scratch, kNoAllocScratchBytes, stream);
    return gdn_forward_segmented(shape, 1, q, k, v, a, b, A_log, dt_bias, state0, mask, o, state_T,
                                 nullptr, 0, scratch, kNoAllocScratchBytes, stream);
}
