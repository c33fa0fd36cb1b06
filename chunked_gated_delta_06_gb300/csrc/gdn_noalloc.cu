// gdn_noalloc.cu -- gdn_chunk_fwd_noalloc: the chunk forward with its scratch
// in a fixed, library-owned device array instead of a caller workspace.
//
// Who needs it: callers that cannot allocate device memory at call time, for
// example code running inside a pre-planned memory arena that forbids new
// allocations after start-up, host plugins that are handed only input and
// output buffers, or latency-critical paths that must not take the device-wide
// synchronisation a cudaMalloc / cudaFree can cause.  They still pass their own
// inputs and outputs; only the scratch moves into the library.
//
// The scratch is one file-scope __device__ array of kScratchBytes (64 MiB).
// Every GPU that loads libgdn.so holds it until the process exits.  Host code
// must not use the array's name as a pointer (on the host it is only a
// stand-in), so the device address is looked up with cudaGetSymbolAddress the
// first time the entry point runs on each device, with that device current,
// and cached per device.  That first call therefore does a little set-up work
// (a symbol lookup, no allocation) and should happen before any stream capture.
//
// Sharing: every call on a device uses the same array, and the array keeps the
// previous call's contents.  Nothing has to start at zero: the forward writes
// every scratch byte it reads (chunk table, status word, WY matrices, per-chunk
// states) earlier in the same call.  Calls whose executions overlap on the GPU
// (different streams, or different host threads, without ordering between
// them) race on the array and give undefined results; order them on one stream.
#include <cuda_runtime.h>
#include <mutex>

#include "../../include/gdn.h"

namespace {

constexpr size_t kScratchBytes = 64u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_fwd_scratch[kScratchBytes];

std::mutex g_lock;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_fwd_scratch on the current device, or nullptr.
void *scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

gdn_status gdn_chunk_fwd_noalloc(const gdn_problem *p, const void *q, const void *k,
                                 const void *v, const float *g, const void *beta,
                                 const float *initial_state, void *o, float *final_state,
                                 gdn_stream_t stream) {
    const size_t need = gdn_chunk_workspace_bytes(p, 0);
    if (need == 0) return GDN_ERR_INVALID_ARG;                // invalid problem
    if (need > kScratchBytes) return GDN_ERR_WORKSPACE_TOO_SMALL;  // beyond the fixed scratch
    void *ws = scratch_on_current_device();
    if (!ws) return GDN_ERR_CUDA;
    return gdn_chunk_fwd(p, q, k, v, g, beta, initial_state, o, final_state, nullptr, ws,
                         kScratchBytes, stream);
}

}  // extern "C"
