// ss_fwd_noalloc: the forward selective scan for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the scan:
// code replayed inside a captured CUDA graph, a custom allocator that owns
// all device memory and must not be bypassed, or an embedding runtime that
// forbids allocation on its hot path.  The regular ss_fwd asks such a caller
// for a workspace whenever the sequence is cut into several time chunks; this
// entry point instead keeps that workspace (the per-chunk carry summaries) in
// a fixed, file-scope device array that the library owns.  The caller still
// passes every input and output.
//
// The array is SS_FWD_NOALLOC_MAX_SCRATCH_BYTES (2 MiB).  Every GPU that
// loads this library reserves it until the process exits.  All calls share
// it, so two calls whose work overlaps on the GPU (different streams, no
// ordering between them) race on it; calls on one stream are safe.  It keeps
// the contents of the last call: every summary the kernels read is first
// written by the same call, so nothing in it needs clearing.
//
// Host code only sees a host-side stand-in for the array's name, never its
// device address.  The address is therefore looked up once per device with
// cudaGetSymbolAddress and cached: the first call on a device that uses the
// scratch (a problem cut into several time chunks) does this set-up with
// that device current.  That first call should come before any stream
// capture begins.  The cache is keyed by device ordinal and assumes the
// runtime's one primary context per device for the life of the process: after
// cudaDeviceReset (which destroys that context and unloads the library's
// device code) the cached address is stale, so a process that resets a device
// must not call this entry point on it again.
#include <cuda_runtime.h>

#include <mutex>

#include "ss.h"
#include "common.cuh"
#include "kernels.h"

using namespace ss;

namespace {

constexpr size_t kScratchBytes = SS_FWD_NOALLOC_MAX_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_fwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_fwd_scratch on the current device (looked up once per device).
int scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SS_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_fwd_scratch) != cudaSuccess || ptr == nullptr) return SS_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return SS_OK;
}

}  // namespace

extern "C" int ss_fwd_noalloc(const void* u, const void* delta, const float* A, const void* B, const void* C,
                              const float* D, const void* z, const float* delta_bias, int softplus, void* y,
                              float* last_state, int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype,
                              void* stream) {
    // Argument checks of ss_fwd, with the built-in scratch in place of a caller workspace.
    if (Bsz < 0 || L < 0 || Dch < 0 || N < 0) return SS_ERR_INVALID_PROBLEM;
    const size_t need = ss_fwd_workspace_bytes(Bsz, L, Dch, N, dtype);
    if (need > kScratchBytes) return SS_ERR_WORKSPACE_TOO_SMALL;
    const bool empty = Bsz == 0 || L == 0 || Dch == 0;
    if (need == 0 || empty) {
        // no chunk carries: the regular entry point needs no workspace either
        return ss_fwd(u, delta, A, B, C, D, z, delta_bias, softplus, y, last_state, Bsz, L, Dch, N, dtype, nullptr, 0,
                      stream);
    }
    void* scratch = nullptr;
    const int rc = scratch_for_current_device(&scratch);
    if (rc != SS_OK) return rc;
    return ss_fwd(u, delta, A, B, C, D, z, delta_bias, softplus, y, last_state, Bsz, L, Dch, N, dtype, scratch,
                  kScratchBytes, stream);
}
