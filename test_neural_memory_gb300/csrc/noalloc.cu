// ttm_titans_fwd_noalloc: the Titans / linear-memory scan for callers that
// cannot allocate device memory.
//
// The tensor-core scan needs device scratch for its per-chunk coefficients.
// ttm_titans_fwd takes that scratch from the caller.  Some callers have no way
// to provide it: code running where allocation is forbidden or unavailable
// (a plugin handed only its input and output buffers, a host that pre-plans
// all device memory up front, or a context where a cudaMalloc would break an
// allocation-free guarantee).  This entry point serves them from a fixed
// block of scratch compiled into the library instead.
//
// The block lives in a file-scope __device__ array, so every GPU that loads
// the library holds it (kNoallocScratchBytes) until the process exits, and
// every call on a device shares it.  Host code may not use the array's name
// as a device address (on the host it only names a stand-in), so the device
// address is looked up once per device with cudaGetSymbolAddress while that
// device is current.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "../../include/ttm.h"

namespace {

constexpr size_t kNoallocScratchBytes = TTM_NOALLOC_SCRATCH_BYTES;   // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices];

// Device address of the scratch block on the current device (set up on the
// first call per device), or nullptr on failure.
void* scratch_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

int ttm_titans_fwd_noalloc(int B, int H, int T, int dk, int dv, int chunk, int dtype,
                           const void* q, const void* k, const void* v, const float* eta,
                           const float* theta, const float* alpha, const float* W0,
                           const float* S0, int w0_shared_over_batch, void* z, float* W_out,
                           float* S_out, void* stream) {
    // Size check first, on the host: a call that needs more scratch than the
    // block holds is refused before anything touches the GPU.
    const size_t need = ttm_linear_workspace_size(B, H, T, dk, dv, chunk, dtype);
    if (need > kNoallocScratchBytes) return TTM_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (need > 0) {
        scratch = scratch_for_current_device();
        if (!scratch) return TTM_ERR_CUDA;
    }
    // The scratch needs no clearing: the coefficient pre-pass writes every
    // record the scan reads before the scan reads it.
    return ttm_titans_fwd(B, H, T, dk, dv, chunk, dtype, q, k, v, eta, theta, alpha, W0, S0,
                          w0_shared_over_batch, z, W_out, S_out, scratch,
                          need > 0 ? kNoallocScratchBytes : 0, stream);
}

}  // extern "C"
