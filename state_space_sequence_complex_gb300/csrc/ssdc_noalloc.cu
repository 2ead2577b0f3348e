// Forward pass for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// moment they run the scan: code inside a custom memory pool or allocator
// hook, real-time paths that forbid allocator calls, or embedders whose
// memory budget is fixed up front. ssd_complex_fwd_noalloc gives them the
// staged paths (exact fp32, or TF32 with staged chunk states) with the
// per-chunk state workspace held in one file-scope device array instead of a
// caller buffer or an allocation. Every GPU that loads the library holds this
// array until the process exits.
#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/ssdc.h"

namespace {

constexpr size_t kScratchBytes = SSDC_NOALLOC_SCRATCH_BYTES;

// The scratch workspace. Its name is a host-side stand-in in host code: the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of g_scratch on the current device, looked up once per
// device (the first call on a device does this).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSDC_ERR_CUDA;
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return SSDC_ERR_CUDA;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return SSDC_OK;
}

}  // namespace

extern "C" int ssd_complex_fwd_noalloc(ssdc_cin x, ssdc_cin A, ssdc_cin B_t, ssdc_cin C_t, const float* dt,
                                       ssdc_dims dims, int chunk_size, ssdc_cout y, ssdc_cout final_state,
                                       cudaStream_t stream) {
    if (dims.precision != SSDC_PREC_FP32 && dims.precision != SSDC_PREC_TF32_STAGED) return SSDC_ERR_UNSUPPORTED;
    const int rc = ssd_complex_fwd_supported(dims, chunk_size);
    if (rc != SSDC_OK) return rc;
    const size_t need = ssd_complex_fwd_workspace_bytes(dims, chunk_size);
    if (need == 0) return SSDC_ERR_INVALID;
    if (need > kScratchBytes) return SSDC_ERR_TOO_LARGE;
    void* ws = nullptr;
    const int arc = scratch_address(&ws);
    if (arc != SSDC_OK) return arc;
    // The staged paths need no zeroed workspace: every chunk state is written
    // before it is read, and the call clears the status word on the stream.
    return ssd_complex_fwd_ws(x, A, B_t, C_t, dt, dims, chunk_size, y, final_state, ws, kScratchBytes, stream);
}

// The status word is the first int of the array (the workspace layout of the
// staged paths); it is copied out by symbol, with no allocation.
extern "C" int ssd_complex_noalloc_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SSDC_ERR_CUDA;
    int status = SSDC_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&status, g_scratch, sizeof(int), 0, cudaMemcpyDeviceToHost) != cudaSuccess)
        return SSDC_ERR_CUDA;
    return status;
}
