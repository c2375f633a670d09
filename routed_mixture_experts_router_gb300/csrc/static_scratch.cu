// moe_layer_forward_static: the whole layer forward for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run the layer: code inside a real-time or latency-critical loop that
// must not take the allocator's locks or risk an out-of-memory failure
// mid-request, plugins hosted by a runtime that owns all device memory and
// hands out none, or tools linked against this library without a memory
// manager of their own.  They still own their inputs and outputs; this entry
// point gives them the layer's scratch (routing results, bucketing, SwiGLU
// activations) from a fixed region compiled into the library.
//
// The region is a file-scope __device__ array of MOE_STATIC_SCRATCH_BYTES
// (8 MiB), so every GPU that loads the library holds those 8 MiB until the
// process exits.  In host code the array's name is only a host-side stand-in
// for the symbol, not a device address; the first call on each device looks
// the real address up with cudaGetSymbolAddress while that device is current
// and caches it, so that first call should happen before any stream capture.
// The cache is per device and lock-free (several host threads may make that
// first call at once; they all store the same address).  It does not survive
// cudaDeviceReset: the reset unloads the module, so a process that resets a
// device must not call this entry point on it again.
// All calls share the one region and it keeps the last call's contents: two
// calls whose work overlaps on the GPU (different streams, or different host
// threads, on the same device) race on it.  Nothing in the region needs to
// start at zero: every call writes each part of it before reading it.
#include <atomic>
#include <limits.h>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];  // zero-initialised (static storage)

}  // namespace

extern "C" MOE_API int moe_layer_forward_static(const float* x, int T, const moe_layer_w* w, int act, int flags,
                                                int residual, float* out, int32_t* status, void* stream) {
    // Argument checks first, exactly as moe_layer_forward makes them: with a
    // null workspace it returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for
    // bad arguments, MOE_OK for T == 0, and MOE_ERR_WORKSPACE only when the
    // arguments are fine, in every case before it enqueues anything.
    const int rc = moe_layer_forward(x, T, w, act, flags, residual, out, nullptr, nullptr, nullptr, nullptr, 0,
                                     status, stream);
    if (rc != MOE_ERR_WORKSPACE) return rc;
    const size_t need = moe_workspace_size(T, w, act, flags);
    if (need == 0) return MOE_ERR_INVALID_ARG;
    if (need > (size_t)MOE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;  // T too large for the fixed region
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    void* base = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (base == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        g_scratch_addr[dev].store(p, std::memory_order_release);
        base = p;
    }
    return moe_layer_forward(x, T, w, act, flags, residual, out, nullptr, nullptr, nullptr, base,
                             (size_t)MOE_STATIC_SCRATCH_BYTES, status, stream);
}
