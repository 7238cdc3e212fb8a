// Fixed device scratch for dp_grad_global_norm_static: the global-norm
// kernels' partial sums live in one file-scope device array instead of a
// workspace the caller allocates.
//
// Every GPU that loads this library keeps the array (kStaticScratchBytes) for
// the life of the process.  All calls share it and it keeps whatever the last
// call wrote; the only field that must start at zero, the finalisation's
// arrival counter, is cleared by the partial-sum kernel at the start of every
// call, and every partial, first-stage sum and the status word are written
// before they are read in the same call.  Two calls whose kernels overlap on
// the GPU (different streams without ordering between them) therefore race
// on the same scratch.
#include <cuda_runtime.h>

#include <atomic>

#include "internal.h"

namespace dpz {

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;   // 4 MiB
constexpr int kMaxDevices = 256;

// The array's device address per device, from the last call outside a stream
// capture on that device.
std::atomic<void*> g_addr[kMaxDevices];

}  // namespace

static __device__ __align__(256) unsigned char g_norm_scratch[kStaticScratchBytes];

size_t static_scratch_bytes() { return kStaticScratchBytes; }

// The array's device address on the current device.  In host code the name
// g_norm_scratch is only a stand-in for the symbol, so the address comes from
// cudaGetSymbolAddress, with the device current.  It is looked up again on
// every call made outside a stream capture (a device reset loads the module
// anew, and the array may then sit elsewhere); while `s` is capturing, the
// lookup is not made and the last one on the device is used, or the call
// fails if there was none.
cudaError_t static_scratch_address(void** ptr, cudaStream_t s)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        (void)cudaGetLastError();     // the query's own error is not the caller's
        cs = cudaStreamCaptureStatusActive;
    }
    if (cs != cudaStreamCaptureStatusNone) {
        void* p = g_addr[dev].load(std::memory_order_acquire);
        if (p == nullptr) return cudaErrorStreamCaptureUnsupported;
        *ptr = p;
        return cudaSuccess;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_norm_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev].store(p, std::memory_order_release);
    *ptr = p;
    return cudaSuccess;
}

}  // namespace dpz
