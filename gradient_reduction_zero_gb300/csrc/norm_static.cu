// Fixed device scratch for dp_grad_global_norm_static: the global-norm
// kernels' partial sums live in one file-scope device array instead of a
// workspace the caller allocates.
//
// Every GPU that loads this library keeps the array (kStaticScratchBytes) for
// the life of the process.  All calls share it and it keeps whatever the last
// call wrote; the only field that must start at zero, the finalisation's
// arrival counter, is cleared by the partial-sum kernel at the start of every
// call.  Two calls whose kernels overlap on the GPU (different streams without
// ordering between them) therefore race on the same scratch.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace dpz {

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;   // 4 MiB
constexpr int kMaxDevices = 256;

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

}  // namespace

static __device__ __align__(256) unsigned char g_norm_scratch[kStaticScratchBytes];

size_t static_scratch_bytes() { return kStaticScratchBytes; }

// The array's device address on the current device.  In host code the name
// g_norm_scratch is only a stand-in for the symbol, so the address is looked
// up with cudaGetSymbolAddress, once per device, with that device current.
cudaError_t static_scratch_address(void** ptr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_norm_scratch);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
    }
    *ptr = g_addr[dev];
    return cudaSuccess;
}

}  // namespace dpz
