/* Device build of the seeded input generator (see gen.h). Fills GPU buffers
 * with exactly the values the host build produces. */
#include <cuda_runtime.h>
#include <stdint.h>

#include "gen.h"

namespace {

template <bool BF16>
__global__ void fill_kernel(void* out, int64_t start, int64_t count,
                            uint64_t key, int kind, double scale,
                            double scale_tail)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < count;
         j += stride) {
        float x = gen_value(kind, key, (uint64_t)(start + j), scale, scale_tail);
        if (BF16)
            static_cast<uint16_t*>(out)[j] = gen_trunc_bf16(x);
        else
            static_cast<float*>(out)[j] = x;
    }
}

int launch(bool bf16, void* out, int64_t start, int64_t count, uint64_t seed,
           uint64_t stream_id, int kind, double scale, double scale_tail,
           void* stream)
{
    if (count <= 0) return 0;
    if (!out) return 1;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (count + 255) / 256;
    if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
    const uint64_t key = gen_key(seed, stream_id);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (bf16)
        fill_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(out, start, count, key,
                                                          kind, scale, scale_tail);
    else
        fill_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(out, start, count, key,
                                                           kind, scale, scale_tail);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace

extern "C" {

__attribute__((visibility("default"))) int gen_fill_f32_dev(
    float* out, int64_t start, int64_t count, uint64_t seed, uint64_t stream_id,
    int kind, double scale, double scale_tail, void* stream)
{
    return launch(false, out, start, count, seed, stream_id, kind, scale,
                  scale_tail, stream);
}

__attribute__((visibility("default"))) int gen_fill_bf16_dev(
    uint16_t* out, int64_t start, int64_t count, uint64_t seed,
    uint64_t stream_id, int kind, double scale, double scale_tail, void* stream)
{
    return launch(true, out, start, count, seed, stream_id, kind, scale,
                  scale_tail, stream);
}

}  // extern "C"
