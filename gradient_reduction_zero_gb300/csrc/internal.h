// Internal interface between the C-ABI layer (api.cpp) and the kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "dpz.h"

#if defined(__CUDACC__)
#define DPZ_HD __host__ __device__
#else
#define DPZ_HD
#endif

namespace dpz {

constexpr int kGroup = 8;             // elements a thread handles at once
constexpr int kBlock = 256;           // threads per block of the streaming kernels
constexpr int kSegment = 32 * kGroup; // elements per norm partial (one warp-iteration)
constexpr int kFinalBlocks = 256;     // most blocks of the norm finalisation
constexpr int kFinalThreads = 512;
constexpr size_t kWsHeaderBytes = 256;

// Start of the workspace (device memory).  Then kFinalBlocks doubles of
// first-stage sums, then one double per 256-element segment of every chunk.
struct WsHeader {
    double sumsq;      // global sum of squares of the averaged gradient
    float norm;        // sqrt(sumsq) rounded to float
    uint32_t nparts;   // segment partials the last norm used
    uint32_t arrive;   // finalisation blocks done (reset by every producer)
    uint32_t status;   // DPZ_STATUS_* bits: written whole by every norm
                       // finalisation, bit DPZ_STATUS_UPDATE_SKIPPED set by the
                       // update kernels that follow it
};
static_assert(offsetof(WsHeader, status) == DPZ_WS_STATUS_OFFSET,
              "the status word sits where dpz.h says");

// A segment partial is a sum of squares: +0 or more, +inf or NaN, never
// negative.  A staged kernel that gives up on a tile writes one of these
// negative markers into the tile's partial slots instead, and the
// finalisation turns them into a NaN norm and status bits.
constexpr double kPartialNormSkipped = -1.0;   // the tile was not read
constexpr double kPartialStepSkipped = -2.0;   // nor was its update written
// Their high 32-bit words (the low words are 0); no sum of squares, not even a
// NaN one, has either as its high word.
constexpr int kPartialNormSkippedHi = (int)0xBFF00000u;
constexpr int kPartialStepSkippedHi = (int)0xC0000000u;

DPZ_HD inline int64_t segments_per_chunk(int64_t C) { return (C + kSegment - 1) / kSegment; }

inline size_t ws_bytes_for(int64_t P, int N)
{
    const int64_t segs = int64_t(N) * segments_per_chunk(P / N);
    size_t b = kWsHeaderBytes + sizeof(double) * (size_t(kFinalBlocks) + size_t(segs));
    return (b + 255) / 256 * 256;
}

inline double* ws_stage1(void* ws)
{
    return reinterpret_cast<double*>(static_cast<char*>(ws) + kWsHeaderBytes);
}

inline double* ws_partials(void* ws) { return ws_stage1(ws) + kFinalBlocks; }

// One arena: N slabs of P elements, chunk C = P / N.
struct Arena {
    int64_t P;
    int64_t C;
    int N;
    int gdt;   // 0 = fp32, 1 = bf16
    int wdt;
};

// Divisor data for the average R(acc / N).
struct Avg {
    float fN;      // (float)N
    float invN;    // 1/N, exact when N is a power of two
    int pow2;      // multiply by invN (same result as dividing) when set
};

// AdamW constants, computed once on the host.
struct AdamArgs {
    float lr, b1, b2, omb1, omb2, bc1, bc2, eps, wd;
    float clip;    // > 0: scale by clip/norm when norm > clip
};

// Which source the AdamW kernel reads the averaged gradient from.
enum class AdamSrc { kLoadOwner, kFold };

// Kernel launchers.  Each launches exactly one kernel on `s` and returns the
// launch status.  Kernels that produce norm partials write one per
// 256-element segment of every chunk (N * segments_per_chunk(C) in chunk
// order), independent of their launch configuration, so the norm is a
// function of the data alone.
cudaError_t launch_reduce(const Arena& a, const Avg& avg, void* grads, bool all_slabs,
                          void* ws, cudaStream_t s);
cudaError_t launch_norm_owned(const Arena& a, const void* grads, void* ws, cudaStream_t s);

// A range [lo, hi) of arena elements to reduce: rank r's value of element e
// at src + r*src_stride + (e - lo), the average of element e (chunk c) stored
// at dst + c*dst_stride + e (strides and offsets in elements).
// max_ctas > 0 caps the blocks of the launch (each then loops over its part
// of the range); 0: one pass.
struct RangeArgs {
    const void* src;
    int64_t src_stride;
    void* dst;
    int64_t dst_stride;
    int64_t lo, hi;
    int max_ctas;
};
cudaError_t launch_reduce_range(const Arena& a, const Avg& avg, const RangeArgs& g, void* ws,
                                cudaStream_t s);
// Every launcher uses programmatic stream serialisation (launch_kernel with
// early = true) and every kernel begins with pdl_enter (bulk.cuh): its blocks
// may be placed while the kernel before it on the stream still runs, and wait
// for that kernel's writes before they touch memory.
cudaError_t launch_norm_finalize(const Arena& a, void* ws, float* norm_out, cudaStream_t s);
// norm_out: where the step's norm went (the bulk-copy staged update writes
// NaN there if it gives up on a tile; may be NULL).
cudaError_t launch_adamw(const Arena& a, const Avg& avg, const AdamArgs& h, AdamSrc src,
                         bool bcast, bool store_avg, void* grads, float* master, float* m,
                         float* v, void* weights, void* ws, cudaStream_t s,
                         int64_t avg_stride, float* norm_out = nullptr);
cudaError_t launch_allgather(const Arena& a, void* weights, cudaStream_t s);

// The whole step without clip, norm included, in one launch of a thread-block
// cluster (up to 8 CTAs, four warps per segment), for arenas of at most
// kSmallStepSegments 256-element segments (adamw.cu).  Same results, bit for
// bit, as the fold kernel plus launch_norm_finalize.
constexpr int64_t kSmallStepSegments = 32;
bool zero1_fits_small_step(const Arena& a);
cudaError_t launch_zero1_small(const Arena& a, const Avg& avg, const AdamArgs& h, bool store_avg,
                               void* grads, float* master, float* m, float* v, void* weights,
                               void* ws, float* norm_out, cudaStream_t s);

// AdamW + cast + all-gather from the stored averages (element e of chunk c
// at grads + c*avg_stride + e), staged through shared memory by bulk copies
// (staged.cu, as is launch_norm_owned).  A tile that does not arrive within
// the wait limit is reported in the workspace's status word and as a NaN in
// norm_out, and sets the device error flag that read_and_clear_pipeline_error
// returns.
cudaError_t launch_adamw_bcast_tma(const Arena& a, const AdamArgs& h, const void* grads,
                                   int64_t avg_stride, float* master, float* m, float* v,
                                   void* weights, void* ws, float* norm_out, cudaStream_t s);
// The step without clip, staged the same way (compile-time fold for N <= 8,
// run-time fold beyond) where zero1_fused_staged holds: N <= 8, or N slab
// tiles that fit shared memory with enough of them resident per SM to keep
// the stream going; other arenas use k_adamw's fold.  ws: norm partials when
// not NULL.
bool zero1_fused_staged(const Arena& a);
cudaError_t launch_zero1_fused_tma(const Arena& a, const Avg& avg, const AdamArgs& h,
                                   bool store_avg, void* grads, float* master, float* m, float* v,
                                   void* weights, void* ws, cudaStream_t s);
cudaError_t read_and_clear_pipeline_error(unsigned* flag);
// Launch one staged kernel (DPZ_SELFTEST_* of dpz.h) on the one-tile arena
// laid out in `buf` (DPZ_SELFTEST_BUF_BYTES), with a barrier that never
// completes and a short wait bound, so that its wait runs out.  Where the
// kernel writes partials, the caller then launches the norm finalisation.
cudaError_t launch_staged_timeout_selftest(int kernel, void* buf, cudaStream_t s);
// The self-test's arena (N = 1, P = 8, bf16 gradients and weights) and its
// layout in the buffer: the workspace at 0, norm_out, then gradients, master,
// m, v and weights at +0, +32, +64, +96 and +128 from kSelftestGrads.
constexpr Arena kSelftestArena{8, 8, 1, 1, 1};
constexpr size_t kSelftestNormOut = 2560;
constexpr size_t kSelftestGrads = 2816;
// Counts the float inputs whose average division by N differs from an
// IEEE division (the whole 2^32 pattern space).
cudaError_t launch_selftest_division(const Avg& avg, unsigned long long* mismatches,
                                     cudaStream_t s);


// The fixed device scratch of dp_grad_global_norm_static (norm_static.cu):
// its size in bytes, and its device address on the current device (looked up
// again on every call made outside a stream capture on `s`).
size_t static_scratch_bytes();
cudaError_t static_scratch_address(void** ptr, cudaStream_t s);

#if defined(__CUDACC__)
// Launch `kernel` on `s` through cudaLaunchKernelEx.  early: with
// programmatic stream serialisation, so that the kernel may begin once the
// blocks of the previous kernel on the stream have exited, before that
// kernel's writes are flushed; the kernel must then execute
// griddepcontrol.wait before it touches anything that earlier work writes or
// reads.
// cluster > 0: the grid's CTAs form thread-block clusters of that many CTAs
// along x (grid.x a multiple of it).
template <class... KArgs, class... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, bool early, unsigned cluster, Args... args)
{
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (early) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 0) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = n > 0 ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
#endif

// Name of the kernel the last launcher call on this thread launched.
const char* last_kernel_name();
void set_last_kernel_name(const char* name);

// Blocks of kBlock threads for a one-shot grid over `segments` 256-element
// segments, U per warp.
inline unsigned blocks_for_segments(int64_t segments, int U)
{
    const int64_t per_block = int64_t(U) * (kBlock / 32);
    const int64_t b = (segments + per_block - 1) / per_block;
    return (unsigned)(b < 1 ? 1 : b);
}

}  // namespace dpz
