// Reduce-side kernels: ring-order reduce-scatter + average (optionally with
// norm partials, optionally written back into every slab = all-reduce),
// the norm of the owner chunks, its finalisation, and the all-gather.
//
// All streaming kernels use the same mapping: chunk-major, and inside chunk c
// a grid-stride loop over 8-element groups, so every thread of a warp works on
// the same chunk (uniform ring order) and consecutive threads touch
// consecutive 16- or 32-byte words of every slab (coalesced).  Block row y
// takes chunks y, y + gridDim.y, ... (one row for large arenas, N rows when
// the chunks are small enough to run side by side).
#include <mutex>
#include <unordered_map>

#include "device.cuh"
#include "internal.h"

namespace dpz {

namespace {

thread_local const char* g_last_kernel = "";

struct DevInfo {
    int sms = 0;
};

std::mutex g_mu;
std::unordered_map<int, DevInfo> g_dev;
std::unordered_map<const void*, int> g_occ;   // kernel -> resident blocks per SM

int blocks_per_sm(const void* fn)
{
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_occ.find(fn);
        if (it != g_occ.end()) return it->second;
    }
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, kBlock, 0) != cudaSuccess || nb < 1)
        nb = 1;
    std::lock_guard<std::mutex> lk(g_mu);
    g_occ[fn] = nb;
    return nb;
}

}  // namespace

int device_sms()
{
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_dev.find(dev);
    if (it != g_dev.end()) return it->second.sms;
    DevInfo d;
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (d.sms <= 0) d.sms = 1;
    g_dev[dev] = d;
    return d.sms;
}

// Grid of a chunk-major streaming kernel.  When the blocks that one chunk
// needs, times N, fit in `waves` resident waves, every chunk gets its own
// row of blocks (grid.y = N) and the chunks run side by side; otherwise a
// single row walks the chunks in turn (grid.y = 1).
dim3 grid_chunks(const void* fn, int64_t threads_per_chunk, int N, int waves)
{
    const int64_t wave = (int64_t)device_sms() * blocks_per_sm(fn) * (waves < 1 ? 1 : waves);
    int64_t per_chunk = (threads_per_chunk + kBlock - 1) / kBlock;
    if (per_chunk < 1) per_chunk = 1;
    if (per_chunk * N <= wave) return dim3((unsigned)per_chunk, (unsigned)N, 1);
    return dim3((unsigned)(per_chunk < wave ? per_chunk : wave), 1, 1);
}

const char* last_kernel_name() { return g_last_kernel; }
void set_last_kernel_name(const char* n) { g_last_kernel = n; }

// ------------------------------------------------------------------ kernels
//
// Loop shape shared by the streaming kernels: for each chunk c of the block's
// row, each warp walks warp-iterations wb = first, first + stride, ... (32
// consecutive groups of 8 elements, all lanes together), lane l taking group
// wb + l.
// Kernels that produce norm partials write, for every warp-iteration, the sum
// of squares of its 256 averaged elements (fixed shuffle tree) into the slot
// of that segment, so the partials do not depend on the grid.

// Segments a warp takes per iteration: two when the loaded words of both fit
// comfortably in registers (more bytes in flight per thread), else one.
template <int GDT, int NT>
struct SegsPerIter {
    static constexpr int kRegsPerSlab = GDT == 0 ? 8 : 4;
    static constexpr int value = (NT > 0 && NT * kRegsPerSlab <= 32) ? 2 : 1;
};

// Ring-order reduce + average of every chunk.  ALL = false: chunk c goes to
// slab c only (reduce-scatter).  ALL = true: to every slab (all-reduce).
// SUMSQ: per-segment sums of squares of the averages.  NT > 0: N == NT known
// at compile time; NT == 0: any N, read from n_rt.
template <int GDT, int NT, bool ALL, bool SUMSQ>
__global__ void __launch_bounds__(kBlock)
k_reduce(char* __restrict__ grads, int64_t P, int64_t C, int n_rt, Avg avg,
         WsHeader* __restrict__ hdr, double* __restrict__ partials)
{
    using G = Group<GDT>;
    constexpr int ES = G::kBytes;
    constexpr int U = SegsPerIter<GDT, NT>::value;
    const int N = NT > 0 ? NT : n_rt;
    const int64_t slab = P * ES;
    const int64_t groups = C / kGroup;
    const int64_t segs = segments_per_chunk(C);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int lane = threadIdx.x & 31;
    const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x - lane;
    if (SUMSQ && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) hdr->arrive = 0u;
    for (int c = blockIdx.y; c < N; c += gridDim.y) {
        constexpr int NS = NT > 0 ? NT : 1;
        const char* src[NS];
        if constexpr (NT > 0) ring_sources<NT>(grads, slab, c, src);
        for (int64_t wb0 = first * U; wb0 < groups; wb0 += stride * U) {
            typename G::Raw raw[U][NS];
            if constexpr (NT > 0) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t gi = wb0 + 32 * u + lane;
                    if (gi < groups) {
                        const int64_t off = (c * C + gi * kGroup) * ES;
#pragma unroll
                        for (int j = 0; j < NT; ++j) raw[u][j] = G::load_raw(src[j] + off);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t wb = wb0 + 32 * u;
                const int64_t gi = wb + lane;
                float ss = 0.0f;
                if (gi < groups) {
                    const int64_t off = (c * C + gi * kGroup) * ES;
                    float acc[8];
                    if constexpr (NT > 0)
                        fold_loaded<GDT, NT>(raw[u], acc);
                    else
                        ring_fold<GDT>(grads, slab, off, c, N, acc);
                    average8<GDT>(acc, avg);
                    if (SUMSQ) ss = sumsq8(acc);
                    const typename G::Raw out = G::pack(acc);
                    if (ALL) {
                        if constexpr (NT > 0) {
#pragma unroll
                            for (int j = 0; j < NT; ++j) G::store_raw(const_cast<char*>(src[j]) + off, out);
                        } else {
                            for (int r = 0; r < N; ++r) G::store_raw(grads + r * slab + off, out);
                        }
                    } else {
                        G::store_raw(grads + c * slab + off, out);
                    }
                }
                if (SUMSQ && wb < groups) {
                    const float t = warp_sum_f32(ss);
                    if (lane == 0) partials[c * segs + wb / 32] = (double)t;
                }
            }
        }
    }
}

// Ring-order reduce + average of the arena elements [lo, hi), for a bucket
// of gradients that is ready before the rest.  Rank r's value of element e is
// read at src + r*src_stride + (e - lo) and the average of element e (chunk
// c = e / C) is written at dst + c*dst_stride + e (elements of the gradient
// dtype).  In place in the arena: src = arena + lo, src_stride = P, dst =
// arena, dst_stride = P.  From a staging bucket into compact shards (ZeRO-2):
// src = staging [N][hi - lo], src_stride = hi - lo, dst = shards [P],
// dst_stride = 0.  Block row y takes the part of the range inside chunk
// c_first + y.  With SUMSQ the range must start and end on 256-element
// segment boundaries of its chunks; the partials of those segments are then
// the ones the whole-arena kernels write.
template <int GDT, int NT, bool SUMSQ>
__global__ void __launch_bounds__(kBlock)
k_reduce_range(const char* __restrict__ src, int64_t src_stride, char* __restrict__ dst,
               int64_t dst_stride, int64_t lo, int64_t hi, int64_t C, int n_rt, int c_first,
               Avg avg, WsHeader* __restrict__ hdr, double* __restrict__ partials)
{
    using G = Group<GDT>;
    constexpr int ES = G::kBytes;
    const int N = NT > 0 ? NT : n_rt;
    const int64_t segs = segments_per_chunk(C);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int lane = threadIdx.x & 31;
    const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x - lane;
    const int64_t sslab = src_stride * ES;
    if (SUMSQ && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) hdr->arrive = 0u;
    const int c = c_first + (int)blockIdx.y;
    const int64_t plo = lo > c * C ? lo : c * C;
    const int64_t phi = hi < (c + 1) * C ? hi : (c + 1) * C;
    if (plo >= phi) return;
    const int64_t groups = (phi - plo) / kGroup;
    const int64_t seg0 = (plo - c * C) / kSegment;          // first segment of the piece
    for (int64_t wb = first; wb < groups; wb += stride) {
        const int64_t gi = wb + lane;
        float ss = 0.0f;
        if (gi < groups) {
            const int64_t e = plo + gi * kGroup;
            const int64_t soff = (e - lo) * ES;
            float acc[8];
            if constexpr (NT > 0) {
                typename G::Raw raw[NT];
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    int r = c + 1 + j;
                    if (r >= NT) r -= NT;
                    raw[j] = G::load_raw(src + r * sslab + soff);
                }
                fold_loaded<GDT, NT>(raw, acc);
            } else {
                ring_fold<GDT>(src, sslab, soff, c, N, acc);
            }
            average8<GDT>(acc, avg);
            if (SUMSQ) ss = sumsq8(acc);
            G::store_raw(dst + (c * dst_stride + e) * ES, G::pack(acc));
        }
        if (SUMSQ) {
            const float t = warp_sum_f32(ss);
            if (lane == 0) partials[c * segs + seg0 + wb / 32] = (double)t;
        }
    }
}

// Segments per warp-iteration for the single-stream kernels (norm of the
// owner chunks, all-gather): one 16- or 32-byte load per lane and segment, so
// several segments keep enough bytes in flight.
template <int DT>
struct StreamSegs {
    static constexpr int value = DT == 0 ? 2 : 4;
};

// Sums of squares of the owner chunks (chunk c of slab c), per segment.
template <int GDT>
__global__ void __launch_bounds__(kBlock)
k_norm_owned(const char* __restrict__ grads, int64_t P, int64_t C, int N,
             WsHeader* __restrict__ hdr, double* __restrict__ partials)
{
    constexpr int ES = Group<GDT>::kBytes;
    constexpr int U = StreamSegs<GDT>::value;
    const int64_t slab = P * ES;
    const int64_t groups = C / kGroup;
    const int64_t segs = segments_per_chunk(C);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int lane = threadIdx.x & 31;
    const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x - lane;
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) hdr->arrive = 0u;
    for (int c = blockIdx.y; c < N; c += gridDim.y) {
        const char* base = grads + c * slab + c * C * ES;
        for (int64_t wb0 = first * U; wb0 < groups; wb0 += stride * U) {
            typename Group<GDT>::Raw raw[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t gi = wb0 + 32 * u + lane;
                if (gi < groups) raw[u] = Group<GDT>::load_raw(base + gi * kGroup * ES);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t wb = wb0 + 32 * u;
                float ss = 0.0f;
                if (wb + lane < groups) {
                    float x[8];
                    Group<GDT>::unpack(raw[u], x);
                    ss = sumsq8(x);
                }
                if (wb < groups) {
                    const float t = warp_sum_f32(ss);
                    if (lane == 0) partials[c * segs + wb / 32] = (double)t;
                }
            }
        }
    }
}

// Sum of the n segment partials in a fixed order, independent of the device:
// block b of F adds the contiguous range [b*L, (b+1)*L) (L = ceil(n/F)) into
// stage1[b]; the last block to arrive (an arrival counter, not an ordering)
// adds stage1[0..F-1] and writes sumsq, the norm and *norm_out.  No block
// waits for another.
__global__ void __launch_bounds__(kFinalThreads)
k_norm_finalize(WsHeader* __restrict__ hdr, double* __restrict__ stage1,
                const double* __restrict__ partials, int64_t n, float* __restrict__ norm_out)
{
    const int F = gridDim.x;
    const int64_t L = (n + F - 1) / F;
    const int64_t lo = (int64_t)blockIdx.x * L;
    const int64_t hi = lo + L < n ? lo + L : n;
    double v = 0.0;
    for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) v += partials[i];
    v = block_sum(v);
    __shared__ bool is_last;
    if (threadIdx.x == 0) {
        stage1[blockIdx.x] = v;
        __threadfence();
        const unsigned prev = atomicAdd(&hdr->arrive, 1u);
        is_last = prev == (unsigned)(F - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    double w = 0.0;
    for (int i = threadIdx.x; i < F; i += blockDim.x) w += __ldcg(&stage1[i]);
    w = block_sum(w);
    if (threadIdx.x == 0) {
        const float nrm = __double2float_rn(__dsqrt_rn(w));
        hdr->sumsq = w;
        hdr->norm = nrm;
        hdr->nparts = (uint32_t)n;
        hdr->arrive = 0u;
        if (norm_out) *norm_out = nrm;
    }
}

// Chunk c of slab c -> chunk c of every other slab.
template <int WDT>
__global__ void __launch_bounds__(kBlock)
k_allgather(char* __restrict__ w, int64_t P, int64_t C, int N)
{
    constexpr int ES = Group<WDT>::kBytes;
    constexpr int U = StreamSegs<WDT>::value;
    const int64_t slab = P * ES;
    const int64_t groups = C / kGroup;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int lane = threadIdx.x & 31;
    const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x - lane;
    for (int c = blockIdx.y; c < N; c += gridDim.y) {
        const int64_t c0 = c * C * ES;
        for (int64_t wb0 = first * U; wb0 < groups; wb0 += stride * U) {
            typename Group<WDT>::Raw x[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t gi = wb0 + 32 * u + lane;
                if (gi < groups) x[u] = Group<WDT>::load_raw(w + c * slab + c0 + gi * kGroup * ES);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t gi = wb0 + 32 * u + lane;
                if (gi < groups)
                    for (int r = 0; r < N; ++r)
                        if (r != c) Group<WDT>::store_raw(w + r * slab + c0 + gi * kGroup * ES, x[u]);
            }
        }
    }
}

// ------------------------------------------------------------------ launchers

template <int GDT, int NT, bool ALL, bool SUMSQ>
static cudaError_t reduce_t(const Arena& a, const Avg& avg, void* grads, void* ws, cudaStream_t s)
{
    auto fn = k_reduce<GDT, NT, ALL, SUMSQ>;
    constexpr int U = SegsPerIter<GDT, NT>::value;
    const dim3 grid = grid_chunks((const void*)fn, (a.C / kGroup + U - 1) / U, a.N, 2);
    set_last_kernel_name(ALL ? "dpz_allreduce_avg" : SUMSQ ? "dpz_rs_avg_sumsq" : "dpz_rs_avg");
    fn<<<grid, kBlock, 0, s>>>(static_cast<char*>(grads), a.P, a.C, a.N, avg,
                               static_cast<WsHeader*>(ws), SUMSQ ? ws_partials(ws) : nullptr);
    return cudaGetLastError();
}

template <int GDT, bool ALL, bool SUMSQ>
static cudaError_t reduce_n(const Arena& a, const Avg& avg, void* grads, void* ws, cudaStream_t s)
{
    switch (a.N) {
    case 1: return reduce_t<GDT, 1, ALL, SUMSQ>(a, avg, grads, ws, s);
    case 2: return reduce_t<GDT, 2, ALL, SUMSQ>(a, avg, grads, ws, s);
    case 4: return reduce_t<GDT, 4, ALL, SUMSQ>(a, avg, grads, ws, s);
    case 8: return reduce_t<GDT, 8, ALL, SUMSQ>(a, avg, grads, ws, s);
    default: return reduce_t<GDT, 0, ALL, SUMSQ>(a, avg, grads, ws, s);
    }
}

cudaError_t launch_reduce(const Arena& a, const Avg& avg, void* grads, bool all_slabs, void* ws,
                          cudaStream_t s)
{
    const bool sumsq = ws != nullptr && !all_slabs;
    if (a.gdt == 2) {
        if (all_slabs) return reduce_n<2, true, false>(a, avg, grads, ws, s);
        return sumsq ? reduce_n<2, false, true>(a, avg, grads, ws, s)
                     : reduce_n<2, false, false>(a, avg, grads, ws, s);
    }
    if (a.gdt == 1) {
        if (all_slabs) return reduce_n<1, true, false>(a, avg, grads, ws, s);
        return sumsq ? reduce_n<1, false, true>(a, avg, grads, ws, s)
                     : reduce_n<1, false, false>(a, avg, grads, ws, s);
    }
    if (all_slabs) return reduce_n<0, true, false>(a, avg, grads, ws, s);
    return sumsq ? reduce_n<0, false, true>(a, avg, grads, ws, s)
                 : reduce_n<0, false, false>(a, avg, grads, ws, s);
}

template <int GDT, int NT, bool SUMSQ>
static cudaError_t range_t(const Arena& a, const Avg& avg, const RangeArgs& g, void* ws,
                           cudaStream_t s)
{
    auto fn = k_reduce_range<GDT, NT, SUMSQ>;
    const int c_first = (int)(g.lo / a.C);
    const int c_last = (int)((g.hi - 1) / a.C);
    const int pieces = c_last - c_first + 1;
    int64_t longest = a.C < g.hi - g.lo ? a.C : g.hi - g.lo;
    dim3 grid = grid_chunks((const void*)fn, longest / kGroup, pieces, 2);
    grid.y = (unsigned)pieces;
    set_last_kernel_name(SUMSQ ? "dpz_rs_range_sumsq" : "dpz_rs_range");
    fn<<<grid, kBlock, 0, s>>>(static_cast<const char*>(g.src), g.src_stride,
                               static_cast<char*>(g.dst), g.dst_stride, g.lo, g.hi, a.C, a.N,
                               c_first, avg, static_cast<WsHeader*>(ws),
                               SUMSQ ? ws_partials(ws) : nullptr);
    return cudaGetLastError();
}

template <int GDT, bool SUMSQ>
static cudaError_t range_n(const Arena& a, const Avg& avg, const RangeArgs& g, void* ws,
                           cudaStream_t s)
{
    switch (a.N) {
    case 1: return range_t<GDT, 1, SUMSQ>(a, avg, g, ws, s);
    case 2: return range_t<GDT, 2, SUMSQ>(a, avg, g, ws, s);
    case 4: return range_t<GDT, 4, SUMSQ>(a, avg, g, ws, s);
    case 8: return range_t<GDT, 8, SUMSQ>(a, avg, g, ws, s);
    default: return range_t<GDT, 0, SUMSQ>(a, avg, g, ws, s);
    }
}

cudaError_t launch_reduce_range(const Arena& a, const Avg& avg, const RangeArgs& g, void* ws,
                                cudaStream_t s)
{
    const bool sumsq = ws != nullptr;
    switch (a.gdt) {
    case 0: return sumsq ? range_n<0, true>(a, avg, g, ws, s) : range_n<0, false>(a, avg, g, ws, s);
    case 1: return sumsq ? range_n<1, true>(a, avg, g, ws, s) : range_n<1, false>(a, avg, g, ws, s);
    default:
        return sumsq ? range_n<2, true>(a, avg, g, ws, s) : range_n<2, false>(a, avg, g, ws, s);
    }
}

cudaError_t launch_norm_owned(const Arena& a, const void* grads, void* ws, cudaStream_t s)
{
    set_last_kernel_name("dpz_norm_owned");
    const char* g = static_cast<const char*>(grads);
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    if (a.gdt != 0) {      // both bf16 modes store bf16 averages
        const dim3 grid = grid_chunks((const void*)k_norm_owned<1>,
                                      a.C / kGroup / StreamSegs<1>::value, a.N, 2);
        k_norm_owned<1><<<grid, kBlock, 0, s>>>(g, a.P, a.C, a.N, hdr, ws_partials(ws));
    } else {
        const dim3 grid = grid_chunks((const void*)k_norm_owned<0>,
                                      a.C / kGroup / StreamSegs<0>::value, a.N, 2);
        k_norm_owned<0><<<grid, kBlock, 0, s>>>(g, a.P, a.C, a.N, hdr, ws_partials(ws));
    }
    return cudaGetLastError();
}

cudaError_t launch_norm_finalize(const Arena& a, void* ws, float* norm_out, cudaStream_t s)
{
    set_last_kernel_name("dpz_norm_finalize");
    const int64_t n = int64_t(a.N) * segments_per_chunk(a.C);
    // blocks: a function of n only, so the summation order is fixed
    int64_t F = (n + 2047) / 2048;
    if (F > kFinalBlocks) F = kFinalBlocks;
    if (F < 1) F = 1;
    k_norm_finalize<<<(int)F, kFinalThreads, 0, s>>>(static_cast<WsHeader*>(ws), ws_stage1(ws),
                                                     ws_partials(ws), n, norm_out);
    return cudaGetLastError();
}

cudaError_t launch_allgather(const Arena& a, void* weights, cudaStream_t s)
{
    set_last_kernel_name("dpz_allgather");
    char* w = static_cast<char*>(weights);
    if (a.wdt == 1) {
        const dim3 grid = grid_chunks((const void*)k_allgather<1>,
                                      a.C / kGroup / StreamSegs<1>::value, a.N, 2);
        k_allgather<1><<<grid, kBlock, 0, s>>>(w, a.P, a.C, a.N);
    } else {
        const dim3 grid = grid_chunks((const void*)k_allgather<0>,
                                      a.C / kGroup / StreamSegs<0>::value, a.N, 2);
        k_allgather<0><<<grid, kBlock, 0, s>>>(w, a.P, a.C, a.N);
    }
    return cudaGetLastError();
}

}  // namespace dpz
