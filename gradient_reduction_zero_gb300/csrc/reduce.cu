// Reduce-side kernels: ring-order reduce-scatter + average (optionally with
// norm partials, optionally written back into every slab = all-reduce), the
// finalisation of the norm, and the all-gather.  (The standalone norm of the
// owner chunks is staged through shared memory: staged.cu.)
//
// All streaming kernels run one-shot grids over the chunk-major list of
// 256-element segments (device.cuh): every thread of a warp works on the
// same chunk (uniform ring order) and consecutive lanes touch consecutive 16-
// or 32-byte words of every slab (coalesced).
#include "bulk.cuh"
#include "device.cuh"
#include "internal.h"

namespace dpz {

namespace {

thread_local const char* g_last_kernel = "";

}  // namespace

const char* last_kernel_name() { return g_last_kernel; }
void set_last_kernel_name(const char* n) { g_last_kernel = n; }

// ------------------------------------------------------------------ kernels
//
// Kernels that produce norm partials write, for every segment, the sum of
// squares of its averaged elements (fixed shuffle tree) into that segment's
// slot, so the partials do not depend on the launch configuration.

// Blocks per SM the reduce kernels are compiled for.  A bf16 lane loads 16
// bytes per slab, so a warp keeps only N x 512 bytes in flight: at 32
// registers eight blocks (64 warps) stay resident, which took the N = 3
// reduce-scatter from 94 to 98 % of the copy peak and left N = 2 and 4-8
// unchanged.  fp32 lanes load 32 bytes per slab; capping the compile-time
// folds cost 0.3-3 % at N = 3-8, so they keep the compiler's choice, as does
// the all-reduce, which also stores N slabs.  The fp32 run-time fold held 88
// to 110 registers (two blocks per SM); at 64 (four blocks) it went from 98 to
// 109 % at N = 12 and from 99 to 108 % at N = 16.  bf16 at N = 2 takes two
// segments per warp (ReduceSegsPerWarp), which does not fit 32 registers: six
// blocks of 40.
template <int GDT, int NT, bool ALL>
struct ReduceBlocksPerSm {
    static constexpr int value = ALL ? 1 : GDT != 0 ? (NT == 2 ? 6 : 8) : NT == 0 ? 4 : 1;
};

// The same for the range kernel, whose extra index arithmetic does not fit
// 32 registers with bf16 storage at N = 7 and 8 (it spills).  Those get the
// tightest cap that does not spill, which is also the occupancy they had
// with no bound: six blocks (40 registers), five (48) for the fp32-accumulating
// mode at N = 8.
template <int GDT, int NT>
struct RangeBlocksPerSm {
    static constexpr int value = GDT == 0 || NT < 7 ? ReduceBlocksPerSm<GDT, NT, false>::value
                                 : GDT == 2 && NT == 8 ? 5 : 6;
};

// Segments per warp of the reduce kernel.  A bf16 lane loads 16 bytes per
// slab, so at N <= 2 one segment per warp keeps too few bytes in flight:
// each warp then takes two consecutive segments of the list and issues all
// their loads before the first add.  On the 1.5B arena that took the
// reduce-scatter from 85.7 to 97.6 % of the copy peak at N = 1 and from 100.4
// to 106.1 % at N = 2, and the all-reduce at N = 1 from 6.51 to 7.10 TB/s.
// The all-reduce at N = 2 did not change, and the reduce-scatter at N = 3
// fell from 98.0 to 94.2 % (two segments need 48 registers, five blocks),
// so both keep one segment per warp.
template <int GDT, int NT, bool ALL>
struct ReduceSegsPerWarp {
    static constexpr int value = GDT != 0 && (NT == 1 || (NT == 2 && !ALL)) ? 2 : 1;
};

// k_reduce's work for SPW > 1 (compile-time N): warp w takes segments
// w*SPW ... w*SPW + SPW-1 of the chunk-major list.  Each segment is folded,
// averaged, stored and summed exactly as with one segment per warp.
template <int GDT, int NT, bool ALL, bool SUMSQ, int SPW>
__device__ __forceinline__ void reduce_segments(char* __restrict__ grads, int64_t slab, int64_t C,
                                                int64_t groups, int64_t segs, const Avg& avg,
                                                double* __restrict__ partials, int lane)
{
    static_assert(NT > 0, "several segments per warp need a compile-time N");
    using G = Group<GDT>;
    constexpr int ES = G::kBytes;
    const int64_t total = (int64_t)NT * segs;
    const int64_t sw0 = global_warp() * SPW;
    if (sw0 >= total) return;                            // whole warps
    SegPos ps[SPW];
    ps[0] = seg_pos(sw0, segs);
#pragma unroll
    for (int u = 1; u < SPW; ++u) {
        ps[u] = ps[u - 1];
        seg_next(ps[u], segs);
        if (sw0 + u >= total) ps[u] = ps[0];             // past the list: a slot left idle
    }
    const char* src[SPW][NT];
    typename G::Raw raw[SPW][NT];
    int64_t off[SPW];
    bool live[SPW];
#pragma unroll
    for (int u = 0; u < SPW; ++u) {                      // every load first
        const int64_t gi = ps[u].seg * 32 + lane;
        live[u] = sw0 + u < total && gi < groups;
        off[u] = (ps[u].c * C + gi * kGroup) * ES;
        ring_sources<NT>(grads, slab, ps[u].c, src[u]);
        if (live[u]) {
#pragma unroll
            for (int j = 0; j < NT; ++j) raw[u][j] = G::load_raw(src[u][j] + off[u]);
        }
    }
#pragma unroll
    for (int u = 0; u < SPW; ++u) {
        if (sw0 + u >= total) break;                     // warp-uniform
        float ss = 0.0f;
        if (live[u]) {
            float acc[8];
            fold_loaded<GDT, NT>(raw[u], acc);
            average8<GDT, NT>(acc, avg);
            if (SUMSQ) ss = sumsq8(acc);
            const typename G::Raw out = G::pack(acc);
            if (ALL) {
#pragma unroll
                for (int j = 0; j < NT; ++j) G::store_raw(const_cast<char*>(src[u][j]) + off[u], out);
            } else {
                G::store_raw(grads + ps[u].c * slab + off[u], out);
            }
        }
        if (SUMSQ) {
            const float t = warp_sum_f32(ss);
            if (lane == 0) partials[ps[u].c * segs + ps[u].seg] = (double)t;
        }
    }
}

// Ring-order reduce + average of every chunk, one segment per warp (two for
// bf16 at N <= 2, ReduceSegsPerWarp).  ALL = false: chunk c goes to slab c
// only (reduce-scatter).  ALL = true: to every slab (all-reduce).  SUMSQ:
// per-segment sums of squares of the averages.  NT > 0: N == NT known at
// compile time; NT == 0: any N, read from n_rt.  Registers per thread follow
// ReduceBlocksPerSm.
template <int GDT, int NT, bool ALL, bool SUMSQ>
__global__ void __launch_bounds__(kBlock, ReduceBlocksPerSm<GDT, NT, ALL>::value)
k_reduce(char* __restrict__ grads, int64_t P, int64_t C, int n_rt, Avg avg,
         WsHeader* __restrict__ hdr, double* __restrict__ partials)
{
    using G = Group<GDT>;
    constexpr int ES = G::kBytes;
    const int N = NT > 0 ? NT : n_rt;
    const int64_t slab = P * ES;
    const int64_t groups = C / kGroup;
    const int64_t segs = segments_per_chunk(C);
    const int lane = threadIdx.x & 31;
    pdl_enter();
    if (SUMSQ && blockIdx.x == 0 && threadIdx.x == 0) hdr->arrive = 0u;
    if constexpr (ReduceSegsPerWarp<GDT, NT, ALL>::value > 1) {
        reduce_segments<GDT, NT, ALL, SUMSQ, ReduceSegsPerWarp<GDT, NT, ALL>::value>(
            grads, slab, C, groups, segs, avg, partials, lane);
        return;
    }
    const int64_t sw = global_warp();
    if (sw >= (int64_t)N * segs) return;                 // whole warps
    const SegPos p = seg_pos(sw, segs);
    const int c = p.c;
    const int64_t gi = p.seg * 32 + lane;
    float ss = 0.0f;
    if (gi < groups) {
        const int64_t off = (c * C + gi * kGroup) * ES;
        float acc[8];
        constexpr int NS = NT > 0 ? NT : 1;
        const char* src[NS];
        if constexpr (NT > 0) {
            ring_sources<NT>(grads, slab, c, src);
            typename G::Raw raw[NT];
#pragma unroll
            for (int j = 0; j < NT; ++j) raw[j] = G::load_raw(src[j] + off);
            fold_loaded<GDT, NT>(raw, acc);
        } else {
            ring_fold<GDT>(grads, slab, off, c, N, acc);
        }
        average8<GDT, NT>(acc, avg);
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
    if (SUMSQ) {
        const float t = warp_sum_f32(ss);
        if (lane == 0) partials[c * segs + p.seg] = (double)t;
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
// c_first + y in 32-group runs, one per warp: one pass when the grid covers
// the piece, else each warp loops with the grid's stride (a capped grid that
// leaves SMs to kernels on other streams).  With SUMSQ the range must start
// and end on 256-element segment boundaries of its chunks; the runs are then
// the segments and their partials are the ones the whole-arena kernels
// write.
template <int GDT, int NT, bool SUMSQ>
__global__ void __launch_bounds__(kBlock, RangeBlocksPerSm<GDT, NT>::value)
k_reduce_range(const char* __restrict__ src, int64_t src_stride, char* __restrict__ dst,
               int64_t dst_stride, int64_t lo, int64_t hi, int64_t C, int n_rt, int c_first,
               Avg avg, WsHeader* __restrict__ hdr, double* __restrict__ partials)
{
    using G = Group<GDT>;
    constexpr int ES = G::kBytes;
    const int N = NT > 0 ? NT : n_rt;
    const int64_t segs = segments_per_chunk(C);
    const int lane = threadIdx.x & 31;
    const int64_t sslab = src_stride * ES;
    pdl_enter();
    if (SUMSQ && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) hdr->arrive = 0u;
    const int c = c_first + (int)blockIdx.y;
    const int64_t plo = lo > c * C ? lo : c * C;
    const int64_t phi = hi < (c + 1) * C ? hi : (c + 1) * C;
    const int64_t groups = (phi - plo) / kGroup;
    if (plo >= phi) return;
    const int64_t seg0 = (plo - c * C) / kSegment;        // first segment of the piece
    const int64_t wstride = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t wp = global_warp(); wp * 32 < groups; wp += wstride) {   // whole warps
        const int64_t gi = wp * 32 + lane;
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
            average8<GDT, NT>(acc, avg);
            if (SUMSQ) ss = sumsq8(acc);
            G::store_raw(dst + (c * dst_stride + e) * ES, G::pack(acc));
        }
        if (SUMSQ) {
            const float t = warp_sum_f32(ss);
            if (lane == 0) partials[c * segs + seg0 + wp] = (double)t;
        }
    }
}

// Segments per warp for the all-gather: one 16- or 32-byte load per lane and
// segment, so several segments keep enough bytes in flight.
template <int DT>
struct StreamSegs {
    static constexpr int value = DT == 0 ? 2 : 4;
};

// Status bits a partial (or a first-stage sum) stands for: none for a sum of
// squares, which is never negative; DPZ_STATUS_NORM_SKIPPED for
// kPartialNormSkipped (-1.0); both bits for kPartialStepSkipped (-2.0).  The
// test compares the high words as integers: GB300's FP64 pipe is narrow, and
// two FP64 compares per partial doubled the finalisation's time.
__device__ __forceinline__ unsigned marker_bits(double x)
{
    const int hi = __double2hiint(x);
    return hi == kPartialNormSkippedHi ? DPZ_STATUS_NORM_SKIPPED
           : hi == kPartialStepSkippedHi ? DPZ_STATUS_NORM_SKIPPED | DPZ_STATUS_UPDATE_SKIPPED
                                         : 0u;
}

// The block-wide OR of the threads' status bits (contains __syncthreads()).
__device__ __forceinline__ unsigned block_or_bits(unsigned b)
{
    const unsigned norm = __syncthreads_or(b & DPZ_STATUS_NORM_SKIPPED) ? DPZ_STATUS_NORM_SKIPPED : 0u;
    const unsigned upd =
        __syncthreads_or(b & DPZ_STATUS_UPDATE_SKIPPED) ? DPZ_STATUS_UPDATE_SKIPPED : 0u;
    return norm | upd;
}

// A partial as the fp32 value it holds.  Every partial is a 256-element sum of
// squares computed in fp32 and stored as a double: +0, or a double whose low
// 29 mantissa bits are zero and whose exponent lies in fp32's normal range.
// The fp32 value is then rebuilt from the double's two words with integer
// operations (a double-to-float conversion runs on the narrow FP64 pipe).  A
// partial of any other form (an fp32 subnormal, inf, NaN, a skipped tile's
// negative marker) leaves a trace in odd_low or odd_exp, and the caller then
// adds that chain in fp64 instead.
constexpr unsigned kOddExpLimit = 254u;

__device__ __forceinline__ float partial_as_f32(double x, unsigned& odd_low, unsigned& odd_exp)
{
    const unsigned h = (unsigned)__double2hiint(x);
    const unsigned l = (unsigned)__double2loint(x);
    odd_low |= l & (h != 0u ? 0x1fffffffu : 0xffffffffu);
    // biased double exponent 897..1150 <=> fp32 exponent field 1..254 (a set
    // sign bit lands far above the limit)
    odd_exp = max(odd_exp, h != 0u ? (h >> 20) - 897u : 0u);
    // (h:l) << 3 keeps the fp32 exponent field plus 896, modulo 2^9, above
    // the 23 mantissa bits; adding 2^30 subtracts 896 << 23 modulo 2^32
    return __uint_as_float(h != 0u ? __funnelshift_l(l, h, 3) + 0x40000000u : 0u);
}

// One step of Sum2 (Ogita, Rump and Oishi, "Accurate sum and dot product",
// SIAM J. Sci. Comput. 26(6), 2005): s += p, and the rounding error of that
// addition, which TwoSum (Knuth) computes exactly, added into c.  After a
// chain of n non-negative terms with exact sum S, s + c (added in fp64)
// differs from S by at most gamma(n-1)^2 * S, gamma(k) = k u / (1 - k u) with
// u = 2^-24, unless s overflowed.  Needs IEEE fp32 addition, round to
// nearest, subnormals kept (the library is built with -ftz=false).
__device__ __forceinline__ void sum2_add(float& s, float& c, float p)
{
    const float t = s + p;
    const float z = t - s;
    c += (s - (t - z)) + (p - z);
    s = t;
}

// Sum of the n segment partials in a fixed order, independent of the device:
// block b of F adds the contiguous range [b*L, (b+1)*L) (L = ceil(n/F)) into
// stage1[b]; the last block to arrive (an arrival counter, not an ordering)
// adds stage1[0..F-1] and writes sumsq, the norm, the status word and
// *norm_out.  No block waits for another.
//
// Each thread adds its terms i, i + 512, ... in that order by Sum2 in fp32,
// then the block adds its threads' s + c in fp64 in a fixed tree.  A chain
// with a partial of another form, or whose fp32 sum overflows, is added
// again in plain fp64 in the same order (inf and NaN propagate as in any
// sum, and a skipped tile's marker makes the norm NaN and sets the status
// bits it stands for).  So the first stage needs no FP64 arithmetic in the
// usual case: on the 1.5B arena's 6.1 M partials the kernel took 23 us per
// launch with fp64 chains, bound by GB300's FP64 pipe, and takes 16 us with
// these, bound by load latency (ncu launch list of the clipped step).  Chains
// of one term (n <= 512 F) give the bits the plain fp64 sum gives.
//
// The kernel is launched early (programmatic dependent launch): its blocks
// are placed while the kernel that writes the partials retires, and wait for
// that kernel's writes before they read anything.
__global__ void __launch_bounds__(kFinalThreads)
k_norm_finalize(WsHeader* __restrict__ hdr, double* __restrict__ stage1,
                const double* __restrict__ partials, int64_t n, float* __restrict__ norm_out)
{
    pdl_enter();
    const int F = gridDim.x;
    const int64_t L = (n + F - 1) / F;
    const int64_t lo = (int64_t)blockIdx.x * L;
    const int64_t hi = lo + L < n ? lo + L : n;
    const int64_t bd = blockDim.x;
    float s = 0.0f, c = 0.0f;
    unsigned odd_low = 0u, odd_exp = 0u;
    int64_t i = lo + threadIdx.x;
    for (; i + 7 * bd < hi; i += 8 * bd) {
        double x[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = __ldcg(&partials[i + k * bd]);
#pragma unroll
        for (int k = 0; k < 8; ++k) sum2_add(s, c, partial_as_f32(x[k], odd_low, odd_exp));
    }
    if (i < hi) {      // the last terms, loaded together (indices clamped to the range)
        double x[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t j = i + k * bd;
            x[k] = __ldcg(&partials[j < hi ? j : hi - 1]);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (i + k * bd < hi) sum2_add(s, c, partial_as_f32(x[k], odd_low, odd_exp));
    }
    double v = 0.0;
    unsigned bits = 0;
    if (odd_low == 0u && odd_exp < kOddExpLimit && isfinite(s)) {
        v = (double)s + (double)c;
    } else {
        for (int64_t q = lo + threadIdx.x; q < hi; q += bd) {
            const double x = __ldcg(&partials[q]);
            v += x;
            bits |= marker_bits(x);
        }
    }
    v = block_sum(v);
    bits = block_or_bits(bits);
    __shared__ bool is_last;
    if (threadIdx.x == 0) {
        stage1[blockIdx.x] = (bits & DPZ_STATUS_UPDATE_SKIPPED) ? kPartialStepSkipped
                             : bits                              ? kPartialNormSkipped
                                                                 : v;
        __threadfence();
        const unsigned prev = atomicAdd(&hdr->arrive, 1u);
        is_last = prev == (unsigned)(F - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    double w = 0.0;
    unsigned wbits = 0;
    for (int k = threadIdx.x; k < F; k += blockDim.x) {
        const double x = __ldcg(&stage1[k]);
        w += x;
        wbits |= marker_bits(x);
    }
    w = block_sum(w);
    wbits = block_or_bits(wbits);
    if (threadIdx.x == 0) {
        float nrm = __double2float_rn(__dsqrt_rn(w));
        if (wbits) {
            w = __longlong_as_double(0x7ff8000000000000LL);
            nrm = __int_as_float(0x7fc00000);
        }
        hdr->sumsq = w;
        hdr->norm = nrm;
        hdr->nparts = (uint32_t)n;
        hdr->status = wbits;
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
    const int64_t segs = segments_per_chunk(C);
    const int64_t total = (int64_t)N * segs;
    const int lane = threadIdx.x & 31;
    const int64_t sw0 = global_warp() * U;
    pdl_enter();
    if (sw0 >= total) return;                             // whole warps
    const SegPos p0 = seg_pos(sw0, segs);
    typename Group<WDT>::Raw x[U];
    SegPos p = p0;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t gi = p.seg * 32 + lane;
        if (sw0 + u < total && gi < groups)
            x[u] = Group<WDT>::load_raw(w + p.c * slab + (p.c * C + gi * kGroup) * ES);
        seg_next(p, segs);
    }
    p = p0;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t gi = p.seg * 32 + lane;
        if (sw0 + u < total && gi < groups) {
            const int64_t off = (p.c * C + gi * kGroup) * ES;
            for (int r = 0; r < N; ++r)
                if (r != p.c) Group<WDT>::store_raw(w + r * slab + off, x[u]);
        }
        seg_next(p, segs);
    }
}

// ------------------------------------------------------------------ launchers

template <int GDT, int NT, bool ALL, bool SUMSQ>
static cudaError_t reduce_t(const Arena& a, const Avg& avg, void* grads, void* ws, cudaStream_t s)
{
    const unsigned blocks = blocks_for_segments(int64_t(a.N) * segments_per_chunk(a.C),
                                                ReduceSegsPerWarp<GDT, NT, ALL>::value);
    set_last_kernel_name(ALL ? "dpz_allreduce_avg" : SUMSQ ? "dpz_rs_avg_sumsq" : "dpz_rs_avg");
    return launch_kernel(k_reduce<GDT, NT, ALL, SUMSQ>, dim3(blocks), dim3(kBlock), 0, s, true, 0u,
                         static_cast<char*>(grads), a.P, a.C, a.N, avg, static_cast<WsHeader*>(ws),
                         SUMSQ ? ws_partials(ws) : nullptr);
}

template <int GDT, bool ALL, bool SUMSQ>
static cudaError_t reduce_n(const Arena& a, const Avg& avg, void* grads, void* ws, cudaStream_t s)
{
    switch (a.N) {       // compile-time folds for N <= 8, the run-time fold beyond
    case 1: return reduce_t<GDT, 1, ALL, SUMSQ>(a, avg, grads, ws, s);
    case 2: return reduce_t<GDT, 2, ALL, SUMSQ>(a, avg, grads, ws, s);
    case 3: return reduce_t<GDT, 3, ALL, SUMSQ>(a, avg, grads, ws, s);
    case 4: return reduce_t<GDT, 4, ALL, SUMSQ>(a, avg, grads, ws, s);
    case 5: return reduce_t<GDT, 5, ALL, SUMSQ>(a, avg, grads, ws, s);
    case 6: return reduce_t<GDT, 6, ALL, SUMSQ>(a, avg, grads, ws, s);
    case 7: return reduce_t<GDT, 7, ALL, SUMSQ>(a, avg, grads, ws, s);
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
    const int c_first = (int)(g.lo / a.C);
    const int c_last = (int)((g.hi - 1) / a.C);
    const int pieces = c_last - c_first + 1;
    const int64_t longest = a.C < g.hi - g.lo ? a.C : g.hi - g.lo;
    dim3 grid(blocks_for_segments(segments_per_chunk(longest), 1), (unsigned)pieces, 1);
    if (g.max_ctas > 0) {
        const unsigned per_piece = g.max_ctas / pieces > 0 ? (unsigned)(g.max_ctas / pieces) : 1u;
        if (grid.x > per_piece) grid.x = per_piece;
    }
    set_last_kernel_name(SUMSQ ? "dpz_rs_range_sumsq" : "dpz_rs_range");
    return launch_kernel(k_reduce_range<GDT, NT, SUMSQ>, grid, dim3(kBlock), 0, s, true, 0u,
                         static_cast<const char*>(g.src), g.src_stride, static_cast<char*>(g.dst),
                         g.dst_stride, g.lo, g.hi, a.C, a.N, c_first, avg,
                         static_cast<WsHeader*>(ws), SUMSQ ? ws_partials(ws) : nullptr);
}

template <int GDT, bool SUMSQ>
static cudaError_t range_n(const Arena& a, const Avg& avg, const RangeArgs& g, void* ws,
                           cudaStream_t s)
{
    switch (a.N) {
    case 1: return range_t<GDT, 1, SUMSQ>(a, avg, g, ws, s);
    case 2: return range_t<GDT, 2, SUMSQ>(a, avg, g, ws, s);
    case 3: return range_t<GDT, 3, SUMSQ>(a, avg, g, ws, s);
    case 4: return range_t<GDT, 4, SUMSQ>(a, avg, g, ws, s);
    case 5: return range_t<GDT, 5, SUMSQ>(a, avg, g, ws, s);
    case 6: return range_t<GDT, 6, SUMSQ>(a, avg, g, ws, s);
    case 7: return range_t<GDT, 7, SUMSQ>(a, avg, g, ws, s);
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

cudaError_t launch_norm_finalize(const Arena& a, void* ws, float* norm_out, cudaStream_t s)
{
    set_last_kernel_name("dpz_norm_finalize");
    const int64_t n = int64_t(a.N) * segments_per_chunk(a.C);
    // blocks: a function of n only, so the summation order is fixed
    int64_t F = (n + 2047) / 2048;
    if (F > kFinalBlocks) F = kFinalBlocks;
    if (F < 1) F = 1;
    return launch_kernel(k_norm_finalize, dim3((unsigned)F), dim3(kFinalThreads), 0, s, true, 0u,
                         static_cast<WsHeader*>(ws), ws_stage1(ws), ws_partials(ws), n, norm_out);
}

cudaError_t launch_allgather(const Arena& a, void* weights, cudaStream_t s)
{
    set_last_kernel_name("dpz_allgather");
    char* w = static_cast<char*>(weights);
    const int64_t nseg = int64_t(a.N) * segments_per_chunk(a.C);
    if (a.wdt == 1)
        return launch_kernel(k_allgather<1>, dim3(blocks_for_segments(nseg, StreamSegs<1>::value)),
                             dim3(kBlock), 0, s, true, 0u, w, a.P, a.C, a.N);
    return launch_kernel(k_allgather<0>, dim3(blocks_for_segments(nseg, StreamSegs<0>::value)),
                         dim3(kBlock), 0, s, true, 0u, w, a.P, a.C, a.N);
}

// ---------------------------------------------------------------------------
// Self-test of the average's division: every float bit pattern a, divided by
// N through divide8 (the compile-time instantiation the kernels use for N <= 8,
// the run-time one beyond), against __fdiv_rn(a, N).  Each thread takes
// kDivGroupsPerThread groups of 8 consecutive patterns and divides each group
// twice: as it stands (the group takes one path as a whole) and as 8 copies of
// one value (so every value that passes markstein_ok is checked on the fast
// path, zero and the smallest normals included).  Two NaNs count as equal.
namespace {

constexpr int kDivGroupsPerThread = 16;
constexpr uint64_t kDivPatterns = 1ull << 32;

__device__ __forceinline__ bool same_quotient(float got, float want)
{
    return __float_as_uint(got) == __float_as_uint(want) || (isnan(got) && isnan(want));
}

template <int NT>
__global__ void __launch_bounds__(kBlock)
k_selftest_division(Avg avg, unsigned long long* mismatches)
{
    const uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    unsigned bad = 0;
    for (int k = 0; k < kDivGroupsPerThread; ++k) {
        const uint32_t base = (uint32_t)((t * kDivGroupsPerThread + k) * 8);
        float x[8], want[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            x[q] = __uint_as_float(base + q);
            want[q] = __fdiv_rn(x[q], avg.fN);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float s[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) s[i] = x[q];
            divide8<NT>(s, avg);
#pragma unroll
            for (int i = 0; i < 8; ++i) bad += !same_quotient(s[i], want[q]);
        }
        divide8<NT>(x, avg);
#pragma unroll
        for (int q = 0; q < 8; ++q) bad += !same_quotient(x[q], want[q]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_down_sync(0xffffffffu, bad, o);
    if ((threadIdx.x & 31) == 0 && bad != 0) atomicAdd(mismatches, (unsigned long long)bad);
}

}  // namespace

cudaError_t launch_selftest_division(const Avg& avg, unsigned long long* mismatches,
                                     cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(mismatches, 0, sizeof(unsigned long long), s);
    if (e != cudaSuccess) return e;
    constexpr uint64_t threads = kDivPatterns / 8 / kDivGroupsPerThread;
    static_assert(threads % kBlock == 0, "the pattern space splits into whole blocks");
    const unsigned blocks = (unsigned)(threads / kBlock);
    switch ((int)avg.fN) {
    case 1: k_selftest_division<1><<<blocks, kBlock, 0, s>>>(avg, mismatches); break;
    case 2: k_selftest_division<2><<<blocks, kBlock, 0, s>>>(avg, mismatches); break;
    case 3: k_selftest_division<3><<<blocks, kBlock, 0, s>>>(avg, mismatches); break;
    case 4: k_selftest_division<4><<<blocks, kBlock, 0, s>>>(avg, mismatches); break;
    case 5: k_selftest_division<5><<<blocks, kBlock, 0, s>>>(avg, mismatches); break;
    case 6: k_selftest_division<6><<<blocks, kBlock, 0, s>>>(avg, mismatches); break;
    case 7: k_selftest_division<7><<<blocks, kBlock, 0, s>>>(avg, mismatches); break;
    case 8: k_selftest_division<8><<<blocks, kBlock, 0, s>>>(avg, mismatches); break;
    default: k_selftest_division<0><<<blocks, kBlock, 0, s>>>(avg, mismatches); break;
    }
    return cudaGetLastError();
}

}  // namespace dpz
