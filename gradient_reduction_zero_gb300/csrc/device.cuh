// Device helpers shared by the streaming kernels: 16- and 32-byte streaming
// loads and stores, bf16 packing with round-to-nearest-even, the ring-order
// fold, the correctly rounded average, the fp32 AdamW element update, the
// fixed warp and block sums (one segment's, or eight segments' at once), and
// thread-block cluster barriers and stores into another CTA's shared memory.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace dpz {

// ------------------------------------------------------------ memory access
//
// Every stream is touched once, so loads ask L2 to fetch whole 256-byte
// segments (the next lanes' data) and stores are marked evict-first.
// (Skipping L1 on the loads with L1::no_allocate measured 11 % slower on the
// reduce kernel.)  fp32 streams use 256-bit accesses (sm_100 and later;
// 32-byte aligned), bf16 streams 128-bit ones.

struct U8 {
    uint32_t x[8];
};

__device__ __forceinline__ uint4 ld16(const void* p)
{
    uint4 r;
    asm volatile("ld.global.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ U8 ld32(const void* p)
{
    U8 r;
    asm volatile("ld.global.L2::256B.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.x[0]), "=r"(r.x[1]), "=r"(r.x[2]), "=r"(r.x[3]), "=r"(r.x[4]),
                   "=r"(r.x[5]), "=r"(r.x[6]), "=r"(r.x[7])
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st16(void* p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st32(void* p, const U8& v)
{
    asm volatile("st.global.cs.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.x[0]),
                 "r"(v.x[1]), "r"(v.x[2]), "r"(v.x[3]), "r"(v.x[4]), "r"(v.x[5]), "r"(v.x[6]),
                 "r"(v.x[7])
                 : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two floats -> two bf16 in one word (lo in the low half), each rounded to
// nearest even; NaN stays NaN, subnormals are kept.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float round_bf16(float x)
{
    return __bfloat162float(__float2bfloat16_rn(x));
}

// Round two floats to bf16 (nearest even) with one paired conversion and
// return them as floats again.
__device__ __forceinline__ void round_bf16x2(float& lo, float& hi)
{
    const uint32_t w = pack_bf16x2(lo, hi);
    lo = bf16_lo(w);
    hi = bf16_hi(w);
}

// A group of 8 elements of one storage type.  DT 0 = fp32 (one 32-byte
// word), DT 1 = bf16 (one 16-byte word), DT 2 = bf16 storage whose ring
// accumulates in fp32.  round8 is the rounding to the storage type;
// hop_round8 the rounding after each ring hop (a bf16 ring rounds once per
// hop; the fp32-accumulating one only at the end).
template <int DT>
struct Group;

template <>
struct Group<1> {
    static constexpr int kBytes = 2;
    struct Raw { uint4 w; };
    static __device__ __forceinline__ Raw load_raw(const char* p) { return {ld16(p)}; }
    static __device__ __forceinline__ void store_raw(char* p, const Raw& r) { st16(p, r.w); }
    static __device__ __forceinline__ void unpack(const Raw& r, float x[8])
    {
        x[0] = bf16_lo(r.w.x); x[1] = bf16_hi(r.w.x);
        x[2] = bf16_lo(r.w.y); x[3] = bf16_hi(r.w.y);
        x[4] = bf16_lo(r.w.z); x[5] = bf16_hi(r.w.z);
        x[6] = bf16_lo(r.w.w); x[7] = bf16_hi(r.w.w);
    }
    static __device__ __forceinline__ Raw pack(const float x[8])
    {
        Raw r;
        r.w.x = pack_bf16x2(x[0], x[1]);
        r.w.y = pack_bf16x2(x[2], x[3]);
        r.w.z = pack_bf16x2(x[4], x[5]);
        r.w.w = pack_bf16x2(x[6], x[7]);
        return r;
    }
    static __device__ __forceinline__ void round8(float x[8])
    {
#pragma unroll
        for (int q = 0; q < 8; q += 2) round_bf16x2(x[q], x[q + 1]);
    }
    static __device__ __forceinline__ void hop_round8(float x[8]) { round8(x); }
};

template <>
struct Group<2> : Group<1> {
    static __device__ __forceinline__ void hop_round8(float[8]) {}
};

template <>
struct Group<0> {
    static constexpr int kBytes = 4;
    using Raw = U8;
    static __device__ __forceinline__ Raw load_raw(const char* p) { return ld32(p); }
    static __device__ __forceinline__ void store_raw(char* p, const Raw& r) { st32(p, r); }
    static __device__ __forceinline__ void unpack(const Raw& r, float x[8])
    {
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = __uint_as_float(r.x[q]);
    }
    static __device__ __forceinline__ Raw pack(const float x[8])
    {
        Raw r;
#pragma unroll
        for (int q = 0; q < 8; ++q) r.x[q] = __float_as_uint(x[q]);
        return r;
    }
    static __device__ __forceinline__ void round8(float[8]) {}
    static __device__ __forceinline__ void hop_round8(float[8]) {}
};

template <int DT>
__device__ __forceinline__ void load_group(const char* p, float x[8])
{
    Group<DT>::unpack(Group<DT>::load_raw(p), x);
}

template <int DT>
__device__ __forceinline__ void store_group(char* p, const float x[8])
{
    Group<DT>::store_raw(p, Group<DT>::pack(x));
}

// ------------------------------------------------------------ one-shot grids
//
// The streaming kernels cut the arena into 256-element segments (32 groups of
// 8), chunk by chunk: the list holds chunk 0's segments, then chunk 1's, and
// so on (the last segment of a chunk may be short).  Warp w of the grid takes
// segments w*U .. w*U + U - 1 of that list, lane l group l of each, and no
// thread loops over the arena.  Blocks are dispatched in index order and
// retire after one pass, so the addresses in flight form one compact window
// that sweeps the arena once.  A persistent grid-stride loop instead lets its
// blocks drift apart over many iterations and lost 5 to 10 % of DRAM
// bandwidth on multi-GB arenas.

__device__ __forceinline__ int64_t global_warp()
{
    return ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
}

struct SegPos {
    int c;          // chunk
    int64_t seg;    // segment inside the chunk
};

// Position of segment sw of the chunk-major list (segs segments per chunk).
__device__ __forceinline__ SegPos seg_pos(int64_t sw, int64_t segs)
{
    const int c = (int)(sw / segs);
    return {c, sw - (int64_t)c * segs};
}

// The next segment of the list.
__device__ __forceinline__ void seg_next(SegPos& p, int64_t segs)
{
    if (++p.seg == segs) {
        p.seg = 0;
        ++p.c;
    }
}

// ------------------------------------------------------------ the ring fold

// Sources of chunk c in ring order: src[j] = slab (c + 1 + j) mod N.
template <int NT>
__device__ __forceinline__ void ring_sources(const char* grads, int64_t slab, int c,
                                             const char* src[NT])
{
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        int r = c + 1 + j;            // <= 2N - 1: one wrap
        if (r >= NT) r -= NT;
        src[j] = grads + (int64_t)r * slab;
    }
}

// Sum of one group over the NT slabs whose raw words are already loaded,
// in ring order:  acc = x[0];  acc = R(acc + x[j]) for j = 1..NT-1.
template <int GDT, int NT>
__device__ __forceinline__ void fold_loaded(const typename Group<GDT>::Raw raw[NT], float acc[8])
{
    using G = Group<GDT>;
    G::unpack(raw[0], acc);
#pragma unroll
    for (int j = 1; j < NT; ++j) {
        float x[8];
        G::unpack(raw[j], x);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = __fadd_rn(acc[q], x[q]);
        G::hop_round8(acc);
    }
}

// The same fold for a run-time N (any N up to 64): for chunk c,
//   acc = x[c+1];  acc = R(acc + x[c+j]) for j = 2..N   (ranks mod N).
// slab: bytes per slab; off: byte offset of the group inside a slab.  One
// slab at a time: few registers, so many warps stay resident and keep loads
// in flight.  A version batching eight loads per thread held 76 registers
// and ran the N = 3 reduce at 28 % of the copy peak; this form, used for
// N > 8 (the compile-time folds take N <= 8), reduces at 102-109 % of it for
// N = 12 to 32.
template <int GDT>
__device__ __forceinline__ void ring_fold(const char* __restrict__ grads, int64_t slab,
                                          int64_t off, int c, int N, float acc[8])
{
    using G = Group<GDT>;
    int r = c + 1;
    if (r >= N) r -= N;
    G::unpack(G::load_raw(grads + (int64_t)r * slab + off), acc);
    for (int j = 2; j <= N; ++j) {
        ++r;
        if (r >= N) r -= N;
        float x[8];
        G::unpack(G::load_raw(grads + (int64_t)r * slab + off), x);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = __fadd_rn(acc[q], x[q]);
        G::hop_round8(acc);
    }
}

// a / N, correctly rounded, for a group of 8 values.
//
// N a power of two: a * (1/N), exact.  Otherwise Markstein's correction
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with y = RN(1/N)
// (avg.invN) and q0 = RN(a*y), the remainder r = a - q0*N is exact in one
// fused multiply-add, and q1 = RN(q0 + r*y) is the correctly rounded a/N.
// The theorem excludes underflow and non-finite operands, so a group holding
// a nonzero value below 1e-30 in magnitude, or one that is not finite, is
// divided instead; a zero gives q0, the exact signed zero.  An exhaustive
// comparison with __fdiv_rn over all 2^32 float inputs for every N from 1
// to 64 finds no difference (dpz_selftest_average_division).
__device__ __forceinline__ bool markstein_ok(float a)
{
    const float ab = fabsf(a);
    return ab < 3.0e38f && (ab >= 1.0e-30f || ab == 0.0f);
}

__device__ __forceinline__ float div_markstein(float a, float fN, float invN)
{
    const float q0 = __fmul_rn(a, invN);
    const float r = __fmaf_rn(-q0, fN, a);
    const float q1 = __fmaf_rn(r, invN, q0);
    return a == 0.0f ? q0 : q1;
}

// NT > 0: N is known at compile time, and only its path is compiled in (the
// power-of-two kernels stay free of the correction's registers).
template <int NT = 0>
__device__ __forceinline__ void divide8(float x[8], const Avg& avg)
{
    constexpr bool kPow2 = NT > 0 && (NT & (NT - 1)) == 0;
    if (kPow2 || (NT == 0 && avg.pow2)) {
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = __fmul_rn(x[q], avg.invN);
        return;
    }
    if constexpr (!kPow2) {
        bool fast = true;
#pragma unroll
        for (int q = 0; q < 8; ++q) fast &= markstein_ok(x[q]);
        if (fast) {
#pragma unroll
            for (int q = 0; q < 8; ++q) x[q] = div_markstein(x[q], avg.fN, avg.invN);
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) x[q] = __fdiv_rn(x[q], avg.fN);
        }
    }
}

// R(acc / N) for the 8 elements (NT as for divide8).
template <int GDT, int NT = 0>
__device__ __forceinline__ void average8(float acc[8], const Avg& avg)
{
    divide8<NT>(acc, avg);
    Group<GDT>::round8(acc);
}

// Sum of squares of 8 values, fp32, fixed pairwise order.
__device__ __forceinline__ float sumsq8(const float x[8])
{
    float s0 = __fadd_rn(__fmul_rn(x[0], x[0]), __fmul_rn(x[1], x[1]));
    float s1 = __fadd_rn(__fmul_rn(x[2], x[2]), __fmul_rn(x[3], x[3]));
    float s2 = __fadd_rn(__fmul_rn(x[4], x[4]), __fmul_rn(x[5], x[5]));
    float s3 = __fadd_rn(__fmul_rn(x[6], x[6]), __fmul_rn(x[7], x[7]));
    return __fadd_rn(__fadd_rn(s0, s1), __fadd_rn(s2, s3));
}

// ------------------------------------------------------------ AdamW

// One element, fp32, every operation rounded to nearest even, in the order the
// C-ABI documents (no contraction into FMA).
__device__ __forceinline__ void adamw_elem(float& theta, float& m, float& v, float g,
                                           const AdamArgs& h)
{
    float mm = __fadd_rn(__fmul_rn(h.b1, m), __fmul_rn(h.omb1, g));
    float vv = __fadd_rn(__fmul_rn(h.b2, v), __fmul_rn(h.omb2, __fmul_rn(g, g)));
    float mhat = __fdiv_rn(mm, h.bc1);
    float vhat = __fdiv_rn(vv, h.bc2);
    float upd = __fdiv_rn(mhat, __fadd_rn(__fsqrt_rn(vhat), h.eps));
    float t = theta;
    theta = __fsub_rn(t, __fmul_rn(h.lr, __fadd_rn(upd, __fmul_rn(h.wd, t))));
    m = mm;
    v = vv;
}

// ------------------------------------------------------------ reductions

// Sum over the 32 lanes of a warp in a fixed tree, fp32; lane 0 holds the
// result.  Used for the 256-element norm segments: with the 8-element sums
// below, each segment is a fixed 8-level pairwise fp32 tree.
__device__ __forceinline__ float warp_sum_f32(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, o));
    return v;
}

// warp_sum_f32 of eight values at once: v[s] is this lane's term of segment
// s, and lane 4s receives segment s's sum.  Each level of the tree pairs the
// same two lanes' values as warp_sum_f32 does, so every segment's sum has the
// same bits; but at each level a lane hands half of its segments to its
// partner and keeps the other half, so the eight trees take 4 + 2 + 1 + 1 + 1
// = 9 shuffles instead of 40.
__device__ __forceinline__ float warp_sum8_f32(const float v[8])
{
    const int lane = threadIdx.x & 31;
    const bool hi16 = lane & 16, hi8 = lane & 8, hi4 = lane & 4;
    float w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {           // lanes l, l^16: segments 0-3 stay below, 4-7 above
        const float keep = hi16 ? v[4 + k] : v[k];
        const float give = hi16 ? v[k] : v[4 + k];
        w[k] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, give, 16));
    }
    float x[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {           // lanes l, l^8: halves of those four
        const float keep = hi8 ? w[2 + k] : w[k];
        const float give = hi8 ? w[k] : w[2 + k];
        x[k] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, give, 8));
    }
    const float keep = hi4 ? x[1] : x[0];   // lanes l, l^4: one segment each
    const float give = hi4 ? x[0] : x[1];
    float y = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, give, 4));
    y = __fadd_rn(y, __shfl_xor_sync(0xffffffffu, y, 2));
    return __fadd_rn(y, __shfl_xor_sync(0xffffffffu, y, 1));
}

// ------------------------------------------------------------ clusters
//
// A thread-block cluster's CTAs run at the same time on different SMs and can
// write each other's shared memory.  Every thread of every CTA of the cluster
// must take part in each barrier.

// Announce that this thread has started (no ordering of its memory accesses).
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

// Announce that this thread's earlier memory accesses are done.
__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

// Wait until every thread of the cluster has arrived; their released accesses
// are then visible to this thread.
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store v into the copy of the shared-memory variable *p that the cluster's
// CTA of the given rank holds.
__device__ __forceinline__ void store_shared_of_rank(double* p, unsigned rank, double v)
{
    const uint32_t local = (uint32_t)__cvta_generic_to_shared(p);
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    asm volatile("st.shared::cluster.f64 [%0], %1;" ::"r"(remote), "d"(v) : "memory");
}

// Sum over the 32 lanes of a warp in a fixed tree; lane 0 holds the result.
__device__ __forceinline__ double warp_sum(double v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
    return v;
}

// Deterministic sum of one double per thread; the result is returned to
// thread 0 (fixed shuffle tree per warp, then warp 0 over the warp sums).
// blockDim.x must be a multiple of 32.  Contains __syncthreads().
__device__ __forceinline__ double block_sum(double v)
{
    __shared__ double warp_sums[32];
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (lane == 0) warp_sums[wid] = v;
    __syncthreads();
    double r = 0.0;
    if (wid == 0) {
        r = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0.0;
        r = warp_sum(r);
    }
    __syncthreads();
    return r;
}

}  // namespace dpz
