// Device helpers shared by the streaming kernels: 16-byte streaming loads and
// stores, bf16 packing with round-to-nearest-even, the ring-order fold, the
// fp32 AdamW element update and a deterministic block sum.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace dpz {

// ------------------------------------------------------------ memory access

__device__ __forceinline__ uint4 ld_stream(const void* p)
{
    return __ldcs(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void st_stream(void* p, uint4 v)
{
    __stcs(reinterpret_cast<uint4*>(p), v);
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

// A group of 8 elements of one storage type.  DT 0 = fp32 (two 16-byte
// words), DT 1 = bf16 (one 16-byte word).
template <int DT>
struct Group;

template <>
struct Group<1> {
    static constexpr int kBytes = 2;
    struct Raw { uint4 w; };
    static __device__ __forceinline__ Raw load_raw(const char* p) { return {ld_stream(p)}; }
    static __device__ __forceinline__ void store_raw(char* p, const Raw& r) { st_stream(p, r.w); }
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
    static __device__ __forceinline__ float round(float x) { return round_bf16(x); }
};

template <>
struct Group<0> {
    static constexpr int kBytes = 4;
    struct Raw { uint4 a, b; };
    static __device__ __forceinline__ Raw load_raw(const char* p)
    {
        return {ld_stream(p), ld_stream(p + 16)};
    }
    static __device__ __forceinline__ void store_raw(char* p, const Raw& r)
    {
        st_stream(p, r.a);
        st_stream(p + 16, r.b);
    }
    static __device__ __forceinline__ void unpack(const Raw& r, float x[8])
    {
        x[0] = __uint_as_float(r.a.x); x[1] = __uint_as_float(r.a.y);
        x[2] = __uint_as_float(r.a.z); x[3] = __uint_as_float(r.a.w);
        x[4] = __uint_as_float(r.b.x); x[5] = __uint_as_float(r.b.y);
        x[6] = __uint_as_float(r.b.z); x[7] = __uint_as_float(r.b.w);
    }
    static __device__ __forceinline__ Raw pack(const float x[8])
    {
        Raw r;
        r.a = make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]),
                         __float_as_uint(x[2]), __float_as_uint(x[3]));
        r.b = make_uint4(__float_as_uint(x[4]), __float_as_uint(x[5]),
                         __float_as_uint(x[6]), __float_as_uint(x[7]));
        return r;
    }
    static __device__ __forceinline__ float round(float x) { return x; }
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

// ------------------------------------------------------------ the ring fold

// Sum of one 8-element group over the N slabs in ring order for chunk c:
//   acc = x[c+1];  acc = R(acc + x[c+j]) for j = 2..N   (ranks mod N)
// slab: bytes per slab; off: byte offset of the group inside a slab.
// Loads are issued in batches so that several slabs are in flight at once.
template <int GDT>
__device__ __forceinline__ void ring_fold(const char* __restrict__ grads, int64_t slab,
                                          int64_t off, int c, int N, float acc[8])
{
    using G = Group<GDT>;
    constexpr int B = GDT == 1 ? 8 : 4;
    int r0 = c + 1;
    if (r0 >= N) r0 -= N;
    typename G::Raw first = G::load_raw(grads + (int64_t)r0 * slab + off);
    for (int j0 = 1; j0 < N; j0 += B) {
        typename G::Raw raw[B];
#pragma unroll
        for (int k = 0; k < B; ++k) {
            int r = c + 1 + j0 + k;            // < 2N + B: at most two wraps
            if (r >= N) r -= N;
            if (r >= N) r -= N;
            if (j0 + k < N) raw[k] = G::load_raw(grads + (int64_t)r * slab + off);
        }
        if (j0 == 1) G::unpack(first, acc);
#pragma unroll
        for (int k = 0; k < B; ++k) {
            if (j0 + k < N) {
                float x[8];
                G::unpack(raw[k], x);
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = G::round(__fadd_rn(acc[q], x[q]));
            }
        }
    }
    if (N == 1) G::unpack(first, acc);
}

// R(acc / N) for the 8 elements.
template <int GDT>
__device__ __forceinline__ void average8(float acc[8], const Avg& avg)
{
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float y = avg.pow2 ? __fmul_rn(acc[q], avg.invN) : __fdiv_rn(acc[q], avg.fN);
        acc[q] = Group<GDT>::round(y);
    }
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
