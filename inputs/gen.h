/*
 * Seeded, counter-based synthetic input generator.
 *
 * This module only makes input data. It holds none of the ZeRO-1 step's
 * arithmetic (no ring, no rounding rule of the method, no optimizer) and is
 * the one piece of code that both the CPU oracle's tests and the GPU runs use:
 * the host build fills arrays for the oracle, the device build fills the same
 * arrays in GPU memory, bit for bit.
 *
 * Definition (value of element i of stream s under seed k):
 *   mix64(z)      SplitMix64 finaliser (Steele, Lea and Flood, 2014):
 *                 z ^= z>>30; z *= 0xBF58476D1CE4E5B9; z ^= z>>27;
 *                 z *= 0x94D049BB133111EB; z ^= z>>31
 *   key(k, s)     mix64(mix64(k + G) + s*G),  G = 0x9E3779B97F4A7C15
 *   draw(key,i,j) mix64(key + (4i + j + 1)*G)        j in 0..3
 *   uniform       ((draw(.,i,0) >> 40) - 2^23) * 2^-23      in [-1, 1)
 *   normal(sigma) Irwin-Hall sum of the twelve 16-bit fields of draws 0..2,
 *                 minus 12*65535/2, times sigma/65536 (mean 0, sd ~sigma),
 *                 computed as one double product, then rounded to float
 *   heavy tail    the normal value uses sigma*100 instead iff
 *                 draw(.,i,3) mod 100 == 0 (about 1 % of the elements)
 *   |normal|      absolute value of the normal draw
 *   bf16 inputs   the float value truncated to its upper 16 bits
 *
 * Only integer operations, one int->double conversion, one double product and
 * one double->float rounding are involved, so host and device agree exactly.
 */
#ifndef DPZ_INPUTS_GEN_H
#define DPZ_INPUTS_GEN_H

#include <stdint.h>

#ifdef __CUDACC__
#define GEN_FN __host__ __device__ __forceinline__
#else
#define GEN_FN static inline
#endif

#define GEN_GOLDEN 0x9E3779B97F4A7C15ull

enum {
    GEN_ZERO = 0,
    GEN_UNIFORM = 1,      /* U[-1, 1) */
    GEN_NORMAL = 2,       /* N(0, sigma) */
    GEN_NORMAL_TAIL = 3,  /* N(0, sigma), 1 % of elements with sigma*100 */
    GEN_ABS_NORMAL = 4    /* |N(0, sigma)| */
};

GEN_FN uint64_t gen_mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

GEN_FN uint64_t gen_key(uint64_t seed, uint64_t stream)
{
    return gen_mix64(gen_mix64(seed + GEN_GOLDEN) + stream * GEN_GOLDEN);
}

GEN_FN uint64_t gen_draw(uint64_t key, uint64_t i, unsigned j)
{
    return gen_mix64(key + (4ull * i + (uint64_t)j + 1ull) * GEN_GOLDEN);
}

GEN_FN int32_t gen_irwin_hall12(uint64_t key, uint64_t i)
{
    int32_t s = 0;
    for (unsigned j = 0; j < 3; ++j) {
        uint64_t h = gen_draw(key, i, j);
        s += (int32_t)(h & 0xffffu) + (int32_t)((h >> 16) & 0xffffu) +
             (int32_t)((h >> 32) & 0xffffu) + (int32_t)(h >> 48);
    }
    return s - 393210;   /* 12 * 65535 / 2 */
}

/* scale = sigma / 65536 and scale_tail = sigma * 100 / 65536 are computed by
 * the caller once, in double, and passed to both builds. */
GEN_FN float gen_value(int kind, uint64_t key, uint64_t i, double scale,
                       double scale_tail)
{
    switch (kind) {
    case GEN_UNIFORM: {
        int32_t u = (int32_t)(gen_draw(key, i, 0) >> 40) - 8388608;
        return (float)((double)u * (1.0 / 8388608.0));
    }
    case GEN_NORMAL:
        return (float)((double)gen_irwin_hall12(key, i) * scale);
    case GEN_NORMAL_TAIL: {
        int tail = (gen_draw(key, i, 3) % 100ull) == 0ull;
        return (float)((double)gen_irwin_hall12(key, i) * (tail ? scale_tail : scale));
    }
    case GEN_ABS_NORMAL: {
        int32_t z = gen_irwin_hall12(key, i);
        return (float)((double)(z < 0 ? -z : z) * scale);
    }
    default:
        return 0.0f;
    }
}

/* bf16 input = the float's upper 16 bits (truncation, not the method's
 * rounding). */
GEN_FN uint16_t gen_trunc_bf16(float x)
{
    union { float f; uint32_t u; } b;
    b.f = x;
    return (uint16_t)(b.u >> 16);
}

#endif
