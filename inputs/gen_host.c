/* Host build of the seeded input generator (see gen.h). */
#include "gen.h"

#include <stdint.h>

void gen_fill_f32(float* out, int64_t start, int64_t count, uint64_t seed,
                  uint64_t stream, int kind, double scale, double scale_tail)
{
    const uint64_t key = gen_key(seed, stream);
    for (int64_t j = 0; j < count; ++j)
        out[j] = gen_value(kind, key, (uint64_t)(start + j), scale, scale_tail);
}

void gen_fill_bf16(uint16_t* out, int64_t start, int64_t count, uint64_t seed,
                   uint64_t stream, int kind, double scale, double scale_tail)
{
    const uint64_t key = gen_key(seed, stream);
    for (int64_t j = 0; j < count; ++j)
        out[j] = gen_trunc_bf16(
            gen_value(kind, key, (uint64_t)(start + j), scale, scale_tail));
}
