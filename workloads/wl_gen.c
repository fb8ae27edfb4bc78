/*
 * wl_gen.c -- seeded synthetic inputs shared by the tests, the smoke check
 * and the benchmark.  It holds none of the compression method's arithmetic:
 * only a counter-based random source and a normal transform.
 *
 *   SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *   generators", OOPSLA 2014): draw(key, i) = mix64(key + (i + 1) * GAMMA).
 *   Uniform in (0, 1]: ((draw >> 11) + 1) * 2^-53.
 *   Normal (Box-Muller, one value per pair of uniforms):
 *     z_i = sqrt(-2 ln u_{2i}) * cos(2 pi u_{2i+1}), in binary64.
 *
 * Being counter-based, any sub-range [start, start + count) of a stream can
 * be produced on its own, which the sampled checks of large inputs use.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* key of the (seed, stream) pair */
static uint64_t key_of(uint64_t seed, uint64_t stream)
{
    return mix64(seed * GAMMA + mix64(stream + 0x632BE59BD9B4E019ULL));
}

static uint64_t draw(uint64_t key, uint64_t i)
{
    return mix64(key + (i + 1) * GAMMA);
}

static double unit(uint64_t r)
{
    return (double)((r >> 11) + 1) * (1.0 / 9007199254740992.0);
}

void wl_u64(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count, uint64_t *out)
{
    uint64_t key = key_of(seed, stream);
    for (uint64_t i = 0; i < count; i++)
        out[i] = draw(key, start + i);
}

void wl_uniform(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count, double *out)
{
    uint64_t key = key_of(seed, stream);
    for (uint64_t i = 0; i < count; i++)
        out[i] = unit(draw(key, start + i));
}

void wl_normal(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count, double *out)
{
    const double two_pi = 6.283185307179586476925286766559;
    uint64_t key = key_of(seed, stream);
    for (uint64_t i = 0; i < count; i++) {
        uint64_t idx = start + i;
        double u1 = unit(draw(key, 2 * idx));
        double u2 = unit(draw(key, 2 * idx + 1));
        out[i] = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
    }
}
