/*
 * synth.c -- seeded, counter-based synthetic input generator.
 *
 * Serves the tests and the benchmark alike; holds none of the SpMV method's
 * arithmetic (no pruning, packing or products).  It only draws numbers.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) used in counter mode: draw n of stream k
 * is mix(key_k + (n + 1) * GAMMA), where key_k = mix(seed ^ mix(k)) and mix is
 * SplitMix64's output function.  Counter mode makes every element a pure
 * function of (seed, stream, index), so any slice can be produced alone and
 * the threads below cannot change the result.
 *
 * Normals: Box-Muller (Box and Muller, 1958), cosine branch, one normal per
 * element from draws 2i and 2i+1; then scaled by sigma and rounded to IEEE
 * binary16 (round to nearest, ties to even) by the routine below.
 *
 * Small integers: draw 2i, reduced to [lo, hi] by a 64x64->128 multiply-high
 * (Lemire's method without rejection; the bias is below 2^-50 for the tiny
 * ranges used), times 2^pow2, converted to binary16 exactly.
 */
#include <math.h>
#include <stdint.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ull

static uint64_t sm64_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream)
{
    return sm64_mix(seed ^ sm64_mix(stream + SM64_GAMMA));
}

static uint64_t draw(uint64_t key, uint64_t n)
{
    return sm64_mix(key + (n + 1) * SM64_GAMMA);
}

/* uniform in [0, 1) with 53 random bits */
static double unit53(uint64_t u)
{
    return (double)(u >> 11) * (1.0 / 9007199254740992.0);
}

/* double -> binary16 bits, round to nearest even (finite inputs of modest
 * size; overflow saturates to inf). */
static uint16_t to_half_bits(double v)
{
    uint16_t sign = (v < 0.0 || (v == 0.0 && signbit(v))) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);
    int e;
    double q;
    if (a < 6.103515625e-05) {               /* below 2^-14: subnormal step */
        q = 5.9604644775390625e-08;          /* 2^-24 */
    } else {
        (void)frexp(a, &e);
        q = ldexp(1.0, e - 11);
    }
    double n = a / q;
    double f = floor(n);
    double d = n - f;
    if (d > 0.5 || (d == 0.5 && fmod(f, 2.0) != 0.0)) f += 1.0;
    /* f * q is now an exact binary16 magnitude; encode it */
    double r = f * q;
    if (r == 0.0) return sign;
    if (r < 6.103515625e-05) return (uint16_t)(sign | (uint16_t)f);
    double m = frexp(r, &e);                 /* r = m 2^e, m in [0.5, 1) */
    int be = e + 14;                         /* biased exponent */
    if (be >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)(be << 10) | (uint16_t)((int)(m * 2048.0) - 1024));
}

void synth_normal_f16(uint64_t seed, uint64_t stream, double sigma, int64_t offset,
                      int64_t n, uint16_t *out)
{
    const uint64_t key = stream_key(seed, stream);
    const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t idx = (uint64_t)(offset + i);
        double u1 = 1.0 - unit53(draw(key, 2 * idx));     /* (0, 1] */
        double u2 = unit53(draw(key, 2 * idx + 1));
        double z = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
        out[i] = to_half_bits(sigma * z);
    }
}

void synth_int_f16(uint64_t seed, uint64_t stream, int lo, int hi, int pow2,
                   int64_t offset, int64_t n, uint16_t *out)
{
    const uint64_t key = stream_key(seed, stream);
    const uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo + 1);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t u = draw(key, 2 * (uint64_t)(offset + i));
        uint64_t k = (uint64_t)(((unsigned __int128)u * span) >> 64);
        double v = ldexp((double)((int64_t)lo + (int64_t)k), pow2);
        out[i] = to_half_bits(v);
    }
}

/* raw 64-bit draws, for choosing sample rows etc. */
void synth_u64(uint64_t seed, uint64_t stream, int64_t offset, int64_t n, uint64_t *out)
{
    const uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = draw(key, (uint64_t)(offset + i));
}
