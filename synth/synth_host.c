/*
 * Seeded synthetic inputs, CPU side.
 *
 * Test and benchmark infrastructure only: this file builds the inputs that
 * both the CPU oracle and the CUDA step receive.  It holds none of the
 * optimizer step's arithmetic.  synth_cuda.cu computes the very same values
 * on the GPU; the two are written independently from the same definition
 * and a GPU test checks that they agree bit for bit.
 *
 * Definition (shared by both sides):
 *   SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 *   generators", OOPSLA 2014): the n-th output (n = 0, 1, ...) of a generator
 *   seeded with s is mix64(s + (n + 1) * 0x9E3779B97F4A7C15), where
 *     mix64(z): z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *               z = (z ^ (z >> 27)) * 0x94D049BB133111EB
 *               return z ^ (z >> 31)            (all arithmetic mod 2^64)
 *   key(seed, stream) = output number `stream` of SplitMix64(seed).
 *   Element i of a stream uses outputs 2i and 2i+1 of SplitMix64(key): a, b.
 *   Irwin-Hall sum of four 32-bit uniforms:
 *     s = lo32(a) + hi32(a) + lo32(b) + hi32(b)          (exact, uint64)
 *     c = s - (2^33 - 2)                                  (exact, int64; mean 0)
 *   The variance of c is (2^64 - 1) / 3, so c / sqrt((2^64 - 1) / 3) has mean
 *   0 and standard deviation 1, with support |z| <= sqrt(3) * 2 = 3.4641.
 *     x = float(c) * scale        (int64 -> fp32 round-to-nearest-even, then
 *                                  one fp32 multiply, round-to-nearest-even)
 *   scale = fp32(sigma / sqrt((2^64 - 1) / 3)), computed once by the caller.
 *   Half-precision outputs round x to nearest even (IEEE 754 binary16, or
 *   bfloat16 = the upper 16 bits of binary32 after rounding).
 */
#include <stdint.h>
#include <string.h>

#define SM_GAMMA 0x9E3779B97F4A7C15ULL

static uint64_t sm_mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static uint64_t sm_output(uint64_t seed, uint64_t n)
{
    return sm_mix64(seed + (n + 1u) * SM_GAMMA);
}

uint64_t synth_key(uint64_t seed, uint64_t stream)
{
    return sm_output(seed, stream);
}

static float synth_value(uint64_t key, uint64_t i, float scale)
{
    uint64_t a = sm_output(key, 2u * i);
    uint64_t b = sm_output(key, 2u * i + 1u);
    uint64_t s = (a & 0xFFFFFFFFULL) + (a >> 32) + (b & 0xFFFFFFFFULL) + (b >> 32);
    int64_t c = (int64_t)s - (int64_t)8589934590LL; /* 2^33 - 2 */
    float f = (float)c;                             /* RNE (default rounding mode) */
    return f * scale;                               /* one fp32 multiply */
}

static uint32_t f32_bits(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    return u;
}

/* binary32 -> binary16, round to nearest, ties to even. */
static uint16_t to_f16_bits(float x)
{
    uint32_t u = f32_bits(x);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t ex = (u >> 23) & 0xFFu;
    uint32_t man = u & 0x7FFFFFu;
    if (ex == 0xFFu) /* Inf or NaN (NaN made quiet) */
        return (uint16_t)(sign | 0x7C00u | (man ? 0x200u | (man >> 13) : 0u));
    int32_t e = (int32_t)ex - 127 + 15; /* biased binary16 exponent */
    if (e >= 31)
        return (uint16_t)(sign | 0x7C00u);
    if (e <= 0) {
        /* subnormal or zero in binary16: the value is full * 2^(e - 14) in
         * units of the smallest subnormal, 2^-24 */
        if (e < -10)
            return sign; /* below half of the smallest subnormal */
        uint32_t full = man | 0x800000u;            /* 24-bit significand */
        uint32_t shift = (uint32_t)(14 - e);        /* bits dropped */
        uint32_t q = full >> shift;
        uint32_t rem = full & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1u);
        if (rem > half || (rem == half && (q & 1u)))
            q += 1u;
        return (uint16_t)(sign | q);
    }
    uint32_t q = ((uint32_t)e << 10) | (man >> 13);
    uint32_t rem = man & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (q & 1u)))
        q += 1u; /* may carry into the exponent; 0x7C00 = Inf is correct */
    return (uint16_t)(sign | q);
}

/* binary32 -> bfloat16, round to nearest, ties to even. */
static uint16_t to_bf16_bits(float x)
{
    uint32_t u = f32_bits(x);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu))
        return (uint16_t)((u >> 16) | 0x40u); /* quiet NaN */
    uint32_t lower = u & 0xFFFFu;
    uint32_t q = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (q & 1u)))
        q += 1u;
    return (uint16_t)q;
}

void synth_fill_f32(uint64_t key, uint64_t first, int64_t n, float scale, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = synth_value(key, first + (uint64_t)i, scale);
}

/* dtype: 0 = binary16, 1 = bfloat16 */
void synth_fill_half(uint64_t key, uint64_t first, int64_t n, float scale, int dtype,
                     uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) {
        float x = synth_value(key, first + (uint64_t)i, scale);
        out[i] = dtype == 0 ? to_f16_bits(x) : to_bf16_bits(x);
    }
}

/* Round an existing fp32 array to half bits (used to seed the initial half
 * parameter buffer from the initial fp32 master weights). */
void synth_round_half(const float *x, int64_t n, int dtype, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = dtype == 0 ? to_f16_bits(x[i]) : to_bf16_bits(x[i]);
}
