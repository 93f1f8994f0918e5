/*
 * CPU oracle for the partitioned mixed-precision ZeRO Adam step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load this code; the product
 * path never does.  It shares no code with the CUDA kernels.
 *
 * Every function is a plain loop over elements, in IEEE binary32 unless
 * stated otherwise, with each operation rounded on its own: the file is
 * compiled with -ffp-contract=off so that no multiply-add is fused.  The
 * optional OpenMP pragmas only split independent elements between threads;
 * they never change a result (the one reduction kept in a fixed order,
 * orc_sumsq, is not parallelised).
 *
 * Sources (the five web pages on DeepSpeed ZeRO):
 *  - "DeepSpeed ZeRO" (formulaic.cloudchewie.com), "ZeRO Stage 1: 切分优化器状态",
 *    sub-sections "权重更新的触发条件" (skip on NaN/Inf, fp32 -> fp16 copy in
 *    place), "以 AdaW 为例" (the m, v, W update) and "具体训练步骤" (local update
 *    of the 1/N_d slice, cast to bf16, all-gather);
 *    "ZeRO Stage 2: 切分梯度" (reduce-scatter of the gradients, fp32 gradients
 *    made from the reduce-scattered half gradients, per-element independence);
 *    "ZeRO Stage 3: 切分参数" / "参数的初始化和切割" (flatten to 1-D and pad).
 *  - "zero-optimizer" (codezrq.github.io), section 2.5 ReduceScatter.
 *  - IEEE 754-2008 binary16 / binary32 formats; bfloat16 is the upper 16 bits
 *    of binary32.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { ORC_F16 = 0, ORC_BF16 = 1 };

/* ------------------------------------------------------------------------ */
/* Format conversions, written from the format definitions.                  */
/* ------------------------------------------------------------------------ */

/* binary16 bits -> binary32 value.  binary16: 1 sign bit, 5 exponent bits
 * (bias 15), 10 fraction bits.  Every binary16 value is exact in binary32. */
float orc_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1F;
    int frac = h & 0x3FF;
    float mag;
    if (ex == 0)
        mag = ldexpf((float)frac, -24); /* subnormal: frac * 2^(1-15-10) */
    else if (ex == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexpf((float)(1024 + frac), ex - 25); /* (1 + frac/2^10) * 2^(ex-15) */
    return sign ? -mag : mag;
}

/* bfloat16 bits -> binary32 value: bfloat16 is the upper half of binary32. */
float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static float half_to_f32(uint16_t x, int dtype)
{
    return dtype == ORC_F16 ? orc_f16_to_f32(x) : orc_bf16_to_f32(x);
}

/*
 * Round a binary32 value to a format with `p` significant bits, minimum
 * normal exponent `emin`, maximum finite value (2 - 2^(1-p)) * 2^emax,
 * to nearest with ties to even, and return the encoded bits.
 *
 * Method: every representable value of the target format with exponent e is
 * k * 2^(e - p + 1) for an integer k.  For finite |x| > 0 take
 * e = max(floor(log2 |x|), emin) and q = |x| / 2^(e - p + 1); scaling by a
 * power of two is exact in double, and rint() (the default rounding mode is
 * round-half-even) gives the nearest k with ties to even.  x is a double, so
 * both binary32 values and exact sums of two half-precision values are
 * rounded once.
 * k = 2^p means the value rounded up into the next binade.
 */
static uint16_t round_to_format(double x, int p, int emin, int emax, int bias, uint16_t qnan)
{
    uint16_t sign = (uint16_t)(signbit(x) ? 0x8000u : 0u);
    int fbits = p - 1; /* stored fraction bits */
    if (isnan(x))
        return (uint16_t)(sign | qnan);
    uint16_t inf_bits = (uint16_t)(((1u << (15 - fbits)) - 1u) << fbits);
    if (isinf(x))
        return (uint16_t)(sign | inf_bits);
    double ax = fabs(x);
    if (ax == 0.0)
        return sign;
    int e2;
    frexp(ax, &e2);     /* ax = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;     /* floor(log2 ax) */
    if (e < emin)
        e = emin;       /* subnormal range shares the minimum exponent */
    int shift = e - fbits;
    double q = ldexp(ax, -shift);
    double k = rint(q);
    if (k == ldexp(1.0, p)) { /* carried into the next binade */
        k = ldexp(1.0, fbits);
        e += 1;
    }
    if (e > emax)
        return (uint16_t)(sign | inf_bits);
    uint32_t kk = (uint32_t)k;
    if (kk < (1u << fbits))  /* subnormal (or rounded to zero) */
        return (uint16_t)(sign | kk);
    uint32_t biased = (uint32_t)(e + bias);
    return (uint16_t)(sign | (biased << fbits) | (kk - (1u << fbits)));
}

/* binary32 -> binary16, round to nearest, ties to even; overflow -> +-Inf. */
uint16_t orc_f32_to_f16(float x)
{
    return round_to_format(x, 11, -14, 15, 15, 0x7E00);
}

/* binary32 -> bfloat16, round to nearest, ties to even; overflow -> +-Inf. */
uint16_t orc_f32_to_bf16(float x)
{
    return round_to_format(x, 8, -126, 127, 127, 0x7FC0);
}

void orc_to_half_array(const float *x, int64_t n, int dtype, uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = dtype == ORC_F16 ? orc_f32_to_f16(x[i]) : orc_f32_to_bf16(x[i]);
}

void orc_from_half_array(const uint16_t *x, int64_t n, int dtype, float *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = half_to_f32(x[i], dtype);
}

/* ------------------------------------------------------------------------ */
/* Step (a2): reduce-scatter sum for one rank.                              */
/* ------------------------------------------------------------------------ */

/*
 * g[j] = sum over q = 0 .. world-1 of float(G_q[offset + j]), for j < n.
 * ReduceScatter ("zero-optimizer", section 2.5; "DeepSpeed ZeRO", ZeRO Stage 2):
 * every rank ends with the element-wise reduction of all ranks' gradients over
 * its own 1/N_d slice.  The reduction is a sum, accumulated in binary32 from
 * +0, in ascending rank order, with no intermediate rounding to half.
 */
void orc_reduce_sum(const uint16_t *const *grads, int world, int dtype, int64_t offset,
                    int64_t n, float *g)
{
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) {
        float acc = 0.0f;
        for (int q = 0; q < world; ++q)
            acc = acc + half_to_f32(grads[q][offset + j], dtype);
        g[j] = acc;
    }
}

/* Gradient accumulation over micro-steps: acc[j] = acc[j] + r[j]
 * in binary32, where r is one micro-step's reduce-scattered sum.  "DeepSpeed
 * ZeRO", "ZeRO-2 在梯度累积场景下的通信量": ZeRO-2 reduce-scatters after every
 * backward and accumulates its 1/N_d slice; the memory section of the same
 * page lists the optional fp32 gradient copy used to accumulate in fp32. */
void orc_accumulate(float *acc, const float *r, int64_t n)
{
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        acc[j] = acc[j] + r[j];
}

/*
 * Step (a2) with the reduction itself in half precision: the
 * running sum is kept in the gradient's type and rounded to nearest even
 * after every addition, in ascending rank order from +0, as a half-precision
 * reduce-scatter produces it ("DeepSpeed ZeRO", ZeRO Stage 2: the fp32
 * gradient slice is made from the reduce-scattered BF16 gradient).  Each
 * addition forms the sum of two half values in binary64 and rounds it to the
 * half type: the binary64 sum is exact for fp16 (exponents span < 42 bits);
 * for bf16 it is exact unless the two exponents differ by more than 45, and
 * then the smaller value lies far below half an ulp of the result, so the
 * single rounding still gives the correctly rounded half-precision sum.
 * Overflow gives +-Inf and Inf + -Inf gives NaN.
 */
void orc_reduce_sum_half(const uint16_t *const *grads, int world, int dtype, int64_t offset,
                         int64_t n, float *g)
{
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int q = 0; q < world; ++q) {
            double exact = acc + (double)half_to_f32(grads[q][offset + j], dtype);
            uint16_t h = dtype == ORC_F16 ? round_to_format(exact, 11, -14, 15, 15, 0x7E00)
                                          : round_to_format(exact, 8, -126, 127, 127, 0x7FC0);
            acc = (double)half_to_f32(h, dtype);
        }
        g[j] = (float)acc;
    }
}

/* Step (a3): unscale by the loss scale S; inv_scale = 1/S (a power of two). */
void orc_unscale(float *g, int64_t n, float inv_scale)
{
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        g[j] = g[j] * inv_scale;
}

/* Step (a4): 1 if any element is NaN or +-Inf ("DeepSpeed ZeRO", ZeRO Stage 1,
 * "权重更新的触发条件": such a step does not update the weights). */
int orc_any_nonfinite(const float *g, int64_t n)
{
    int found = 0;
#pragma omp parallel for schedule(static) reduction(| : found)
    for (int64_t j = 0; j < n; ++j)
        found |= !isfinite(g[j]);
    return found;
}

/* Step (a5): the sum of squares sum_j g_j^2 behind the global L2 gradient norm
 * ("zero-optimizer", "一. 优化前": gradient-norm computation over fused
 * buffers), continued from (*sum, *comp).  Each square is exact in binary64; the squares are added in sequence with
 * Neumaier's compensated summation (Kahan-Babuska), which keeps the rounding
 * error of every addition in *comp, so *sum + *comp is within a few ulps of
 * the exact sum for any length (a plain sequential binary64 sum drifts by
 * ~1e-9 relative over 1e9 such terms). */
void orc_sumsq(const float *g, int64_t n, double *sum, double *comp)
{
    double s = *sum, c = *comp;
    for (int64_t j = 0; j < n; ++j) {
        double d = (double)g[j];
        double t = d * d;
        double u = s + t;
        if (fabs(s) >= fabs(t))
            c = c + ((s - u) + t);
        else
            c = c + ((t - u) + s);
        s = u;
    }
    *sum = s;
    *comp = c;
}

/* Step (a5), clip: g = g * c in binary32. */
void orc_scale(float *g, int64_t n, float c)
{
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        g[j] = g[j] * c;
}

/* ------------------------------------------------------------------------ */
/* Step (a6): Adam / AdamW on the fp32 master weights, momentum, variance.   */
/* ------------------------------------------------------------------------ */

/*
 * Per-step binary32 scalars, computed by the caller in double and rounded
 * once:  b1 = beta1, omb1 = 1 - beta1, b2 = beta2, omb2 = 1 - beta2,
 * step = lr / (1 - beta1^t), rbc2 = sqrt(1 - beta2^t), eps, decay = 1 - lr*wd
 * (decoupled decay), wd (coupled L2 decay, used when adamw == 0).
 */
typedef struct {
    float b1, omb1, b2, omb2, step, rbc2, eps, decay, wd;
    int32_t adamw;
} orc_scalars;

/*
 * "DeepSpeed ZeRO", ZeRO Stage 1, "以 AdaW 为例":
 *   m_t = beta1 m_{t-1} + (1 - beta1) g
 *   v_t = beta2 v_{t-1} + (1 - beta2) g^2
 *   W_t = W_{t-1} - eta m_t / (sqrt(v_t) + eps)
 * with the bias correction of Kingma and Ba (Algorithm 1) folded into
 * step = eta / (1 - beta1^t) and sqrt(v_t) / sqrt(1 - beta2^t), and, for
 * AdamW (Loshchilov and Hutter), the decoupled decay W <- W (1 - eta wd)
 * applied before the Adam update.  Each binary32 operation is rounded alone.
 */
void orc_adam(const float *g_in, float *w, float *m, float *v, int64_t n, const orc_scalars *s)
{
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) {
        float g = g_in[j];
        float wj = w[j];
        if (!s->adamw && s->wd != 0.0f)
            g = g + s->wd * wj; /* coupled L2 term (Adam with weight decay) */
        float mj = s->b1 * m[j] + s->omb1 * g;
        float vj = s->b2 * v[j] + s->omb2 * (g * g);
        if (s->adamw)
            wj = wj * s->decay;
        float den = sqrtf(vj) / s->rbc2 + s->eps;
        wj = wj - s->step * (mj / den);
        m[j] = mj;
        v[j] = vj;
        w[j] = wj;
    }
}
