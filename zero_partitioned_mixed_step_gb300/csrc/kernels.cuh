// Device helpers of the step kernels: 16-byte loads and stores, the
// rank-ordered reduction of one 8-element unit, the per-step scalars, the
// Adam update, the round-to-nearest-even cast and the deterministic
// sum-of-squares reduction.
//
// Arithmetic conventions (they make the GPU results reproduce the CPU
// oracle's bits): every binary32 operation is an explicitly rounded
// intrinsic (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn ...), so nothing is
// contracted into a fused multiply-add; per-step scalars are computed in
// binary64 with IEEE division and square root and rounded once to binary32.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "internal.h"

namespace zs {

// ------------------------------------------------------------------ memory
//
// Every stream is touched once per step and a step moves far more than the
// L2, so all accesses skip L1 and are marked evict-first in L2.  16-byte
// accesses take the hint through an L2 cache policy; 256-bit accesses carry
// it directly.

__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// The same hint the other way round, for data that a second pass reads again
// while it can still be in L2 (the tail of a clipped step's first pass).
__device__ __forceinline__ uint64_t evict_last_policy()
{
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16 bytes of one rank's gradient (read-only during the kernel).
__device__ __forceinline__ uint4 ld_stream(const uint16_t *p, uint64_t pol)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p), "l"(pol));
    return r;
}

// ld_stream issued where it is written (not moved past a later barrier).
__device__ __forceinline__ uint4 ld_stream_now(const uint16_t *p, uint64_t pol)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(pol));
    return r;
}

// 8 fp32 values (32 bytes, 32-byte aligned) in one 256-bit access.  The
// coherent path is used because a clipped step may update the state in place.
__device__ __forceinline__ void load8(const float *p, float x[8])
{
    uint32_t u[8];
    asm("ld.global.L1::no_allocate.L2::evict_first.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7])
        : "l"(p));
#pragma unroll
    for (int i = 0; i < 8; ++i)
        x[i] = __uint_as_float(u[i]);
}

// load8 issued where it is written (not moved past a later barrier).
__device__ __forceinline__ void load8_now(const float *p, float x[8])
{
    uint32_t u[8];
    asm volatile(
        "ld.global.L1::no_allocate.L2::evict_first.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7])
        : "l"(p));
#pragma unroll
    for (int i = 0; i < 8; ++i)
        x[i] = __uint_as_float(u[i]);
}

__device__ __forceinline__ void store8(float *p, const float x[8])
{
    asm volatile(
        "st.global.L1::no_allocate.L2::evict_first.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
        :
        : "l"(p), "r"(__float_as_uint(x[0])), "r"(__float_as_uint(x[1])),
          "r"(__float_as_uint(x[2])), "r"(__float_as_uint(x[3])), "r"(__float_as_uint(x[4])),
          "r"(__float_as_uint(x[5])), "r"(__float_as_uint(x[6])), "r"(__float_as_uint(x[7]))
        : "memory");
}

// load8 / store8 marked evict-last in L2.
__device__ __forceinline__ void load8_keep(const float *p, float x[8])
{
    uint32_t u[8];
    asm("ld.global.L1::no_allocate.L2::evict_last.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7])
        : "l"(p));
#pragma unroll
    for (int i = 0; i < 8; ++i)
        x[i] = __uint_as_float(u[i]);
}

__device__ __forceinline__ void store8_keep(float *p, const float x[8])
{
    asm volatile(
        "st.global.L1::no_allocate.L2::evict_last.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
        :
        : "l"(p), "r"(__float_as_uint(x[0])), "r"(__float_as_uint(x[1])),
          "r"(__float_as_uint(x[2])), "r"(__float_as_uint(x[3])), "r"(__float_as_uint(x[4])),
          "r"(__float_as_uint(x[5])), "r"(__float_as_uint(x[6])), "r"(__float_as_uint(x[7]))
        : "memory");
}

// Drop the 128-byte L2 line at p (128-byte aligned) without writing it back:
// its contents become undefined.  Used on a scratch line whose last reader
// has read it, so that a line the step no longer needs is not written back if
// it is still dirty.  (Measured with warm caches on the 124M-element clipped
// step, L2 had already written back all but ~7 MB of the 64 MB kept tail by
// the end of the first pass, so this saves little; the kept tail's gain is
// the second pass's reads.)
__device__ __forceinline__ void discard_l2_line(const void *p)
{
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// The same 8 fp32 values in pinned host memory, reached over the host link:
// two ordinary 16-byte accesses (zero-copy), evict-first in L2.
__device__ __forceinline__ void load8_host(const float *p, float x[8])
{
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4 *>(p + 4));
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void store8_host(float *p, const float x[8])
{
    __stcs(reinterpret_cast<float4 *>(p), make_float4(x[0], x[1], x[2], x[3]));
    __stcs(reinterpret_cast<float4 *>(p + 4), make_float4(x[4], x[5], x[6], x[7]));
}

// 16 bytes of half-precision parameters.
__device__ __forceinline__ void st_half8(uint16_t *p, uint4 v, uint64_t pol)
{
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;"
                 :
                 : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

// 4 fp32 values (16-byte aligned).
__device__ __forceinline__ float4 ld_state4(const float *p)
{
    return __ldcs(reinterpret_cast<const float4 *>(p));
}

// ------------------------------------------------------------------ conversions

// DT is a zero_dtype: bit 0 selects bfloat16 (else binary16), bit 1 a
// reduction carried out in that type instead of in fp32.
__host__ __device__ constexpr bool is_bf16(int dt) { return (dt & 1) != 0; }
__host__ __device__ constexpr bool half_reduce(int dt) { return (dt & 2) != 0; }

// Add the 8 half-precision values of x (exactly converted to fp32) to acc.
template <int DT>
__device__ __forceinline__ void add_half8(float acc[8], const uint4 x)
{
    const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float lo, hi;
        if constexpr (!is_bf16(DT)) {
            __half2 h = *reinterpret_cast<const __half2 *>(&u[j]);
            float2 f = __half22float2(h);
            lo = f.x;
            hi = f.y;
        } else {
            lo = __uint_as_float(u[j] << 16);
            hi = __uint_as_float(u[j] & 0xFFFF0000u);
        }
        acc[2 * j] = __fadd_rn(acc[2 * j], lo);
        acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], hi);
    }
}

// Round 8 fp32 values to half precision, nearest even, packed little-endian.
template <int DT>
__device__ __forceinline__ uint4 pack_half8(const float w[8])
{
    uint32_t u[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if constexpr (!is_bf16(DT)) {
            __half2 h = __floats2half2_rn(w[2 * j], w[2 * j + 1]);
            u[j] = *reinterpret_cast<uint32_t *>(&h);
        } else {
            __nv_bfloat162 b = __floats2bfloat162_rn(w[2 * j], w[2 * j + 1]);
            u[j] = *reinterpret_cast<uint32_t *>(&b);
        }
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
}

// Half-precision running sums: acc holds 4 packed pairs in the gradient's type;
// add the 8 values of x with one round-to-nearest-even addition per element.
template <int DT>
__device__ __forceinline__ void add_half8_in_half(uint32_t acc[4], const uint4 x)
{
    const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if constexpr (!is_bf16(DT)) {
            __half2 a = *reinterpret_cast<const __half2 *>(&acc[j]);
            a = __hadd2(a, *reinterpret_cast<const __half2 *>(&u[j]));
            acc[j] = *reinterpret_cast<uint32_t *>(&a);
        } else {
            __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&acc[j]);
            a = __hadd2(a, *reinterpret_cast<const __nv_bfloat162 *>(&u[j]));
            acc[j] = *reinterpret_cast<uint32_t *>(&a);
        }
    }
}

__device__ __forceinline__ bool nonfinite(float x)
{
    return (__float_as_uint(x) & 0x7F800000u) == 0x7F800000u;
}

// ------------------------------------------------------------------ reduce-scatter

template <int MAXW>
struct GradTable {
    const uint16_t *p[MAXW];
};

// acc[i] = sum over q of float(grads[q][gi + i]), i < 8, in ascending q from +0.
// W > 0: the group size is known at compile time and loads are issued in
// batches of up to 16 ranks before they are summed; W == 0: `world` at run time.
template <int DT, int W, int MAXW>
__device__ __forceinline__ void reduce_unit(const GradTable<MAXW> &t, int world, int64_t gi,
                                            float acc[8], uint64_t pol)
{
    if constexpr (half_reduce(DT)) {
        // running sums in the half type, from +0, one rounding per addition
        uint32_t h[4] = {0u, 0u, 0u, 0u};
        int q = 0;
        for (; q + 8 <= world; q += 8) {
            uint4 x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                x[j] = ld_stream(t.p[q + j] + gi, pol);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                add_half8_in_half<DT>(h, x[j]);
        }
        for (; q < world; ++q)
            add_half8_in_half<DT>(h, ld_stream(t.p[q] + gi, pol));
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[i] = 0.0f;
        add_half8<DT>(acc, make_uint4(h[0], h[1], h[2], h[3]));  // exact widening
        return;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        acc[i] = 0.0f;
    if constexpr (W > 0) {
        constexpr int CH = W < 16 ? W : 16;
#pragma unroll
        for (int q0 = 0; q0 < W; q0 += CH) {
            uint4 x[CH];
#pragma unroll
            for (int j = 0; j < CH; ++j)
                x[j] = ld_stream(t.p[q0 + j] + gi, pol);
#pragma unroll
            for (int j = 0; j < CH; ++j)
                add_half8<DT>(acc, x[j]);
        }
    } else {
        int q = 0;
        for (; q + 8 <= world; q += 8) {
            uint4 x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                x[j] = ld_stream(t.p[q + j] + gi, pol);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                add_half8<DT>(acc, x[j]);
        }
        for (; q < world; ++q)
            add_half8<DT>(acc, ld_stream(t.p[q] + gi, pol));
    }
}

// ------------------------------------------------------------------ element mapping

// Which elements a launch covers.  A launch walks units u = 0 .. units - 1
// with a grid stride over a one-dimensional grid.
//  - every rank at once (all_ranks): the union of the partitions is the whole
//    padded flat vector, so unit u is flat elements 8u .. 8u + 7 and the
//    state buffers are flat too;
//  - one rank r: unit u is r's u-th group of 8 owned elements; its flat
//    position follows the partition (or bucket-slice) layout, and the state
//    buffers hold r's elements in order.
struct View {
    int64_t units;         // units the launch covers
    int64_t part;          // owned_numel (flat stride between partitions, not bucketed)
    int64_t bucket;        // elements per bucket, 0 = not bucketed
    int64_t slice;         // a rank's elements in a full bucket
    int64_t slice_units;   // slice / 8
    int64_t full_units;    // units in the full buckets: (num_buckets - 1) * slice_units
    int64_t last_base;     // flat start of the last bucket
    int64_t last_slice;    // a rank's elements in the last bucket
    int32_t rank;          // the simulated rank when !all_ranks
    int32_t all_ranks;
    int32_t grads_are_slices;
    int32_t world;
};

// Flat element index of rank r's owned unit k (one-rank view).
__device__ __forceinline__ int64_t flat_of(const View &v, int r, int64_t k)
{
    const int64_t e = k * kUnit;
    if (v.bucket == 0)
        return (int64_t)r * v.part + e;
    if (k < v.full_units) {
        int64_t b;
        if (v.full_units < (INT64_C(1) << 32))
            b = (int64_t)((uint32_t)k / (uint32_t)v.slice_units);
        else
            b = k / v.slice_units;
        return b * v.bucket + (int64_t)r * v.slice + (e - b * v.slice);
    }
    return v.last_base + (int64_t)r * v.last_slice + (e - v.full_units * kUnit);
}

// Flat index f, state index si and gradient index gi of unit u.
template <bool ALL>
__device__ __forceinline__ void locate(const View &v, int64_t u, int64_t &f, int64_t &si,
                                       int64_t &gi)
{
    if constexpr (ALL) {
        f = si = gi = u * kUnit;
    } else {
        f = flat_of(v, v.rank, u);
        si = u * kUnit;
        gi = v.grads_are_slices ? si : f;
    }
}

// ------------------------------------------------------------------ per-step scalars

struct Scalars {
    float inv_s, b1, omb1, b2, omb2, step, rbc2, eps, decay, wd, coef;
    int32_t adamw, clip, skip;
};

// Clip coefficient min(1, max_norm / (sqrt(sumsq) + 1e-6)), binary64 rounded
// once to binary32.
__device__ __forceinline__ float clip_coefficient(double sumsq, double max_norm)
{
    return __double2float_rn(fmin(1.0, __ddiv_rn(max_norm, __dadd_rn(__dsqrt_rn(sumsq), 1e-6))));
}

// One entry of zero_step_state::scalar_cache: the bias-correction scalars of
// one step and every input they were formed from.
struct ScalarCacheEntry {
    double lr, beta1, beta2;
    double beta1_pow, beta2_pow;  // the state's beta powers at the start of that step
    float step, rbc2;
    uint32_t tag, pad0;
    uint64_t pad1;
};
static_assert(sizeof(ScalarCacheEntry) == 64, "two entries fill scalar_cache");
static_assert(offsetof(zero_step_state, scalar_cache) == 64 && sizeof(zero_step_state) == 192,
              "zero_step_state layout");
constexpr uint32_t kScalarCacheTag = 0x5a530c01u;  // marks an entry the library wrote

__device__ __forceinline__ bool same_bits(double a, double b)
{
    return __double_as_longlong(a) == __double_as_longlong(b);
}

// step = lr / (1 - beta1^t) and rbc2 = sqrt(1 - beta2^t) from the beta powers
// at the start of the step (beta^t = beta_pow * beta), in binary64 rounded
// once to binary32.
__device__ __forceinline__ float bias_step(const CfgDev &c, double beta1_pow)
{
    return __double2float_rn(__ddiv_rn(c.lr, __dsub_rn(1.0, __dmul_rn(beta1_pow, c.beta1))));
}

__device__ __forceinline__ float bias_rbc2(const CfgDev &c, double beta2_pow)
{
    return __double2float_rn(__dsqrt_rn(__dsub_rn(1.0, __dmul_rn(beta2_pow, c.beta2))));
}

// Scalars of step t + 1 from the state at the start of the step.  Thread 0
// reads the state's flags and the slot; step and rbc2 come from the scalar
// cache entry of the slot when that entry was formed from exactly this
// step's lr, betas and beta powers (the values are then the ones the formula
// gives), else thread 0 forms step and thread 32 rbc2 here, in different
// warps so that the binary64 division and square root (slow on GB300's
// binary64 pipe) overlap.  Each of the two threads loads both entries along
// with the state, so that no load waits on the slot index.  Thread 64 forms
// the clip coefficient when `total` (the step's global sum of squares) is
// given.  ADAM = false (a first pass) forms only the flags, the slot and
// 1/S.  The configuration-only values were rounded on the host (make_cfg_dev).
// A barrier must follow before sh is read; every CTA has at least 96 threads.
template <bool ADAM>
__device__ __forceinline__ void form_scalars(const CfgDev &c, const zero_step_state *st,
                                             const double *total, Scalars &sh, int &sh_cur)
{
    const ScalarCacheEntry *e = reinterpret_cast<const ScalarCacheEntry *>(st->scalar_cache);
    if (threadIdx.x == 0) {
        sh.b1 = c.b1;
        sh.omb1 = c.omb1;
        sh.b2 = c.b2;
        sh.omb2 = c.omb2;
        sh.eps = c.eps;
        sh.decay = c.decay;
        sh.wd = c.wd;
        sh.adamw = c.adamw;
        sh.clip = c.max_norm > 0.0;
        sh.inv_s = __fdiv_rn(1.0f, st->loss_scale);
        sh.skip = st->found_inf & 1;
        const int cur = st->cur;
        sh_cur = cur;
        if (ADAM) {
            if (!c.bias_correction) {
                sh.step = c.lr_f;
            } else {
                const double p = st->beta1_pow;
                const uint32_t t0 = e[0].tag, t1 = e[1].tag;
                const double l0 = e[0].lr, l1 = e[1].lr;
                const double b0 = e[0].beta1, b1 = e[1].beta1;
                const double q0 = e[0].beta1_pow, q1 = e[1].beta1_pow;
                const float s0 = e[0].step, s1 = e[1].step;
                const bool hit = cur ? t1 == kScalarCacheTag && same_bits(l1, c.lr) &&
                                           same_bits(b1, c.beta1) && same_bits(q1, p)
                                     : t0 == kScalarCacheTag && same_bits(l0, c.lr) &&
                                           same_bits(b0, c.beta1) && same_bits(q0, p);
                if (hit)
                    sh.step = cur ? s1 : s0;
                else
                    sh.step = bias_step(c, p);
            }
        }
    } else if (threadIdx.x == 32) {
        if (ADAM) {
            if (!c.bias_correction) {
                sh.rbc2 = 1.0f;
            } else {
                const int cur = st->cur;
                const double p = st->beta2_pow;
                const uint32_t t0 = e[0].tag, t1 = e[1].tag;
                const double b0 = e[0].beta2, b1 = e[1].beta2;
                const double q0 = e[0].beta2_pow, q1 = e[1].beta2_pow;
                const float r0 = e[0].rbc2, r1 = e[1].rbc2;
                const bool hit = cur ? t1 == kScalarCacheTag && same_bits(b1, c.beta2) &&
                                           same_bits(q1, p)
                                     : t0 == kScalarCacheTag && same_bits(b0, c.beta2) &&
                                           same_bits(q0, p);
                if (hit)
                    sh.rbc2 = cur ? r1 : r0;
                else
                    sh.rbc2 = bias_rbc2(c, p);
            }
        }
    } else if (threadIdx.x == 64) {
        sh.coef = total && c.max_norm > 0.0 ? clip_coefficient(__ldcg(total), c.max_norm) : 1.0f;
    }
}

// One thread of a kernel that updates with the state read at its start, before
// the kernel counts itself in found_inf (so before anything can end the
// step): forms the scalars of the NEXT step as they will be if this step
// commits (beta powers advanced by one factor, same configuration) into the
// cache entry of slot 1 - cur, the slot the next step reads after a commit,
// unless that entry holds them already.  If this step is skipped, the next
// step reads slot cur again, whose entry still matches its unchanged beta
// powers.  No reader uses entry 1 - cur while this step runs, and several
// launches of one step (bucket ranges) write the same values.  The slot and
// the beta powers are read here, not kept from the prologue, so that nothing
// stays live across the kernel's main loop for it.
__device__ __forceinline__ void form_next_scalars(const CfgDev &c, zero_step_state *st)
{
    if (!c.bias_correction)
        return;
    const int cur = st->cur;
    const double p1 = __dmul_rn(st->beta1_pow, c.beta1);
    const double p2 = __dmul_rn(st->beta2_pow, c.beta2);
    ScalarCacheEntry *e = reinterpret_cast<ScalarCacheEntry *>(st->scalar_cache) + (cur ^ 1);
    if (e->tag == kScalarCacheTag && same_bits(e->lr, c.lr) && same_bits(e->beta1, c.beta1) &&
        same_bits(e->beta2, c.beta2) && same_bits(e->beta1_pow, p1) &&
        same_bits(e->beta2_pow, p2))
        return;
    const float step = bias_step(c, p1);
    const float rbc2 = bias_rbc2(c, p2);
    e->lr = c.lr;
    e->beta1 = c.beta1;
    e->beta2 = c.beta2;
    e->beta1_pow = p1;
    e->beta2_pow = p2;
    e->step = step;
    e->rbc2 = rbc2;
    e->tag = kScalarCacheTag;
}

// ------------------------------------------------------------------ end of step

// What ending a step needs from the optimizer configuration.
struct FinCfg {
    double beta1, beta2, backoff, growth, min_scale;
    int32_t dynamic, interval;
};

inline FinCfg fin_cfg(const zero_adam_cfg &c)
{
    return FinCfg{c.beta1, c.beta2, c.backoff, c.growth, c.min_scale, c.dynamic_scale ? 1 : 0,
                  c.growth_interval};
}

// Step (a8) on the device state, one thread: skip (found = 1: count it, back
// the dynamic loss scale off) or commit (t + 1, beta powers, slot flip, good
// steps and loss-scale growth); found_inf is cleared either way.
__device__ __forceinline__ void end_step(const FinCfg &c, zero_step_state *st, int flip,
                                         int found)
{
    if (found) {
        st->overflow = 1;
        st->skipped += 1;
        if (c.dynamic) {
            const double s = __dmul_rn((double)st->loss_scale, c.backoff);
            st->loss_scale = __double2float_rn(s > c.min_scale ? s : c.min_scale);
            st->good_steps = 0;
        }
    } else {
        st->overflow = 0;
        st->t += 1;
        st->beta1_pow = __dmul_rn(st->beta1_pow, c.beta1);
        st->beta2_pow = __dmul_rn(st->beta2_pow, c.beta2);
        if (flip)
            st->cur ^= 1;
        st->good_steps += 1;
        if (c.dynamic && st->good_steps == c.interval) {
            st->loss_scale = __double2float_rn(__dmul_rn((double)st->loss_scale, c.growth));
            st->good_steps = 0;
        }
    }
    st->found_inf = 0;
}

// The end of a kernel, called by every thread of every CTA: OR the CTA's
// non-finite flag into bit 0 of found_inf and, when the launch is the step's
// last, count the CTA in the bits above; the CTA whose count completes the
// grid ends the step (commit or skip, a8), so no separate launch is needed.
// One thread does both atomics, the OR first: one thread's atomics on one
// word stay in order, so the count the last CTA sees carries every CTA's
// flag, and no fence is needed (what the step wrote reaches the next kernel
// through the kernel boundary).  found_inf is 0 between steps (end_step
// clears it), and every CTA reads the state it needs when it starts, before
// it counts itself, so the commit never races a reader.
__device__ __forceinline__ void finish_cta(bool bad, bool ends, const FinCfg &c,
                                           zero_step_state *st)
{
    const int any = __syncthreads_or(bad ? 1 : 0);
    if (threadIdx.x != 0)
        return;
    if (any)
        atomicOr(&st->found_inf, 1);
    if (!ends)
        return;
    const int32_t old = atomicAdd(&st->found_inf, 2);
    if ((old >> 1) == (int32_t)gridDim.x - 1)
        end_step(c, st, 1, old & 1);
}

// ------------------------------------------------------------------ Adam

// One AdamW / Adam step on one element (binary32, each operation rounded):
//   [coupled L2: g += wd w]
//   m = b1 m + (1 - b1) g;  v = b2 v + (1 - b2) g^2
//   [decoupled: w = w (1 - lr wd)]
//   w = w - step * (m / (sqrt(v) / sqrt(1 - b2^t) + eps)),  step = lr / (1 - b1^t)
__device__ __forceinline__ void adam1(float g, float &w, float &m, float &v, const Scalars &s)
{
    if (!s.adamw && s.wd != 0.0f)
        g = __fadd_rn(g, __fmul_rn(s.wd, w));
    const float mi = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
    const float vi = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
    float wi = s.adamw ? __fmul_rn(w, s.decay) : w;
    const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(vi), s.rbc2), s.eps);
    wi = __fsub_rn(wi, __fmul_rn(s.step, __fdiv_rn(mi, den)));
    m = mi;
    v = vi;
    w = wi;
}

__device__ __forceinline__ void adam8(const float g[8], float w[8], float m[8], float v[8],
                                      const Scalars &s)
{
#pragma unroll
    for (int i = 0; i < 8; ++i)
        adam1(g[i], w[i], m[i], v[i], s);
}

template <int DT>
__device__ __forceinline__ uint16_t round_half1(float w)
{
    if constexpr (!is_bf16(DT))
        return __half_as_ushort(__float2half_rn(w));
    else
        return __bfloat16_as_ushort(__float2bfloat16_rn(w));
}

// ------------------------------------------------------------------ sum of squares
//
// Squares are summed in pairs of binary32 values (hi, lo) whose sum carries
// about 48 significant bits, without binary64 arithmetic in the streaming
// loops (GB300 issues binary64 at a small fraction of the binary32 rate):
// each square is split exactly into p + e (p = fl(g*g), e = fma(g, g, -p)),
// a unit's p are added with Knuth's TwoSum so their rounding errors are kept,
// and pairs are added with a TwoSum on the high parts followed by a
// renormalisation.  All terms are squares, so no cancellation occurs and the
// relative error of every pair addition stays at a few units of 2^-48.  A
// pair becomes binary64 only at the end of a chunk (one binary64 addition).
// Squares below binary32's range (|g| < ~1e-23) are lost; they can matter
// only for a norm below ~1e-19, where the clip coefficient is 1.

struct FF {
    float hi, lo;
};

__device__ __forceinline__ FF ff_add(FF a, FF b)
{
    const float s = __fadd_rn(a.hi, b.hi);
    const float v = __fsub_rn(s, a.hi);
    float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, v)), __fsub_rn(b.hi, v));
    e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
    const float hi = __fadd_rn(s, e);
    return FF{hi, __fsub_rn(e, __fsub_rn(hi, s))};
}

struct SumSq {
    FF acc{0.0f, 0.0f};

    __device__ __forceinline__ void add8(const float g[8])
    {
        float hi = 0.0f, lo = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float p = __fmul_rn(g[i], g[i]);
            const float e = __fmaf_rn(g[i], g[i], -p);
            const float s = __fadd_rn(hi, p);
            const float bb = __fsub_rn(s, hi);
            const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(p, bb));
            hi = s;
            lo = __fadd_rn(lo, __fadd_rn(err, e));
        }
        acc = ff_add(acc, FF{hi, lo});
    }
};

// Sum of n doubles in a fixed order, the result valid in every lane of the
// calling (whole) warp: lane l adds p[l], p[l + 32], p[l + 64] ... in index
// order from +0 (the loads are issued eight at a time; the order of the
// additions does not change), then a fixed butterfly combines the lanes.
// The values may have been written by other CTAs of the running kernel, so
// they are read from L2 (ld.global.cg), past this SM's L1.
__device__ __forceinline__ double warp_fixed_sum(const double *p, int64_t n)
{
    const int lane = threadIdx.x & 31;
    double x = 0.0;
    int64_t i = lane;
    for (; i + 7 * 32 < n; i += 8 * 32) {
        double y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            y[j] = __ldcg(p + i + 32 * j);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            x = __dadd_rn(x, y[j]);
    }
    for (; i < n; i += 32)
        x = __dadd_rn(x, __ldcg(p + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x = __dadd_rn(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
    return x;
}

// ------------------------------------------------------------------ the norm's tree
//
// Chunks, superchunks, ranks (see NormPlan in internal.h).  A first pass
// walks its chunks with a grid stride, so that at any moment the CTAs stream
// neighbouring memory (every-rank launches take the chunks bucket by bucket
// and rank by rank inside a bucket: the flat order); a whole CTA sums one
// chunk, and a barrier per chunk keeps the CTA's warps on the same chunk:
// each of its 256-unit rows is then read by all 8 warps at once (4 KB of
// each gradient, 8 KB of each fp32 array), which measured 10 % faster on an
// 8-billion-element first pass than letting the warps drift apart.  After
// the barrier warp 0 adds the warps' pairs and stores the chunk's sum.
// Nothing waits for another CTA.

// Where a chunk lies and where its sum goes.
struct ChunkLoc {
    int64_t r;        // rank, relative to the launch (0 for one rank's view)
    int64_t bl;       // bucket, relative to the launch
    int64_t u0, n_u;  // its units within the rank's slice of that bucket
    int64_t ci;       // its slot among the chunks (rank by rank, in element order)
};

__device__ __forceinline__ ChunkLoc locate_chunk(const NormPlan &np, int64_t pi)
{
    ChunkLoc L;
    const bool has_last = np.b0 + np.nbl == np.nb;
    const int64_t per_bucket = (int64_t)np.ranks * np.cps;
    const int64_t n_full = (np.nbl - (has_last ? 1 : 0)) * per_bucket;
    int64_t c, ub, k;
    if (pi < n_full) {
        L.bl = pi / per_bucket;
        const int64_t rem = pi - L.bl * per_bucket;
        L.r = rem / np.cps;
        c = rem - L.r * np.cps;
        ub = np.slice_units;
        k = (np.b0 + L.bl) * np.cps + c;
    } else {
        const int64_t rem = pi - n_full;
        L.r = rem / np.cps_last;
        c = rem - L.r * np.cps_last;
        L.bl = np.nbl - 1;
        ub = np.last_slice_units;
        k = (np.nb - 1) * np.cps + c;
    }
    L.u0 = c * np.cu;
    L.n_u = ub - L.u0 < np.cu ? ub - L.u0 : np.cu;
    L.ci = L.r * np.cpr + k;
    return L;
}

// A first pass's walk over its chunks, called by every thread.  chunk_fn(L)
// sums the squares of this thread's units of chunk L (units L.u0 +
// threadIdx.x, + 256, ...) and returns the pair.
template <class ChunkFn>
__device__ __forceinline__ void norm_walk(const NormPlan &np, ChunkFn &&chunk_fn)
{
    __shared__ FF warp_sum[2][kThreads / 32];  // double-buffered by chunk parity
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int parity = 0;
    for (int64_t pi = blockIdx.x; pi < np.launch_chunks; pi += gridDim.x, parity ^= 1) {
        const ChunkLoc L = locate_chunk(np, pi);
        FF x = chunk_fn(L);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const FF y{__shfl_xor_sync(0xFFFFFFFFu, x.hi, o),
                       __shfl_xor_sync(0xFFFFFFFFu, x.lo, o)};
            x = ff_add(x, y);
        }
        if (lane == 0)
            warp_sum[parity][warp] = x;
        __syncthreads();
        if (threadIdx.x == 0) {
            FF t = warp_sum[parity][0];
#pragma unroll
            for (int w = 1; w < kThreads / 32; ++w)
                t = ff_add(t, warp_sum[parity][w]);
            np.partials[L.ci] = __dadd_rn((double)t.hi, (double)t.lo);
        }
    }
}

// Report a non-finite gradient of this warp once.
__device__ __forceinline__ void flag_nonfinite(bool bad, int32_t *flag)
{
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && (threadIdx.x & 31) == 0)
        atomicOr(flag, 1);
}

}  // namespace zs
