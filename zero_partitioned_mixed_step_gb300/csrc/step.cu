// The streaming kernels of the step and the entry points zero_step_fused,
// zero_step_fused_accumulated, zero_step_fused_buckets,
// zero_step_buckets_pass1 / _norm / _pass2, zero_reduce_scatter_sum and
// zero_reduce_scatter_accumulate.
//
// One kernel template covers the passes over the data.  Each thread handles
// 8-element units (16-byte loads of each rank's half gradient, 32-byte loads
// and stores of each fp32 state array) with a grid stride; the grid is one
// wave: exactly as many CTAs as the SMs hold at once (every CTA does the same
// share of the work, so a second, partial wave would only add a tail).
//   FUSED      (a2)-(a7) in one pass: reduce, unscale, flag, Adam from slot
//              cur into slot 1 - cur, cast into the parameter buffer.
//   PASS1      (a2)-(a5) of a clipped step: reduce, unscale, flag, the
//              chunk sums of the norm's fixed tree (internal.h: chunks of the
//              layout, not of the grid; the tree kernel then forms the
//              total in the workspace), optionally keep g in a staging
//              buffer.
//   PASS2_*    (a5 clip)-(a7) of a clipped step, skipped when pass 1 flagged
//              an overflow; it reads the total pass 1 formed; g is reduced
//              again or read from the stage.  It walks the units backwards,
//              starting on the first pass's last units, whose data pass 1
//              left in L2.
//   RS         (a2) alone: the reduced fp32 gradient.
//   RS_ACC     (a2) into an fp32 accumulator (gradient accumulation).
//   ACC_*      the step with the gradient read from an fp32 accumulator (the
//              sum of micro-steps' reduced, still scaled gradients) instead of
//              the N_d half buffers: FUSED, PASS1 and PASS2 as above.
// The last launch of a step (FUSED, a second pass, ACC_FUSED) also ends it:
// the CTA that finishes last commits or skips the step (a8).  Gradient
// buffers may be device memory or page-locked host memory, which these
// kernels load over the host link.
#include <atomic>
#include <cstdlib>

#include "kernels.cuh"
#include "staged.cuh"

namespace zs {

enum Mode {
    M_FUSED = 0, M_PASS1 = 1, M_PASS2_RECOMPUTE = 2, M_PASS2_STAGED = 3, M_RS = 4,
    M_RS_ACC = 5, M_ACC_FUSED = 6, M_ACC_PASS1 = 7, M_ACC_PASS2 = 8
};

// What each mode does with a unit.
__host__ __device__ constexpr bool reads_half_grads(int m)
{
    return m == M_FUSED || m == M_PASS1 || m == M_PASS2_RECOMPUTE || m == M_RS || m == M_RS_ACC;
}
__host__ __device__ constexpr bool reads_accumulator(int m)
{
    return m == M_ACC_FUSED || m == M_ACC_PASS1 || m == M_ACC_PASS2;
}
__host__ __device__ constexpr bool flags_overflow(int m)
{
    return m == M_FUSED || m == M_PASS1 || m == M_ACC_FUSED || m == M_ACC_PASS1;
}
__host__ __device__ constexpr bool sums_squares(int m) { return m == M_PASS1 || m == M_ACC_PASS1; }
__host__ __device__ constexpr bool second_pass(int m)
{
    return m == M_PASS2_RECOMPUTE || m == M_PASS2_STAGED || m == M_ACC_PASS2;
}
__host__ __device__ constexpr bool reduces_only(int m) { return m == M_RS || m == M_RS_ACC; }
// Modes that can be the last kernel of a step (and then end it themselves).
__host__ __device__ constexpr bool ends_step(int m)
{
    return m == M_FUSED || m == M_ACC_FUSED || second_pass(m);
}

template <int MAXW>
struct StepParams {
    GradTable<MAXW> grads;
    View view;
    CfgDev cfg;
    zero_step_state *state;
    const float *w0, *w1, *m0, *m1, *v0, *v1;  // ping-pong slots (reads)
    float *wo0, *wo1, *mo0, *mo1, *vo0, *vo1;   // ping-pong slots (writes)
    uint16_t *par0, *par1;                      // parameter buffer slots
    float *stage;      // PASS1 output / PASS2_STAGED input / RS output / accumulator
    NormPlan norm;     // first passes: the chunks of the norm's tree this launch forms
    const double *norm_total;  // second passes: the sum of squares the first pass formed
    int32_t add;       // RS_ACC: add to the accumulator (else overwrite it)
    // Clipped steps: the first pass marks what it reads or writes for units
    // u >= keep_from evict-last in L2 (the stage it writes, else the
    // accumulator or the gradients it reads), and the second pass walks the
    // units backwards, so it starts on what is still in L2.  keep_from is a
    // multiple of 4 (= units when nothing is kept).  discard: the second pass
    // drops the stage's kept lines from L2 after reading them (the stage is
    // 128-byte aligned), so a line still dirty is not written back to DRAM.
    int64_t keep_from;
    int32_t discard;
    // The step's last kernel: the CTA that finishes last ends the step (a8).
    int32_t end_step;
    int32_t host_grads;  // the gradients are in page-locked host memory (host side only)
    FinCfg fin;
};

// A first pass's walk over its chunks of the norm's tree: each chunk's units
// go through `unit` (which adds their squares to ss), then the chunk's sum is
// stored (norm_walk in kernels.cuh).
template <bool ALL, class UnitFn>
__device__ __forceinline__ void norm_loop(const NormPlan &np, const View &vw, SumSq &ss,
                                          UnitFn &unit)
{
    norm_walk(np, [&](const ChunkLoc &L) {
        int64_t ubase;  // the launch's unit index of the chunk's first unit
        if constexpr (ALL) {
            int64_t flat;
            if (vw.bucket == 0)
                flat = L.r * vw.part;
            else
                flat = L.bl * vw.bucket + L.r * (L.bl == np.nbl - 1 ? vw.last_slice : vw.slice);
            ubase = flat / kUnit + L.u0;
        } else {
            ubase = L.bl * vw.slice_units + L.u0;
        }
        ss.acc = FF{0.0f, 0.0f};
        for (int64_t k = threadIdx.x; k < L.n_u; k += kThreads)
            unit(ubase + k);
        return ss.acc;
    });
}

// Instances with a lead CTA (step_body): the one-pass steps over at most 4
// ranks, the small steps, where the prologue's binary64 division and square
// root are a visible share of the step (1M elements over 2 ranks, median of
// 300 steps with L2 flushed: 13.9 -> 12.3 us on one GB300, 12.4-12.6 -> 12.3
// us on another).  A larger step forms them in its prologue (microseconds
// against milliseconds).  The branch is compiled
// into these instances only: in the others it changed ptxas' register
// allocation (the 64-rank shard's instance went from 80 to 64 registers and
// from 2.57 to 2.62 ms per step; a writer at the end of a grid-stride CTA took
// another from 80 to 112).
__host__ __device__ constexpr bool has_lead(int dt, int w, int mode, bool host_state)
{
    return mode == M_FUSED && !host_state && w > 0 && w <= 4 && !half_reduce(dt);
}

// The body of the streaming kernels (the __global__ wrappers below differ
// only in their launch bounds).
template <int DT, int W, int MAXW, int MODE, bool ALL, bool HOST_STATE>
__device__ __forceinline__ void step_body(const StepParams<MAXW> &p)
{
    __shared__ Scalars sh;
    __shared__ int sh_cur;
    Scalars s{};
    int cur = 0;
    const View &vw = p.view;
    // A one-pass step over at most 4 ranks whose units fit in one wave forms
    // the next step's bias-correction scalars (form_next_scalars) in a CTA
    // of its own, off the step's critical path: launch_one adds a CTA to the
    // grid, and that CTA 0 ("lead") does only this, alongside the work CTAs
    // 1, 2, ...  The grid tells: more CTAs than units / 256.  (See has_lead.)
    constexpr bool kLead = has_lead(DT, W, MODE, HOST_STATE);
    const int lead = kLead && (int64_t)gridDim.x > (vw.units + kThreads - 1) / kThreads ? 1 : 0;
    if constexpr (kLead) {
        if (lead && blockIdx.x == 0) {
            if (threadIdx.x == 0)
                form_next_scalars(p.cfg, p.state);
            finish_cta(false, ends_step(MODE) && p.end_step, p.fin, p.state);
            return;
        }
    }
    const int64_t cta = (int64_t)blockIdx.x - lead;  // among the work CTAs
    const int64_t stride = ((int64_t)gridDim.x - lead) * kThreads;
    const uint64_t pol = evict_first_policy();
    // One-pass steps over at most 4 ranks issue their first unit's loads
    // before the prologue's barrier (the gradients need nothing, the state
    // only the slot index), so that they are in flight while thread 0 forms
    // the step's scalars.  (At 8 and 16 ranks the loads held across the
    // barrier took ptxas from 78 and 71 registers to 90 and 119, a CTA per SM
    // fewer; at 2 ranks it went from 78 to 64, a CTA per SM more.)
    constexpr bool kEarly = MODE == M_FUSED && !HOST_STATE && W > 0 && W <= 4 &&
                            !half_reduce(DT);
    const int64_t u_first = cta * kThreads + threadIdx.x;
    uint4 early_g[kEarly ? W : 1];
    float early_w[8], early_m[8], early_v[8];
    int64_t early_f = 0, early_si = 0;
    if constexpr (kEarly) {
        if (u_first < vw.units) {
            int64_t gi;
            locate<ALL>(vw, u_first, early_f, early_si, gi);
            const int c0 = p.state->cur;
            load8_now((c0 ? p.w1 : p.w0) + early_si, early_w);
            load8_now((c0 ? p.m1 : p.m0) + early_si, early_m);
            load8_now((c0 ? p.v1 : p.v0) + early_si, early_v);
#pragma unroll
            for (int q = 0; q < W; ++q)
                early_g[q] = ld_stream_now(p.grads.p[q] + gi, pol);
        }
    }
    if constexpr (!reduces_only(MODE)) {
        // A second pass also forms the clip coefficient from the global sum
        // of squares the first pass formed; the first work CTA publishes both
        // in the state when the step is not skipped.
        form_scalars<!sums_squares(MODE)>(p.cfg, p.state,
                                          second_pass(MODE) ? p.norm_total : nullptr, sh,
                                          sh_cur);
        __syncthreads();
        s = sh;
        cur = sh_cur;
        if constexpr (second_pass(MODE)) {
            if (cta == 0 && threadIdx.x == 0 && !s.skip) {
                p.state->sumsq = __ldcg(p.norm_total);
                p.state->clip_coef = s.coef;
            }
        }
    }
    bool work = true;
    if constexpr (second_pass(MODE)) {
        if (s.skip) {  // the whole step is skipped: write nothing
            work = false;
            if constexpr (MODE == M_PASS2_STAGED) {
                if (p.discard)  // the kept stage lines are not needed either
                    for (int64_t u = p.keep_from + 4 * (cta * kThreads + threadIdx.x);
                         u + 4 <= vw.units; u += 4 * stride)
                        discard_l2_line(p.stage + u * kUnit);
            }
        }
    }
    const float *w_src = cur ? p.w1 : p.w0;
    const float *m_src = cur ? p.m1 : p.m0;
    const float *v_src = cur ? p.v1 : p.v0;
    float *w_dst = cur ? p.wo0 : p.wo1;
    float *m_dst = cur ? p.mo0 : p.mo1;
    float *v_dst = cur ? p.vo0 : p.vo1;
    uint16_t *out = cur ? p.par0 : p.par1;

    uint64_t keep_pol = pol;
    if constexpr (sums_squares(MODE))
        keep_pol = evict_last_policy();
    bool bad = false;
    SumSq ss;
    // One unit: the whole per-element work of the mode.
    auto unit = [&](int64_t u) {
        int64_t f, si, gi;
        locate<ALL>(vw, u, f, si, gi);
        const bool keep = sums_squares(MODE) && u >= p.keep_from;
        // The state loads are issued before the gradient loads, so that a
        // unit's whole input is in flight at once (1.3 % faster on the 64-rank
        // shard, no change at 16 ranks).
        float w[8], m[8], v[8];
        if constexpr (!reduces_only(MODE) && !sums_squares(MODE)) {
            if constexpr (HOST_STATE) {
                load8_host(w_src + si, w);
                load8_host(m_src + si, m);
                load8_host(v_src + si, v);
            } else {
                load8(w_src + si, w);
                load8(m_src + si, m);
                load8(v_src + si, v);
            }
        }
        float g[8];
        if constexpr (MODE == M_PASS2_STAGED) {
            load8(p.stage + si, g);  // already unscaled by pass 1
        } else if constexpr (reads_accumulator(MODE)) {
            if (keep)
                load8_keep(p.stage + si, g);
            else
                load8(p.stage + si, g);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                g[i] = __fmul_rn(g[i], s.inv_s);
        } else {
            // a first pass that will reduce again keeps its tail's gradients
            const bool keep_grads = keep && MODE == M_PASS1 && !p.stage;
            reduce_unit<DT, W, MAXW>(p.grads, vw.world, gi, g, keep_grads ? keep_pol : pol);
            if constexpr (MODE == M_RS) {
                store8(p.stage + si, g);
                return;
            }
            if constexpr (MODE == M_RS_ACC) {
                if (p.add) {
                    float a[8];
                    load8(p.stage + si, a);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        g[i] = __fadd_rn(a[i], g[i]);
                }
                store8(p.stage + si, g);
                return;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
                g[i] = __fmul_rn(g[i], s.inv_s);
        }
        if constexpr (flags_overflow(MODE)) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                bad |= nonfinite(g[i]);
        }
        if constexpr (sums_squares(MODE)) {
            ss.add8(g);
            if (MODE == M_PASS1 && p.stage) {
                if (keep)
                    store8_keep(p.stage + si, g);
                else
                    store8(p.stage + si, g);
            }
            return;
        }
        if constexpr (second_pass(MODE)) {
            if (s.coef < 1.0f) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    g[i] = __fmul_rn(g[i], s.coef);
            }
        }
        adam8(g, w, m, v, s);
        if constexpr (HOST_STATE) {
            store8_host(w_dst + si, w);
            store8_host(m_dst + si, m);
            store8_host(v_dst + si, v);
        } else {
            store8(w_dst + si, w);
            store8(m_dst + si, m);
            store8(v_dst + si, v);
        }
        st_half8(out + f, pack_half8<DT>(w), pol);
    };

    const int64_t base = cta * kThreads;
    if constexpr (sums_squares(MODE)) {
        norm_loop<ALL>(p.norm, vw, ss, unit);
    } else if constexpr (second_pass(MODE)) {
        // Backwards over the grid-stride sequence: the units the first pass
        // reached last come first, while their lines can still be in L2.
        if (work && base < vw.units) {
            for (int64_t k = (vw.units - 1 - base) / stride; k >= 0; --k) {
                const int64_t first = base + k * stride;  // the CTA's first unit this round
                const int64_t u = first + threadIdx.x;
                if (u < vw.units)
                    unit(u);
                if constexpr (MODE == M_PASS2_STAGED) {
                    if (p.discard && first + kThreads > p.keep_from) {  // uniform in the CTA
                        // lanes 4j .. 4j + 3 read the four units of one line
                        __syncwarp();
                        if ((threadIdx.x & 3) == 0 && u >= p.keep_from && u + 4 <= vw.units)
                            discard_l2_line(p.stage + u * kUnit);
                    }
                }
            }
        }
    } else {
        int64_t u = base + threadIdx.x;
        if constexpr (kEarly) {
            if (u < vw.units) {  // the unit whose loads were issued before the barrier
                float g[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    g[i] = 0.0f;
#pragma unroll
                for (int q = 0; q < W; ++q)
                    add_half8<DT>(g, early_g[q]);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    g[i] = __fmul_rn(g[i], s.inv_s);
                    bad |= nonfinite(g[i]);
                }
                adam8(g, early_w, early_m, early_v, s);
                store8(w_dst + early_si, early_w);
                store8(m_dst + early_si, early_m);
                store8(v_dst + early_si, early_v);
                st_half8(out + early_f, pack_half8<DT>(early_w), pol);
            }
            u += stride;
        }
        for (; u < vw.units; u += stride)
            unit(u);
    }
    if constexpr (flags_overflow(MODE) || ends_step(MODE))
        finish_cta(bad, ends_step(MODE) && p.end_step, p.fin, p.state);
}

// Device-resident state: the launch bound names only the block size, and
// ptxas keeps these instances at 46-80 registers (3 CTAs of 256 threads per
// SM).  A minimum of one CTA per SM in the bound lets it spend up to 255
// (252 for the 64-rank shard), which costs two thirds of the warps.
template <int DT, int W, int MAXW, int MODE, bool ALL>
__global__ void __launch_bounds__(kThreads)
    step_kernel(const __grid_constant__ StepParams<MAXW> p)
{
    step_body<DT, W, MAXW, MODE, ALL, false>(p);
}

// Master, m and v in pinned host memory (offload): held to 5 resident CTAs
// per SM (at most 51 registers).  Host accesses take microseconds, so more
// warps in flight pay: timed on the 1.5B, 16-rank offloaded step, 156 ms at 5
// CTAs/SM against 174 ms at the natural 3 (225 ms at 4, 196 ms at 6: the
// register caps also reorder the loads).  When the gradients are in host
// memory too, the launch takes at most kHostAllCtasPerSm CTAs per SM.
template <int DT, int W, int MAXW, int MODE, bool ALL>
__global__ void __launch_bounds__(kThreads, 5)
    step_kernel_host_state(const __grid_constant__ StepParams<MAXW> p)
{
    step_body<DT, W, MAXW, MODE, ALL, true>(p);
}

// ------------------------------------------------------------------ launch

// CTAs per SM at most when the state and the gradients are all in page-locked
// host memory.  The 1.5B, 16-rank offloaded step with its gradients in host
// memory, one box: 760 CTAs (5 per SM) 985 ms per step, the host link read at
// 67 GB/s; 456 CTAs (3 per SM) and 152 CTAs 322 ms, 205 GB/s (the link's
// rate).  Too many loads to host memory in flight collapse the link's rate.
constexpr int kHostAllCtasPerSm = 3;

// CTAs per SM of a first pass at most (when more fit).  Swept on the 8B
// clipped step (bf16, 8 ranks) and the 124M one, same box: 3 per SM 61.95 /
// 0.988 ms, 4 per SM 61.16 / 0.963 ms, 5 per SM 61.23 / 0.949 ms, all that fit
// (6) 61.64 / 0.947 ms.
constexpr int kFirstPassCtasPerSm = 5;

template <int DT, int W, int MAXW, int MODE, bool HOST_STATE = false>
int launch_one(const StepParams<MAXW> &p, cudaStream_t stream, int *gx_out)
{
    void (*kern)(StepParams<MAXW>);
    if constexpr (HOST_STATE)
        kern = p.view.all_ranks ? step_kernel_host_state<DT, W, MAXW, MODE, true>
                                : step_kernel_host_state<DT, W, MAXW, MODE, false>;
    else
        kern = p.view.all_ranks ? step_kernel<DT, W, MAXW, MODE, true>
                                : step_kernel<DT, W, MAXW, MODE, false>;
    int target = target_ctas(reinterpret_cast<const void *>(kern));
    if (sums_squares(MODE) && target > device_sms() * kFirstPassCtasPerSm)
        target = device_sms() * kFirstPassCtasPerSm;
    if (HOST_STATE && p.host_grads && target > device_sms() * kHostAllCtasPerSm)
        target = device_sms() * kHostAllCtasPerSm;
    const int64_t want = sums_squares(MODE) ? p.norm.launch_chunks
                                            : (p.view.units + kThreads - 1) / kThreads;
    int64_t gx = want < 1 ? 1 : (want < target ? want : target);
    // A small one-pass step whose units fit in one wave with a CTA to spare
    // gets a lead CTA that forms the next step's bias-correction scalars
    // (step_body tells it from the grid: more CTAs than units / 256).
    if (has_lead(DT, W, MODE, HOST_STATE) && p.cfg.bias_correction && want + 1 <= target)
        gx = want + 1;
    if (gx_out)
        *gx_out = (int)gx;
    kern<<<(unsigned)gx, kThreads, 0, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ZERO_OK : cuda_error(e);
}

template <int DT, int MAXW, int MODE>
int dispatch_world(const StepParams<MAXW> &p, cudaStream_t stream, int *gx)
{
    if constexpr (!reads_half_grads(MODE) || half_reduce(DT)) {
        // no gradient loads, or the half-precision reduction: one instance
        // with the group size read at run time
        return launch_one<DT, 0, MAXW, MODE>(p, stream, gx);
    } else if constexpr (MAXW == 64) {
        switch (p.view.world) {
        case 2: return launch_one<DT, 2, MAXW, MODE>(p, stream, gx);
        case 4: return launch_one<DT, 4, MAXW, MODE>(p, stream, gx);
        case 8: return launch_one<DT, 8, MAXW, MODE>(p, stream, gx);
        case 16: return launch_one<DT, 16, MAXW, MODE>(p, stream, gx);
        case 32: return launch_one<DT, 32, MAXW, MODE>(p, stream, gx);
        case 64: return launch_one<DT, 64, MAXW, MODE>(p, stream, gx);
        default: return launch_one<DT, 0, MAXW, MODE>(p, stream, gx);
        }
    } else {
        return launch_one<DT, 0, MAXW, MODE>(p, stream, gx);
    }
}

template <int MAXW>
int dispatch(const StepParams<MAXW> &p, zero_dtype dt, int mode, cudaStream_t s, int *gx)
{
#define ZS_MODES(DT)                                                              \
    switch (mode) {                                                               \
    case M_FUSED: return dispatch_world<DT, MAXW, M_FUSED>(p, s, gx);             \
    case M_PASS1: return dispatch_world<DT, MAXW, M_PASS1>(p, s, gx);             \
    case M_PASS2_RECOMPUTE: return dispatch_world<DT, MAXW, M_PASS2_RECOMPUTE>(p, s, gx); \
    case M_RS_ACC: return dispatch_world<DT, MAXW, M_RS_ACC>(p, s, gx);           \
    default: return dispatch_world<DT, MAXW, M_RS>(p, s, gx);                     \
    }
#define ZS_NO_GRAD_MODES(DT)                                                      \
    switch (mode) {                                                               \
    case M_PASS2_STAGED: return dispatch_world<DT, MAXW, M_PASS2_STAGED>(p, s, gx); \
    case M_ACC_FUSED: return dispatch_world<DT, MAXW, M_ACC_FUSED>(p, s, gx);     \
    case M_ACC_PASS1: return dispatch_world<DT, MAXW, M_ACC_PASS1>(p, s, gx);     \
    default: return dispatch_world<DT, MAXW, M_ACC_PASS2>(p, s, gx);              \
    }
    const bool grads = mode == M_FUSED || mode == M_PASS1 || mode == M_PASS2_RECOMPUTE ||
                       mode == M_RS || mode == M_RS_ACC;
    if (!grads) {  // only the parameters' storage type matters
        if (is_bf16(dt)) {
            ZS_NO_GRAD_MODES(ZERO_BF16)
        } else {
            ZS_NO_GRAD_MODES(ZERO_F16)
        }
    }
    switch (dt) {
    case ZERO_F16: ZS_MODES(ZERO_F16)
    case ZERO_BF16: ZS_MODES(ZERO_BF16)
    case ZERO_F16_HALF_REDUCE: ZS_MODES(ZERO_F16_HALF_REDUCE)
    default: ZS_MODES(ZERO_BF16_HALF_REDUCE)
    }
#undef ZS_MODES
#undef ZS_NO_GRAD_MODES
}

// Everything a pass needs besides the per-mode pointers.
struct PassArgs {
    const void *const *grads = nullptr;
    int grads_are_slices = 0;
    zero_dtype dtype = ZERO_F16;
    const zero_layout *lay = nullptr;  // the launch's (sub-)layout; buffers start at its origin
    int rank = -1;
    const zero_adam_cfg *cfg = nullptr;
    zero_step_state *state = nullptr;
    float *const *master = nullptr, *const *m = nullptr, *const *v = nullptr;
    void *const *params = nullptr;
    float *stage = nullptr;
    int add = 0;
    bool host_state = false;       // master/m/v in pinned host memory (one-pass step only)
    bool grads_on_device = true;   // every gradient buffer is device memory
    NormPlan norm{};               // first passes: their chunks of the norm's tree
    const double *norm_total = nullptr;  // second passes: the first pass's total
    int64_t keep_from = INT64_MAX;  // clipped steps: see StepParams
    bool discard = false;
    bool end_step = false;    // the launch is the step's last: it ends the step
};

// The one-pass step with the optimizer state in pinned host memory: one
// instance per storage type, group size read at run time.
template <int MAXW>
int dispatch_host_state(const StepParams<MAXW> &p, zero_dtype dt, cudaStream_t s, int *gx)
{
    switch (dt) {
    case ZERO_F16: return launch_one<ZERO_F16, 0, MAXW, M_FUSED, true>(p, s, gx);
    case ZERO_BF16: return launch_one<ZERO_BF16, 0, MAXW, M_FUSED, true>(p, s, gx);
    case ZERO_F16_HALF_REDUCE:
        return launch_one<ZERO_F16_HALF_REDUCE, 0, MAXW, M_FUSED, true>(p, s, gx);
    default: return launch_one<ZERO_BF16_HALF_REDUCE, 0, MAXW, M_FUSED, true>(p, s, gx);
    }
}

template <int MAXW>
int run_pass(const PassArgs &a, int mode, cudaStream_t stream, int *gx)
{
    StepParams<MAXW> p{};
    const zero_layout &L = *a.lay;
    const int world = L.world;
    if (a.grads)
        for (int q = 0; q < world; ++q)
            p.grads.p[q] = static_cast<const uint16_t *>(a.grads[q]);
    View &v = p.view;
    v.units = (a.rank < 0 ? L.padded_numel : L.owned_numel) / kUnit;
    v.part = L.owned_numel;
    v.bucket = L.bucket_numel;
    v.slice = L.slice_numel;
    v.slice_units = L.slice_numel / kUnit;
    v.full_units = L.bucket_numel ? (L.num_buckets - 1) * (L.slice_numel / kUnit) : 0;
    v.last_base = L.bucket_numel ? (L.num_buckets - 1) * L.bucket_numel : 0;
    v.last_slice = L.last_slice_numel;
    v.rank = a.rank < 0 ? 0 : a.rank;
    v.all_ranks = a.rank < 0;
    v.grads_are_slices = a.grads_are_slices;
    v.world = world;
    if (a.cfg) {
        const zero_adam_cfg &c = *a.cfg;
        p.cfg = make_cfg_dev(c);
    }
    p.state = a.state;
    if (a.master) {
        p.w0 = p.wo0 = a.master[0];
        p.w1 = p.wo1 = a.master[1];
        p.m0 = p.mo0 = a.m[0];
        p.m1 = p.mo1 = a.m[1];
        p.v0 = p.vo0 = a.v[0];
        p.v1 = p.vo1 = a.v[1];
        p.par0 = static_cast<uint16_t *>(a.params[0]);
        p.par1 = static_cast<uint16_t *>(a.params[1]);
    }
    p.stage = a.stage;
    p.norm = a.norm;
    p.norm_total = a.norm_total;
    p.add = a.add;
    p.keep_from = a.keep_from < v.units ? a.keep_from : v.units;
    p.discard = a.discard && p.keep_from < v.units ? 1 : 0;
    p.end_step = a.end_step ? 1 : 0;
    p.host_grads = a.grads && !a.grads_on_device ? 1 : 0;
    if (a.cfg)
        p.fin = fin_cfg(*a.cfg);
    if (a.host_state)
        return dispatch_host_state<MAXW>(p, a.dtype, stream, gx);
    return dispatch<MAXW>(p, a.dtype, mode, stream, gx);
}

int run(const PassArgs &a, int mode, cudaStream_t stream, int *gx)
{
    if (a.lay->world <= 64)
        return run_pass<64>(a, mode, stream, gx);
    return run_pass<ZERO_MAX_WORLD>(a, mode, stream, gx);
}

int check_grads(const void *const *grads, int grads_are_slices, zero_dtype dtype,
                const zero_layout *lay, int rank)
{
    int rc = check_layout(lay);
    if (rc)
        return rc;
    if (!grads || dtype < ZERO_F16 || dtype > ZERO_BF16_HALF_REDUCE || rank < -1 ||
        rank >= lay->world ||
        (grads_are_slices && rank < 0))
        return ZERO_EINVAL;
    for (int q = 0; q < lay->world; ++q) {
        if (!grads[q] && lay->padded_numel)
            return ZERO_EINVAL;
        if (!aligned16(grads[q]))
            return ZERO_EALIGN;
    }
    return ZERO_OK;
}

// Where a buffer lives: 1 page-locked host memory, 0 memory of device `dev`
// (or managed memory), -1 anything else (pageable host memory, an unknown
// pointer, another device's memory).
int residence(const void *p, int dev)
{
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    if (attr.type == cudaMemoryTypeManaged)
        return 0;
    if (attr.type == cudaMemoryTypeDevice)
        return attr.device == dev ? 0 : -1;
    return attr.type == cudaMemoryTypeHost ? 1 : -1;
}

int current_device(int *dev)
{
    const cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return cuda_error(e);
    }
    return ZERO_OK;
}

// Every gradient buffer must be memory the kernels can load: device memory
// of the current device or page-locked host memory.  One query per buffer;
// *all_device tells whether the bulk-copy (staged) kernel may take them.
int check_grad_residence(const void *const *grads, int world, bool *all_device)
{
    int dev = 0, rc = current_device(&dev);
    if (rc)
        return rc;
    bool on_device = true;
    for (int q = 0; q < world; ++q) {
        const int r = residence(grads[q], dev);
        if (r < 0)
            return ZERO_EINVAL;
        on_device = on_device && r == 0;
    }
    *all_device = on_device;
    return ZERO_OK;
}

// 1 when all six master/m/v slots are pinned host memory (offload), 0 when
// all are device memory, ZERO_EINVAL otherwise.
int state_residence(float *const master[2], float *const m[2], float *const v[2])
{
    int dev = 0, rc = current_device(&dev);
    if (rc)
        return rc;
    const void *ptrs[6] = {master[0], master[1], m[0], m[1], v[0], v[1]};
    const int first = residence(ptrs[0], dev);
    for (int i = 1; i < 6; ++i)
        if (ptrs[i] != ptrs[i - 1] && residence(ptrs[i], dev) != first)
            return ZERO_EINVAL;
    return first < 0 ? ZERO_EINVAL : first;
}

// Checks of the ping-pong slots and the state shared by the fused entry points.
int check_pingpong(const zero_layout *layout, const zero_adam_cfg *cfg, float *const master[2],
                   float *const m[2], float *const v[2], void *const params[2],
                   const zero_step_state *state_dev)
{
    if (!master || !m || !v || !params || !state_dev)
        return ZERO_EINVAL;
    const bool clip = cfg->max_grad_norm > 0.0;
    const bool empty = layout->padded_numel == 0;  // nothing to read or write
    for (int s = 0; s < 2; ++s) {
        if (!empty && (!master[s] || !m[s] || !v[s] || !params[s]))
            return ZERO_EINVAL;
        if (!aligned32(master[s]) || !aligned32(m[s]) || !aligned32(v[s]) || !aligned16(params[s]))
            return ZERO_EALIGN;
    }
    if (!clip && !empty &&
        (master[0] == master[1] || m[0] == m[1] || v[0] == v[1] || params[0] == params[1]))
        return ZERO_EINVAL;  // a one-pass step needs distinct slots to be able to skip
    if (reinterpret_cast<uintptr_t>(state_dev) & 7u)
        return ZERO_EALIGN;
    return ZERO_OK;
}

// The workspace of a step on `layout`.
int check_ws(const zero_layout *layout, const void *ws, size_t ws_bytes)
{
    if (!ws)
        return ZERO_EINVAL;
    if (!aligned16(ws))
        return ZERO_EALIGN;
    if (ws_bytes < zero_workspace_bytes(layout))
        return ZERO_ESPACE;
    return ZERO_OK;
}

// check_pingpong, plus the stage and the workspace.
int check_slots(const zero_layout *layout, const zero_adam_cfg *cfg, float *const master[2],
                float *const m[2], float *const v[2], void *const params[2], const float *stage,
                bool stage_allowed, const zero_step_state *state_dev, const void *ws,
                size_t ws_bytes)
{
    if (!ws)
        return ZERO_EINVAL;
    const int rc = check_pingpong(layout, cfg, master, m, v, params, state_dev);
    if (rc)
        return rc;
    if (stage && !stage_allowed)
        return ZERO_EINVAL;
    if (stage && !aligned32(stage))
        return ZERO_EALIGN;
    return check_ws(layout, ws, ws_bytes);
}

// The norm's tree for launches over buckets [b0, b0 + nbl) of `L` (the whole
// layout), in workspace ws.
NormPlan layout_plan(const zero_layout &L, int rank, int64_t b0, int64_t nbl, void *ws)
{
    const bool bucketed = L.bucket_numel > 0;
    const int64_t nb = bucketed ? L.num_buckets : 1;
    const int64_t su = (bucketed ? L.slice_numel : L.owned_numel) / kUnit;
    const int64_t lsu = L.last_slice_numel / kUnit;
    return norm_plan(norm_geometry(su, lsu, nb), su, lsu, nb, b0, nbl, rank < 0 ? L.world : 1,
                     ws, nullptr);
}

// Polls of the staged kernel's stage waits; a test may lower the limit with
// ZERO_TEST_STAGED_WAIT_LIMIT (read once per process), and then also makes
// every wait run out (see staged.cuh).
long long staged_test_wait_limit()
{
    static const long long n = [] {
        const char *t = std::getenv("ZERO_TEST_STAGED_WAIT_LIMIT");
        const long long v = t ? std::atoll(t) : 0;
        return v > 0 ? v : 0LL;
    }();
    return n;
}

// Resident CTAs per SM of the staged kernel on device `dev` after raising its
// dynamic shared-memory limit there (the attribute belongs to the device):
// found once per device; 0 when the kernel cannot run there.
constexpr int kStagedDevices = 64;

template <int DT, int W>
int staged_resident(int dev)
{
    static std::atomic<int> cache[kStagedDevices];  // 0 unknown, -1 unusable, > 0 CTAs per SM
    if (dev >= 0 && dev < kStagedDevices) {
        const int c = cache[dev].load(std::memory_order_acquire);
        if (c != 0)
            return c > 0 ? c : 0;
    }
    int occ = 0;
    if (cudaFuncSetAttribute(staged_fused_kernel<DT, W>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kStagedSmemBudget) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, staged_fused_kernel<DT, W>,
                                                      kStagedThreads, kStagedSmemBudget) !=
            cudaSuccess) {
        (void)cudaGetLastError();
        occ = 0;
    }
    if (dev >= 0 && dev < kStagedDevices)
        cache[dev].store(occ > 0 ? occ : -1, std::memory_order_release);
    return occ > 0 ? occ : 0;
}

// The staged one-pass step (staged.cuh), when it applies: every rank at once,
// fp32 reduction, device-resident state and gradients, N_d = 16.  Returns 1
// when it does not apply or cannot be launched (the caller then uses the
// register path).
template <int DT, int W>
int launch_staged_w(const StagedParams &p, cudaStream_t stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 1;
    }
    const int resident = staged_resident<DT, W>(dev);
    if (resident < 1)
        return 1;
    const int64_t tiles = (p.n + kStagedTile - 1) / kStagedTile;
    int64_t want = (int64_t)device_sms() * resident;
    const int cap = test_grid_cap();
    if (cap > 0 && want > cap)
        want = cap;
    const unsigned grid = (unsigned)(tiles < want ? tiles : want);
    staged_fused_kernel<DT, W>
        <<<grid, kStagedThreads, p.stages * staged_stage_bytes(W), stream>>>(p);
    if (cudaGetLastError() != cudaSuccess)
        return 1;  // not launched: the register kernel takes the step
    return ZERO_OK;
}

int launch_staged(const PassArgs &a, cudaStream_t stream)
{
    const zero_layout &L = *a.lay;
    const int stages = staged_stages(L.world);
    // The bulk copies serve gradients in device memory; gradients in
    // page-locked host memory are loaded by the register kernel.
    if (a.rank >= 0 || a.host_state || !a.grads_on_device || half_reduce(a.dtype) ||
        L.world != kStagedWorld || stages < 2 || L.padded_numel <= 0)
        return 1;
    StagedParams p{};
    for (int q = 0; q < L.world; ++q)
        p.g[q] = static_cast<const uint16_t *>(a.grads[q]);
    p.stages = stages;
    p.n = L.padded_numel;
    const zero_adam_cfg &c = *a.cfg;
    p.cfg = make_cfg_dev(c);
    p.state = a.state;
    p.w0 = p.wo0 = a.master[0];
    p.w1 = p.wo1 = a.master[1];
    p.m0 = p.mo0 = a.m[0];
    p.m1 = p.mo1 = a.m[1];
    p.v0 = p.vo0 = a.v[0];
    p.v1 = p.vo1 = a.v[1];
    p.par0 = static_cast<uint16_t *>(a.params[0]);
    p.par1 = static_cast<uint16_t *>(a.params[1]);
    p.end_step = a.end_step ? 1 : 0;
    p.fin = fin_cfg(c);
    p.spin_limit = kStageSpinLimit;
    p.tx_extra = 0;
    if (const long long n = staged_test_wait_limit()) {  // tests only
        p.spin_limit = n;
        p.tx_extra = 16;
    }
    return is_bf16(a.dtype) ? launch_staged_w<ZERO_BF16, kStagedWorld>(p, stream)
                            : launch_staged_w<ZERO_F16, kStagedWorld>(p, stream);
}

// Bytes of a clipped step's first-pass data (the stage it writes, else the
// accumulator or the gradients it reads) left in L2 for the second pass: about
// half of GB300's 126 MB L2.
#ifndef ZS_KEEP_MB
#define ZS_KEEP_MB 64
#endif
constexpr int64_t kKeepBytes = (int64_t)ZS_KEEP_MB << 20;

// One whole step (one or two passes) in the given modes on a.lay.  The step's
// last launch also ends the step (a8: its last CTA commits or skips); an empty
// vector runs no pass and ends the step with the one-thread kernel.  A clipped
// step's first pass stores the norm's chunk sums in ws, the tree kernel sums
// them and the second pass reads the total.
int run_step(PassArgs &a, bool clip, int one_pass, int pass1, int pass2, void *ws,
             cudaStream_t stream)
{
    int rc, gx = 1;
    const zero_layout &L = *a.lay;
    if (L.padded_numel == 0)
        return launch_finalize(a.cfg, a.state, 1, stream);
    if (!clip) {
        a.end_step = true;
        rc = one_pass == M_FUSED ? launch_staged(a, stream) : 1;
        if (rc == 1)
            rc = run(a, one_pass, stream, &gx);
        return rc;
    }
    const int64_t units = (a.rank < 0 ? L.padded_numel : L.owned_numel) / kUnit;
    const bool regrads = pass1 == M_PASS1 && !a.stage;  // pass 2 reduces again
    const int64_t kept = kKeepBytes / (regrads ? 2 * kUnit * (int64_t)L.world : 4 * kUnit);
    int64_t from = units > kept ? units - kept : 0;
    from = (from + 3) / 4 * 4;
    a.keep_from = from < units ? from : units;
    a.discard = a.stage && pass2 == M_PASS2_STAGED &&
                (reinterpret_cast<uintptr_t>(a.stage) & 127u) == 0;
    a.norm = layout_plan(L, a.rank, 0, L.bucket_numel ? L.num_buckets : 1, ws);
    a.norm_total = norm_total_slot(ws);
    a.end_step = false;
    if ((rc = run(a, pass1, stream, &gx)))
        return rc;
    if ((rc = launch_norm_tree(a.norm, stream)))
        return rc;
    a.end_step = true;
    return run(a, pass2, stream, &gx);
}

// A range of buckets [first, first + n) of L as a layout of its own, with the
// offsets of its first element in flat buffers, in rank-order buffers and in
// the gradient buffers.
struct Range {
    zero_layout lay;
    int64_t flat_off, owned_off, state_off, grad_off;
};

Range bucket_range(const zero_layout &L, int rank, int grads_are_slices, int64_t first, int64_t n)
{
    Range R{L, 0, 0, 0, 0};
    if (L.bucket_numel > 0) {
        zero_layout &S = R.lay;
        const int64_t end = first + n;
        S.num_buckets = n;
        S.last_slice_numel = end == L.num_buckets ? L.last_slice_numel : L.slice_numel;
        S.owned_numel = (n - 1) * L.slice_numel + S.last_slice_numel;
        S.padded_numel = S.owned_numel * L.world;
        S.numel = S.flat_numel = S.padded_numel;
        R.flat_off = first * L.bucket_numel;
        R.owned_off = first * L.slice_numel;
    }
    R.state_off = rank < 0 ? R.flat_off : R.owned_off;
    R.grad_off = grads_are_slices ? R.owned_off : R.flat_off;
    return R;
}

// Checks of a bucket range.
int check_range(const zero_layout &L, int64_t first, int64_t n)
{
    if (first < 0 || n < 0 || first > L.num_buckets - n)
        return ZERO_EINVAL;
    return ZERO_OK;
}

// Buffers offset to a range's first element.
struct RangeBuffers {
    const void *g[ZERO_MAX_WORLD];
    float *w[2], *m[2], *v[2];
    void *par[2];
};

void offset_buffers(const Range &R, const void *const *grads, int world, float *const master[2],
                    float *const m[2], float *const v[2], void *const params[2], RangeBuffers &B)
{
    if (grads)
        for (int q = 0; q < world; ++q)
            B.g[q] = static_cast<const uint16_t *>(grads[q]) + R.grad_off;
    for (int s = 0; s < 2; ++s) {
        B.w[s] = master ? master[s] + R.state_off : nullptr;
        B.m[s] = m ? m[s] + R.state_off : nullptr;
        B.v[s] = v ? v[s] + R.state_off : nullptr;
        B.par[s] = params ? static_cast<uint16_t *>(params[s]) + R.flat_off : nullptr;
    }
}

}  // namespace zs

using namespace zs;

extern "C" int zero_reduce_scatter_sum(const void *const *grads, int grads_are_slices,
                                       zero_dtype dtype, const zero_layout *layout, int rank,
                                       float *g_out, zero_stream_t stream)
{
    int rc = check_grads(grads, grads_are_slices, dtype, layout, rank);
    if (rc)
        return rc;
    if (!g_out)
        return ZERO_EINVAL;
    if (!aligned32(g_out))
        return ZERO_EALIGN;
    if (layout->padded_numel == 0)
        return ZERO_OK;
    bool on_device;
    if ((rc = check_grad_residence(grads, layout->world, &on_device)))
        return rc;
    PassArgs a;
    a.grads = grads;
    a.grads_are_slices = grads_are_slices;
    a.dtype = dtype;
    a.lay = layout;
    a.rank = rank;
    a.stage = g_out;
    int gx;
    return run(a, M_RS, stream, &gx);
}

extern "C" int zero_reduce_scatter_accumulate(const void *const *grads, int grads_are_slices,
                                              zero_dtype dtype, const zero_layout *layout,
                                              int rank, float *acc, int add, zero_stream_t stream)
{
    int rc = check_grads(grads, grads_are_slices, dtype, layout, rank);
    if (rc)
        return rc;
    if (!acc && layout->padded_numel)
        return ZERO_EINVAL;
    if (!aligned32(acc))
        return ZERO_EALIGN;
    if (layout->padded_numel == 0)
        return ZERO_OK;
    bool on_device;
    if ((rc = check_grad_residence(grads, layout->world, &on_device)))
        return rc;
    PassArgs a;
    a.grads = grads;
    a.grads_are_slices = grads_are_slices;
    a.dtype = dtype;
    a.lay = layout;
    a.rank = rank;
    a.stage = acc;
    a.add = add ? 1 : 0;
    int gx;
    return run(a, M_RS_ACC, stream, &gx);
}

extern "C" int zero_step_fused(const void *const *grads, int grads_are_slices, zero_dtype dtype,
                               const zero_layout *layout, int rank, float *const master[2],
                               float *const m[2], float *const v[2], void *const params[2],
                               float *g_stage, const zero_adam_cfg *cfg,
                               zero_step_state *state_dev, void *ws, size_t ws_bytes,
                               zero_stream_t stream)
{
    int rc = check_grads(grads, grads_are_slices, dtype, layout, rank);
    if (rc)
        return rc;
    if ((rc = check_cfg(cfg)))
        return rc;
    const bool clip = cfg->max_grad_norm > 0.0;
    if ((rc = check_slots(layout, cfg, master, m, v, params, g_stage, clip, state_dev, ws,
                          ws_bytes)))
        return rc;
    PassArgs a;
    a.grads = grads;
    a.grads_are_slices = grads_are_slices;
    a.dtype = dtype;
    a.lay = layout;
    a.rank = rank;
    a.cfg = cfg;
    a.state = state_dev;
    a.master = master;
    a.m = m;
    a.v = v;
    a.params = params;
    a.stage = g_stage;
    if (layout->padded_numel > 0) {
        if ((rc = check_grad_residence(grads, layout->world, &a.grads_on_device)))
            return rc;
        const int where = state_residence(master, m, v);
        if (where < 0 || (where == 1 && clip))
            return ZERO_EINVAL;  // mixed residence, or offloaded state with the clip
        a.host_state = where == 1;
    }
    return run_step(a, clip, M_FUSED, M_PASS1, g_stage ? M_PASS2_STAGED : M_PASS2_RECOMPUTE, ws,
                    stream);
}

extern "C" int zero_step_fused_accumulated(const float *acc, zero_dtype dtype,
                                           const zero_layout *layout, int rank,
                                           float *const master[2], float *const m[2],
                                           float *const v[2], void *const params[2],
                                           const zero_adam_cfg *cfg, zero_step_state *state_dev,
                                           void *ws, size_t ws_bytes, zero_stream_t stream)
{
    int rc = check_layout(layout);
    if (rc)
        return rc;
    if (dtype < ZERO_F16 || dtype > ZERO_BF16_HALF_REDUCE || rank < -1 ||
        rank >= layout->world || (!acc && layout->padded_numel))
        return ZERO_EINVAL;
    if (!aligned32(acc))
        return ZERO_EALIGN;
    if ((rc = check_cfg(cfg)))
        return rc;
    const bool clip = cfg->max_grad_norm > 0.0;
    if ((rc = check_slots(layout, cfg, master, m, v, params, nullptr, false, state_dev, ws,
                          ws_bytes)))
        return rc;
    PassArgs a;
    a.dtype = dtype;
    a.lay = layout;
    a.rank = rank;
    a.cfg = cfg;
    a.state = state_dev;
    a.master = master;
    a.m = m;
    a.v = v;
    a.params = params;
    a.stage = const_cast<float *>(acc);
    return run_step(a, clip, M_ACC_FUSED, M_ACC_PASS1, M_ACC_PASS2, ws, stream);
}

extern "C" int zero_step_fused_buckets(const void *const *grads, int grads_are_slices,
                                       zero_dtype dtype, const zero_layout *layout, int rank,
                                       int64_t first_bucket, int64_t n_buckets,
                                       float *const master[2], float *const m[2],
                                       float *const v[2], void *const params[2],
                                       const zero_adam_cfg *cfg, zero_step_state *state_dev,
                                       zero_stream_t stream)
{
    int rc = check_grads(grads, grads_are_slices, dtype, layout, rank);
    if (rc)
        return rc;
    if ((rc = check_cfg(cfg)))
        return rc;
    const zero_layout &L = *layout;
    if (cfg->max_grad_norm > 0.0 || check_range(L, first_bucket, n_buckets))
        return ZERO_EINVAL;
    if ((rc = check_pingpong(layout, cfg, master, m, v, params, state_dev)))
        return rc;
    if (n_buckets == 0 || L.padded_numel == 0)
        return ZERO_OK;
    // The buckets of the range as a layout of their own; the buffers are
    // offset to the range's first element.  Each bucket's rank slices lie
    // inside it, so the range is a self-contained bucketed vector.
    const Range R = bucket_range(L, rank, grads_are_slices, first_bucket, n_buckets);
    RangeBuffers B;
    offset_buffers(R, grads, L.world, master, m, v, params, B);
    PassArgs a;
    a.grads = B.g;
    a.grads_are_slices = grads_are_slices;
    a.dtype = dtype;
    a.lay = &R.lay;
    a.rank = rank;
    a.cfg = cfg;
    a.state = state_dev;
    a.master = B.w;
    a.m = B.m;
    a.v = B.v;
    a.params = B.par;
    if ((rc = check_grad_residence(B.g, L.world, &a.grads_on_device)))
        return rc;
    const int where = state_residence(B.w, B.m, B.v);
    if (where < 0)
        return ZERO_EINVAL;  // mixed residence
    a.host_state = where == 1;
    rc = launch_staged(a, stream);
    if (rc == 1) {
        int gx;
        rc = run(a, M_FUSED, stream, &gx);
    }
    return rc;
}

// Checks shared by the two passes of a clipped step on a range of buckets.
static int check_range_pass(const void *const *grads, int grads_are_slices, zero_dtype dtype,
                            const zero_layout *layout, int rank, int64_t first_bucket,
                            int64_t n_buckets, const zero_adam_cfg *cfg,
                            const zero_step_state *state_dev, const void *ws, size_t ws_bytes)
{
    int rc = grads ? check_grads(grads, grads_are_slices, dtype, layout, rank)
                   : check_layout(layout);
    if (rc)
        return rc;
    if (dtype < ZERO_F16 || dtype > ZERO_BF16_HALF_REDUCE || rank < -1 ||
        rank >= layout->world || (grads_are_slices && rank < 0))
        return ZERO_EINVAL;
    if ((rc = check_cfg(cfg)))
        return rc;
    if (!(cfg->max_grad_norm > 0.0) || !state_dev ||
        check_range(*layout, first_bucket, n_buckets))
        return ZERO_EINVAL;
    if (reinterpret_cast<uintptr_t>(state_dev) & 7u)
        return ZERO_EALIGN;
    return check_ws(layout, ws, ws_bytes);
}

extern "C" int zero_step_buckets_pass1(const void *const *grads, int grads_are_slices,
                                       zero_dtype dtype, const zero_layout *layout, int rank,
                                       int64_t first_bucket, int64_t n_buckets, float *g_stage,
                                       const zero_adam_cfg *cfg, zero_step_state *state_dev,
                                       void *ws, size_t ws_bytes, zero_stream_t stream)
{
    if (!grads)
        return ZERO_EINVAL;
    int rc = check_range_pass(grads, grads_are_slices, dtype, layout, rank, first_bucket,
                              n_buckets, cfg, state_dev, ws, ws_bytes);
    if (rc)
        return rc;
    if (g_stage && !aligned32(g_stage))
        return ZERO_EALIGN;
    const zero_layout &L = *layout;
    if (n_buckets == 0 || L.padded_numel == 0)
        return ZERO_OK;
    const Range R = bucket_range(L, rank, grads_are_slices, first_bucket, n_buckets);
    RangeBuffers B;
    offset_buffers(R, grads, L.world, nullptr, nullptr, nullptr, nullptr, B);
    PassArgs a;
    a.grads = B.g;
    a.grads_are_slices = grads_are_slices;
    a.dtype = dtype;
    a.lay = &R.lay;
    a.rank = rank;
    a.cfg = cfg;
    a.state = state_dev;
    a.stage = g_stage ? g_stage + R.state_off : nullptr;
    if ((rc = check_grad_residence(B.g, L.world, &a.grads_on_device)))
        return rc;
    a.norm = layout_plan(L, rank, first_bucket, n_buckets, ws);
    int gx;
    return run(a, M_PASS1, stream, &gx);
}

extern "C" int zero_step_buckets_norm(const zero_layout *layout, int rank, void *ws,
                                     size_t ws_bytes, zero_stream_t stream)
{
    int rc = check_layout(layout);
    if (rc)
        return rc;
    if (rank < -1 || rank >= layout->world)
        return ZERO_EINVAL;
    if ((rc = check_ws(layout, ws, ws_bytes)))
        return rc;
    const zero_layout &L = *layout;
    if (L.padded_numel == 0)
        return ZERO_OK;
    return launch_norm_tree(layout_plan(L, rank, 0, L.bucket_numel ? L.num_buckets : 1, ws),
                            stream);
}

extern "C" int zero_step_buckets_pass2(const void *const *grads, int grads_are_slices,
                                       zero_dtype dtype, const zero_layout *layout, int rank,
                                       int64_t first_bucket, int64_t n_buckets,
                                       float *const master[2], float *const m[2],
                                       float *const v[2], void *const params[2],
                                       const float *g_stage, const zero_adam_cfg *cfg,
                                       zero_step_state *state_dev, const void *ws,
                                       size_t ws_bytes, zero_stream_t stream)
{
    if (!grads == !g_stage)
        return ZERO_EINVAL;  // exactly one source of the gradient
    int rc = check_range_pass(grads, grads_are_slices, dtype, layout, rank, first_bucket,
                              n_buckets, cfg, state_dev, ws, ws_bytes);
    if (rc)
        return rc;
    if ((rc = check_pingpong(layout, cfg, master, m, v, params, state_dev)))
        return rc;
    if (g_stage && !aligned32(g_stage))
        return ZERO_EALIGN;
    const zero_layout &L = *layout;
    if (n_buckets == 0 || L.padded_numel == 0)
        return ZERO_OK;
    const Range R = bucket_range(L, rank, grads_are_slices, first_bucket, n_buckets);
    RangeBuffers B;
    offset_buffers(R, grads, L.world, master, m, v, params, B);
    PassArgs a;
    a.grads = grads ? B.g : nullptr;
    a.grads_are_slices = grads_are_slices;
    a.dtype = dtype;
    a.lay = &R.lay;
    a.rank = rank;
    a.cfg = cfg;
    a.state = state_dev;
    a.master = B.w;
    a.m = B.m;
    a.v = B.v;
    a.params = B.par;
    a.stage = g_stage ? const_cast<float *>(g_stage) + R.state_off : nullptr;
    if (grads && (rc = check_grad_residence(B.g, L.world, &a.grads_on_device)))
        return rc;
    if (state_residence(B.w, B.m, B.v) != 0)
        return ZERO_EINVAL;  // the clipped step keeps its state in device memory
    a.norm_total = norm_total_slot(const_cast<void *>(ws));
    int gx;
    return run(a, g_stage ? M_PASS2_STAGED : M_PASS2_RECOMPUTE, stream, &gx);
}
