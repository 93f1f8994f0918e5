// The streaming kernels of the step and the entry points zero_step_fused,
// zero_step_fused_accumulated, zero_step_fused_buckets,
// zero_reduce_scatter_sum and zero_reduce_scatter_accumulate.
//
// One kernel template covers the passes over the data.  Each thread handles
// 8-element units (16-byte loads of each rank's half gradient, 32-byte loads
// and stores of each fp32 state array) with a grid stride; the grid is one
// wave: exactly as many CTAs as the SMs hold at once (every CTA does the same
// share of the work, so a second, partial wave would only add a tail).
//   FUSED      (a2)-(a7) in one pass: reduce, unscale, flag, Adam from slot
//              cur into slot 1 - cur, cast into the parameter buffer.
//   PASS1      (a2)-(a5) of a clipped step: reduce, unscale, flag, per-CTA
//              sums of squares, optionally keep g in a staging buffer.
//   PASS2_*    (a5 clip)-(a7) of a clipped step, skipped when pass 1 flagged
//              an overflow; every CTA first reduces pass 1's per-CTA sums of
//              squares in one fixed order; g is reduced again or read from
//              the stage.  It walks the units backwards, starting on the
//              first pass's last units, whose data pass 1 left in L2.
//   RS         (a2) alone: the reduced fp32 gradient.
//   RS_ACC     (a2) into an fp32 accumulator (gradient accumulation).
//   ACC_*      the step with the gradient read from an fp32 accumulator (the
//              sum of micro-steps' reduced, still scaled gradients) instead of
//              the N_d half buffers: FUSED, PASS1 and PASS2 as above.
// The last launch of a step (FUSED, a second pass, ACC_FUSED) also ends it:
// the CTA that finishes last commits or skips the step (a8).  Gradient
// buffers may be device memory or page-locked host memory, which these
// kernels load over the host link.
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
    double *partials;  // PASS1: one per CTA; second passes reduce them
    int32_t n_partials;  // second passes: CTAs of the first pass
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
    FinCfg fin;
};

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
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    if constexpr (!reduces_only(MODE)) {
        if constexpr (second_pass(MODE)) {
            // The global sum of squares, reduced by every CTA from the first
            // pass's per-CTA partials in one fixed order (all CTAs get the
            // same bits); CTA 0 publishes it in the state.
            if (threadIdx.x < 32) {
                const double x = warp_fixed_sum(p.partials, p.n_partials);
                if (threadIdx.x == 0) {
                    const double total = __dadd_rn(0.0, x);
                    compute_scalars(p.cfg, p.state, total, sh);
                    sh_cur = p.state->cur;
                    if (blockIdx.x == 0 && !sh.skip) {
                        p.state->sumsq = total;
                        p.state->clip_coef = sh.coef;
                    }
                }
            }
        } else if (threadIdx.x == 0) {
            compute_scalars(p.cfg, p.state, p.state->sumsq, sh);
            sh_cur = p.state->cur;
        }
        __syncthreads();
        s = sh;
        cur = sh_cur;
    }
    bool work = true;
    if constexpr (second_pass(MODE)) {
        if (s.skip) {  // the whole step is skipped: write nothing
            work = false;
            if constexpr (MODE == M_PASS2_STAGED) {
                if (p.discard)  // the kept stage lines are not needed either
                    for (int64_t u = p.keep_from +
                                     4 * ((int64_t)blockIdx.x * kThreads + threadIdx.x);
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

    const uint64_t pol = evict_first_policy();
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

    const int64_t base = (int64_t)blockIdx.x * kThreads;
    if constexpr (second_pass(MODE)) {
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
        for (int64_t u = base + threadIdx.x; u < vw.units; u += stride)
            unit(u);
    }
    if constexpr (flags_overflow(MODE))
        flag_nonfinite(bad, &p.state->found_inf);
    if constexpr (sums_squares(MODE)) {
        const double tot = block_sum(ss.acc);
        if (threadIdx.x == 0)
            p.partials[blockIdx.x] = tot;
    }
    if constexpr (ends_step(MODE)) {
        if (p.end_step)
            arrive_and_end_step(p.fin, p.state);
    }
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
// register caps also reorder the loads).
template <int DT, int W, int MAXW, int MODE, bool ALL>
__global__ void __launch_bounds__(kThreads, 5)
    step_kernel_host_state(const __grid_constant__ StepParams<MAXW> p)
{
    step_body<DT, W, MAXW, MODE, ALL, true>(p);
}

// ------------------------------------------------------------------ launch

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
    const int target = target_ctas(reinterpret_cast<const void *>(kern));
    const int64_t want = (p.view.units + kThreads - 1) / kThreads;
    const int64_t gx = want < 1 ? 1 : (want < target ? want : target);
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
    const void *const *grads;
    int grads_are_slices;
    zero_dtype dtype;
    const zero_layout *lay;
    int rank;
    const zero_adam_cfg *cfg;
    zero_step_state *state;
    float *const *master, *const *m, *const *v;
    void *const *params;
    float *stage;
    double *partials;
    int add;
    bool host_state = false;  // master/m/v in pinned host memory (one-pass step only)
    int n_partials = 0;       // second passes: CTAs of the first pass
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
        p.cfg = CfgDev{c.lr, c.beta1, c.beta2, c.eps, c.weight_decay, c.max_grad_norm,
                       c.adamw ? 1 : 0, c.bias_correction ? 1 : 0};
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
    p.partials = a.partials;
    p.n_partials = a.n_partials;
    p.add = a.add;
    p.keep_from = a.keep_from < v.units ? a.keep_from : v.units;
    p.discard = a.discard && p.keep_from < v.units ? 1 : 0;
    p.end_step = a.end_step ? 1 : 0;
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

// Where a buffer lives: 1 pinned host memory, 0 device memory, -1 neither
// (pageable host memory or an unknown pointer).
int residence(const void *p)
{
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    if (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged)
        return 0;
    return attr.type == cudaMemoryTypeHost ? 1 : -1;
}

// 1 when all six master/m/v slots are pinned host memory (offload), 0 when
// all are device memory, ZERO_EINVAL otherwise.
int state_residence(float *const master[2], float *const m[2], float *const v[2])
{
    const void *ptrs[6] = {master[0], master[1], m[0], m[1], v[0], v[1]};
    int first = residence(ptrs[0]);
    for (int i = 1; i < 6; ++i)
        if (residence(ptrs[i]) != first)
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
    if ((stage && !aligned32(stage)) || !aligned16(ws))
        return ZERO_EALIGN;
    if (ws_bytes < zero_workspace_bytes(layout->world))
        return ZERO_ESPACE;
    return ZERO_OK;
}

// The staged one-pass step (staged.cuh), when it applies: every rank at once,
// fp32 reduction, device-resident state, N_d = 16.  Returns 1 when it does not
// apply (the caller then uses the register path).
template <int DT, int W>
int launch_staged_w(const StagedParams &p, cudaStream_t stream)
{
    static const int resident = [] {
        if (cudaFuncSetAttribute(staged_fused_kernel<DT, W>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kStagedSmemBudget) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, staged_fused_kernel<DT, W>,
                                                          kStagedThreads, kStagedSmemBudget) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        return occ;
    }();
    if (resident < 1)
        return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    const int64_t tiles = (p.n + kStagedTile - 1) / kStagedTile;
    const int64_t want = (int64_t)sms * resident;
    const unsigned grid = (unsigned)(tiles < want ? tiles : want);
    staged_fused_kernel<DT, W>
        <<<grid, kStagedThreads, p.stages * staged_stage_bytes(W), stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ZERO_OK : cuda_error(e);
}

int launch_staged(const PassArgs &a, cudaStream_t stream)
{
    const zero_layout &L = *a.lay;
    const int stages = staged_stages(L.world);
    if (a.rank >= 0 || a.host_state || half_reduce(a.dtype) || L.world != kStagedWorld ||
        stages < 2 || L.padded_numel <= 0)
        return 1;
    // The bulk copies serve gradients in device memory; gradients in
    // page-locked host memory are loaded by the register kernel.
    for (int q = 0; q < L.world; ++q)
        if (residence(a.grads[q]) != 0)
            return 1;
    StagedParams p{};
    for (int q = 0; q < L.world; ++q)
        p.g[q] = static_cast<const uint16_t *>(a.grads[q]);
    p.stages = stages;
    p.n = L.padded_numel;
    const zero_adam_cfg &c = *a.cfg;
    p.cfg = CfgDev{c.lr, c.beta1, c.beta2, c.eps, c.weight_decay, c.max_grad_norm,
                   c.adamw ? 1 : 0, c.bias_correction ? 1 : 0};
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
    if (const char *t = std::getenv("ZERO_TEST_STAGED_WAIT_LIMIT")) {  // tests only
        const long long n = std::atoll(t);
        if (n > 0) {
            p.spin_limit = n;
            p.tx_extra = 16;
        }
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

// One step (one or two passes) in the given modes.  With commit the step's
// last launch also ends the step (a8: its last CTA commits or skips); an empty
// vector runs no pass and ends the step with the one-thread kernel.  A clipped
// step's second pass reduces the first pass's per-CTA sums of squares itself
// (there is no separate norm kernel).
int run_step(PassArgs &a, bool clip, int one_pass, int pass1, int pass2, cudaStream_t stream,
             bool commit = true)
{
    int rc, gx = 1;
    const zero_layout &L = *a.lay;
    if (L.padded_numel == 0)
        return commit ? launch_finalize(a.cfg, a.state, 1, stream) : ZERO_OK;
    if (!clip) {
        a.end_step = commit;
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
    a.end_step = false;
    if ((rc = run(a, pass1, stream, &gx)))
        return rc;
    a.n_partials = gx;
    a.end_step = commit;
    return run(a, pass2, stream, &gx);
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
    PassArgs a{grads, grads_are_slices, dtype, layout, rank, nullptr, nullptr,
               nullptr, nullptr, nullptr, nullptr, g_out, nullptr, 0};
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
    PassArgs a{grads, grads_are_slices, dtype, layout, rank, nullptr, nullptr,
               nullptr, nullptr, nullptr, nullptr, acc, nullptr, add ? 1 : 0};
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
    double *partials = reinterpret_cast<double *>(static_cast<char *>(ws) + kWsHeader);
    PassArgs a{grads, grads_are_slices, dtype, layout, rank, cfg, state_dev,
               master, m, v, params, g_stage, partials, 0};
    if (layout->padded_numel > 0) {
        const int where = state_residence(master, m, v);
        if (where < 0 || (where == 1 && clip))
            return ZERO_EINVAL;  // mixed residence, or offloaded state with the clip
        a.host_state = where == 1;
    }
    return run_step(a, clip, M_FUSED, M_PASS1, g_stage ? M_PASS2_STAGED : M_PASS2_RECOMPUTE,
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
    double *partials = reinterpret_cast<double *>(static_cast<char *>(ws) + kWsHeader);
    PassArgs a{nullptr, 0, dtype, layout, rank, cfg, state_dev,
               master, m, v, params, const_cast<float *>(acc), partials, 0};
    return run_step(a, clip, M_ACC_FUSED, M_ACC_PASS1, M_ACC_PASS2, stream);
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
    if (cfg->max_grad_norm > 0.0 || first_bucket < 0 || n_buckets < 0 ||
        first_bucket > L.num_buckets - n_buckets)
        return ZERO_EINVAL;
    if ((rc = check_pingpong(layout, cfg, master, m, v, params, state_dev)))
        return rc;
    if (n_buckets == 0 || L.padded_numel == 0)
        return ZERO_OK;
    // The buckets of the range as a layout of their own; the buffers are
    // offset to the range's first element.  Each bucket's rank slices lie
    // inside it, so the range is a self-contained bucketed vector.
    zero_layout S = L;
    int64_t flat_off = 0, owned_off = 0;
    if (L.bucket_numel > 0) {
        const int64_t end = first_bucket + n_buckets;
        S.num_buckets = n_buckets;
        S.last_slice_numel = end == L.num_buckets ? L.last_slice_numel : L.slice_numel;
        S.owned_numel = (n_buckets - 1) * L.slice_numel + S.last_slice_numel;
        S.padded_numel = S.owned_numel * L.world;
        S.numel = S.flat_numel = S.padded_numel;
        flat_off = first_bucket * L.bucket_numel;
        owned_off = first_bucket * L.slice_numel;
    }
    const int64_t state_off = rank < 0 ? flat_off : owned_off;
    const int64_t grad_off = grads_are_slices ? owned_off : flat_off;
    const void *g[ZERO_MAX_WORLD];
    for (int q = 0; q < L.world; ++q)
        g[q] = static_cast<const uint16_t *>(grads[q]) + grad_off;
    float *w2[2] = {master[0] + state_off, master[1] + state_off};
    float *m2[2] = {m[0] + state_off, m[1] + state_off};
    float *v2[2] = {v[0] + state_off, v[1] + state_off};
    void *p2[2] = {static_cast<uint16_t *>(params[0]) + flat_off,
                   static_cast<uint16_t *>(params[1]) + flat_off};
    PassArgs a{g, grads_are_slices, dtype, &S, rank, cfg, state_dev,
               w2, m2, v2, p2, nullptr, nullptr, 0};
    const int where = state_residence(w2, m2, v2);
    if (where < 0)
        return ZERO_EINVAL;  // mixed residence
    a.host_state = where == 1;
    return run_step(a, false, M_FUSED, M_PASS1, M_PASS2_RECOMPUTE, stream, false);
}
