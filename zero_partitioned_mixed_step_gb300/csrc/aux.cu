// The unfused entry points (zero_check_overflow, zero_grad_norm,
// zero_adam_step, zero_step_finalize) and the small single-CTA kernels that
// end a step.
#include <atomic>
#include <cmath>
#include <cstdlib>

#include "kernels.cuh"

namespace zs {

// Resident CTAs per SM of each kernel, looked up once per kernel (the value
// depends only on the kernel and the architecture), and the SM count of each
// device: both are read-only after the first launch, so launches do not pay
// for the queries again.
namespace {

constexpr int kOccSlots = 512;
struct OccSlot {
    std::atomic<const void *> kernel{nullptr};
    std::atomic<int> occ{0};
};
OccSlot occ_slots[kOccSlots];
constexpr int kSmDevices = 64;
std::atomic<int> sm_count[kSmDevices];

int resident_ctas(const void *kernel)
{
    const size_t h = (reinterpret_cast<uintptr_t>(kernel) >> 4) % kOccSlots;
    for (size_t i = 0; i < kOccSlots; ++i) {
        OccSlot &s = occ_slots[(h + i) % kOccSlots];
        const void *k = s.kernel.load(std::memory_order_acquire);
        if (k == kernel) {
            const int occ = s.occ.load(std::memory_order_acquire);
            if (occ > 0)
                return occ;
            break;  // another thread is filling this slot: query directly
        }
        if (k == nullptr) {
            int occ = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, 0) !=
                    cudaSuccess || occ < 1)
                return 1;
            const void *expected = nullptr;
            if (s.kernel.compare_exchange_strong(expected, kernel, std::memory_order_acq_rel))
                s.occ.store(occ, std::memory_order_release);
            return occ;
        }
    }
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, 0) != cudaSuccess ||
        occ < 1)
        occ = 1;
    return occ;
}

}  // namespace

int device_sms()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 1;
    if (dev >= 0 && dev < kSmDevices && (sms = sm_count[dev].load(std::memory_order_acquire)) > 0)
        return sms;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms < 1)
        return 1;
    if (dev >= 0 && dev < kSmDevices)
        sm_count[dev].store(sms, std::memory_order_release);
    return sms;
}

int test_grid_cap()
{
    static const int cap = [] {
        const char *t = std::getenv("ZERO_TEST_MAX_CTAS");
        const long v = t ? std::atol(t) : 0;
        return v > 0 && v < kMaxCtas ? (int)v : 0;
    }();
    return cap;
}

int target_ctas(const void *kernel)
{
    int64_t t = (int64_t)device_sms() * resident_ctas(kernel);
    if (t > kMaxCtas)
        t = kMaxCtas;
    const int cap = test_grid_cap();
    return (int)(cap > 0 && t > cap ? cap : t);
}

// ------------------------------------------------------------------ end of step

__global__ void finalize_kernel(FinCfg c, zero_step_state *st, int flip)
{
    if (threadIdx.x != 0 || blockIdx.x != 0)
        return;
    end_step(c, st, flip, st->found_inf & 1);
}

int launch_finalize(const zero_adam_cfg *cfg, zero_step_state *state, int flip, cudaStream_t s)
{
    finalize_kernel<<<1, 32, 0, s>>>(fin_cfg(*cfg), state, flip);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ZERO_OK : cuda_error(e);
}

// ------------------------------------------------------------------ element-wise kernels

static int grid_for(const void *kernel, int64_t units)
{
    const int target = target_ctas(kernel);
    const int64_t want = (units + kThreads - 1) / kThreads;
    return (int)(want < 1 ? 1 : (want < target ? want : target));
}

__global__ void __launch_bounds__(kThreads)
    overflow_kernel(const float *g, int64_t n, float inv_s, int32_t *flag)
{
    bool bad = false;
    const int64_t n4 = n / 4;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t k = (int64_t)blockIdx.x * kThreads + threadIdx.x; k < n4; k += stride) {
        const float4 x = ld_state4(g + 4 * k);
        bad |= nonfinite(__fmul_rn(x.x, inv_s)) | nonfinite(__fmul_rn(x.y, inv_s)) |
               nonfinite(__fmul_rn(x.z, inv_s)) | nonfinite(__fmul_rn(x.w, inv_s));
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 3))
        bad |= nonfinite(__fmul_rn(g[4 * n4 + threadIdx.x], inv_s));
    flag_nonfinite(bad, flag);
}

// The tree above the chunk sums that a first pass (or the first passes of
// all the bucket ranges of a step) stored: every warp sums superchunks (lane
// l adds chunks l and l + 32 of the superchunk from +0, then a fixed
// butterfly); the CTA that finishes last adds each rank's superchunks (the
// same lane order) and then the ranks in ascending order from +0, writes the
// total and returns the counter to zero.
__global__ void __launch_bounds__(kThreads) norm_tree_kernel(NormPlan np)
{
    __shared__ double rank_sum[ZERO_MAX_WORLD];
    __shared__ int last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t nsc = (int64_t)np.ranks * np.spr;
    const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
    for (int64_t sc = (int64_t)blockIdx.x * (kThreads / 32) + warp; sc < nsc; sc += warps) {
        const int64_t r = sc / np.spr, s = sc - r * np.spr;
        const int64_t left = np.cpr - s * kNormSuper;
        const double x = warp_fixed_sum(np.partials + r * np.cpr + s * kNormSuper,
                                        left < kNormSuper ? left : kNormSuper);
        if (lane == 0)
            np.sc_partials[sc] = x;
    }
    __threadfence();  // this CTA's superchunk sums before its count
    __syncthreads();
    if (threadIdx.x == 0)
        last = atomicAdd(np.done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last)
        return;
    __threadfence();
    for (int r = warp; r < np.ranks; r += kThreads / 32) {
        const double x = warp_fixed_sum(np.sc_partials + (int64_t)r * np.spr, np.spr);
        if (lane == 0)
            rank_sum[r] = x;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double total = 0.0;
        for (int r = 0; r < np.ranks; ++r)
            total = __dadd_rn(total, rank_sum[r]);
        *np.total = total;
        *np.done = 0u;
    }
}

int launch_norm_tree(const NormPlan &np, cudaStream_t stream)
{
    const int64_t nsc = (int64_t)np.ranks * np.spr;
    const int64_t want = (nsc + kThreads / 32 - 1) / (kThreads / 32);
    const int target = target_ctas(reinterpret_cast<const void *>(norm_tree_kernel));
    const int gx = (int)(want < 1 ? 1 : (want < target ? want : target));
    norm_tree_kernel<<<gx, kThreads, 0, stream>>>(np);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ZERO_OK : cuda_error(e);
}

// The chunk sums of the squares of g * inv_s, the vector taken as one rank's
// single slice of ceil(n / 8) units (the last one padded with zeros).
__global__ void __launch_bounds__(kThreads)
    norm_kernel(const float *g, int64_t n, float inv_s, NormPlan np)
{
    const int64_t full = n / kUnit;
    norm_walk(np, [&](const ChunkLoc &L) {
        SumSq ss;
        for (int64_t k = threadIdx.x; k < L.n_u; k += kThreads) {
            const int64_t u = L.u0 + k;
            float x[8];
            if (u < full) {
                load8(g + u * kUnit, x);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    x[i] = u * kUnit + i < n ? g[u * kUnit + i] : 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
                x[i] = __fmul_rn(x[i], inv_s);
            ss.add8(x);
        }
        return ss.acc;
    });
}

// zero_grad_norm's two launches (the chunk sums, then the tree) with the tree in
// `ws`, a workspace of ws_bytes bytes whose counter is zero.
static int launch_norm(const float *g, int64_t n, float inv_scale, double *sumsq_dev, void *ws,
                       size_t ws_bytes, cudaStream_t stream)
{
    if (n == 0) {  // an empty sum: +0
        const cudaError_t e = cudaMemsetAsync(sumsq_dev, 0, sizeof(double), stream);
        return e == cudaSuccess ? ZERO_OK : cuda_error(e);
    }
    const int64_t units = (n + kUnit - 1) / kUnit;
    const NormGeom geo = norm_geometry(units, units, 1);
    if (norm_ws_bytes(1, geo) > ws_bytes)
        return ZERO_ESPACE;
    const NormPlan np = norm_plan(geo, units, units, 1, 0, 1, 1, ws, sumsq_dev);
    const int target = target_ctas(reinterpret_cast<const void *>(norm_kernel));
    const int gx = (int)(np.launch_chunks < target ? np.launch_chunks : target);
    norm_kernel<<<gx, kThreads, 0, stream>>>(g, n, inv_scale, np);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_error(e);
    return launch_norm_tree(np, stream);
}

template <int DT>
__global__ void __launch_bounds__(kThreads)
    adam_kernel(const float *g, float *w, float *m, float *v, uint16_t *out, int64_t n,
                CfgDev cfg, const zero_step_state *st)
{
    __shared__ Scalars sh;
    __shared__ int sh_cur;
    form_scalars<true>(cfg, st, &st->sumsq, sh, sh_cur);
    __syncthreads();
    const Scalars s = sh;
    if (s.skip)
        return;
    const uint64_t pol = evict_first_policy();
    const bool scale = s.clip && s.coef < 1.0f;
    const int64_t units = n / kUnit;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t k = (int64_t)blockIdx.x * kThreads + threadIdx.x; k < units; k += stride) {
        const int64_t e = k * kUnit;
        float gg[8], ww[8], mm[8], vv[8];
        load8(g + e, gg);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            gg[i] = __fmul_rn(gg[i], s.inv_s);
            if (scale)
                gg[i] = __fmul_rn(gg[i], s.coef);
        }
        load8(w + e, ww);
        load8(m + e, mm);
        load8(v + e, vv);
        adam8(gg, ww, mm, vv, s);
        store8(w + e, ww);
        store8(m + e, mm);
        store8(v + e, vv);
        st_half8(out + e, pack_half8<DT>(ww), pol);
    }
    if (blockIdx.x == 0 && threadIdx.x < (n % kUnit)) {
        const int64_t e = units * kUnit + threadIdx.x;
        float gg = __fmul_rn(g[e], s.inv_s);
        if (scale)
            gg = __fmul_rn(gg, s.coef);
        float ww = w[e], mm = m[e], vv = v[e];
        adam1(gg, ww, mm, vv, s);
        w[e] = ww;
        m[e] = mm;
        v[e] = vv;
        out[e] = round_half1<DT>(ww);
    }
}

}  // namespace zs

using namespace zs;

extern "C" {

int zero_check_overflow(const float *g, int64_t n, float inv_scale, int32_t *flag_dev,
                        zero_stream_t stream)
{
    if (n < 0 || !flag_dev || (n > 0 && !g) || !(inv_scale > 0.0f) || !std::isfinite(inv_scale))
        return ZERO_EINVAL;
    if (!aligned16(g) || (reinterpret_cast<uintptr_t>(flag_dev) & 3u))
        return ZERO_EALIGN;
    if (n == 0)
        return ZERO_OK;
    const int gx = grid_for(reinterpret_cast<const void *>(overflow_kernel), n / 4);
    overflow_kernel<<<gx, kThreads, 0, stream>>>(g, n, inv_scale, flag_dev);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ZERO_OK : cuda_error(e);
}

int zero_grad_norm(const float *g, int64_t n, float inv_scale, double *sumsq_dev, void *ws,
                   size_t ws_bytes, zero_stream_t stream)
{
    if (n < 0 || !sumsq_dev || !ws || (n > 0 && !g) || !(inv_scale > 0.0f) ||
        !std::isfinite(inv_scale))
        return ZERO_EINVAL;
    if (!aligned32(g) || !aligned16(ws) || (reinterpret_cast<uintptr_t>(sumsq_dev) & 7u))
        return ZERO_EALIGN;
    if (ws_bytes < zero_workspace_bytes(nullptr))
        return ZERO_ESPACE;
    return launch_norm(g, n, inv_scale, sumsq_dev, ws, ws_bytes, stream);
}

int zero_adam_step(const float *g, float *master, float *m, float *v, void *half_out,
                   zero_dtype dtype, int64_t n, const zero_adam_cfg *cfg,
                   const zero_step_state *state_dev, zero_stream_t stream)
{
    int rc = check_cfg(cfg);
    if (rc)
        return rc;
    if (n < 0 || !state_dev || dtype < ZERO_F16 || dtype > ZERO_BF16_HALF_REDUCE ||
        (n > 0 && (!g || !master || !m || !v || !half_out)))
        return ZERO_EINVAL;
    if (!aligned32(g) || !aligned32(master) || !aligned32(m) || !aligned32(v) ||
        !aligned16(half_out) || (reinterpret_cast<uintptr_t>(state_dev) & 7u))
        return ZERO_EALIGN;
    if (n == 0)
        return ZERO_OK;
    const CfgDev c = make_cfg_dev(*cfg);
    uint16_t *out = static_cast<uint16_t *>(half_out);
    if (!is_bf16(dtype)) {  // the output's storage type
        const int gx = grid_for(reinterpret_cast<const void *>(adam_kernel<ZERO_F16>), n / kUnit);
        adam_kernel<ZERO_F16><<<gx, kThreads, 0, stream>>>(g, master, m, v, out, n, c, state_dev);
    } else {
        const int gx = grid_for(reinterpret_cast<const void *>(adam_kernel<ZERO_BF16>), n / kUnit);
        adam_kernel<ZERO_BF16><<<gx, kThreads, 0, stream>>>(g, master, m, v, out, n, c, state_dev);
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ZERO_OK : cuda_error(e);
}

int zero_step_finalize(const zero_adam_cfg *cfg, zero_step_state *state_dev, int flip_slot,
                       zero_stream_t stream)
{
    int rc = check_cfg(cfg);
    if (rc)
        return rc;
    if (!state_dev)
        return ZERO_EINVAL;
    if (reinterpret_cast<uintptr_t>(state_dev) & 7u)
        return ZERO_EALIGN;
    return launch_finalize(cfg, state_dev, flip_slot ? 1 : 0, stream);
}

}  // extern "C"

// ------------------------------------------------------------------ no-allocation norm
//
// zero_grad_norm_noalloc: zero_grad_norm's kernel with the norm's tree in a
// library-owned device array instead of a caller-provided workspace.

namespace zs {

static_assert(kNormWsAnyVector == ZERO_NOALLOC_SCRATCH_BYTES,
              "the static scratch holds the tree of any vector");

// The tree of one call: its counter (zero when the library is loaded, and
// returned to zero by every call that completes), chunk and superchunk sums.  Every GPU that loads the library holds this array
// until the process exits.  In host code the name is only a host-side
// stand-in for the device array: kernels must be given the address
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char noalloc_ws[ZERO_NOALLOC_SCRATCH_BYTES];

constexpr int kNoallocDevices = 64;
static std::atomic<void *> noalloc_ptr[kNoallocDevices];

// The device address of noalloc_ws on device `dev` (the current device),
// looked up on the first call for that device and cached.
static int noalloc_scratch(int dev, void **out)
{
    if (dev >= 0 && dev < kNoallocDevices) {
        void *p = noalloc_ptr[dev].load(std::memory_order_acquire);
        if (p) {
            *out = p;
            return ZERO_OK;
        }
    }
    void *addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, noalloc_ws);
    if (e != cudaSuccess || !addr) {
        (void)cudaGetLastError();
        return cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    }
    if (dev >= 0 && dev < kNoallocDevices)
        noalloc_ptr[dev].store(addr, std::memory_order_release);
    *out = addr;
    return ZERO_OK;
}

}  // namespace zs

extern "C" int zero_grad_norm_noalloc(const float *g, int64_t n, float inv_scale,
                                      double *sumsq_dev, zero_stream_t stream)
{
    using namespace zs;
    if (n < 0 || !sumsq_dev || (n > 0 && !g) || !(inv_scale > 0.0f) || !std::isfinite(inv_scale))
        return ZERO_EINVAL;
    if (!aligned32(g) || (reinterpret_cast<uintptr_t>(sumsq_dev) & 7u))
        return ZERO_EALIGN;
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return cuda_error(e);
    }
    void *scratch = nullptr;
    const int rc = noalloc_scratch(dev, &scratch);
    if (rc)
        return rc;
    // a vector whose tree needs more than the array holds is ZERO_ESPACE
    // (none does: the chunks grow with the vector)
    return launch_norm(g, n, inv_scale, sumsq_dev, scratch, ZERO_NOALLOC_SCRATCH_BYTES, stream);
}
