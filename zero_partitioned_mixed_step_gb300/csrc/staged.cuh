// The one-pass fused step (a2)-(a7), and (a8) when the launch ends the step,
// with its inputs staged through shared memory by the Tensor Memory
// Accelerator's bulk copies.
//
// Used for every-rank launches over the flat vector with the reduction in
// fp32, state and gradients in device memory and N_d = 16 (a compile-time
// constant, so the shared-memory reads and the copies unroll).  Measured on
// GB300 against the register kernel on the same buffers, it is 0.9 % faster
// at N_d = 16 with fp16 gradients (1.8 % with bf16) and slower at N_d = 8
// (1 %) and N_d = 4 (8 %), where the fp32 state dominates the traffic; with
// 256 threads and one CTA per SM it lost at every N_d.
// Each CTA (128 threads, two per SM) walks tiles of 1024 elements with a grid
// stride.  For a tile, one thread issues N_d + 3 one-dimensional bulk copies
// (cp.async.bulk, marked evict-first in L2): each rank's 2 KB gradient slice
// and the 4 KB slices of master, m and v of the current ping-pong slot, all
// completing on the stage's mbarrier.  The next tile's copies are in flight
// while the threads reduce, update and store the current one (two 44 KB
// stages per CTA).  Results leave with 256-bit stores
// (state) and 16-byte stores (parameters) to the other slot.  The arithmetic
// is exactly the register path's, so the two give the same bits.
//
// Waits are bounded: a CTA that polls a stage's mbarrier kStageSpinLimit
// times without completion records the error in the step state, marks the
// step as overflowed (so it is skipped and nothing changes), stops issuing
// copies, waits (again bounded) for the copies it still has in flight, and
// finishes.  When the launch ends the step, the CTA that finishes last
// commits or skips it.  A test exercises that path on the GPU: with the
// environment variable ZERO_TEST_STAGED_WAIT_LIMIT=n the launch polls a stage
// at most n times and announces 16 bytes more to each stage's mbarrier than
// its copies bring, so the first wait runs out.  The drain then retires the
// 16 bytes itself (mbarrier.complete_tx), so its wait ends exactly when the
// stage's real copies have landed: no copy is in flight when the CTA
// finishes.
#pragma once

#include "kernels.cuh"

namespace zs {

constexpr int kStagedThreads = 128;
constexpr int kStagedTile = kStagedThreads * kUnit;  // elements per tile
constexpr int kStagedMaxStages = 8;
constexpr int kStagedWorld = 16;                  // the one N_d it serves
constexpr int kStagedSmemBudget = 100 * 1024;     // dynamic shared memory per CTA
constexpr long long kStageSpinLimit = 1ll << 26;  // polls of try_wait (seconds)

// Bytes of one stage for a group of `world` ranks.
__host__ __device__ constexpr int staged_stage_bytes(int world)
{
    return world * kStagedTile * 2 + 3 * kStagedTile * 4;
}

inline int staged_stages(int world)
{
    const int n = kStagedSmemBudget / staged_stage_bytes(world);
    return n < 2 ? 0 : (n > kStagedMaxStages ? kStagedMaxStages : n);
}

struct StagedParams {
    const uint16_t *g[kStagedWorld];
    int32_t stages;
    int64_t n;  // padded flat elements (a multiple of 64)
    CfgDev cfg;
    zero_step_state *state;
    const float *w0, *w1, *m0, *m1, *v0, *v1;
    float *wo0, *wo1, *mo0, *mo1, *vo0, *vo1;
    uint16_t *par0, *par1;
    int32_t end_step;  // the CTA that finishes last ends the step (a8)
    FinCfg fin;
    long long spin_limit;  // polls of a stage's mbarrier before giving up
    uint32_t tx_extra;     // 0; > 0 only when a test makes every wait run out
};

__device__ __forceinline__ bool stage_ready(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        :
        : "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

template <int DT, int W>
__global__ void __launch_bounds__(kStagedThreads, 1)
    staged_fused_kernel(const __grid_constant__ StagedParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full[kStagedMaxStages];
    __shared__ Scalars sh;
    __shared__ int sh_cur;
    __shared__ int abort_flag;
    const int tid = threadIdx.x;
    constexpr int world = W;
    constexpr int sb = staged_stage_bytes(W);
    constexpr int gbytes = W * kStagedTile * 2;
    const int nst = p.stages;
    const int64_t tiles = (p.n + kStagedTile - 1) / kStagedTile;
    form_scalars<true>(p.cfg, p.state, nullptr, sh, sh_cur);
    if (tid == 0) {
        abort_flag = 0;
        for (int st = 0; st < nst; ++st) {
            const uint32_t a = (uint32_t)__cvta_generic_to_shared(&full[st]);
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(a) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const Scalars s = sh;
    const int cur = sh_cur;
    const float *w_src = cur ? p.w1 : p.w0;
    const float *m_src = cur ? p.m1 : p.m0;
    const float *v_src = cur ? p.v1 : p.v0;
    float *w_dst = cur ? p.wo0 : p.wo1;
    float *m_dst = cur ? p.mo0 : p.mo1;
    float *v_dst = cur ? p.vo0 : p.vo1;
    uint16_t *out = cur ? p.par0 : p.par1;
    const uint64_t pol = evict_first_policy();

    // Tile k of this CTA into stage k % nst (thread 0 only).
    auto issue = [&](int64_t k) {
        const int64_t t = blockIdx.x + k * gridDim.x;
        if (t >= tiles)
            return;
        const int st = (int)(k % nst);
        const int64_t e0 = t * kStagedTile;
        const int64_t left = p.n - e0;
        const uint32_t len = (uint32_t)(left < kStagedTile ? left : kStagedTile);  // multiple of 64
        const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&full[st]);
        const uint32_t base = (uint32_t)__cvta_generic_to_shared(smem + st * sb);
        // the threads' earlier reads of this stage come before the copies' writes
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                     "r"(len * 2u * (uint32_t)world + 3u * len * 4u + p.tx_extra)
                     : "memory");
#pragma unroll
        for (int q = 0; q < W; ++q)
            bulk_copy(base + q * kStagedTile * 2, p.g[q] + e0, len * 2u, bar, pol);
        bulk_copy(base + gbytes, w_src + e0, len * 4u, bar, pol);
        bulk_copy(base + gbytes + kStagedTile * 4, m_src + e0, len * 4u, bar, pol);
        bulk_copy(base + gbytes + 2 * kStagedTile * 4, v_src + e0, len * 4u, bar, pol);
    };

    if (tid == 0)
        for (int k = 0; k < nst; ++k)
            issue(k);
    bool bad = false;
    int64_t k = 0;
    for (;; ++k) {
        const int64_t t = blockIdx.x + k * gridDim.x;
        if (t >= tiles)
            break;
        const int st = (int)(k % nst);
        const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&full[st]);
        const uint32_t parity = (uint32_t)((k / nst) & 1);
        bool ready = false;
        for (long long it = 0; it < p.spin_limit; ++it)
            if (stage_ready(bar, parity)) {
                ready = true;
                break;
            }
        if (!ready)
            abort_flag = 1;
        __syncthreads();
        if (abort_flag)
            break;
        const uint8_t *stage = smem + st * sb;
        const int64_t e = t * kStagedTile + (int64_t)tid * kUnit;
        if (e < p.n) {
            float g[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                g[i] = 0.0f;
            uint4 x[W];
#pragma unroll
            for (int q = 0; q < W; ++q)
                x[q] = reinterpret_cast<const uint4 *>(stage + q * kStagedTile * 2)[tid];
#pragma unroll
            for (int q = 0; q < W; ++q)
                add_half8<DT>(g, x[q]);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                g[i] = __fmul_rn(g[i], s.inv_s);
                bad |= nonfinite(g[i]);
            }
            float w[8], m[8], v[8];
            const float4 *sw = reinterpret_cast<const float4 *>(stage + gbytes) + 2 * tid;
            const float4 *sm = reinterpret_cast<const float4 *>(stage + gbytes + kStagedTile * 4) +
                               2 * tid;
            const float4 *sv =
                reinterpret_cast<const float4 *>(stage + gbytes + 2 * kStagedTile * 4) + 2 * tid;
            const float4 a0 = sw[0], a1 = sw[1], b0 = sm[0], b1 = sm[1], c0 = sv[0], c1 = sv[1];
            w[0] = a0.x; w[1] = a0.y; w[2] = a0.z; w[3] = a0.w;
            w[4] = a1.x; w[5] = a1.y; w[6] = a1.z; w[7] = a1.w;
            m[0] = b0.x; m[1] = b0.y; m[2] = b0.z; m[3] = b0.w;
            m[4] = b1.x; m[5] = b1.y; m[6] = b1.z; m[7] = b1.w;
            v[0] = c0.x; v[1] = c0.y; v[2] = c0.z; v[3] = c0.w;
            v[4] = c1.x; v[5] = c1.y; v[6] = c1.z; v[7] = c1.w;
            adam8(g, w, m, v, s);
            store8(w_dst + e, w);
            store8(m_dst + e, m);
            store8(v_dst + e, v);
            st_half8(out + e, pack_half8<DT>(w), pol);
        }
        __syncthreads();  // every thread is done with this stage
        if (tid == 0)
            issue(k + nst);
    }
    if (abort_flag) {
        if (tid == 0) {
            atomicOr(&p.state->error, 1);     // error: a stage never completed
            atomicOr(&p.state->found_inf, 1);  // skip the step: nothing changes
            for (int64_t kk = k; kk < k + nst; ++kk) {  // copies still in flight
                const int64_t t = blockIdx.x + kk * gridDim.x;
                if (t >= tiles)
                    break;
                const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&full[kk % nst]);
                if (p.tx_extra)  // the announced extra bytes never come: retire them
                    asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(bar),
                                 "r"(p.tx_extra)
                                 : "memory");
                for (long long it = 0; it < kStageSpinLimit; ++it)
                    if (stage_ready(bar, (uint32_t)((kk / nst) & 1)))
                        break;
            }
        }
    }
    // the next step's bias-correction scalars, by the last CTA (the least work)
    if (blockIdx.x == gridDim.x - 1 && tid == 0)
        form_next_scalars(p.cfg, p.state);
    finish_cta(abort_flag || bad, p.end_step != 0, p.fin, p.state);
}

}  // namespace zs
