// Host-only entry points: the partition layout (step a1), the initial step
// state, the workspace size, page-locked host blocks and the error strings.
#include <cmath>
#include <cstring>

#include <cuda_runtime.h>
#include <vector_types.h>

#include "internal.h"

namespace zs {

static int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

int check_layout(const zero_layout *lay)
{
    if (!lay || lay->world < 1 || lay->world > ZERO_MAX_WORLD || lay->align_elems < 8 ||
        lay->align_elems % 8 || lay->padded_numel < 0 || lay->owned_numel < 0)
        return ZERO_EINVAL;
    const int64_t w = lay->world;
    if (lay->owned_numel * w != lay->padded_numel || lay->padded_numel % (w * 8))
        return ZERO_EINVAL;
    if (lay->bucket_numel == 0) {
        if (lay->slice_numel != lay->owned_numel || lay->last_slice_numel != lay->owned_numel)
            return ZERO_EINVAL;
        return ZERO_OK;
    }
    if (lay->bucket_numel < 0 || lay->bucket_numel % (w * 8) || lay->num_buckets < 0 ||
        lay->slice_numel * w != lay->bucket_numel || lay->last_slice_numel % 8)
        return ZERO_EINVAL;
    if (lay->num_buckets == 0)
        return lay->padded_numel == 0 ? ZERO_OK : ZERO_EINVAL;
    if ((lay->num_buckets - 1) * lay->slice_numel + lay->last_slice_numel != lay->owned_numel)
        return ZERO_EINVAL;
    return ZERO_OK;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

NormGeom norm_geometry(int64_t slice_units, int64_t last_slice_units, int64_t nb)
{
    NormGeom g{};
    const int64_t rank_units = (nb > 0 ? nb - 1 : 0) * slice_units + last_slice_units;
    g.cu = round_up(ceil_div(rank_units, kNormChunksPerRank), kThreads);
    if (g.cu < kNormChunkMinUnits)
        g.cu = kNormChunkMinUnits;
    g.cps_last = ceil_div(last_slice_units, g.cu);
    g.cps = nb > 1 ? ceil_div(slice_units, g.cu) : g.cps_last;
    g.cpr = (nb > 0 ? nb - 1 : 0) * g.cps + g.cps_last;
    g.spr = ceil_div(g.cpr, kNormSuper);
    return g;
}

size_t norm_ws_bytes(int64_t ranks, const NormGeom &g)
{
    return (size_t)(kWsHeader + ranks * (g.cpr + g.spr) * (int64_t)sizeof(double));
}

NormPlan norm_plan(const NormGeom &g, int64_t slice_units, int64_t last_slice_units, int64_t nb,
                   int64_t b0, int64_t nbl, int32_t ranks, void *ws, double *total)
{
    NormPlan p{};
    p.cu = g.cu;
    p.cps = g.cps;
    p.cps_last = g.cps_last;
    p.cpr = g.cpr;
    p.spr = g.spr;
    p.slice_units = slice_units;
    p.last_slice_units = last_slice_units;
    p.nb = nb;
    p.b0 = b0;
    p.nbl = nbl;
    const bool has_last = b0 + nbl == nb;
    p.launch_chunks = (int64_t)ranks * ((nbl - (has_last ? 1 : 0)) * g.cps +
                                        (has_last ? g.cps_last : 0));
    p.ranks = ranks;
    char *base = static_cast<char *>(ws);
    p.done = reinterpret_cast<uint32_t *>(base);
    p.partials = reinterpret_cast<double *>(base + kWsHeader);
    p.sc_partials = p.partials + (int64_t)ranks * g.cpr;
    p.total = total ? total : norm_total_slot(ws);
    return p;
}

CfgDev make_cfg_dev(const zero_adam_cfg &c)
{
    CfgDev d{};
    d.lr = c.lr;
    d.beta1 = c.beta1;
    d.beta2 = c.beta2;
    d.max_norm = c.max_grad_norm;
    d.b1 = (float)c.beta1;
    d.omb1 = (float)(1.0 - c.beta1);
    d.b2 = (float)c.beta2;
    d.omb2 = (float)(1.0 - c.beta2);
    d.eps = (float)c.eps;
    const double lr_wd = c.lr * c.weight_decay;  // rounded on its own (no contraction)
    d.decay = (float)(1.0 - lr_wd);
    d.wd = (float)c.weight_decay;
    d.lr_f = (float)c.lr;
    d.adamw = c.adamw ? 1 : 0;
    d.bias_correction = c.bias_correction ? 1 : 0;
    return d;
}

static bool power_of_two(double x)
{
    int e;
    return x > 0.0 && std::isfinite(x) && std::frexp(x, &e) == 0.5;
}

int check_cfg(const zero_adam_cfg *c)
{
    if (!c)
        return ZERO_EINVAL;
    if (!(c->lr >= 0.0) || !(c->beta1 >= 0.0 && c->beta1 < 1.0) ||
        !(c->beta2 >= 0.0 && c->beta2 < 1.0) || !(c->eps > 0.0) || !(c->weight_decay >= 0.0) ||
        !(c->max_grad_norm >= 0.0) || !std::isfinite(c->max_grad_norm))
        return ZERO_EINVAL;
    // powers of two keep the loss scale, and so the unscale, exact
    if (c->dynamic_scale &&
        (c->growth_interval < 1 || !(c->backoff <= 1.0) || !power_of_two(c->backoff) ||
         !(c->growth >= 1.0) || !power_of_two(c->growth) || !power_of_two(c->min_scale)))
        return ZERO_EINVAL;
    return ZERO_OK;
}

}  // namespace zs

extern "C" {

const char *zero_strerror(int code)
{
    switch (code) {
    case ZERO_OK: return "ok";
    case ZERO_EINVAL: return "invalid argument";
    case ZERO_EALIGN: return "buffer not aligned (32 bytes for fp32, 16 for half)";
    case ZERO_ESPACE: return "workspace too small";
    default: return code <= ZERO_ECUDA_BASE ? "CUDA call failed" : "unknown error";
    }
}

int zero_version(void) { return 3; }

int zero_partition_layout(int n_tensors, const int64_t *numel, int world, int align_elems,
                          int64_t bucket_numel, int64_t *tensor_offset_out, zero_layout *out)
{
    if (!out || n_tensors < 0 || (n_tensors > 0 && !numel) || world < 1 ||
        world > ZERO_MAX_WORLD || align_elems < 8 || align_elems % 8 || bucket_numel < 0 ||
        (bucket_numel > 0 && bucket_numel % ((int64_t)world * 8)))
        return ZERO_EINVAL;
    const int64_t limit = INT64_C(1) << 52;  // keeps every derived size far from overflow
    int64_t off = 0, total = 0;
    for (int k = 0; k < n_tensors; ++k) {
        if (numel[k] < 0 || numel[k] > limit)
            return ZERO_EINVAL;
        off = zs::round_up(off, align_elems);
        if (tensor_offset_out)
            tensor_offset_out[k] = off;
        off += numel[k];
        total += numel[k];
        if (off > limit)
            return ZERO_EINVAL;
    }
    zero_layout L;
    std::memset(&L, 0, sizeof L);
    L.numel = total;
    L.flat_numel = off;
    L.world = world;
    L.align_elems = align_elems;
    L.bucket_numel = bucket_numel;
    const int64_t unit = (int64_t)world * align_elems;
    if (bucket_numel == 0) {
        L.padded_numel = zs::round_up(off, unit);
        L.owned_numel = L.padded_numel / world;
        L.num_buckets = L.padded_numel ? 1 : 0;
        L.slice_numel = L.last_slice_numel = L.owned_numel;
    } else {
        L.slice_numel = bucket_numel / world;
        if (off > 0) {
            L.num_buckets = (off + bucket_numel - 1) / bucket_numel;
            const int64_t last = off - (L.num_buckets - 1) * bucket_numel;
            const int64_t last_pad = zs::round_up(last, unit);
            L.padded_numel = (L.num_buckets - 1) * bucket_numel + last_pad;
            L.last_slice_numel = last_pad / world;
            L.owned_numel = (L.num_buckets - 1) * L.slice_numel + L.last_slice_numel;
        }
    }
    *out = L;
    return ZERO_OK;
}

int zero_state_init(zero_step_state *s, float loss_scale)
{
    if (!s || !(loss_scale > 0.0f) || !std::isfinite(loss_scale))
        return ZERO_EINVAL;
    int e;
    if (std::frexp(loss_scale, &e) != 0.5f)  // a power of two keeps 1/S exact
        return ZERO_EINVAL;
    std::memset(s, 0, sizeof *s);
    s->beta1_pow = 1.0;
    s->beta2_pow = 1.0;
    s->loss_scale = loss_scale;
    s->clip_coef = 1.0f;
    return ZERO_OK;
}

size_t zero_workspace_bytes(const zero_layout *layout)
{
    if (!layout)
        return zs::norm_ws_bytes_any_vector();
    if (zs::check_layout(layout))
        return 0;
    const zero_layout &L = *layout;
    const int64_t nb = L.bucket_numel ? L.num_buckets : (L.padded_numel ? 1 : 0);
    const int64_t su = (L.bucket_numel ? L.slice_numel : L.owned_numel) / zs::kUnit;
    const zs::NormGeom g = zs::norm_geometry(su, L.last_slice_numel / zs::kUnit, nb);
    const size_t need = zs::norm_ws_bytes(L.world, g);
    return need > (size_t)zs::kWsHeader ? need : (size_t)zs::kWsHeader;
}

int zero_host_alloc(size_t bytes, void **out)
{
    if (!out)
        return ZERO_EINVAL;
    *out = nullptr;
    if (bytes == 0)
        return ZERO_OK;
    // portable: page-locked for every device's context, not only the current one
    const cudaError_t e = cudaHostAlloc(out, bytes, cudaHostAllocPortable | cudaHostAllocMapped);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        *out = nullptr;
        return zs::cuda_error(e);
    }
    return ZERO_OK;
}

int zero_host_free(void *p)
{
    if (!p)
        return ZERO_OK;
    const cudaError_t e = cudaFreeHost(p);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return zs::cuda_error(e);
    }
    return ZERO_OK;
}

}  // extern "C"
