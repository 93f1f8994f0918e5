// Internal declarations shared by the translation units of libzerostep.
#pragma once

#include <cstdint>

#include <vector_types.h>

#include "zerostep.h"

namespace zs {

constexpr int kThreads = 256;      // threads per CTA of the streaming kernels
constexpr int kUnit = 8;           // elements per thread-unit: 16 bytes of half, 32 of fp32
constexpr int kMaxCtas = 4096;     // upper bound on CTAs of one streaming grid
constexpr int kWsHeader = 256;     // bytes at the start of the workspace (norm counters, result)

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

inline int cuda_error(int err) { return ZERO_ECUDA_BASE - err; }

// Checks shared by the entry points; each returns ZERO_OK or an error code.
int check_layout(const zero_layout *lay);
int check_cfg(const zero_adam_cfg *cfg);

// The optimizer configuration as the kernels use it: the values the step
// needs in binary64 (lr and the betas, for the bias corrections; the clip
// threshold), and the values that depend on the configuration alone, formed
// on the host in binary64 and rounded once to binary32 (the library's host
// code is compiled without floating-point contraction).
struct CfgDev {
    double lr, beta1, beta2, max_norm;
    float b1, omb1, b2, omb2, eps, decay, wd, lr_f;  // beta1, 1 - beta1, ..., 1 - lr wd, wd, lr
    int32_t adamw, bias_correction;
};
CfgDev make_cfg_dev(const zero_adam_cfg &c);

// ------------------------------------------------------------------ the norm's summation tree
//
// The global sum of squares is formed over a tree whose shape depends only on
// the layout (never on the device or the grid), so every launch shape, every
// split of the buckets into ranges and every GPU give the same bits:
//   chunk      kNormChunkMinUnits .. units of one rank's slice of one bucket
//              (chunks restart at every slice boundary), summed by one CTA:
//              thread t takes units t, t + 256, ...; each warp adds its
//              lanes with a fixed butterfly, then the 8 warps' pairs are
//              added in warp order and the pair rounded to binary64;
//   superchunk kNormSuper consecutive chunks of one rank, in a fixed lane
//              order;
//   rank       its superchunks in a fixed lane order;
//   total      the ranks' sums added in ascending rank order from +0.
// The first pass stores the chunk sums only (no synchronisation between
// CTAs); the tree kernel (launch_norm_tree) forms the rest.  One rank's view forms its
// own rank sum only; an every-rank launch gives exactly the rank-order sum of
// the per-rank results.
constexpr int64_t kNormChunkMinUnits = 512;      // 4096 elements
constexpr int64_t kNormChunksPerRank = 32768;    // target upper bound per rank
constexpr int kNormSuper = 64;                   // chunks per superchunk

// Chunk geometry of one rank's elements.
struct NormGeom {
    int64_t cu;        // units per chunk (a multiple of 256, at least kNormChunkMinUnits)
    int64_t cps;       // chunks in the slice of a full bucket
    int64_t cps_last;  // chunks in the slice of the last bucket (the whole partition if unbucketed)
    int64_t cpr;       // chunks per rank
    int64_t spr;       // superchunks per rank
};

// slice_units / last_slice_units: units of a rank's slice of a full bucket and
// of the last bucket; nb buckets (1 when not bucketed: the partition is the
// "last" slice).
NormGeom norm_geometry(int64_t slice_units, int64_t last_slice_units, int64_t nb);
// Workspace bytes of the tree for `ranks` ranks of that geometry.
size_t norm_ws_bytes(int64_t ranks, const NormGeom &g);

// What a launch needs to put its chunks into the tree.
struct NormPlan {
    int64_t cu, cps, cps_last, cpr, spr;
    int64_t slice_units, last_slice_units;  // of the whole layout
    int64_t nb;             // buckets of the whole layout
    int64_t b0, nbl;        // the launch covers buckets b0 .. b0 + nbl - 1
    int64_t launch_chunks;  // chunks the launch computes
    int32_t ranks;          // ranks whose sums are formed (world, or 1 for one rank's view)
    int32_t pad_;
    uint32_t *done;         // the tree kernel's finished CTAs (zero between launches)
    double *partials;       // chunk sums
    double *sc_partials;    // superchunk sums
    double *total;          // where the total goes
};

// The plan of a launch over buckets [b0, b0 + nbl) of nb (slices of
// slice_units / last_slice_units units), forming the sums of `ranks` ranks,
// with the tree in workspace `ws`; the total goes to `total`, or to the
// workspace's result slot when `total` is null.  Only the counter at the
// start of the workspace must be zero when a tree kernel starts (it returns
// it to zero); every other slot is written before it is read.
NormPlan norm_plan(const NormGeom &g, int64_t slice_units, int64_t last_slice_units, int64_t nb,
                   int64_t b0, int64_t nbl, int32_t ranks, void *ws, double *total);
// Bytes zero_grad_norm needs for a vector of any length (one rank, one slice:
// at most kNormChunksPerRank chunks, as the chunk grows with the vector).
constexpr size_t kNormWsAnyVector = kWsHeader + kNormChunksPerRank * 8 +
                                    (kNormChunksPerRank / kNormSuper) * 8;
inline size_t norm_ws_bytes_any_vector() { return kNormWsAnyVector; }
// The workspace's result slot (written by the tree kernel).
inline double *norm_total_slot(void *ws)
{
    return reinterpret_cast<double *>(static_cast<char *>(ws) + 8);
}
// The tree kernel: chunks -> superchunks -> ranks -> total (aux.cu).
int launch_norm_tree(const NormPlan &np, struct CUstream_st *stream);

}  // namespace zs

namespace zs {

// Launch the device-side end of a step (aux.cu).
int launch_finalize(const zero_adam_cfg *cfg, zero_step_state *state, int flip,
                    struct CUstream_st *stream);
// CTAs for one streaming kernel: SM count x resident CTAs per SM, capped (and
// capped further by test_grid_cap()).
int target_ctas(const void *kernel);
// SM count of the current device (cached per device).
int device_sms();
// 0, or the grid cap a test sets with ZERO_TEST_MAX_CTAS (read once per
// process): results must not depend on it.
int test_grid_cap();

}  // namespace zs
