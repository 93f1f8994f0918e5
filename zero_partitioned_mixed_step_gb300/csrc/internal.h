// Internal declarations shared by the translation units of libzerostep.
#pragma once

#include <cstdint>

#include "zerostep.h"

namespace zs {

constexpr int kThreads = 256;      // threads per CTA of the streaming kernels
constexpr int kUnit = 8;           // elements per thread-unit: 16 bytes of half, 32 of fp32
constexpr int kMaxCtas = 4096;     // upper bound on CTAs of one reduction grid
constexpr int kWsHeader = 256;     // bytes at the start of the workspace (unused header)

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

inline int cuda_error(int err) { return ZERO_ECUDA_BASE - err; }

// Checks shared by the entry points; each returns ZERO_OK or an error code.
int check_layout(const zero_layout *lay);
int check_cfg(const zero_adam_cfg *cfg);

}  // namespace zs

namespace zs {

// Launch the device-side end of a step (aux.cu).
int launch_finalize(const zero_adam_cfg *cfg, zero_step_state *state, int flip,
                    struct CUstream_st *stream);
// Reduce per-CTA partial sums of squares (gy rows of gx) in a fixed order:
// per rank (row), then ranks in ascending order.  Writes *out_sumsq when not
// null and, when state is not null and no overflow was found, state->sumsq and
// state->clip_coef (max_norm > 0).
int launch_norm_finalize(const double *partials, int gx, int gy, double max_norm,
                         zero_step_state *state, double *out_sumsq, struct CUstream_st *stream);
// CTAs for one streaming kernel: SM count x resident CTAs per SM, capped.
int target_ctas(const void *kernel);

}  // namespace zs
