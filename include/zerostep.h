/*
 * zerostep.h — C ABI of the partitioned mixed-precision ZeRO Adam step on one
 * GB300 GPU (sm_103a).
 *
 * The operation (the data-parallel hot path of ZeRO stages 1-3):
 *   N_d data-parallel ranks each hold a half-precision (fp16 or bf16)
 *   gradient of the whole flat parameter vector.  Rank r owns a 1/N_d
 *   partition of that vector.  One step
 *     (a2) reduce-scatters the gradients: rank r's fp32 gradient is the
 *          element-wise sum over all ranks of their gradients on r's
 *          partition;
 *     (a3) multiplies it by 1/S (S = the loss scale, a power of two);
 *     (a4) skips the whole step if any element of any partition is NaN/Inf,
 *          leaving every buffer bit-for-bit unchanged (only a dynamic loss
 *          scale is lowered);
 *     (a5) optionally scales the gradient by min(1, max_norm / (||g||_2 + 1e-6)),
 *          the norm taken over all partitions;
 *     (a6) applies Adam or AdamW to the partition's fp32 master weights,
 *          momentum and variance;
 *     (a7) rounds the new master weights to half precision (nearest, ties to
 *          even) and writes them at the partition's place in the flat
 *          half-precision parameter buffer, i.e. the layout an all-gather of
 *          all partitions produces;
 *     (a8) commits the step (t <- t + 1) or records the skip.
 *   Sources — five web pages on DeepSpeed ZeRO:
 *     "DeepSpeed ZeRO" (formulaic.cloudchewie.com): "ZeRO Stage 1: 切分优化器状态"
 *       ("权重更新的触发条件": skip on NaN/Inf and in-place fp32 -> fp16 copy;
 *       "以 AdaW 为例": the m, v, W update; "具体训练步骤": local update of the
 *       1/N_d slice, cast, all-gather), "ZeRO Stage 2: 切分梯度" (reduce-scatter;
 *       fp32 gradient slice made from the reduce-scattered half gradient;
 *       per-element independence of the update), "ZeRO Stage 3: 切分参数"
 *       ("参数的初始化和切割": flatten, pad, [start, end) per rank), "相关分析"
 *       ("Constant Size Buffer": fixed-size buckets), "配置说明" (loss scale);
 *     "zero-optimizer" (codezrq.github.io), 2.5 ReduceScatter and 2.6 AllGather;
 *       "一. 优化前" (gradient-norm computation in fused buffers);
 *     "ZeRO 技术原理：基础与实现" (jianzhnie.github.io), 3.1.1 ZeRO-1 and
 *       3.3.1 "初始化——模型参数的分割" (per-rank [start, end) of a flat tensor);
 *     "千亿参数模型如何塞进有限显卡：ZeRO如何用分片消除数据并行的内存冗余"
 *       (answer.freetools.me), "Stage 2：梯度分片" (Reduce-Scatter to the owner).
 *   Where the pages are silent the library takes these readings: the reduction
 *   is a sum in fp32, in ascending rank order from +0, with no rounding to
 *   half in between; Adam is bias-corrected (Kingma and Ba) unless
 *   bias_correction = 0; AdamW decay is decoupled, W <- W (1 - lr wd), applied
 *   before the update; the overflow test is on the reduced unscaled gradient.
 *
 * Simulation on one GPU: the N_d ranks' gradient buffers all live in this
 * GPU's memory.  A call either processes every rank's partition at once
 * (rank = -1) or one rank's partition (rank = r).
 *
 * Conventions for every entry point:
 *  - The caller allocates and owns every buffer.  The library allocates no
 *    memory except the blocks zero_host_alloc hands to the caller.  Between
 *    calls it keeps only read-only device properties (SM counts, resident CTAs
 *    per kernel, cached on first use) and the one static array that
 *    zero_grad_norm_noalloc documents.  Pointers named *_dev or documented as
 *    device pointers must be CUDA device pointers of the current device; all
 *    others are host pointers read during the call only.
 *  - Device work is enqueued on `stream` (NULL = the legacy default stream)
 *    and runs asynchronously; nothing synchronises the host.  Calls that use
 *    the same workspace or state must be ordered (one stream, or events),
 *    except the bucket-range calls of one step, which may run concurrently
 *    as their descriptions say.
 *  - Arguments are validated on the host before anything is enqueued; on an
 *    error nothing is enqueued.  Return values: ZERO_OK (0) or a negative
 *    code below.  A value <= ZERO_ECUDA_BASE is ZERO_ECUDA_BASE - cudaError_t
 *    of a failed launch.  Kernels never trap: numerical overflow is reported
 *    through zero_step_state, not as an error.
 *  - fp32 vector buffers (master, m, v, gradients in fp32, stages) must be
 *    32-byte aligned and half-precision buffers 16-byte aligned (ZERO_EALIGN
 *    otherwise): the kernels move 8 elements per access.
 */
#ifndef ZEROSTEP_H
#define ZEROSTEP_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__) || defined(__clang__)
/* The library is built with hidden visibility: only the entry points below
 * are exported, so two copies loaded in one process keep their own state. */
#define ZERO_API __attribute__((visibility("default")))
#else
#define ZERO_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *zero_stream_t; /* the same type as cudaStream_t */

enum {
    ZERO_OK = 0,
    ZERO_EINVAL = -1,        /* null pointer, bad size, world, rank, dtype, config or layout */
    ZERO_EALIGN = -2,        /* a buffer is not aligned (32 bytes fp32, 16 bytes half) */
    ZERO_ESPACE = -3,        /* workspace smaller than zero_workspace_bytes() */
    ZERO_ECUDA_BASE = -1000  /* ZERO_ECUDA_BASE - cudaError_t */
};

#define ZERO_MAX_WORLD 1024

/* Gradient / parameter precision.  With ZERO_F16 or ZERO_BF16 the gradients
 * are reduced in fp32.  The _HALF_REDUCE codes keep the same storage type but
 * reduce in it: every partial sum over ranks is rounded to nearest even in
 * the half type, in ascending rank order, as a half-precision reduce-scatter
 * produces it ("DeepSpeed ZeRO", ZeRO Stage 2: the fp32 gradient slice is
 * made from the reduce-scattered BF16 gradient); a partial sum beyond the
 * type's range becomes +-Inf and skips the step. */
typedef enum {
    ZERO_F16 = 0,
    ZERO_BF16 = 1,
    ZERO_F16_HALF_REDUCE = 2,
    ZERO_BF16_HALF_REDUCE = 3
} zero_dtype;

/*
 * Partition layout of the flat parameter vector (step a1).
 * Tensor k starts at offset_k = round_up(offset_{k-1} + numel_{k-1}, align).
 * Not bucketed (bucket_numel = 0): the vector is padded to a multiple of
 * world * align and rank r owns [r * owned, (r + 1) * owned).
 * Bucketed: the vector is cut into buckets of bucket_numel elements (the last
 * one padded to a multiple of world * align); rank r owns slice r of every
 * bucket, so its elements are, in order, bucket 0 slice r, bucket 1 slice r, ...
 * Padding elements must be zero in every gradient, master and moment buffer
 * (they then stay zero).
 */
typedef struct {
    int64_t numel;            /* sum of tensor sizes (unpadded) */
    int64_t flat_numel;       /* end of the last tensor, alignment gaps included */
    int64_t padded_numel;     /* length of the padded flat vector */
    int64_t owned_numel;      /* elements each rank owns */
    int64_t bucket_numel;     /* 0: one contiguous partition per rank */
    int64_t num_buckets;      /* 1 when not bucketed (0 for an empty vector) */
    int64_t slice_numel;      /* a rank's slice of a full bucket (= owned_numel if not bucketed) */
    int64_t last_slice_numel; /* a rank's slice of the last bucket (= owned_numel if not bucketed) */
    int32_t world;            /* N_d, 1 .. ZERO_MAX_WORLD */
    int32_t align_elems;      /* tensor alignment in elements, a multiple of 8 */
} zero_layout;

/* Optimizer configuration.  Field names follow DeepSpeed's JSON config
 * ("DeepSpeed ZeRO", "配置说明": lr, betas, eps, weight_decay; fp16.loss_scale
 * = 0 selects the dynamic loss scale). */
typedef struct {
    double lr;
    double beta1, beta2;
    double eps;
    double weight_decay;
    int32_t adamw;           /* 1: decoupled decay (AdamW); 0: coupled L2 term added to g */
    int32_t bias_correction; /* 1: Kingma-Ba bias correction; 0: the pages' formula as printed */
    double max_grad_norm;    /* > 0: clip by the global L2 norm (two passes); 0: no clipping */
    int32_t dynamic_scale;   /* 1: S <- max(S * backoff, min_scale) on overflow and
                                S <- S * growth after growth_interval good steps in a row */
    int32_t growth_interval;
    double backoff, growth, min_scale;
} zero_adam_cfg;

/*
 * Step state, DEVICE-resident (192 bytes, 8-byte aligned), owned by the
 * caller.  Initialise a host copy with zero_state_init and copy it to the
 * device.  The kernels read it at the start of a step and zero_step_finalize
 * (or the last kernel of zero_step_fused / zero_step_fused_accumulated)
 * updates it at the end.  The first 64 bytes are the step's state proper;
 * scalar_cache is the library's own (below).
 */
typedef struct {
    int64_t t;          /* committed (not skipped) steps */
    double beta1_pow;   /* beta1^t as a running product in binary64 */
    double beta2_pow;   /* beta2^t as a running product in binary64 */
    double sumsq;       /* global sum of squares of the unscaled gradient (last clip step) */
    float loss_scale;   /* S, a power of two */
    float clip_coef;    /* clip coefficient of the last clipped step */
    int32_t good_steps; /* good steps since the last overflow or growth */
    int32_t overflow;   /* 1 if the last step was skipped */
    int32_t found_inf;  /* bit 0: OR of the non-finite flags of the step in progress;
                           while the last kernel of a fused step runs, the bits above
                           count its finished CTAs (the last one ends the step); 0
                           between steps */
    int32_t cur;        /* ping-pong slot (0/1) holding the current master/m/v/params */
    int32_t skipped;    /* number of skipped steps */
    int32_t error;      /* nonzero if a kernel gave up waiting for its own memory copies
                           (never expected; that step was skipped); 0 at init */
    /* Library-internal: the bias-correction scalars of the next step
       (lr / (1 - beta1^t) and sqrt(1 - beta2^t), each rounded to binary32),
       formed by one thread of the step before, off the step's critical path,
       so that the next step's CTAs need no binary64 division or square root.
       The one-pass kernels of small steps over at most 4 ranks and the
       N_d = 16 staged kernel form them; other kernels leave the cache as it
       is.  Two entries, one per ping-pong slot; each records every input of
       its values (lr, beta1, beta2, beta1_pow, beta2_pow) and is used only
       when all of them are bit for bit the step's own, otherwise the step
       forms the scalars itself: a changed learning rate or betas, a restored
       state or a skipped step never see stale values.  zero_state_init
       zero-fills it; keep it as the library left it (copying the whole
       struct is fine). */
    uint64_t scalar_cache[16];
} zero_step_state;

/* Human-readable text for a return code (static storage). */
ZERO_API const char *zero_strerror(int code);

/* ABI version: 3 (2: zero_workspace_bytes takes the layout, the clipped
 * step's bucket-range passes; 3: zero_step_state carries the scalar cache and
 * is 192 bytes). */
ZERO_API int zero_version(void);

/*
 * Step (a1): the partition layout.  Host-only, pure.
 *  numel[n_tensors]: tensor sizes (>= 0).  world: N_d in 1 .. ZERO_MAX_WORLD.
 *  align_elems: tensor alignment in elements, a positive multiple of 8
 *  (64 gives 128-byte aligned fp16/bf16 tensors).  bucket_numel: 0 or a
 *  positive multiple of world * 8.  tensor_offset_out[n_tensors] (may be NULL)
 *  receives each tensor's flat offset.
 * Pages: "DeepSpeed ZeRO", "ZeRO Stage 3", "参数的初始化和切割" (flatten, pad so
 * the length divides by the data-parallel size, [start, end) per rank);
 * "ZeRO 技术原理", 3.3.1 (partition_size per rank, start = partition_size *
 * rank; the floor division there is read as padding so no element is lost);
 * "DeepSpeed ZeRO", "Constant Size Buffer" (buckets).
 */
ZERO_API int zero_partition_layout(int n_tensors, const int64_t *numel, int world,
                                   int align_elems, int64_t bucket_numel,
                                   int64_t *tensor_offset_out, zero_layout *out);

/* Fill *host_state with the state before the first step: t = 0, beta powers
 * 1, loss_scale (a positive power of two), clip_coef 1, everything else 0. */
ZERO_API int zero_state_init(zero_step_state *host_state, float loss_scale);

/*
 * Bytes of device workspace a step on `layout` needs (zero_step_fused,
 * zero_step_fused_accumulated, zero_step_buckets_pass1 / _pass2), or, with
 * layout = NULL, the bytes zero_grad_norm needs for a vector of any length
 * (266,496).  0 for an invalid layout.
 * The workspace holds the tree over which the global sum of squares is
 * formed: chunks of at least 4096 elements of one rank's slice of one bucket
 * (about 32768 chunks per rank for large partitions), 64 chunks to a
 * superchunk, then ranks.  It takes about 8 bytes per chunk (2.1 MB for 8
 * billion parameters over 8 ranks).  Its shape depends
 * only on the layout, so the sum's bits do not depend on the GPU, the grid,
 * or how the buckets are split into ranges.  ZERO-FILL THE WORKSPACE ONCE
 * before its first use: it holds one counter, which every call that runs to
 * completion returns to zero.
 */
ZERO_API size_t zero_workspace_bytes(const zero_layout *layout);

/*
 * Page-locked host memory for the buffers a step exchanges with the host:
 * gradients that the caller copies in before a step, or the fp32 master
 * weights and moments kept in CPU memory as in ZeRO-Offload ("千亿参数模型如何
 * 塞进有限显卡…", "ZeRO-Offload：利用CPU内存").  The memory is mapped into the
 * device's address space, so a kernel may also read or write it directly
 * (zero_step_fused does so for offloaded state).  The calls give C callers
 * that have no framework allocator the same blocks a framework's pinned
 * allocator would give.
 *  zero_host_alloc: *out = a new block of `bytes` bytes (at least 256-byte
 *    aligned, contents undefined); bytes = 0 gives *out = NULL and ZERO_OK.
 *    ZERO_EINVAL if out is NULL; a failed allocation returns
 *    ZERO_ECUDA_BASE - cudaError_t with *out = NULL.
 *  zero_host_free: releases a block from zero_host_alloc (NULL is a no-op).
 *    It synchronises with the device like cudaFreeHost: no copy or kernel
 *    may still use the block.  The caller owns each block until it frees it.
 * The pages have no counterpart for this call; it is the runtime's memory
 * management for the host side of the step.
 */
ZERO_API int zero_host_alloc(size_t bytes, void **out);
ZERO_API int zero_host_free(void *p);

/*
 * Step (a2): reduce-scatter sum, g[j] = sum over q = 0 .. world-1 of
 * float(grads[q][.]) in ascending q, fp32, not unscaled.
 *  grads: HOST array of `world` pointers, one gradient buffer per rank: device
 *    memory, or page-locked host memory mapped into the device's address
 *    space (zero_host_alloc, cudaHostAlloc, cudaHostRegister), which the
 *    kernels then load directly over the host link (no copy into device
 *    memory; on GB300 the loads of 16 such buffers ran at 210 GB/s, the
 *    link's rate, where copy engines gave 94-155 GB/s).
 *  grads_are_slices: 0 = each buffer is the full padded flat vector;
 *    1 = each buffer holds only the elements `rank` owns, in order (needs rank >= 0).
 *  rank = -1: every partition; g_out (device, padded_numel floats) is in flat
 *    order.  rank = r: r's partition; g_out (owned_numel floats) in r's order.
 * Pages: "zero-optimizer", 2.5 ReduceScatter; "DeepSpeed ZeRO", ZeRO Stage 2.
 */
ZERO_API int zero_reduce_scatter_sum(const void *const *grads, int grads_are_slices,
                                     zero_dtype dtype, const zero_layout *layout, int rank,
                                     float *g_out, zero_stream_t stream);

/*
 * Step (a4): *flag_dev |= 1 if any g[j] * inv_scale (j < n) is NaN or +-Inf;
 * otherwise *flag_dev is left as it is (clear it before the first call; pass
 * &state->found_inf to feed zero_adam_step).  g: device, n floats, 16-byte
 * aligned.
 * Pages: "DeepSpeed ZeRO", ZeRO Stage 1, "权重更新的触发条件".
 */
ZERO_API int zero_check_overflow(const float *g, int64_t n, float inv_scale, int32_t *flag_dev,
                                 zero_stream_t stream);

/*
 * Step (a5): *sumsq_dev = sum over j < n of (g[j] * inv_scale)^2.  The
 * squares are formed exactly and summed in pairs of binary32 values (about
 * 48 significant bits) within chunks, then in binary64 over a fixed tree
 * (see zero_workspace_bytes): the order depends on n only, so every GPU and
 * every call give the same bits, and for g a rank's reduced gradient of an
 * unbucketed layout the result is that rank's sum in the fused step's tree.
 * Relative error about 1e-13 or better.  g: device, 32-byte aligned;
 * sumsq_dev: device double; ws: device workspace of ws_bytes >=
 * zero_workspace_bytes(NULL), zero-filled before its first use (the call
 * leaves its counter at zero).  Two launches: the chunk sums, then the tree (a
 * memset for n = 0: *sumsq_dev = +0).
 * Pages: "zero-optimizer", "一. 优化前" (gradient-norm computation over fused
 * buffers); the clip rule itself is a reading (see zero_adam_cfg).
 */
ZERO_API int zero_grad_norm(const float *g, int64_t n, float inv_scale, double *sumsq_dev, void *ws,
                            size_t ws_bytes, zero_stream_t stream);

/*
 * Gradient accumulation, one micro-step: the reduce-scatter sum of the N_d
 * half-precision gradients (as zero_reduce_scatter_sum: fp32, ascending rank
 * order from +0, not unscaled) added to an fp32 accumulator:
 *   acc[j] = (add ? acc[j] : 0) + sum_q float(grads[q][.])
 * (the micro-step's sum over ranks is formed first, then added once).
 *  grads, grads_are_slices, dtype, layout, rank: as zero_reduce_scatter_sum.
 *  acc: device fp32, padded_numel (rank = -1, flat order) or owned_numel
 *  (rank = r, r's order), 32-byte aligned.  add = 0 starts a new accumulation.
 * Pages: "DeepSpeed ZeRO", "ZeRO-2 在梯度累积场景下的通信量" (ZeRO-2 reduce-scatters
 * after every backward and accumulates its 1/N_d slice) and the page's memory
 * section (the optional fp32 gradient copy for accumulating in fp32).
 */
ZERO_API int zero_reduce_scatter_accumulate(const void *const *grads, int grads_are_slices,
                                            zero_dtype dtype, const zero_layout *layout, int rank,
                                            float *acc, int add, zero_stream_t stream);

/*
 * The whole step (a3)-(a8) with the gradient taken from an fp32 accumulator
 * (after micro-steps of zero_reduce_scatter_accumulate) instead of the N_d
 * half-precision buffers: unscale, overflow test (NaN/Inf in any micro-step
 * skips the step), optional clip, Adam/AdamW, cast, commit.  dtype is the
 * parameter buffer's type; acc, layout and rank as in
 * zero_reduce_scatter_accumulate; master, m, v, params, cfg, state_dev, ws as
 * zero_step_fused (one pass with distinct ping-pong slots without clipping;
 * two passes over acc, slots may alias, with clipping).
 * Pages: as zero_step_fused and zero_reduce_scatter_accumulate.
 */
ZERO_API int zero_step_fused_accumulated(const float *acc, zero_dtype dtype,
                                         const zero_layout *layout, int rank,
                                         float *const master[2], float *const m[2],
                                         float *const v[2], void *const params[2],
                                         const zero_adam_cfg *cfg, zero_step_state *state_dev,
                                         void *ws, size_t ws_bytes, zero_stream_t stream);

/*
 * zero_grad_norm for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is an interface variant, not a step of the method.
 * Some callers have no way to provide the workspace zero_grad_norm needs:
 * plain-C plugins that are handed device pointers by a host framework but
 * have no allocator of their own, code inside a framework whose caching
 * allocator already owns the device memory (a direct cudaMalloc can fail
 * there although the framework has free memory), and loops that cannot
 * afford the device-wide synchronisation cudaMalloc and cudaFree can cause.
 * This entry point allocates nothing and calls no allocating routine.
 *  Result, arguments and summation order: as zero_grad_norm (the same kernel
 *  and the same tree, so the same bits), without ws / ws_bytes.
 *  Scratch: the tree lives in a library-owned static device array of
 *  ZERO_NOALLOC_SCRATCH_BYTES (266,496 bytes: the tree of a vector of any
 *  length) that every GPU which loads the library holds until the process
 *  exits.  A vector whose tree would not fit is rejected with ZERO_ESPACE
 *  (none is: the chunks grow with the vector).  The array's one counter is
 *  zero when the library is loaded and every call returns it to zero; the
 *  other slots are written before they are read.  All calls share the array, so
 *  calls that can overlap on the GPU (different streams, or different host
 *  threads, without ordering between them) race and must not be issued.
 *  Set-up: the first call on each device looks up the array's device
 *  address for the current device (cudaGetSymbolAddress) and caches it; make
 *  that first call before any stream capture.
 */
#define ZERO_NOALLOC_SCRATCH_BYTES 266496
ZERO_API int zero_grad_norm_noalloc(const float *g, int64_t n, float inv_scale, double *sumsq_dev,
                                    zero_stream_t stream);

/*
 * Steps (a3), (a5 clip), (a6), (a7) on n elements in place, for the reduced
 * gradient g that zero_reduce_scatter_sum produced (not yet unscaled).
 * Reads from state_dev: loss_scale, t and the beta powers (the update is step
 * t + 1), found_inf (if set the call changes nothing) and, when
 * cfg->max_grad_norm > 0, sumsq (from zero_grad_norm) for the clip.
 * master, m, v: device fp32 (n); half_out: device fp16/bf16 (n) receiving
 * round-to-nearest-even of the new master weights.  Call zero_step_finalize
 * afterwards to commit the step.
 * Pages: "DeepSpeed ZeRO", ZeRO Stage 1, "以 AdaW 为例" and "权重更新的触发条件".
 */
ZERO_API int zero_adam_step(const float *g, float *master, float *m, float *v, void *half_out,
                            zero_dtype dtype, int64_t n, const zero_adam_cfg *cfg,
                            const zero_step_state *state_dev, zero_stream_t stream);

/*
 * Step (a8): end a step.  If state_dev->found_inf: overflow = 1, skipped += 1,
 * and with a dynamic scale S <- max(S * backoff, min_scale), good_steps = 0.
 * Otherwise: overflow = 0, t += 1, beta powers advance, good_steps += 1 (and
 * S <- S * growth after growth_interval of them), and if flip_slot the
 * ping-pong slot cur is toggled.  found_inf is cleared either way.
 * Pages: "DeepSpeed ZeRO", ZeRO Stage 1, "权重更新的触发条件"; "配置说明".
 */
ZERO_API int zero_step_finalize(const zero_adam_cfg *cfg, zero_step_state *state_dev, int flip_slot,
                                zero_stream_t stream);

/*
 * The whole step (a2)-(a8), fused.
 *  grads, grads_are_slices, dtype, layout, rank: as zero_reduce_scatter_sum.
 *  master[2], m[2], v[2]: HOST arrays of two DEVICE pointers each (ping-pong
 *    slots) to fp32 buffers of padded_numel (rank = -1, flat order) or
 *    owned_numel (rank = r, r's order) elements.
 *  params[2]: HOST array of two DEVICE pointers to the flat half-precision
 *    parameter buffer (padded_numel elements, all-gather layout); the step
 *    writes the elements of the partitions it processes.
 *  The step reads slot state->cur and writes slot 1 - cur, then toggles cur
 *  when the step commits; a skipped step writes only the unused slot, so the
 *  current slot stays bit-for-bit unchanged.
 *  Without clipping (cfg->max_grad_norm == 0) the step is ONE pass over the
 *  data: the slots must be distinct buffers.  With clipping it is two passes
 *  (norm, then update); the two slots may then be the same buffer (in place).
 *  g_stage: NULL, or (clip only) a device fp32 buffer with the length of
 *    master that keeps the reduced gradient between the passes instead of
 *    reducing it twice (2 * N_d bytes read per element are replaced by 8).
 *    It is scratch: its contents after the call are undefined (the second
 *    pass drops the lines it no longer needs from L2 without writing back
 *    any that are still dirty).
 *  state_dev: device step state.  ws: device workspace of ws_bytes >=
 *    zero_workspace_bytes(layout), zero-filled before its first use (the
 *    clipped step's first pass forms the global sum of squares over the
 *    workspace's fixed tree, rank by rank, then the ranks in ascending order).
 * Offload: master, m and v (all six slots) may instead be
 *  pinned host memory (cudaHostAlloc / cudaHostRegister) that the GPU reads
 *  and writes over the host link while gradients and parameters stay in
 *  device memory, as in ZeRO-Offload, where the optimizer state lives in CPU
 *  memory ("千亿参数模型如何塞进有限显卡…", "ZeRO-Offload：利用CPU内存"; "DeepSpeed
 *  ZeRO", "配置说明": offload_optimizer.device = cpu).  The residence is
 *  detected per call (cudaPointerGetAttributes); mixed residence, or
 *  offloaded state together with the clip, is ZERO_EINVAL.
 * CUDA graphs: the call synchronises nothing and ends the step on the device,
 *  so it can be captured on a stream and replayed (gradients refreshed in the
 *  same buffers); do one step of the same kind outside any capture first,
 *  which fills the library's per-kernel caches.
 * Pages: all of the above; the ping-pong slots are this library's way to
 * skip a step bit-exactly without a second pass over the gradients.
 */
ZERO_API int zero_step_fused(const void *const *grads, int grads_are_slices, zero_dtype dtype,
                             const zero_layout *layout, int rank, float *const master[2],
                             float *const m[2], float *const v[2], void *const params[2],
                             float *g_stage, const zero_adam_cfg *cfg,
                             zero_step_state *state_dev, void *ws, size_t ws_bytes,
                             zero_stream_t stream);

/*
 * The one-pass step (a2)-(a7) on buckets [first_bucket, first_bucket +
 * n_buckets) of a layout, WITHOUT the commit (a8).  Call it once per range,
 * so that every bucket of the layout is covered exactly once per step.  The
 * ranges may go to different streams and run concurrently, since they touch
 * disjoint elements.  After all of them, call zero_step_finalize(cfg,
 * state_dev, 1, stream) on a stream ordered after every range.  The result
 * is then bit for bit the zero_step_fused result.
 * A range's half-precision parameters are final as soon as that range's work
 * completes, so a caller can start that bucket's all-gather while later
 * buckets are still being updated.  A NaN/Inf found in any range makes the
 * commit skip the whole step, as the unused ping-pong slot is the only one
 * written.  This is DeepSpeed's overlap of the optimizer step with the
 * parameter all-gather ("DeepSpeed ZeRO", ZeRO Stage 1, 通信与计算重叠: start
 * the all-gather of each updated part while the rest is still updating) over
 * its constant-size buffers ("相关分析", Constant Size Buffer).
 *  Arguments as zero_step_fused, except:
 *  first_bucket, n_buckets: 0 <= first_bucket, first_bucket + n_buckets <=
 *    layout->num_buckets (a layout without buckets has one bucket, the whole
 *    vector).  n_buckets = 0 enqueues nothing.
 *  There is no g_stage and no workspace: a clipped step needs the global norm
 *    before any update, so cfg->max_grad_norm > 0 is ZERO_EINVAL.
 * Every bucket must be processed before the commit, and none twice: after the
 * commit, a bucket left out would hold the slot's older contents.  That is
 * the caller's contract; the library does not track it.
 */
ZERO_API int zero_step_fused_buckets(const void *const *grads, int grads_are_slices,
                                     zero_dtype dtype, const zero_layout *layout, int rank,
                                     int64_t first_bucket, int64_t n_buckets,
                                     float *const master[2], float *const m[2],
                                     float *const v[2], void *const params[2],
                                     const zero_adam_cfg *cfg, zero_step_state *state_dev,
                                     zero_stream_t stream);

/*
 * The CLIPPED step (cfg->max_grad_norm > 0) on ranges of buckets, in two
 * passes with one global norm between them:
 *   1. zero_step_buckets_pass1 on every bucket of the layout, exactly once,
 *      in ranges [first_bucket, first_bucket + n_buckets): (a2) reduce, (a3)
 *      unscale, (a4) flag NaN/Inf in state_dev->found_inf, (a5) the squares'
 *      chunk sums into the workspace's fixed tree, and, with g_stage, keep the
 *      unscaled gradient there.  A range can run as soon as its buckets'
 *      gradients are ready (during the backward pass), and ranges may run
 *      concurrently on different streams.
 *   2. zero_step_buckets_norm once, on a stream ordered after EVERY pass-1
 *      range: the tree above the chunk sums in its fixed order
 *      (superchunks, each rank, then the ranks in ascending order) gives the
 *      global sum of squares, kept in the workspace.
 *   3. zero_step_buckets_pass2 on every bucket, exactly once, in ranges, each
 *      on a stream ordered after step 2: (a5) the clip with c = min(1,
 *      max_norm / (sqrt(total) + 1e-6)), (a6) Adam/AdamW, (a7) the cast; a
 *      range's parameters are final (ready for its all-gather) as soon as the
 *      range completes.  Skipped (nothing written) when pass 1 flagged
 *      NaN/Inf.  The ranges may run concurrently.
 *   4. zero_step_finalize(cfg, state_dev, 1, stream) after every pass-2 range:
 *      commits (t + 1, cur toggled) or skips the step.
 * The result is bit for bit that of zero_step_fused with the clip on the
 * same buffers, whatever the split into ranges, and state_dev->sumsq /
 * clip_coef are set as zero_step_fused sets them.  This is DeepSpeed's
 * overlap of the optimizer step with the parameter all-gather ("DeepSpeed
 * ZeRO", ZeRO Stage 1, 通信与计算重叠) over constant-size buffers
 * ("相关分析", Constant Size Buffer), with the gradient norm of the page
 * "zero-optimizer" ("一. 优化前") taken over all buckets before any update.
 *  Arguments as zero_step_fused_buckets, plus:
 *  g_stage: NULL, or a device fp32 buffer with the length of master (the
 *    whole layout's, not the range's): pass 1 writes the range's unscaled
 *    gradient there and pass 2 reads it.  Pass 2 takes exactly one source:
 *    grads (reduced again) or g_stage.
 *  ws, ws_bytes: the step's workspace (zero_workspace_bytes(layout),
 *    zero-filled before first use), the same for every call of the step.
 *  master/m/v/params (pass 2): ping-pong slots as zero_step_fused; they may
 *    alias (in place), and must be device memory.
 * Every bucket must go through each pass exactly once per step; a bucket left
 * out of pass 1 leaves stale chunk sums in the tree.
 */
ZERO_API int zero_step_buckets_pass1(const void *const *grads, int grads_are_slices,
                                     zero_dtype dtype, const zero_layout *layout, int rank,
                                     int64_t first_bucket, int64_t n_buckets, float *g_stage,
                                     const zero_adam_cfg *cfg, zero_step_state *state_dev,
                                     void *ws, size_t ws_bytes, zero_stream_t stream);
ZERO_API int zero_step_buckets_norm(const zero_layout *layout, int rank, void *ws,
                                    size_t ws_bytes, zero_stream_t stream);
ZERO_API int zero_step_buckets_pass2(const void *const *grads, int grads_are_slices,
                                     zero_dtype dtype, const zero_layout *layout, int rank,
                                     int64_t first_bucket, int64_t n_buckets,
                                     float *const master[2], float *const m[2],
                                     float *const v[2], void *const params[2],
                                     const float *g_stage, const zero_adam_cfg *cfg,
                                     zero_step_state *state_dev, const void *ws,
                                     size_t ws_bytes, zero_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ZEROSTEP_H */
