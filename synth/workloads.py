"""The five synthetic workloads of the step, as input recipes.

Each recipe gives the tensor list, the simulated data-parallel group, the
gradient distribution, the optimizer hyper-parameters, the number of steps
and where NaN/Inf is injected.  Inputs are seeded: the master weights are
N(0, 0.02) (stream 10000 of the workload seed), the gradients of rank q at
step s are N(0, grad_sigma) times the loss scale (stream q of seed
``seed * 10**6 + s``), both drawn with the counter-based generator of this
package.  Gradient elements are indexed by their flat position, so a rank's
slice of a buffer equals the same range of the full buffer.

The tensor lists are architecture shapes only (no weights are loaded):
GPT-2 small with a tied output head (124,439,808 parameters) and an 8B
decoder with grouped-query attention and an untied head (8,030,261,248).
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Tuple

from . import F16, BF16, key


def gpt2_small_numels() -> Tuple[int, ...]:
    d, vocab, ctx, layers = 768, 50257, 1024, 12
    t = [vocab * d, ctx * d]
    for _ in range(layers):
        t += [d, d,                      # ln_1 weight, bias
              d * 3 * d, 3 * d,          # attention qkv weight, bias
              d * d, d,                  # attention output projection
              d, d,                      # ln_2
              d * 4 * d, 4 * d,          # mlp up
              4 * d * d, d]              # mlp down
    t += [d, d]                          # final layer norm
    return tuple(t)


def decoder_8b_numels() -> Tuple[int, ...]:
    d, ffn, vocab, layers, kv = 4096, 14336, 128256, 32, 1024
    t = [vocab * d]                      # token embedding
    for _ in range(layers):
        t += [d,                         # attention norm
              d * d, kv * d, kv * d,     # q, k, v projections
              d * d,                     # output projection
              d,                         # ffn norm
              ffn * d, ffn * d, d * ffn]  # gate, up, down
    t += [d, vocab * d]                  # final norm, untied lm head
    return tuple(t)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    numels: Tuple[int, ...]
    world: int
    dtype: int
    grad_sigma: float
    loss_scale: float
    dynamic_scale: bool
    lr: float
    beta1: float
    beta2: float
    eps: float
    weight_decay: float
    adamw: bool
    max_grad_norm: float
    steps: int
    seed: int
    bucket: int = 0
    rank: Optional[int] = None           # None: all ranks simulated at once
    grads_are_slices: bool = False       # gradient buffers hold only `rank`'s elements
    master_sigma: float = 0.02
    align: int = 64
    inject_every: int = 0                # inject +Inf at steps that are multiples of this
    inject_at: Tuple[Tuple[int, int, int], ...] = ()   # (step, rank, flat index)
    micro_steps: int = 1                 # gradient-accumulation micro-steps per step
    half_reduce: bool = False            # reduce in the gradients' half type, not fp32
    offload_state: bool = False          # master/m/v in pinned host memory
    per_bucket: bool = False             # one launch per bucket (per pass) on two streams, then the commit

    @property
    def numel(self) -> int:
        return sum(self.numels)

    def grad_seed(self, step: int) -> int:
        return self.seed * 1_000_000 + step

    def master_key(self) -> int:
        return key(self.seed, 10_000)

    def grad_key(self, step: int, q: int, micro: int = 0) -> int:
        """Rank q's gradient at a step (1-based) and micro-step (0-based)."""
        return key(self.grad_seed(step), q + 1024 * micro)

    def injections(self, step: int) -> Tuple[Tuple[int, int], ...]:
        """(rank, flat index) pairs that receive +Inf before ``step`` (1-based)."""
        out = [(r, i) for s, r, i in self.inject_at if s == step]
        if self.inject_every and step % self.inject_every == 0:
            r = step % self.world
            i = key(self.seed, 777_000 + step) % self.numel
            out.append((r, i))
        return tuple(out)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


ADAMW = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, adamw=True)

# 1M flat parameters, 2 ranks, fp16, static loss scale 1024, AdamW, 3 steps,
# +Inf at rank 0 element 500,000 in step 2 (the step is skipped).
CFG1 = Workload("flat-1M-nd2-fp16", (1_000_000,), 2, F16, 1e-3, 1024.0, False,
                max_grad_norm=0.0, steps=3, seed=1001, inject_at=((2, 0, 500_000),), **ADAMW)

# GPT-2 small tensor list (128-byte aligned tensors), 8 ranks, bf16, no loss
# scale, AdamW, global-norm clip 1.0, 10 steps.
CFG2 = Workload("gpt2-small-124M-nd8-bf16-clip", gpt2_small_numels(), 8, BF16, 1e-3, 1.0, False,
                max_grad_norm=1.0, steps=10, seed=1002, **ADAMW)

# 1.5B flat, 16 ranks, fp16 scaled by 2^12, dynamic loss scale, Adam without
# weight decay, 100 steps, +Inf every 50th step.
CFG3 = Workload("flat-1.5B-nd16-fp16-dynamic", (1_500_000_000,), 16, F16, 1e-3, 4096.0, True,
                lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, adamw=False,
                max_grad_norm=0.0, steps=100, seed=1003, inject_every=50)

# 7.5B flat, 64 ranks, ZeRO-2 view of rank 0 alone: 64 fp16 buffers holding
# only rank 0's slice, static loss scale 1024, AdamW, 20 steps.
CFG4 = Workload("7.5B-shard-nd64-rank0-fp16", (7_500_000_000,), 64, F16, 1e-3, 1024.0, False,
                max_grad_norm=0.0, steps=20, seed=1004, rank=0, grads_are_slices=True, **ADAMW)

# 8B decoder tensor list, 8 ranks, bf16, 25M-element buckets, AdamW,
# global-norm clip 1.0 across buckets, 10 steps.
CFG5 = Workload("8B-decoder-nd8-bf16-bucket25M-clip", decoder_8b_numels(), 8, BF16, 1e-3, 1.0,
                False, max_grad_norm=1.0, steps=10, seed=1005, bucket=25_000_000, **ADAMW)

ALL = (CFG1, CFG2, CFG3, CFG4, CFG5)

# A smaller case of the 1.5B workload for detailed profiles: 64M elements
# with the same 16 ranks; one launch still streams ~3.7 GB (far above L2)
# while the buffers hold ~4 GB of device memory.
PROFILE_CFG3 = CFG3.replace(name="flat-64M-nd16-fp16-dynamic", numels=(64_000_000,))

# Gradient accumulation (four micro-steps of reduce-scatter into an fp32
# accumulator per optimizer step) on the 1.5B, 16-rank workload.
ACCUM_CFG3 = CFG3.replace(name="flat-1.5B-nd16-fp16-accum4", micro_steps=4, steps=20,
                          inject_every=0)

# The 1.5B, 16-rank workload with the reduction in fp16 (each partial sum
# rounded to fp16), as a half-precision reduce-scatter would produce it.
HALFRED_CFG3 = CFG3.replace(name="flat-1.5B-nd16-fp16-halfreduce", half_reduce=True)

# ZeRO-Offload style: the 1.5B, 16-rank workload with the fp32 master weights
# and moments in Grace memory, reached by the GPU over NVLink-C2C.
OFFLOAD_CFG3 = CFG3.replace(name="flat-1.5B-nd16-fp16-offload", offload_state=True, steps=10,
                            inject_every=0)

# A smaller case of the 7.5B rank-0 shard for detailed profiles: a 600M flat
# vector over the same 64 ranks gives rank 0 9.375M elements (one launch
# streams 1.44 GB, far above L2; ~4 GB on the device, most of it the two
# slots of the full half-precision parameter vector).
PROFILE_CFG4 = CFG4.replace(name="600M-shard-nd64-rank0-fp16", numels=(600_000_000,))

# The 1.5B, 16-rank workload cut into 60 buckets of 25,000,064 elements (the
# multiple of 16 x 8 nearest 25M): as one launch, and as one launch per
# bucket alternating between two streams with one commit at the end (the
# optimizer step whose finished buckets an all-gather can take while later
# buckets update).
BUCKET_CFG3 = CFG3.replace(name="flat-1.5B-nd16-fp16-bucket25M", bucket=25_000_064)
PERBUCKET_CFG3 = BUCKET_CFG3.replace(name="flat-1.5B-nd16-fp16-bucket25M-perbucket",
                                     per_bucket=True)

# The 8B clipped workload run bucket by bucket: the first pass on each of the
# 322 buckets (one launch each, alternating between two streams), then the
# second pass on each bucket in the same way, then the commit; bucket 0's
# parameters are final once its second pass ends.
PERBUCKET_CFG5 = CFG5.replace(name="8B-decoder-nd8-bf16-bucket25M-clip-perbucket",
                              per_bucket=True)

BY_NAME = {w.name: w for w in ALL + (PROFILE_CFG3, PROFILE_CFG4, ACCUM_CFG3, HALFRED_CFG3,
                                     OFFLOAD_CFG3, BUCKET_CFG3, PERBUCKET_CFG3,
                                     PERBUCKET_CFG5)}
