"""Small problems shared by the GPU tests of the norm's tree and of the
clipped step on bucket ranges (and by their child processes)."""
from synth.workloads import CFG1, CFG2, CFG5
import synth


def small_gpt2():
    d, vocab, ctx = 64, 1000, 128
    t = [vocab * d, ctx * d]
    for _ in range(2):
        t += [d, d, d * 3 * d, 3 * d, d * d, d, d, d, d * 4 * d, 4 * d, 4 * d * d, d]
    return tuple(t + [d, d])


def small_decoder():
    d, ffn, vocab, kv = 64, 224, 1000, 16
    t = [vocab * d]
    for _ in range(2):
        t += [d, d * d, kv * d, kv * d, d * d, d, ffn * d, ffn * d, d * ffn]
    return tuple(t + [d, vocab * d])


# (workload, Lockstep keyword arguments)
NORM_CASES = {
    "gpt2-nd8-bf16-staged": (CFG2.replace(numels=small_gpt2(), steps=2), dict(stage=True)),
    "decoder-nd8-buckets-recompute": (CFG5.replace(numels=small_decoder(), bucket=8 * 8 * 1000,
                                                   steps=2), dict(stage=False)),
    "decoder-rank5-view": (CFG5.replace(numels=small_decoder(), bucket=8 * 8 * 1000, steps=2,
                                        rank=5), {}),
    "flat-nd16-fp16-clip": (CFG1.replace(numels=(3_000_001,), world=16, max_grad_norm=0.05,
                                         steps=2, inject_at=()), {}),
}

# Clipped workloads for the bucket-range passes: (workload, stage), each with
# at least three buckets; step 2 gets +Inf in bucket 2.
RANGE_CASES = {
    "decoder-nd8-bf16-staged": (CFG5.replace(numels=small_decoder(), bucket=8 * 8 * 1000,
                                             steps=3), True),
    "decoder-nd8-bf16-recompute": (CFG5.replace(numels=small_decoder(), bucket=8 * 8 * 1000,
                                                steps=3), False),
    "nd3-fp16-dynamic": (CFG1.replace(world=3, bucket=3 * 8 * 4096, max_grad_norm=0.5,
                                      dynamic_scale=True, steps=3), False),
    "nd4-rank1-slices": (CFG1.replace(world=4, bucket=4 * 8 * 8192, rank=1,
                                      grads_are_slices=True, max_grad_norm=0.2, steps=3), False),
    "nd8-bf16-halfreduce": (CFG2.replace(numels=(300_000, 77, 1000), bucket=8 * 8 * 2048,
                                         half_reduce=True, steps=3), True),
    "nd2-unbucketed": (CFG1.replace(numels=(1_000_003,), max_grad_norm=0.3, steps=3), True),
}
