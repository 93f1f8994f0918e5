"""The benchmark's host-side bookkeeping on the CPU: the algorithmic bytes a
step is credited with, the launch count it claims, the kernel it names, and
the source hash that keeps a recorded ncu traffic figure tied to the code it
was measured on."""
import bench
from synth.workloads import BY_NAME, CFG1, CFG2, CFG3, CFG4, CFG5


def test_algorithmic_bytes_per_element():
    """Read N_d half gradients, read and write fp32 master, m and v, write the
    half parameter: 2 N_d + 26 bytes.  A clipped step adds the fp32 stage
    written and read back (8) or the gradients read again (2 N_d)."""
    for world in (1, 2, 8, 16, 64, 1024):
        assert bench.algorithmic_bytes_per_elem(world, False, False) == 2 * world + 26
        assert bench.algorithmic_bytes_per_elem(world, True, True) == 2 * world + 26 + 8
        assert bench.algorithmic_bytes_per_elem(world, True, False) == 4 * world + 26
    # the workloads' figures quoted in the design notes
    assert bench.algorithmic_bytes_per_elem(16, False, False) == 58
    assert bench.algorithmic_bytes_per_elem(64, False, False) == 154
    assert bench.algorithmic_bytes_per_elem(8, True, True) == 50


def test_algorithmic_bytes_with_accumulation():
    """K micro-steps: each reads the N_d gradients and writes the fp32
    accumulator, all but the first also read it; then the step reads the
    accumulator (twice with the clip) and moves the state and parameters."""
    for world in (2, 16):
        for k in (2, 4):
            per_micro = 2 * world + 4
            reads_acc = 4 * (k - 1)
            step = 4 + 24 + 2
            assert bench.algorithmic_bytes_per_elem(world, False, False, k) == \
                k * per_micro + reads_acc + step
            assert bench.algorithmic_bytes_per_elem(world, True, False, k) == \
                k * per_micro + reads_acc + step + 4


def test_dominant_kernel_follows_the_library_rule():
    """The shared-memory staged kernel carries every-rank one-pass steps at
    16 ranks with the fp32 reduction and device state; everything else runs
    the register kernel."""
    assert bench.dominant_kernel(CFG3).startswith("staged_fused_kernel")
    assert bench.dominant_kernel(CFG1).startswith("step_kernel")
    assert bench.dominant_kernel(CFG4).startswith("step_kernel")
    assert "two passes" in bench.dominant_kernel(CFG2)
    assert "two passes" in bench.dominant_kernel(CFG5)
    assert bench.dominant_kernel(BY_NAME["flat-1.5B-nd16-fp16-halfreduce"]).startswith(
        "step_kernel")
    assert bench.dominant_kernel(BY_NAME["flat-1.5B-nd16-fp16-offload"]).startswith(
        "step_kernel")


def test_source_hash_ignores_comments_only():
    """Editing comments or whitespace keeps the hash; editing code changes it."""
    import os
    csrc = os.path.join(bench.ROOT, "zero_partitioned_mixed_step_gb300", "csrc")
    src = {}
    for name in bench.STEP_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            src[name] = f.read()
    base = bench.kernel_source_hash(read=lambda n: src[n])
    assert base == bench.kernel_source_hash()
    commented = dict(src)
    commented["step.cu"] = (b"// a new comment line\n/* and a block\n comment */\n" +
                            src["step.cu"].replace(b"\n", b"  \n", 3))
    assert bench.kernel_source_hash(read=lambda n: commented[n]) == base
    changed = dict(src)
    changed["kernels.cuh"] = src["kernels.cuh"].replace(b"evict_first", b"evict_last", 1)
    assert bench.kernel_source_hash(read=lambda n: changed[n]) != base


def test_recorded_traffic_is_tied_to_the_code():
    """The committed traffic figure is returned only for a workload recorded
    at the current code's hash."""
    assert bench.recorded_traffic("no-such-workload") is None
    t = bench.recorded_traffic(CFG3.name)
    if t is not None:  # recorded at this code: about the algorithmic bytes
        alg = 1_500_000_256 * 58
        assert 0.95 * alg < t < 1.02 * alg
