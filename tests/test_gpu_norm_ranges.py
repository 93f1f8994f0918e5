"""The global sum of squares over the norm's fixed tree, and the clipped step
run as bucket ranges, through the C ABI.

The tree's shape depends on the layout only (chunks of each rank's bucket
slices, superchunks, ranks in ascending order), so:
  * the bits do not depend on the grid (a child process caps every grid at
    7 CTAs and gets the same bits and buffers);
  * an every-rank step's sum is the rank-order sum of the per-rank views'
    sums, as an all-reduce of per-rank sums in rank order would give it,
    and zero_grad_norm of a rank's reduced gradient is that rank's sum;
  * splitting the clipped step into bucket ranges on two streams (pass 1 on
    every range, the norm, pass 2 on every range, the commit) gives the
    fused step's bits, including a step skipped for an Inf in a middle
    bucket ("DeepSpeed ZeRO", ZeRO Stage 1: overlap of the optimizer step
    with the all-gather, over the constant-size buffers of "相关分析")."""
import json
import os
import struct
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import zero_partitioned_mixed_step_gb300 as zs
from gpu_norm_cases import NORM_CASES, RANGE_CASES
from zs_harness import (INF_BITS, SUMSQ_RTOL, Lockstep, gen_grads, rank_index, state_proper,
                        to_dev_half)

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _child(name, **env):
    e = dict(os.environ)
    e.pop("ZERO_TEST_MAX_CTAS", None)
    e.pop("ZERO_TEST_STAGED_WAIT_LIMIT", None)
    e.update(env)
    r = subprocess.run([sys.executable, os.path.join(HERE, "gpu_children.py"), name],
                       capture_output=True, text=True, env=e, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_norm_bits_do_not_depend_on_the_grid():
    """Every streaming grid capped at 7 CTAs (instead of SMs x resident CTAs)
    gives the same sums of squares, buffers and zero_grad_norm bits."""
    full = _child("norm_bits")
    small = _child("norm_bits", ZERO_TEST_MAX_CTAS="7")
    assert small.pop("cap") == "7" and full.pop("cap") is None
    assert small == full


def _bits(x: float) -> str:
    return struct.pack("<d", x).hex()


@pytest.mark.parametrize("name", ["gpt2-nd8-bf16-staged", "decoder-nd8-buckets-recompute",
                                  "flat-nd16-fp16-clip"])
def test_every_rank_sum_is_the_rank_order_sum_of_rank_views(name):
    wl, kw = NORM_CASES[name]
    full = Lockstep(wl, **kw)
    views = [Lockstep(wl.replace(rank=r), **kw) for r in range(wl.world)]
    for s in (1, 2):
        grads = gen_grads(wl, full.lay, s, full.st.loss_scale)
        full.step(grads)
        for ls in views:
            ls.step(grads)
        st = full.check()
        total = 0.0
        sums = []
        for ls in views:
            sums.append(ls.check().sumsq)
            total = total + sums[-1]
        assert _bits(st.sumsq) == _bits(total), (s, st.sumsq, total)
        assert abs(st.sumsq - full.st.sumsq) <= SUMSQ_RTOL * full.st.sumsq
    if wl.bucket == 0:
        # zero_grad_norm of rank r's reduced gradient (unscaled) is rank r's sum
        gd = [to_dev_half(g, wl.dtype) for g in grads]
        zl, _ = zs.zero_partition_layout(wl.numels, wl.world, wl.align)
        ws = zs.new_workspace()
        for r, ls in enumerate(views):
            g = torch.empty(zl.owned_numel, dtype=torch.float32, device="cuda")
            zs.zero_reduce_scatter_sum(gd, zl, g, rank=r)
            out = torch.zeros(1, dtype=torch.float64, device="cuda")
            zs.zero_grad_norm(g, oracle.f32(1.0 / ls.st.loss_scale), out.data_ptr(), ws)
            assert _bits(float(out.item())) == _bits(sums[r]), r


def _ranges(nb):
    if nb < 3:
        return [(0, nb)]
    return [(0, 1), (1, nb // 2 - 1), (nb // 2, nb - nb // 2)] if nb >= 4 else \
        [(0, 1), (1, 1), (2, nb - 2)]


@pytest.mark.parametrize("where", ["device", "host"], ids=["grads-on-device", "grads-in-host"])
@pytest.mark.parametrize("name", list(RANGE_CASES))
def test_clipped_bucket_ranges_equal_fused_step(name, where):
    """The ranges may also load the gradients straight from page-locked host
    memory (the first pass, and the second pass when it reduces again)."""
    base, stage = RANGE_CASES[name]
    lay = oracle.layout(base.numels, base.world, base.align, base.bucket)
    nb = lay.num_buckets if base.bucket else 1
    r = 0 if base.rank is None else base.rank
    if base.bucket:
        inf_at = 2 * base.bucket + r * lay.slice + 5  # in bucket 2, rank r's slice
    else:
        inf_at = r * lay.owned + lay.owned // 2
    wl = base.replace(inject_at=((2, 0, inf_at),))
    ref, alt = Lockstep(wl, stage=stage), Lockstep(wl, stage=stage)
    ranges = [(f, n) for f, n in _ranges(nb) if n > 0]
    assert sum(n for _, n in ranges) == nb
    s0 = torch.cuda.current_stream()
    side = [torch.cuda.Stream(), torch.cuda.Stream()]

    def fork():
        ev = torch.cuda.Event()
        ev.record(s0)
        for st in side:
            st.wait_event(ev)

    def join():
        for st in side:
            ev = torch.cuda.Event()
            ev.record(st)
            s0.wait_event(ev)

    for s in range(1, wl.steps + 1):
        grads = gen_grads(wl, ref.lay, s, ref.st.loss_scale)
        ref.step(grads)
        gd = [to_dev_half(g, wl.dtype) for g in grads]
        if where == "host":
            gd = [zs.host_empty(g.numel(), g.dtype).copy_(g.cpu()) for g in gd]
        fork()
        for i, (f, n) in enumerate(ranges):
            alt.z.pass1_buckets(gd, f, n, side[i % 2])
        join()
        alt.z.norm_buckets(s0)
        fork()
        for i, (f, n) in enumerate(reversed(ranges)):
            alt.z.pass2_buckets(gd, f, n, side[i % 2])
        join()
        alt.z.commit(s0)
        torch.cuda.synchronize()
        a, b = ref.z.read_state(), alt.z.read_state()
        assert state_proper(a) == state_proper(b), s
        assert b.overflow == (1 if s == 2 else 0) and b.error == 0
        for x, y in zip(ref.z.current(), alt.z.current()):
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), s
        ref.check()
    assert ref.st.skipped == 1 and ref.st.t == wl.steps - 1
    assert ref.st.coef < 1.0  # the clip was active


def test_one_norm_workspace_serves_any_sequence_of_lengths():
    """zero_grad_norm with one workspace over vectors of growing and
    shrinking length (their trees have different numbers of chunks) gives
    each vector the bits a fresh workspace gives it."""
    import synth
    ws = zs.new_workspace()
    for n in (37, 300_000_001, 1000, 6_000_005, 300_000_001, 8):
        g = torch.empty(n, dtype=torch.float32, device="cuda")
        synth.gpu_fill_f32(synth.key(5, n), 0, g, 1e-2)
        a = torch.zeros(1, dtype=torch.float64, device="cuda")
        b = torch.zeros(1, dtype=torch.float64, device="cuda")
        zs.zero_grad_norm(g, 1.0, a.data_ptr(), ws)
        zs.zero_grad_norm(g, 1.0, b.data_ptr(), zs.new_workspace())
        assert _bits(float(a.item())) == _bits(float(b.item())), n
        del g
        torch.cuda.empty_cache()


def test_one_step_workspace_serves_every_view():
    """The clipped step's workspace shared by an every-rank group and a
    one-rank group of the same layout, alternating steps: each gets the bits
    it gets with a workspace of its own."""
    wl, kw = NORM_CASES["decoder-nd8-buckets-recompute"]
    view = wl.replace(rank=3)
    shared_all, shared_one = Lockstep(wl, **kw), Lockstep(view, **kw)
    own_all, own_one = Lockstep(wl, **kw), Lockstep(view, **kw)
    shared_one.z.ws = shared_all.z.ws
    for s in (1, 2, 3):
        grads = gen_grads(wl, own_all.lay, s, own_all.st.loss_scale)
        for ls in (shared_all, shared_one, own_all, own_one):
            ls.step(grads)
        torch.cuda.synchronize()
        for a, b in ((shared_all, own_all), (shared_one, own_one)):
            assert state_proper(a.z.read_state()) == state_proper(b.z.read_state()), s
            for x, y in zip(a.z.current(), b.z.current()):
                assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), s
    own_all.check()
    own_one.check()
