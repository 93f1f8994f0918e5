"""The CUDA step (through the C ABI) against the CPU oracle, element by
element, on the same seeded inputs, step after step.

Sizes are small enough for the oracle to finish in seconds but span many
CTAs, several ranks and ragged tails; every workload's structure (tensor
list, alignment, buckets, rank view, dtype, loss scaling, clipping,
overflow injection) is exercised.  Full-size workloads are in
test_gpu_fullsize.py."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.workloads import CFG1, CFG2, CFG3, CFG4, CFG5, decoder_8b_numels, gpt2_small_numels
import zero_partitioned_mixed_step_gb300 as zs
from zs_harness import (SUMSQ_RTOL, Lockstep, assert_close, gen_grads, half_bits, lib_cfg,
                        oracle_cfg, rank_index, state_proper, to_dev_half)

pytestmark = pytest.mark.gpu


def _small_gpt2():
    d, vocab, ctx = 64, 1000, 128
    t = [vocab * d, ctx * d]
    for _ in range(2):
        t += [d, d, d * 3 * d, 3 * d, d * d, d, d, d, d * 4 * d, 4 * d, 4 * d * d, d]
    return tuple(t + [d, d])


def _small_decoder():
    d, ffn, vocab, kv = 64, 224, 1000, 16
    t = [vocab * d]
    for _ in range(2):
        t += [d, d * d, kv * d, kv * d, d * d, d, ffn * d, ffn * d, d * ffn]
    return tuple(t + [d, vocab * d])


SMALL = {
    # the whole first workload: 1M parameters, 2 ranks, Inf in step 2
    "cfg1": CFG1,
    # GPT-2-shaped list, 8 ranks, bf16, clip 1.0
    "cfg2-small": CFG2.replace(numels=_small_gpt2(), steps=4),
    # flat ragged vector, 16 ranks, fp16 x 2^12, dynamic scale, Inf every 2nd step
    "cfg3-small": CFG3.replace(numels=(3_000_001,), steps=5, inject_every=2),
    # rank 0 of 64, gradient buffers hold rank 0's slice only
    "cfg4-small": CFG4.replace(numels=(64 * 50_000 + 13,), steps=3,
                               inject_at=((2, 5, 1234),)),
    # 8B-shaped list in buckets, 8 ranks, bf16, clip across buckets
    "cfg5-small": CFG5.replace(numels=_small_decoder(), bucket=8 * 8 * 1000, steps=3),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_workload_lockstep(name):
    wl = SMALL[name]
    ls = Lockstep(wl)
    for _ in range(wl.steps):
        ls.step()
        ls.check()
    assert ls.st.t + ls.st.skipped == wl.steps


@pytest.mark.parametrize("stage", [True, False])
def test_clip_staged_and_recomputed_agree(stage):
    """The two-pass clipped step gives the same bits whether the reduced
    gradient is kept in fp32 between the passes or reduced again."""
    wl = SMALL["cfg2-small"].replace(steps=2)
    ls = Lockstep(wl, stage=stage)
    for _ in range(2):
        ls.step()
        ls.check()


@pytest.mark.parametrize("offset_floats", [0, 8], ids=["stage-128B-aligned", "stage-32B-off"])
@pytest.mark.parametrize("numels,world", [((8 * 1001 + 3,), 1), ((3 * 8 * 777 + 5,), 3)],
                         ids=["one-rank", "three-ranks"])
def test_clip_stage_alignment_and_ragged_units(numels, world, offset_floats):
    """The clipped step's second pass drops the kept stage lines from L2 only
    when the stage is 128-byte aligned, and only whole 128-byte lines inside
    the buffer.  A stage 32 bytes off a 128-byte boundary (no line is
    dropped) and vectors whose count of 8-element units is not a multiple of
    4 (8-element tensor alignment: the last line is partial) give the
    oracle's results all the same, step after step."""
    wl = CFG2.replace(numels=numels, world=world, align=8, max_grad_norm=0.01, steps=3)
    ls = Lockstep(wl, stage=True)
    n = ls.z.g_stage.numel()
    assert (n // 8) % 4 != 0  # a partial last line
    buf = torch.empty(n + 32, dtype=torch.float32, device="cuda")
    ls.z.g_stage = buf[offset_floats:offset_floats + n]
    assert (ls.z.g_stage.data_ptr() % 128 == 0) == (offset_floats == 0)
    for _ in range(wl.steps):
        ls.step()
        st = ls.check()
        assert st.clip_coef < 1.0  # the clip is active


EDGE = {
    "one-rank": CFG1.replace(numels=(70_001,), world=1, steps=2, inject_at=()),
    "three-ranks-generic": CFG1.replace(numels=(100_003, 17), world=3, steps=3,
                                        inject_at=((2, 1, 50_000),)),
    "hundred-ranks": CFG1.replace(numels=(100 * 640 + 8,), world=100, steps=2, inject_at=()),
    # the largest group the ABI accepts; the Inf is in the last rank's gradient, at the
    # vector's last element (owned by rank 682)
    "max-world-1024": CFG1.replace(numels=(1024 * 128 + 8,), world=1024, steps=2,
                                   inject_at=((2, 1023, 1024 * 128 + 7),)),
    # zero gradients: the moments stay zero and only the decoupled decay moves w
    "zero-gradients": CFG1.replace(numels=(40_000,), world=4, grad_sigma=0.0, steps=2,
                                   inject_at=()),
    "psi-below-world": CFG1.replace(numels=(5,), world=8, steps=2, inject_at=()),
    "tiny-tensors-gaps": CFG2.replace(numels=(1, 2, 3, 65, 127, 4096, 7), world=4, steps=3),
    "bf16-dynamic": CFG3.replace(numels=(200_000,), world=8, dtype=synth.BF16, steps=4,
                                 inject_every=3),
    "bucketed-rank-view": CFG5.replace(numels=_small_decoder(), bucket=8 * 8 * 1000, steps=2,
                                       rank=5),
    "bucketed-rank-slices": CFG5.replace(numels=_small_decoder(), bucket=8 * 8 * 1000,
                                         steps=2, rank=3, grads_are_slices=True,
                                         max_grad_norm=0.0),
    "rank-view-full-buffers": CFG4.replace(numels=(16 * 4096 + 100,), world=16, rank=7,
                                           grads_are_slices=False, steps=2),
    "clip-never-active": CFG2.replace(numels=(50_000,), world=2, max_grad_norm=1e6, steps=2),
    # the norm's tree over the most ranks the ABI accepts (1024 rank sums added in order),
    # and over 100 ranks in buckets whose superchunks span several buckets
    "clip-world-1024": CFG2.replace(numels=(1024 * 512 + 8,), world=1024, steps=2,
                                    max_grad_norm=0.05),
    "clip-world-100-buckets": CFG2.replace(numels=(100 * 8 * 700 + 13, 999), world=100,
                                           bucket=100 * 8 * 64, steps=2, max_grad_norm=0.05),
}


@pytest.mark.parametrize("name", list(EDGE))
def test_edge_lockstep(name):
    wl = EDGE[name]
    ls = Lockstep(wl)
    for _ in range(wl.steps):
        ls.step()
        ls.check()


@pytest.mark.parametrize("kw", [dict(adamw=False, weight_decay=0.05),
                                dict(bias_correction=False),
                                dict(dynamic_scale=True, growth_interval=2)],
                         ids=["coupled-l2", "literal-adam", "scale-growth"])
def test_optimizer_variants(kw):
    wl = CFG1.replace(numels=(300_000,), steps=5, inject_at=((3, 1, 7),))
    ls = Lockstep(wl, **kw)
    for _ in range(wl.steps):
        ls.step()
        ls.check()


@pytest.mark.parametrize("bits,where", [(0x7C00, "first"), (0xFC00, "boundary"),
                                        (0x7E00, "last-real"), (0x7C01, "padding")])
def test_overflow_anywhere_skips_bit_exactly(bits, where):
    """NaN, +Inf or -Inf in any rank's buffer (first element, a partition
    boundary, the last real element, a padding element) skips the step: the
    current slot of every buffer is unchanged bit for bit."""
    wl = CFG1.replace(numels=(100_001,), world=4, steps=2, inject_at=(), dtype=synth.F16,
                      dynamic_scale=True)
    ls = Lockstep(wl)
    ls.step()
    ls.check()
    before = [t.clone() for t in ls.z.current()]
    g = gen_grads(wl, ls.lay, 2, ls.st.loss_scale)
    P = ls.lay.owned
    pos = {"first": (0, 0), "boundary": (2, 2 * P - 1), "last-real": (3, 100_000),
           "padding": (1, ls.lay.padded - 1)}[where]
    g[pos[0]][pos[1]] = bits
    ls.step(g)
    st = ls.check()
    assert st.overflow == 1 and st.t == 1 and st.loss_scale == wl.loss_scale / 2
    for a, b in zip(before, ls.z.current()):
        assert torch.equal(a.view(torch.uint8) if a.dtype != torch.float32 else a.view(torch.int32),
                           b.view(torch.uint8) if b.dtype != torch.float32 else b.view(torch.int32))


def test_empty_vector():
    cfg = zs.adam_cfg()
    z = zs.ZeroStep((), 4, synth.F16, cfg)
    assert z.layout.padded_numel == 0
    grads = [torch.empty(0, dtype=torch.float16, device="cuda") for _ in range(4)]
    z.step(grads)
    torch.cuda.synchronize()
    st = z.read_state()
    assert st.t == 1 and st.overflow == 0


def test_unfused_entry_points_match_oracle_and_fused():
    """reduce-scatter -> overflow check -> norm -> Adam -> finalize through the
    separate entry points: the reduced gradient is bit-exact, the norm within
    tolerance, and the result equals the fused step's."""
    wl = CFG2.replace(numels=(123_457, 999), world=8, steps=1)
    lay = oracle.layout(wl.numels, wl.world)
    zl, _ = zs.zero_partition_layout(wl.numels, wl.world)
    grads = gen_grads(wl, lay, 1, 1.0)
    gd = [to_dev_half(g, wl.dtype) for g in grads]
    dev = "cuda"
    # (a2) all ranks and one rank
    g_all = torch.empty(lay.padded, dtype=torch.float32, device=dev)
    zs.zero_reduce_scatter_sum(gd, zl, g_all)
    want = oracle.reduce_sum(grads, wl.dtype, 0, lay.padded)
    assert np.array_equal(g_all.cpu().numpy().view(np.uint32), want.view(np.uint32))
    g3 = torch.empty(lay.owned, dtype=torch.float32, device=dev)
    zs.zero_reduce_scatter_sum(gd, zl, g3, rank=3)
    assert np.array_equal(g3.cpu().numpy(), want[rank_index(lay, 3)])
    # (a4)
    state = zs.new_state(1.0)
    zs.zero_check_overflow(g_all, 1.0, zs.state_field_ptr(state, "found_inf"))
    assert zs.read_state(state).found_inf == 0
    bad = g_all.clone()
    bad[lay.padded - 1] = float("nan")
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    zs.zero_check_overflow(bad, 1.0, flag.data_ptr())
    assert int(flag.item()) == 1
    odd = g_all[:13].clone()
    odd[12] = float("-inf")
    flag.zero_()
    zs.zero_check_overflow(odd, 1.0, flag.data_ptr())
    assert int(flag.item()) == 1
    # (a5)
    ws = zs.new_workspace()
    zs.zero_grad_norm(g_all, 1.0, zs.state_field_ptr(state, "sumsq"), ws)
    s = zs.read_state(state).sumsq
    ref = oracle.sumsq_value(oracle.sumsq(want))
    assert abs(s - ref) <= SUMSQ_RTOL * ref
    for n in (0, 1, 7, 9, 1001):
        out = torch.zeros(1, dtype=torch.float64, device=dev)
        zs.zero_grad_norm(g_all[:n].clone(), 0.5, out.data_ptr(), ws)
        h = want[:n].copy()
        oracle.unscale(h, 0.5)
        r = oracle.sumsq_value(oracle.sumsq(h))
        assert abs(float(out.item()) - r) <= SUMSQ_RTOL * max(r, 1e-300)
    # (a6)-(a8) with the clip
    cfg = lib_cfg(wl)
    master = gen_master_flat(wl, lay)
    w = torch.from_numpy(master.copy()).to(dev)
    m = torch.zeros_like(w)
    v = torch.zeros_like(w)
    out = torch.empty(lay.padded, dtype=zs.torch_dtype(wl.dtype), device=dev)
    zs.zero_adam_step(g_all, w, m, v, out, cfg, state)
    zs.zero_step_finalize(cfg, state)
    torch.cuda.synchronize()
    ost = oracle.State()
    wo, mo, vo = master.copy(), np.zeros_like(master), np.zeros_like(master)
    ho = np.zeros(lay.padded, np.uint16)
    oracle.step(grads, wl.dtype, lay, oracle_cfg(wl), ost, wo, mo, vo, ho)
    assert_close("master", w.cpu().numpy(), wo)
    assert_close("m", m.cpu().numpy(), mo)
    assert_close("v", v.cpu().numpy(), vo)
    st = zs.read_state(state)
    assert st.t == 1 and st.cur == 0
    # the fused step gives the same bits when its clip coefficient (from a
    # per-rank norm) rounds to the same binary32 value
    ls = Lockstep(wl)
    ls.step(grads)
    fst = ls.check()
    fw, fm, fv, fp = ls.z.current()
    if fst.clip_coef == oracle.clip_coef(s, wl.max_grad_norm):
        assert torch.equal(fw.view(torch.int32), w.view(torch.int32))
        assert torch.equal(fv.view(torch.int32), v.view(torch.int32))
        assert np.array_equal(half_bits(fp), half_bits(out))


def gen_master_flat(wl, lay):
    from zs_harness import gen_master
    return gen_master(wl, lay)


def test_adam_step_skips_on_flag_and_tail():
    """zero_adam_step changes nothing when the state's flag is set, and
    handles a length that is not a multiple of 8."""
    n = 1003
    dev = "cuda"
    g = torch.randn(n, device=dev) * 1e-3
    w0 = torch.randn(n, device=dev) * 0.02
    w, m, v = w0.clone(), torch.zeros(n, device=dev), torch.zeros(n, device=dev)
    out = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    cfg = zs.adam_cfg(weight_decay=0.01)
    state = zs.new_state(1.0)
    off = zs.StepState.found_inf.offset
    state[off:off + 4].copy_(torch.ones(1, dtype=torch.int32, device=dev).view(torch.uint8))
    zs.zero_adam_step(g, w, m, v, out, cfg, state)
    torch.cuda.synchronize()
    assert torch.equal(w, w0) and not m.any() and not out.view(torch.int16).any()
    zs.zero_step_finalize(cfg, state)
    st = zs.read_state(state)
    assert st.overflow == 1 and st.t == 0 and st.found_inf == 0
    zs.zero_adam_step(g, w, m, v, out, cfg, state)
    torch.cuda.synchronize()
    sc = oracle.step_scalars(oracle.AdamCfg(weight_decay=0.01), oracle.State())
    wo, mo, vo = w0.cpu().numpy().copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    oracle.adam(g.cpu().numpy().copy(), wo, mo, vo, sc)
    assert_close("master", w.cpu().numpy(), wo)
    assert np.array_equal(half_bits(out), oracle.f32_to_half(wo, oracle.BF16))


def test_generators_agree():
    """The GPU input generator gives the CPU generator's bits."""
    dev = "cuda"
    for dtype in (synth.F16, synth.BF16):
        k = synth.key(1234, 5)
        n = 100_003
        cpu = synth.fill_half(k, 777, n, 4.1, dtype)
        gpu = torch.empty(n, dtype=torch.int16, device=dev)
        synth.gpu_fill_half(k, 777, gpu, 4.1, dtype)
        assert np.array_equal(gpu.cpu().numpy().view(np.uint16), cpu)
    k = synth.key(99, 10_000)
    cpu = synth.fill_f32(k, 0, 50_001, 0.02)
    gpu = torch.empty(50_001, dtype=torch.float32, device=dev)
    synth.gpu_fill_f32(k, 0, gpu, 0.02)
    assert np.array_equal(gpu.cpu().numpy().view(np.uint32), cpu.view(np.uint32))
    x = torch.randn(4099, device=dev) * 100
    for dtype in (synth.F16, synth.BF16):
        out = torch.empty(4099, dtype=torch.int16, device=dev)
        synth.gpu_round_half(x, out, dtype)
        assert np.array_equal(out.cpu().numpy().view(np.uint16),
                              synth.round_half(x.cpu().numpy(), dtype))


# ----------------------------------------------------------------- gradient accumulation

ACCUM = {
    "flat-nd16-4micro": CFG3.replace(numels=(1_000_003,), steps=3, micro_steps=4,
                                     inject_every=0, inject_at=((2, 3, 4321),)),
    "gpt2-nd8-clip-3micro": SMALL["cfg2-small"].replace(steps=2, micro_steps=3),
    "bucketed-rank-slices-2micro": EDGE["bucketed-rank-slices"].replace(micro_steps=2),
    "rank0-of-64-2micro": SMALL["cfg4-small"].replace(steps=2, micro_steps=2),
    "halfreduce-bf16-3micro": SMALL["cfg2-small"].replace(steps=2, micro_steps=3,
                                                          half_reduce=True),
}


@pytest.mark.parametrize("name", list(ACCUM))
def test_accumulation_lockstep(name):
    """K micro-steps of zero_reduce_scatter_accumulate, then
    zero_step_fused_accumulated, against the oracle, step after step; the
    injected +Inf (in one micro-step) skips that step."""
    from zs_harness import INF_BITS, gen_master, half_bits
    wl = ACCUM[name]
    ls = Lockstep(wl)
    for s in range(1, wl.steps + 1):
        S = ls.st.loss_scale
        n_acc = ls.lay.padded if wl.rank is None else ls.lay.owned
        acc = np.zeros(n_acc, np.float32)
        for k in range(wl.micro_steps):
            grads = gen_grads(wl, ls.lay, s, S)  # step s, then vary per micro-step
            if k:
                grads = _micro_grads(wl, ls.lay, s, k, S)
            ls.z.accumulate([to_dev_half(g, wl.dtype) for g in grads], add=k > 0)
            oracle.reduce_scatter_accumulate(grads, wl.dtype, ls.lay, acc, k > 0, rank=wl.rank,
                                             grads_are_slices=wl.grads_are_slices,
                                             half_reduce=wl.half_reduce)
        ls.z.step_accumulated()
        oracle.step_accumulated(acc, wl.dtype, ls.lay, ls.ocfg, ls.st, ls.w, ls.m, ls.v, ls.half,
                                rank=wl.rank)
        ls.steps += 1
        torch.cuda.synchronize()
        assert np.array_equal(ls.z.acc.cpu().numpy().view(np.uint32), acc.view(np.uint32))
        ls.check()
    if name == "flat-nd16-4micro":
        assert ls.st.skipped == 1


def _micro_grads(wl, lay, step, micro, loss_scale):
    from zs_harness import tensor_mask, rank_index
    mask = tensor_mask(lay)
    out = []
    for q in range(wl.world):
        g = synth.fill_half(wl.grad_key(step, q, micro), 0, lay.padded,
                            wl.grad_sigma * loss_scale, wl.dtype)
        g[~mask] = 0
        out.append(g)
    if wl.grads_are_slices:
        idx = rank_index(lay, wl.rank)
        out = [g[idx].copy() for g in out]
    return out


def test_one_micro_step_equals_the_fused_step():
    """Accumulating a single micro-step and stepping from it gives the fused
    step's bits."""
    wl = CFG1.replace(numels=(200_003,), world=4, steps=2, inject_at=())
    a, b = Lockstep(wl), Lockstep(wl)
    for s in range(1, 3):
        grads = gen_grads(wl, a.lay, s, a.st.loss_scale)
        a.step(grads)
        b.z.accumulate([to_dev_half(g, wl.dtype) for g in grads], add=False)
        b.z.step_accumulated()
    torch.cuda.synchronize()
    for x, y in zip(a.z.current(), b.z.current()):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


# ----------------------------------------------------------------- half-precision reduction

HALFRED = {
    "fp16-nd16-dynamic": SMALL["cfg3-small"].replace(half_reduce=True),
    "bf16-nd8-clip": SMALL["cfg2-small"].replace(half_reduce=True, steps=3),
    "fp16-rank0-of-64-slices": SMALL["cfg4-small"].replace(half_reduce=True),
    "bucketed-bf16-clip": SMALL["cfg5-small"].replace(half_reduce=True),
    "three-ranks": EDGE["three-ranks-generic"].replace(half_reduce=True),
}


@pytest.mark.parametrize("name", list(HALFRED))
def test_half_reduce_lockstep(name):
    """The reduction in the gradients' own half type (every partial sum
    rounded to nearest even) against the oracle, step after step."""
    wl = HALFRED[name]
    ls = Lockstep(wl)
    for _ in range(wl.steps):
        ls.step()
        ls.check()


def test_half_reduce_overflow_skips_where_fp32_does_not():
    """fp16 gradients near the top of the range: a partial sum overflows in
    fp16 (the step is skipped) although the fp32 reduction stays finite."""
    wl = CFG1.replace(numels=(50_000,), world=4, steps=1, inject_at=(), loss_scale=2.0 ** 24,
                      dynamic_scale=True)
    fp32, half = Lockstep(wl), Lockstep(wl.replace(half_reduce=True))
    fp32.step()
    half.step()
    a, b = fp32.check(), half.check()
    assert a.overflow == 0 and a.t == 1
    assert b.overflow == 1 and b.t == 0 and b.loss_scale == 2.0 ** 23


# ----------------------------------------------------------------- offloaded optimizer state

OFFLOAD = {
    "fp16-nd16-dynamic": SMALL["cfg3-small"].replace(offload_state=True),
    "bf16-rank0-of-64-slices": SMALL["cfg4-small"].replace(offload_state=True,
                                                           dtype=synth.BF16),
    "bucketed-rank-view": EDGE["bucketed-rank-slices"].replace(offload_state=True),
    "fp16-halfreduce": CFG1.replace(numels=(300_003,), world=8, offload_state=True,
                                    half_reduce=True, inject_at=((2, 7, 123),)),
}


@pytest.mark.parametrize("name", list(OFFLOAD))
def test_offloaded_state_lockstep(name):
    """The one-pass step with master, m and v in pinned host memory (read and
    written by the GPU over the host link) against the oracle."""
    wl = OFFLOAD[name]
    ls = Lockstep(wl)
    assert ls.z.master[0].is_pinned() and not ls.z.master[0].is_cuda
    for _ in range(wl.steps):
        ls.step()
        ls.check()


def test_mixed_residence_is_rejected():
    cfg = zs.adam_cfg()
    z = zs.ZeroStep((1000,), 2, synth.F16, cfg)
    grads = [torch.zeros(z.grad_numel(), dtype=torch.float16, device="cuda")] * 2
    host = torch.zeros_like(z.master[1], device="cpu").pin_memory()
    with pytest.raises(zs.ZeroError):
        zs.zero_step_fused(grads, z.layout, [z.master[0], host], z.m, z.v, z.params, cfg,
                           z.state, z.ws)


# ----------------------------------------------------------------- staged (TMA bulk-copy) path

@pytest.mark.parametrize("world,dtype", [(16, synth.F16), (16, synth.BF16), (8, synth.BF16)])
def test_staged_path_matches_register_path(world, dtype):
    """An every-rank one-pass step (the shared-memory staged kernel at
    N_d = 16) equals, bit for bit, the same step run rank by rank (the
    register kernel of one-rank views), over a ragged vector.  (No overflow
    is injected: a one-rank view tests only its own partition for NaN/Inf.)"""
    wl = CFG1.replace(numels=(777_777, 4097, 3), world=world, dtype=dtype, steps=3,
                      inject_at=())
    full = Lockstep(wl)
    parts = [Lockstep(wl.replace(rank=r)) for r in range(world)]
    for s in range(1, wl.steps + 1):
        grads = gen_grads(wl, full.lay, s, full.st.loss_scale)
        full.step(grads)
        for ls in parts:
            ls.step(grads)
    full.check()
    fw, fm, fv, fp = full.z.current()
    pb = half_bits(fp)
    for r, ls in enumerate(parts):
        ls.check()
        idx = torch.from_numpy(rank_index(full.lay, r)).cuda()
        w, m, v, p = ls.z.current()
        assert torch.equal(fw[idx].view(torch.int32), w.view(torch.int32))
        assert torch.equal(fm[idx].view(torch.int32), m.view(torch.int32))
        assert torch.equal(fv[idx].view(torch.int32), v.view(torch.int32))
        assert np.array_equal(pb[idx.cpu().numpy()], half_bits(p)[idx.cpu().numpy()])


def test_staged_wait_that_runs_out_skips_the_step_and_reports():
    """Every mbarrier wait of the shared-memory staged kernel is bounded.
    With ZERO_TEST_STAGED_WAIT_LIMIT set (read once per process, so the
    check runs in a child process: tests/gpu_children.py), each stage is
    announced 16 bytes more than its copies bring, so every CTA's first wait
    runs out after 1000 polls: the kernel records state.error, skips the step
    (every buffer's current slot unchanged bit for bit, the dynamic loss
    scale backed off), retires the extra bytes, waits for its own copies and
    finishes; a second step does the same, and the process then keeps using
    the GPU."""
    import json
    import subprocess
    import sys
    env = dict(os.environ, ZERO_TEST_STAGED_WAIT_LIMIT="1000")
    env.pop("ZERO_TEST_MAX_CTAS", None)
    here = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, os.path.join(here, "gpu_children.py"), "staged_wait"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert json.loads(r.stdout.strip().splitlines()[-1]) == {"ok": True}


GRAPHED = {
    "nd4-register-kernel": CFG1.replace(numels=(300_001,), world=4, steps=4,
                                        inject_at=((3, 1, 7),)),
    "nd16-staged-kernel": CFG1.replace(numels=(200_001,), world=16, steps=4,
                                       inject_at=((2, 15, 200_000),)),
    "nd8-clip-two-passes": CFG2.replace(numels=_small_gpt2(), steps=3),
}


@pytest.mark.parametrize("name", list(GRAPHED))
def test_fused_step_replays_from_a_cuda_graph(name):
    """The fused step synchronises nothing on the host and ends itself on
    the device, so a training loop can capture it once in a CUDA graph:
    replayed on gradients refreshed in the same device buffers, it gives the
    same bits and the same step state as the step launched directly (which
    the oracle checks), including a skipped step and the slot flips."""
    wl = GRAPHED[name]
    kw = dict(stage=True) if wl.max_grad_norm > 0 else {}
    a, b = Lockstep(wl, **kw), Lockstep(wl, **kw)
    warm = Lockstep(wl, **kw)  # fills the library's per-kernel caches outside the capture
    warm.step()
    torch.cuda.synchronize()
    bufs = [to_dev_half(g, wl.dtype) for g in gen_grads(wl, b.lay, 1, wl.loss_scale)]
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=side):
        b.z.step(bufs, side)
    torch.cuda.synchronize()
    assert b.z.read_state().t == 0  # capturing ran nothing
    for s in range(1, wl.steps + 1):
        grads = gen_grads(wl, a.lay, s, a.st.loss_scale)
        a.step(grads)
        for buf, g in zip(bufs, grads):
            buf.copy_(to_dev_half(g, wl.dtype))
        graph.replay()
        torch.cuda.synchronize()
        a.check()
        sa, sb = a.z.read_state(), b.z.read_state()
        assert bytes(sa) == bytes(sb), s
        for x, y in zip(a.z.current(), b.z.current()):
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    assert a.st.skipped == (1 if wl.inject_at else 0)


# ----------------------------------------------------------------- page-locked host blocks

def test_host_blocks_round_trip():
    """host_empty gives page-locked host tensors (zero_host_alloc) that the
    copy engines move in both directions without change, and the one-pass
    step reads gradients copied from them like gradients made on the device."""
    n = (1 << 20) + 64
    h = zs.host_empty(n, torch.float16)
    assert h.is_pinned() and h.numel() == n and h.data_ptr() % 256 == 0
    src = torch.randn(n, dtype=torch.float32).to(torch.float16)
    h.copy_(src)
    d = torch.empty(n, dtype=torch.float16, device="cuda")
    d.copy_(h, non_blocking=True)
    back = zs.host_empty(n, torch.float16)
    back.copy_(d, non_blocking=True)
    torch.cuda.synchronize()
    assert torch.equal(back.view(torch.int16), src.view(torch.int16))
    del h, back  # blocks are released with their last tensor


FROM_HOST = {
    # 16 ranks, every rank: on the device this is the shared-memory staged kernel
    "nd16-all-ranks": CFG1.replace(numels=(200_001,), world=16, steps=2, inject_at=((2, 9, 77),)),
    "nd4-fp16": CFG1.replace(numels=(300_001,), world=4, steps=2, inject_at=()),
    "nd8-bf16-clip-staged": CFG2.replace(numels=_small_gpt2(), steps=2),
    "nd4-rank2-slices": CFG4.replace(numels=(4 * 40_000 + 8,), world=4, rank=2, steps=2,
                                     inject_at=()),
    "nd8-bf16-halfreduce": CFG1.replace(numels=(100_000,), world=8, dtype=synth.BF16,
                                        half_reduce=True, steps=2, inject_at=()),
}


@pytest.mark.parametrize("copy", [False, True], ids=["loaded-from-host", "copied-in"])
@pytest.mark.parametrize("name", list(FROM_HOST))
def test_step_from_host_matches_device_step(name, copy):
    """step_from_host with each rank's gradient in a page-locked host block,
    either loaded by the step's kernels straight over the host link or
    copied into device buffers first, gives the same bits as the step on
    gradients in device memory (which the oracle checks), including a
    skipped step."""
    wl = FROM_HOST[name]
    a = Lockstep(wl, stage=True) if wl.max_grad_norm > 0 else Lockstep(wl)
    b = Lockstep(wl, stage=True) if wl.max_grad_norm > 0 else Lockstep(wl)
    for s in range(1, wl.steps + 1):
        grads = gen_grads(wl, a.lay, s, a.st.loss_scale)
        a.step(grads)
        src = [to_dev_half(g, wl.dtype) for g in grads]
        host = [zs.host_empty(g.numel(), g.dtype).copy_(g.cpu()) for g in src]
        dev = [torch.empty_like(g) for g in src] if copy else None
        st = b.z.step_from_host(host, dev)
        assert st.error == 0 and st.t + st.skipped == s
    a.check()
    for x, y in zip(a.z.current(), b.z.current()):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    assert a.z.read_state().t == b.z.read_state().t


def test_accumulation_from_host_matches_device():
    """Micro-steps whose gradients the accumulation kernel loads straight
    from page-locked host blocks give the same bits as from device buffers."""
    wl = CFG1.replace(numels=(100_003,), world=8, steps=1, inject_at=())
    a, b = Lockstep(wl), Lockstep(wl)
    micro = 3
    src = [[to_dev_half(g, wl.dtype) for g in gen_grads(wl, a.lay, k + 1, wl.loss_scale)]
           for k in range(micro)]
    for k in range(micro):
        a.z.accumulate(src[k], k > 0)
        host = [zs.host_empty(g.numel(), g.dtype).copy_(g.cpu()) for g in src[k]]
        b.z.accumulate(host, k > 0)
        torch.cuda.synchronize()
    a.z.step_accumulated()
    b.z.step_accumulated()
    torch.cuda.synchronize()
    assert torch.equal(a.z.acc.view(torch.int32), b.z.acc.view(torch.int32))
    for x, y in zip(a.z.current(), b.z.current()):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


# ----------------------------------------------------------------- per-bucket step, then commit

BUCKETED = {
    "nd16-fp16-staged": CFG1.replace(world=16, bucket=16 * 8 * 512),
    "nd3-bf16": CFG1.replace(world=3, dtype=synth.BF16, bucket=3 * 8 * 512),
    "nd4-fp16-rank1-slices": CFG1.replace(world=4, bucket=4 * 8 * 1024, rank=1,
                                          grads_are_slices=True),
    "nd8-bf16-halfreduce": CFG1.replace(world=8, dtype=synth.BF16, bucket=8 * 8 * 512,
                                        half_reduce=True),
    "nd2-fp16-offload": CFG1.replace(world=2, bucket=2 * 8 * 4096, offload_state=True),
}


@pytest.mark.parametrize("where", ["device", "host"], ids=["grads-on-device", "grads-in-host"])
@pytest.mark.parametrize("name", list(BUCKETED))
def test_bucket_ranges_then_commit_equal_fused_step(name, where):
    """The step run as ranges of buckets on two streams, then one commit,
    gives the fused step's bits (and both follow the oracle), including a
    step skipped for an Inf that lies in a middle bucket; the ranges may
    also load the gradients from page-locked host blocks."""
    base = BUCKETED[name]
    lay = oracle.layout(base.numels, base.world, base.align, base.bucket)
    nb = lay.num_buckets
    assert nb >= 3
    r = 0 if base.rank is None else base.rank
    inf_at = 2 * base.bucket + r * (base.bucket // base.world) + 5  # in bucket 2, r's slice
    wl = base.replace(numels=base.numels, steps=3, inject_at=((2, 0, inf_at),))
    ref, alt = Lockstep(wl), Lockstep(wl)
    ranges = [(0, 1), (1, nb // 2 - 1), (nb // 2, nb - nb // 2)]
    ranges = [(f, n) for f, n in ranges if n > 0]
    assert sum(n for _, n in ranges) == nb
    s0 = torch.cuda.current_stream()
    side = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in range(1, wl.steps + 1):
        grads = gen_grads(wl, ref.lay, s, ref.st.loss_scale)
        ref.step(grads)
        gd = [to_dev_half(g, wl.dtype) for g in grads]
        if where == "host":
            gd = [zs.host_empty(g.numel(), g.dtype).copy_(g.cpu()) for g in gd]
        ready = torch.cuda.Event()
        ready.record(s0)
        for st in side:
            st.wait_event(ready)
        for i, (f, n) in enumerate(ranges):
            alt.z.step_buckets(gd, f, n, side[i % 2])
        for st in side:
            done = torch.cuda.Event()
            done.record(st)
            s0.wait_event(done)
        alt.z.commit(s0)
        torch.cuda.synchronize()
        a, b = ref.z.read_state(), alt.z.read_state()
        assert state_proper(a) == state_proper(b)
        assert b.overflow == (1 if s == 2 else 0) and b.error == 0
        for x, y in zip(ref.z.current(), alt.z.current()):
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    ref.check()
