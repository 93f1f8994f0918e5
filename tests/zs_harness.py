"""Helpers shared by the GPU parity tests: seeded inputs for a workload, the
CUDA step and the CPU oracle run side by side, element-wise comparison."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
import zero_partitioned_mixed_step_gb300 as zs

INF_BITS = {synth.F16: 0x7C00, synth.BF16: 0x7F80}

# Tolerances: fp32 master/m/v within 1e-6 relative plus 1e-12 absolute;
# half-precision parameters within 1 ulp; flags and layout bit-exact.
RTOL = 1e-6
ATOL = 1e-12
# The global sum of squares: the oracle's compensated sum is within a few
# ulps of the exact value; the GPU adds exact per-unit squares (error-free
# transformations in binary32) into binary64 per thread (~10^4 terms) and
# then in a fixed tree, which bounds its error near 1e-14 relative.
SUMSQ_RTOL = 1e-11


def oracle_cfg(wl) -> oracle.AdamCfg:
    return oracle.AdamCfg(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
                          weight_decay=wl.weight_decay, adamw=wl.adamw,
                          max_grad_norm=wl.max_grad_norm, dynamic_scale=wl.dynamic_scale)


def lib_cfg(wl, **kw):
    args = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
                weight_decay=wl.weight_decay, adamw=wl.adamw, max_grad_norm=wl.max_grad_norm,
                dynamic_scale=wl.dynamic_scale)
    args.update(kw)
    return zs.adam_cfg(**args)


def state_proper(st: "zs.StepState") -> bytes:
    """The step state's own fields (the 64 bytes before the library's scalar
    cache, which depends on which kernels ran, not on the step's result)."""
    return bytes(st)[:zs.StepState.scalar_cache.offset]


def tensor_mask(lay: oracle.Layout) -> np.ndarray:
    mask = np.zeros(lay.padded, bool)
    for o, n in zip(lay.offsets, lay.numels):
        mask[o:o + n] = True
    return mask


def rank_index(lay: oracle.Layout, r: int) -> np.ndarray:
    segs = lay.segments[r]
    if not segs:
        return np.zeros(0, np.int64)
    return np.concatenate([np.arange(fs, fs + ln, dtype=np.int64) for fs, ln in segs])


def gen_master(wl, lay) -> np.ndarray:
    master = synth.fill_f32(wl.master_key(), 0, lay.padded, wl.master_sigma)
    master[~tensor_mask(lay)] = 0
    return master


def gen_grads(wl, lay, step: int, loss_scale: float):
    """Every rank's gradient for a step (1-based), as fp16/bf16 bits: full
    flat buffers, or only ``wl.rank``'s elements when grads_are_slices."""
    mask = tensor_mask(lay)
    sigma = wl.grad_sigma * loss_scale
    out = []
    idx = rank_index(lay, wl.rank) if wl.grads_are_slices else None
    for q in range(wl.world):
        g = synth.fill_half(wl.grad_key(step, q), 0, lay.padded, sigma, wl.dtype)
        g[~mask] = 0
        out.append(g)
    for q, i in wl.injections(step):
        out[q][i] = INF_BITS[wl.dtype]
    if idx is not None:
        out = [g[idx].copy() for g in out]
    return out


def to_dev_half(bits: np.ndarray, dtype: int) -> torch.Tensor:
    return torch.from_numpy(bits.view(np.int16)).to("cuda").view(zs.torch_dtype(dtype))


def half_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in units in the last place between half-precision bit patterns."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a) - ordered(b))


def assert_close(name: str, got: np.ndarray, want: np.ndarray) -> int:
    """Element-wise |got - want| <= RTOL |want| + ATOL; returns how many are
    bit-identical (reported in failures)."""
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    same = int(np.count_nonzero(got.view(np.uint32) == want.view(np.uint32)))
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    tol = RTOL * np.abs(want.astype(np.float64)) + ATOL
    bad = ~(err <= tol)
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError(f"{name}: {int(bad.sum())} of {got.size} elements out of tolerance "
                             f"(first at {i}: got {got[i]!r}, want {want[i]!r}); "
                             f"{same} bit-identical")
    return same


def assert_half_close(name: str, got: np.ndarray, want: np.ndarray) -> int:
    d = ulp_distance(got, want)
    assert d.max(initial=0) <= 1, f"{name}: {int((d > 1).sum())} elements more than 1 ulp apart"
    return int(np.count_nonzero(d == 0))


class Lockstep:
    """The CUDA fused step and the oracle on the same seeded inputs."""

    def __init__(self, wl, stage=None, **cfg_kw):
        self.wl = wl
        self.lay = oracle.layout(wl.numels, wl.world, wl.align, wl.bucket)
        self.ocfg = oracle_cfg(wl)
        for k, v in cfg_kw.items():
            setattr(self.ocfg, k, v)
        self.zcfg = lib_cfg(wl, **{k: v for k, v in cfg_kw.items()})
        rank = -1 if wl.rank is None else wl.rank
        self.z = zs.ZeroStep(wl.numels, wl.world, wl.dtype, self.zcfg, loss_scale=wl.loss_scale,
                             rank=rank, bucket_numel=wl.bucket, align_elems=wl.align,
                             grads_are_slices=wl.grads_are_slices, stage_grad=stage,
                             half_reduce=wl.half_reduce, offload_state=wl.offload_state)
        L = self.z.layout
        assert (L.padded_numel, L.owned_numel) == (self.lay.padded, self.lay.owned)
        master = gen_master(wl, self.lay)
        self.idx = None if wl.rank is None else rank_index(self.lay, wl.rank)
        self.w = master.copy() if self.idx is None else master[self.idx].copy()
        self.m = np.zeros_like(self.w)
        self.v = np.zeros_like(self.w)
        self.half = synth.round_half(master, wl.dtype)
        self.z.master[0].copy_(torch.from_numpy(self.w))
        self.z.params[0].copy_(to_dev_half(self.half, wl.dtype))
        self.st = oracle.State(loss_scale=wl.loss_scale)
        self.steps = 0
        self.identical = {}

    def step(self, grads=None):
        self.steps += 1
        wl = self.wl
        if grads is None:
            grads = gen_grads(wl, self.lay, self.steps, self.st.loss_scale)
        self.z.step([to_dev_half(g, wl.dtype) for g in grads])
        oracle.step(grads, wl.dtype, self.lay, self.ocfg, self.st, self.w, self.m, self.v,
                    self.half, rank=wl.rank, grads_are_slices=wl.grads_are_slices,
                    half_reduce=wl.half_reduce)

    def check(self):
        torch.cuda.synchronize()
        zs_ = self.z.read_state()
        st = self.st
        assert zs_.overflow == st.overflow, (zs_.overflow, st.overflow)
        assert zs_.t == st.t and zs_.skipped == st.skipped
        assert zs_.beta1_pow == st.bp1 and zs_.beta2_pow == st.bp2
        assert zs_.loss_scale == st.loss_scale and zs_.good_steps == st.good_steps
        assert zs_.found_inf == 0 and zs_.error == 0
        if self.ocfg.max_grad_norm > 0 and st.t > 0:
            assert abs(zs_.sumsq - st.sumsq) <= SUMSQ_RTOL * st.sumsq, (zs_.sumsq, st.sumsq)
            assert abs(zs_.clip_coef - st.coef) <= 2.0 ** -23 * st.coef, (zs_.clip_coef, st.coef)
        w, m, v, p = self.z.current()
        self.identical["master"] = assert_close("master", w.cpu().numpy(), self.w)
        self.identical["m"] = assert_close("m", m.cpu().numpy(), self.m)
        self.identical["v"] = assert_close("v", v.cpu().numpy(), self.v)
        pb = half_bits(p)
        if self.idx is None:
            self.identical["params"] = assert_half_close("params", pb, self.half)
        else:  # a rank alone writes only its own elements of the parameter buffer
            self.identical["params"] = assert_half_close("params", pb[self.idx],
                                                         self.half[self.idx])
        return zs_
