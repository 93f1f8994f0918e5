"""CPU oracle for the partitioned mixed-precision ZeRO Adam step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import this package.  The product
path (``zero_partitioned_mixed_step_gb300``) never imports it, and this package
never imports the product: the two share no code.

The per-element loops live in ``oracle.c`` (plain C, binary32 with every
operation rounded alone, compiled with ``-ffp-contract=off``).  This module
holds the layout, the per-step scalars (double, rounded once to binary32) and
the order of the steps, which follows the pages:

* "DeepSpeed ZeRO" (formulaic.cloudchewie.com), "ZeRO Stage 1: 切分优化器状态":
  "权重更新的触发条件" (a step whose gradients hold NaN/Inf updates nothing: the
  moments are not created, fp32 is not copied to fp16), "以 AdaW 为例" (the m, v,
  W update), "具体训练步骤" (each rank updates its 1/N_d fp32 slice, casts it to
  half and all-gathers it).
* Same page, "ZeRO Stage 2: 切分梯度": reduce-scatter of the gradients; the fp32
  gradient slice comes from the reduce-scattered half gradients; Adam is
  per-element, so rank i needs only its own slice of gradient and state.
* Same page, "ZeRO Stage 3: 切分参数", "参数的初始化和切割": flatten to 1-D, pad so
  the length divides by the data-parallel size, give each rank [start, end).
* Same page, "相关分析", "Constant Size Buffer": fixed-size buckets.
* Same page, "配置说明": fp16.loss_scale = 0 means dynamic loss scaling.
* "zero-optimizer" (codezrq.github.io), section 2.5 ReduceScatter.

Readings where the pages are silent or disagree (each one is listed with its
reason in the design notes): bias-corrected Adam, decoupled AdamW decay
applied before the update, a sum (not a mean) in the reduction, binary32
accumulation in ascending rank order, padding instead of floor division,
64-element tensor alignment, overflow checked on the reduced unscaled
gradient across all ranks, t counting committed steps only, loss-scale
backoff 0.5 / growth 2 after ``growth_interval`` good steps, and the clip
coefficient min(1, max_norm / (||g||_2 + 1e-6)).

Parity status: every function here is pinned by a test under ``tests/``
(``test_oracle_*.py``); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import tempfile
from typing import List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")

F16 = 0
BF16 = 1

_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def _lib_path(openmp: bool) -> str:
    return os.path.join(_BUILD, "liboracle_omp.so" if openmp else "liboracle.so")


def build(force: bool = False) -> None:
    """Compile the oracle's C (single-threaded and OpenMP builds) with gcc."""
    os.makedirs(_BUILD, exist_ok=True)
    for openmp in (False, True):
        out = _lib_path(openmp)
        if (not force and os.path.exists(out)
                and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
            continue
        fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD)
        os.close(fd)
        cmd = ["gcc", *_CFLAGS, *(["-fopenmp"] if openmp else []), _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)


class _Scalars(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in
                ("b1", "omb1", "b2", "omb2", "step", "rbc2", "eps", "decay", "wd")] + [
                    ("adamw", ctypes.c_int32)]


_LIBS = {}


def _lib(openmp: bool = False):
    if openmp not in _LIBS:
        build()
        lib = ctypes.CDLL(_lib_path(openmp))
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.orc_f16_to_f32.restype = ctypes.c_float
        lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f32.restype = ctypes.c_float
        lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
        lib.orc_f32_to_f16.restype = ctypes.c_uint16
        lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.orc_f32_to_bf16.restype = ctypes.c_uint16
        lib.orc_to_half_array.argtypes = [P, I64, ctypes.c_int, P]
        lib.orc_from_half_array.argtypes = [P, I64, ctypes.c_int, P]
        lib.orc_reduce_sum.argtypes = [P, ctypes.c_int, ctypes.c_int, I64, I64, P]
        lib.orc_reduce_sum_half.argtypes = [P, ctypes.c_int, ctypes.c_int, I64, I64, P]
        lib.orc_unscale.argtypes = [P, I64, ctypes.c_float]
        lib.orc_accumulate.argtypes = [P, P, I64]
        lib.orc_any_nonfinite.argtypes = [P, I64]
        lib.orc_any_nonfinite.restype = ctypes.c_int
        lib.orc_sumsq.argtypes = [P, I64, ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_double)]
        lib.orc_scale.argtypes = [P, I64, ctypes.c_float]
        lib.orc_adam.argtypes = [P, P, P, P, I64, ctypes.POINTER(_Scalars)]
        _LIBS[openmp] = lib
    return _LIBS[openmp]


def f32(x: float) -> float:
    """Round a Python float (binary64) to binary32, to nearest even."""
    return float(np.float32(x))


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# --------------------------------------------------------------------------
# Conversions
# --------------------------------------------------------------------------

def half_to_f32(h: np.ndarray, dtype: int, openmp: bool = False) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    _lib(openmp).orc_from_half_array(_ptr(h), h.size, dtype, _ptr(out))
    return out


def f32_to_half(x: np.ndarray, dtype: int, openmp: bool = False) -> np.ndarray:
    """IEEE round-to-nearest-even to binary16 (F16) or bfloat16 (BF16), as bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    _lib(openmp).orc_to_half_array(_ptr(x), x.size, dtype, _ptr(out))
    return out


# --------------------------------------------------------------------------
# Step (a1): partition layout
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Layout:
    numels: Tuple[int, ...]
    world: int
    align: int
    bucket: int                 # 0 = one contiguous partition per rank
    offsets: Tuple[int, ...]    # flat start of every tensor
    numel: int                  # sum of tensor sizes (unpadded)
    flat_end: int               # end of the last tensor, alignment gaps included
    padded: int                 # padded flat length
    owned: int                  # elements each rank owns
    num_buckets: int
    slice: int                  # a rank's slice of a full bucket (bucketed)
    last_slice: int             # a rank's slice of the last bucket (bucketed)
    segments: Tuple[Tuple[Tuple[int, int], ...], ...]  # per rank: (flat start, length)


def _round_up(x: int, a: int) -> int:
    return -(-x // a) * a


def layout(numels: Sequence[int], world: int, align: int = 64, bucket: int = 0) -> Layout:
    """Flatten the tensors into one 1-D vector and split it among ``world`` ranks.

    "DeepSpeed ZeRO", "ZeRO Stage 3: 切分参数", "参数的初始化和切割": flatten to 1-D,
    pad so the length divides by the data-parallel size, give each rank its
    [start, end).  Readings: every tensor starts at a multiple of ``align``
    elements; the flat vector is padded to a multiple of world * align, so
    every partition starts on an ``align`` boundary; rank r owns
    [r P, (r + 1) P).  With ``bucket`` > 0 (the constant-size buffers of the
    same page's "Constant Size Buffer") the vector is cut into buckets of
    ``bucket`` elements, the last one padded to a multiple of world * align,
    and rank r owns slice r of every bucket.
    """
    if world < 1 or align < 1:
        raise ValueError("world and align must be >= 1")
    offsets = []
    off = 0
    for n in numels:
        if n < 0:
            raise ValueError("negative tensor size")
        off = _round_up(off, align)
        offsets.append(off)
        off += n
    flat_end = off
    unit = world * align
    if bucket == 0:
        padded = _round_up(flat_end, unit)
        P = padded // world
        segs = tuple(((r * P, P),) if P else () for r in range(world))
        return Layout(tuple(numels), world, align, 0, tuple(offsets), sum(numels), flat_end,
                      padded, P, 1 if P else 0, P, P, segs)
    if bucket % world:
        raise ValueError("bucket size must divide by world")
    nb = max(1, -(-flat_end // bucket)) if flat_end else 0
    if nb == 0:
        return Layout(tuple(numels), world, align, bucket, tuple(offsets), 0, 0, 0, 0, 0,
                      bucket // world, 0, tuple(() for _ in range(world)))
    last = flat_end - (nb - 1) * bucket
    last_pad = _round_up(last, unit)
    padded = (nb - 1) * bucket + last_pad
    s, ls = bucket // world, last_pad // world
    segs = []
    for r in range(world):
        seg = [(b * bucket + r * s, s) for b in range(nb - 1)]
        seg.append(((nb - 1) * bucket + r * ls, ls))
        segs.append(tuple(seg))
    return Layout(tuple(numels), world, align, bucket, tuple(offsets), sum(numels), flat_end,
                  padded, (nb - 1) * s + ls, nb, s, ls, tuple(segs))


# --------------------------------------------------------------------------
# Optimizer configuration and step state
# --------------------------------------------------------------------------

@dataclasses.dataclass
class AdamCfg:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    adamw: bool = True              # decoupled decay (AdamW); False = coupled L2
    bias_correction: bool = True    # False = the pages' formula taken literally
    max_grad_norm: float = 0.0      # 0 = no clipping
    dynamic_scale: bool = False
    backoff: float = 0.5
    growth: float = 2.0
    growth_interval: int = 1000
    min_scale: float = 1.0


@dataclasses.dataclass
class State:
    t: int = 0                 # committed steps
    bp1: float = 1.0           # beta1 ** t as a running product (binary64)
    bp2: float = 1.0           # beta2 ** t as a running product (binary64)
    loss_scale: float = 1.0    # S, a power of two
    good_steps: int = 0
    overflow: int = 0          # 1 if the last step was skipped
    skipped: int = 0
    sumsq: float = 0.0         # last step's global sum of squares (unscaled, unclipped)
    coef: float = 1.0          # last step's clip coefficient


def step_scalars(cfg: AdamCfg, st: State) -> _Scalars:
    """Per-step binary32 scalars for step t + 1, each computed in binary64 and
    rounded once.  beta^t is the running product of the committed steps."""
    bp1 = st.bp1 * cfg.beta1
    bp2 = st.bp2 * cfg.beta2
    if cfg.bias_correction:
        step = f32(cfg.lr / (1.0 - bp1))
        rbc2 = f32(math.sqrt(1.0 - bp2))
    else:
        step = f32(cfg.lr)
        rbc2 = 1.0
    return _Scalars(f32(cfg.beta1), f32(1.0 - cfg.beta1), f32(cfg.beta2), f32(1.0 - cfg.beta2),
                    step, rbc2, f32(cfg.eps), f32(1.0 - cfg.lr * cfg.weight_decay),
                    f32(cfg.weight_decay), 1 if cfg.adamw else 0)


def clip_coef(sumsq: float, max_grad_norm: float) -> float:
    """c = min(1, max_norm / (||g||_2 + 1e-6)) in binary64, rounded to binary32."""
    return f32(min(1.0, max_grad_norm / (math.sqrt(sumsq) + 1e-6)))


def skip(cfg: AdamCfg, st: State) -> None:
    """An overflow step: nothing but the loss scale changes."""
    st.overflow = 1
    st.skipped += 1
    if cfg.dynamic_scale:
        st.loss_scale = max(st.loss_scale * cfg.backoff, cfg.min_scale)
        st.good_steps = 0


def commit(cfg: AdamCfg, st: State) -> None:
    """A good step: t advances, the running beta products advance, and the
    dynamic loss scale grows after growth_interval good steps in a row."""
    st.overflow = 0
    st.t += 1
    st.bp1 = st.bp1 * cfg.beta1
    st.bp2 = st.bp2 * cfg.beta2
    st.good_steps += 1
    if cfg.dynamic_scale and st.good_steps == cfg.growth_interval:
        st.loss_scale = st.loss_scale * cfg.growth
        st.good_steps = 0


# --------------------------------------------------------------------------
# Element-wise primitives (thin wrappers over oracle.c)
# --------------------------------------------------------------------------

def reduce_sum(grads: Sequence[np.ndarray], dtype: int, offset: int, n: int,
               openmp: bool = False, half_reduce: bool = False) -> np.ndarray:
    """Step (a2): g[j] = sum_q float(grads[q][offset + j]) in ascending q, in
    binary32, or with ``half_reduce`` in the gradient's half type (every
    partial sum rounded to nearest even)."""
    arr = (ctypes.c_void_p * len(grads))(*[_ptr(g) for g in grads])
    for g in grads:
        assert g.dtype == np.uint16 and g.size >= offset + n
    out = np.empty(n, np.float32)
    fn = _lib(openmp).orc_reduce_sum_half if half_reduce else _lib(openmp).orc_reduce_sum
    fn(arr, len(grads), dtype, offset, n, _ptr(out))
    return out


def accumulate(acc: np.ndarray, r: np.ndarray, openmp: bool = False) -> None:
    """acc += r element-wise in binary32 (one micro-step into the accumulator)."""
    assert acc.dtype == np.float32 and r.dtype == np.float32 and acc.size == r.size
    _lib(openmp).orc_accumulate(_ptr(acc), _ptr(r), acc.size)


def unscale(g: np.ndarray, inv_scale: float, openmp: bool = False) -> None:
    _lib(openmp).orc_unscale(_ptr(g), g.size, inv_scale)


def any_nonfinite(g: np.ndarray, openmp: bool = False) -> bool:
    return bool(_lib(openmp).orc_any_nonfinite(_ptr(g), g.size))


def sumsq(g: np.ndarray, acc: Tuple[float, float] = (0.0, 0.0)) -> Tuple[float, float]:
    """Step (a5): continue the compensated sum of squares ``acc`` = (sum,
    compensation) over g; ``sumsq_value`` turns it into a number."""
    s = ctypes.c_double(acc[0])
    c = ctypes.c_double(acc[1])
    _lib(False).orc_sumsq(_ptr(g), g.size, ctypes.byref(s), ctypes.byref(c))
    return (s.value, c.value)


def sumsq_value(acc: Tuple[float, float]) -> float:
    return acc[0] + acc[1]


def scale(g: np.ndarray, c: float, openmp: bool = False) -> None:
    _lib(openmp).orc_scale(_ptr(g), g.size, c)


def adam(g: np.ndarray, w: np.ndarray, m: np.ndarray, v: np.ndarray, sc: _Scalars,
         openmp: bool = False) -> None:
    """Step (a6) in place on w, m, v."""
    n = g.size
    assert w.size == n and m.size == n and v.size == n
    _lib(openmp).orc_adam(_ptr(g), _ptr(w), _ptr(m), _ptr(v), n, ctypes.byref(sc))


# --------------------------------------------------------------------------
# The whole step
# --------------------------------------------------------------------------

def _ranks(lay: Layout, rank: Optional[int]) -> List[int]:
    return list(range(lay.world)) if rank is None else [rank]


def step(grads: Sequence[np.ndarray], dtype: int, lay: Layout, cfg: AdamCfg, st: State,
         master: np.ndarray, m: np.ndarray, v: np.ndarray, half: np.ndarray,
         rank: Optional[int] = None, grads_are_slices: bool = False,
         openmp: bool = False, half_reduce: bool = False) -> None:
    """One partitioned mixed-precision step, in place.

    ``rank`` None simulates all ranks: ``grads[q]`` are the ranks' full padded
    flat gradient buffers and master/m/v are flat (rank r's partition at its
    flat positions).  ``rank`` = r simulates rank r alone: master/m/v hold the
    elements r owns, in order, and ``grads[q]`` are either full buffers or
    (``grads_are_slices``) only the elements r owns.  ``half`` is always the
    full flat parameter buffer in the all-gather layout.  ``half_reduce``
    reduces in the gradient's half type (see ``reduce_sum``).
    """
    ranks = _ranks(lay, rank)
    inv_s = f32(1.0 / st.loss_scale)
    parts = []  # (rank, flat start, state index, g)
    for r in ranks:
        local = 0
        for fs, ln in lay.segments[r]:
            goff = local if (rank is not None and grads_are_slices) else fs
            g = reduce_sum(grads, dtype, goff, ln, openmp, half_reduce)  # (a2)
            unscale(g, inv_s, openmp)                                # (a3)
            parts.append((r, fs, fs if rank is None else local, g))
            local += ln
    if any(any_nonfinite(g, openmp) for _, _, _, g in parts):       # (a4)
        skip(cfg, st)
        return
    if cfg.max_grad_norm > 0:                                        # (a5)
        total = 0.0
        for r in ranks:
            acc = (0.0, 0.0)
            for rr, _, _, g in parts:
                if rr == r:
                    acc = sumsq(g, acc)
            total = total + sumsq_value(acc)
        st.sumsq = total
        st.coef = clip_coef(total, cfg.max_grad_norm)
        if st.coef < 1.0:
            for _, _, _, g in parts:
                scale(g, st.coef, openmp)
    sc = step_scalars(cfg, st)
    for _, fs, si, g in parts:                                       # (a6), (a7)
        n = g.size
        adam(g, master[si:si + n], m[si:si + n], v[si:si + n], sc, openmp)
        half[fs:fs + n] = f32_to_half(master[si:si + n], dtype, openmp)
    commit(cfg, st)                                                  # (a8)


def scan_scalars(grad_chunks, dtype: int, lay: Layout, inv_scale: float, want_sumsq: bool,
                 openmp: bool = False, ranks: Optional[Sequence[int]] = None,
                 chunk: int = 1 << 24, half_reduce: bool = False) -> Tuple[bool, float]:
    """The step's global scalars (overflow flag, sum of squares) for gradients
    too large to hold at once.  ``grad_chunks(r, flat_start, n)`` returns the
    world gradient arrays for flat elements [flat_start, flat_start + n);
    chunks are taken in each rank's element order, so the sum of squares is
    the same compensated sum ``step`` forms.  ``ranks``: the simulated ranks
    (all by default)."""
    flag = False
    total = 0.0
    for r in (range(lay.world) if ranks is None else ranks):
        acc = (0.0, 0.0)
        for fs, ln in lay.segments[r]:
            for chunk_start in range(fs, fs + ln, chunk):
                n = min(chunk, fs + ln - chunk_start)
                gs = grad_chunks(r, chunk_start, n)
                g = reduce_sum(gs, dtype, 0, n, openmp, half_reduce)
                unscale(g, inv_scale, openmp)
                flag = flag or any_nonfinite(g, openmp)
                if want_sumsq:
                    acc = sumsq(g, acc)
        total = total + sumsq_value(acc)
    return flag, total


def window_step(grads: Sequence[np.ndarray], dtype: int, cfg: AdamCfg, st: State, flag: bool,
                total_sumsq: float, master: np.ndarray, m: np.ndarray, v: np.ndarray,
                half_reduce: bool = False) -> Optional[np.ndarray]:
    """Steps (a2)-(a7) for one contiguous window of a rank's elements, given
    the step's global scalars (the update is element-wise once they are known:
    "DeepSpeed ZeRO", ZeRO Stage 2, the per-element independence of Adam).
    ``grads[q]`` hold the window's gradient elements.  Updates master/m/v in
    place and returns the half output, or None when the step is skipped.
    Does not advance ``st``; call ``skip``/``commit`` once per step."""
    g = reduce_sum(grads, dtype, 0, master.size, half_reduce=half_reduce)
    unscale(g, f32(1.0 / st.loss_scale))
    if flag:
        return None
    if cfg.max_grad_norm > 0:
        c = clip_coef(total_sumsq, cfg.max_grad_norm)
        if c < 1.0:
            scale(g, c)
    sc = step_scalars(cfg, st)
    adam(g, master, m, v, sc)
    return f32_to_half(master, dtype)


def finish_window_step(cfg: AdamCfg, st: State, flag: bool, total_sumsq: float) -> None:
    """Step (a8) after every window of a step has gone through
    ``window_step``: skip when the scan found NaN/Inf, else record the step's
    sum of squares and clip coefficient (when clipping) and commit."""
    if flag:
        skip(cfg, st)
        return
    if cfg.max_grad_norm > 0:
        st.sumsq = total_sumsq
        st.coef = clip_coef(total_sumsq, cfg.max_grad_norm)
    commit(cfg, st)


# --------------------------------------------------------------------------
# Gradient accumulation
# --------------------------------------------------------------------------

def reduce_scatter_accumulate(grads: Sequence[np.ndarray], dtype: int, lay: Layout,
                              acc: np.ndarray, add: bool, rank: Optional[int] = None,
                              grads_are_slices: bool = False, openmp: bool = False,
                              half_reduce: bool = False) -> None:
    """One micro-step: acc = (acc if add else 0) + reduce-scatter sum.

    "DeepSpeed ZeRO", "ZeRO-2 在梯度累积场景下的通信量": with gradient
    accumulation ZeRO-2 reduce-scatters after every backward and accumulates
    its 1/N_d slice.  The micro-step's sum over ranks is formed first (from
    +0, ascending rank order), then added to the accumulator in binary32.
    ``acc`` is flat (rank None) or rank r's elements in order (rank r)."""
    for r in _ranks(lay, rank):
        local = 0
        for fs, ln in lay.segments[r]:
            goff = local if (rank is not None and grads_are_slices) else fs
            red = reduce_sum(grads, dtype, goff, ln, openmp, half_reduce)
            si = fs if rank is None else local
            if add:
                accumulate(acc[si:si + ln], red, openmp)
            else:
                acc[si:si + ln] = red
            local += ln


def step_accumulated(acc: np.ndarray, dtype: int, lay: Layout, cfg: AdamCfg, st: State,
                     master: np.ndarray, m: np.ndarray, v: np.ndarray, half: np.ndarray,
                     rank: Optional[int] = None, openmp: bool = False) -> None:
    """The step of ``step`` with the gradient taken from an fp32 accumulator
    (the sum of the micro-steps' reduced, still scaled gradients) instead of
    the N_d half-precision buffers: unscale, overflow test, clip, Adam, cast,
    commit, in the same order."""
    ranks = _ranks(lay, rank)
    inv_s = f32(1.0 / st.loss_scale)
    parts = []
    for r in ranks:
        local = 0
        for fs, ln in lay.segments[r]:
            si = fs if rank is None else local
            g = np.array(acc[si:si + ln], dtype=np.float32, copy=True)
            unscale(g, inv_s, openmp)
            parts.append((r, fs, si, g))
            local += ln
    if any(any_nonfinite(g, openmp) for _, _, _, g in parts):
        skip(cfg, st)
        return
    if cfg.max_grad_norm > 0:
        total = 0.0
        for r in ranks:
            a = (0.0, 0.0)
            for rr, _, _, g in parts:
                if rr == r:
                    a = sumsq(g, a)
            total = total + sumsq_value(a)
        st.sumsq = total
        st.coef = clip_coef(total, cfg.max_grad_norm)
        if st.coef < 1.0:
            for _, _, _, g in parts:
                scale(g, st.coef, openmp)
    sc = step_scalars(cfg, st)
    for _, fs, si, g in parts:
        n = g.size
        adam(g, master[si:si + n], m[si:si + n], v[si:si + n], sc, openmp)
        half[fs:fs + n] = f32_to_half(master[si:si + n], dtype, openmp)
    commit(cfg, st)

