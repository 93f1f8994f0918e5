"""ctypes declarations of libzerostep.so (include/zerostep.h)."""
from __future__ import annotations

import ctypes
import os

from . import _build

F16 = 0
BF16 = 1

OK = 0
EINVAL = -1
EALIGN = -2
ESPACE = -3
ECUDA_BASE = -1000
MAX_WORLD = 1024
NOALLOC_SCRATCH_BYTES = 266496


class Layout(ctypes.Structure):
    _fields_ = [("numel", ctypes.c_int64), ("flat_numel", ctypes.c_int64),
                ("padded_numel", ctypes.c_int64), ("owned_numel", ctypes.c_int64),
                ("bucket_numel", ctypes.c_int64), ("num_buckets", ctypes.c_int64),
                ("slice_numel", ctypes.c_int64), ("last_slice_numel", ctypes.c_int64),
                ("world", ctypes.c_int32), ("align_elems", ctypes.c_int32)]


class AdamCfg(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double),
                ("adamw", ctypes.c_int32), ("bias_correction", ctypes.c_int32),
                ("max_grad_norm", ctypes.c_double), ("dynamic_scale", ctypes.c_int32),
                ("growth_interval", ctypes.c_int32), ("backoff", ctypes.c_double),
                ("growth", ctypes.c_double), ("min_scale", ctypes.c_double)]


class StepState(ctypes.Structure):
    _fields_ = [("t", ctypes.c_int64), ("beta1_pow", ctypes.c_double),
                ("beta2_pow", ctypes.c_double), ("sumsq", ctypes.c_double),
                ("loss_scale", ctypes.c_float), ("clip_coef", ctypes.c_float),
                ("good_steps", ctypes.c_int32), ("overflow", ctypes.c_int32),
                ("found_inf", ctypes.c_int32), ("cur", ctypes.c_int32),
                ("skipped", ctypes.c_int32), ("error", ctypes.c_int32),
                ("scalar_cache", ctypes.c_uint64 * 16)]


assert ctypes.sizeof(StepState) == 192
assert ctypes.sizeof(Layout) == 72

# Every symbol include/zerostep.h declares, with its ctypes signature.
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
SIGNATURES = {
    "zero_strerror": ([_I], ctypes.c_char_p),
    "zero_version": ([], _I),
    "zero_partition_layout": ([_I, ctypes.POINTER(ctypes.c_int64), _I, _I, _I64,
                               ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(Layout)], _I),
    "zero_state_init": ([ctypes.POINTER(StepState), ctypes.c_float], _I),
    "zero_workspace_bytes": ([ctypes.POINTER(Layout)], ctypes.c_size_t),
    "zero_host_alloc": ([ctypes.c_size_t, ctypes.POINTER(ctypes.c_void_p)], _I),
    "zero_host_free": ([_P], _I),
    "zero_reduce_scatter_sum": ([_P, _I, _I, ctypes.POINTER(Layout), _I, _P, _P], _I),
    "zero_check_overflow": ([_P, _I64, ctypes.c_float, _P, _P], _I),
    "zero_grad_norm": ([_P, _I64, ctypes.c_float, _P, _P, ctypes.c_size_t, _P], _I),
    "zero_grad_norm_noalloc": ([_P, _I64, ctypes.c_float, _P, _P], _I),
    "zero_adam_step": ([_P, _P, _P, _P, _P, _I, _I64, ctypes.POINTER(AdamCfg), _P, _P], _I),
    "zero_step_finalize": ([ctypes.POINTER(AdamCfg), _P, _I, _P], _I),
    "zero_step_fused": ([_P, _I, _I, ctypes.POINTER(Layout), _I, _P, _P, _P, _P, _P,
                         ctypes.POINTER(AdamCfg), _P, _P, ctypes.c_size_t, _P], _I),
    "zero_reduce_scatter_accumulate": ([_P, _I, _I, ctypes.POINTER(Layout), _I, _P, _I, _P], _I),
    "zero_step_fused_buckets": ([_P, _I, _I, ctypes.POINTER(Layout), _I, _I64, _I64, _P, _P, _P,
                                 _P, ctypes.POINTER(AdamCfg), _P, _P], _I),
    "zero_step_fused_accumulated": ([_P, _I, ctypes.POINTER(Layout), _I, _P, _P, _P, _P,
                                     ctypes.POINTER(AdamCfg), _P, _P, ctypes.c_size_t, _P], _I),
    "zero_step_buckets_pass1": ([_P, _I, _I, ctypes.POINTER(Layout), _I, _I64, _I64, _P,
                                 ctypes.POINTER(AdamCfg), _P, _P, ctypes.c_size_t, _P], _I),
    "zero_step_buckets_norm": ([ctypes.POINTER(Layout), _I, _P, ctypes.c_size_t, _P], _I),
    "zero_step_buckets_pass2": ([_P, _I, _I, ctypes.POINTER(Layout), _I, _I64, _I64, _P, _P, _P,
                                 _P, _P, ctypes.POINTER(AdamCfg), _P, _P, ctypes.c_size_t, _P],
                                _I),
}

_lib = None


def lib():
    """Load the in-tree libzerostep.so.  There is no fallback: without the
    built library every call fails with an ImportError."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise ImportError(
                "libzerostep.so is not built; run `python -c 'import __graft_entry__ as g; "
                "g.build()'` (nvcc, sm_103a) first")
        so = ctypes.CDLL(_build.LIB)
        for name, (args, res) in SIGNATURES.items():
            f = getattr(so, name)
            f.argtypes = args
            f.restype = res
        _lib = so
    return _lib


class ZeroError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {code} ({lib().zero_strerror(code).decode()})")


def check(fn: str, code: int) -> None:
    if code != OK:
        raise ZeroError(fn, code)
