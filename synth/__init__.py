"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This package builds inputs only; it holds none of the optimizer step's
arithmetic.  Each value is defined by a counter-based generator (SplitMix64
outputs combined into an Irwin-Hall sum; the full definition is at the top of
``synth_host.c``), so any element can be computed on its own, on the CPU
(``synth_host.c``) or on the GPU (``synth_cuda.cu``), and both give the same
bits.  The oracle receives the CPU values, the CUDA step the GPU values; a GPU
test checks that the two generators agree bit for bit.
"""
from __future__ import annotations

import ctypes
import math
import os
import shutil
import subprocess
import tempfile
from typing import Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_HOST_SRC = os.path.join(_HERE, "synth_host.c")
_CUDA_SRC = os.path.join(_HERE, "synth_cuda.cu")
_HOST_LIB = os.path.join(_BUILD, "libsynth_host.so")
_CUDA_LIB = os.path.join(_BUILD, "libsynth_cuda.so")

F16 = 0
BF16 = 1

# Standard deviation of the centred Irwin-Hall sum of four uniform 32-bit integers.
IRWIN_HALL_SD = math.sqrt((2.0 ** 64 - 1.0) / 3.0)
# Every generated value lies within this many standard deviations of 0.
SUPPORT_SIGMAS = 2.0 * math.sqrt(3.0)


def _stale(out: str, src: str) -> bool:
    return not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src)


def _compile(cmd_for_tmp, out: str) -> None:
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD)
    os.close(fd)
    subprocess.run(cmd_for_tmp(tmp), check=True)
    os.replace(tmp, out)


def build(force: bool = False, cuda: bool = True) -> None:
    """Compile the CPU generator (gcc) and, when nvcc exists, the GPU one."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or _stale(_HOST_LIB, _HOST_SRC):
        _compile(lambda o: ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                            _HOST_SRC, "-o", o], _HOST_LIB)
    if cuda and shutil.which("nvcc") and (force or _stale(_CUDA_LIB, _CUDA_SRC)):
        _compile(lambda o: ["nvcc", "-O3", "-shared", "-Xcompiler", "-fPIC", "-cudart", "shared",
                            "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
                            _CUDA_SRC, "-o", o], _CUDA_LIB)


_host = None
_cuda = None


def _host_lib():
    global _host
    if _host is None:
        build(cuda=False)
        lib = ctypes.CDLL(_HOST_LIB)
        U64, I64, P = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        lib.synth_key.argtypes = [U64, U64]
        lib.synth_key.restype = U64
        lib.synth_fill_f32.argtypes = [U64, U64, I64, ctypes.c_float, P]
        lib.synth_fill_half.argtypes = [U64, U64, I64, ctypes.c_float, ctypes.c_int, P]
        lib.synth_round_half.argtypes = [P, I64, ctypes.c_int, P]
        _host = lib
    return _host


def _cuda_lib():
    global _cuda
    if _cuda is None:
        if not os.path.exists(_CUDA_LIB):
            raise RuntimeError("synth GPU generator not built: run __graft_entry__.build()")
        lib = ctypes.CDLL(_CUDA_LIB)
        U64, I64, P = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        lib.synth_gpu_fill_f32.argtypes = [U64, U64, I64, ctypes.c_float, P, P]
        lib.synth_gpu_fill_half.argtypes = [U64, U64, I64, ctypes.c_float, ctypes.c_int, P, P]
        lib.synth_gpu_round_half.argtypes = [P, I64, ctypes.c_int, P, P]
        _cuda = lib
    return _cuda


def scale_for(sigma: float) -> float:
    """The binary32 multiplier that gives standard deviation ``sigma``."""
    return float(np.float32(sigma / IRWIN_HALL_SD))


def key(seed: int, stream: int) -> int:
    return int(_host_lib().synth_key(seed & (2 ** 64 - 1), stream & (2 ** 64 - 1)))


def max_abs(sigma: float) -> float:
    """An upper bound on |value| for standard deviation ``sigma`` (before any
    rounding to half precision, which can only move a value to a neighbour)."""
    return SUPPORT_SIGMAS * sigma * 1.0001


# ---------------------------------------------------------------- CPU side

def fill_f32(k: int, first: int, n: int, sigma: float) -> np.ndarray:
    out = np.empty(n, np.float32)
    _host_lib().synth_fill_f32(k, first, n, scale_for(sigma), out.ctypes.data)
    return out


def fill_half(k: int, first: int, n: int, sigma: float, dtype: int) -> np.ndarray:
    out = np.empty(n, np.uint16)
    _host_lib().synth_fill_half(k, first, n, scale_for(sigma), dtype, out.ctypes.data)
    return out


def round_half(x: np.ndarray, dtype: int) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.size, np.uint16)
    _host_lib().synth_round_half(x.ctypes.data, x.size, dtype, out.ctypes.data)
    return out


# ---------------------------------------------------------------- GPU side

def _stream_ptr(stream) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"{what}: CUDA error {rc}")


def gpu_fill_f32(k: int, first: int, out, sigma: float, stream=None) -> None:
    """Fill a contiguous CUDA float32 tensor with elements first .. first+n-1."""
    _check(_cuda_lib().synth_gpu_fill_f32(k, first, out.numel(), scale_for(sigma),
                                          out.data_ptr(), _stream_ptr(stream)), "synth fill f32")


def gpu_fill_half(k: int, first: int, out, sigma: float, dtype: int, stream=None) -> None:
    """Fill a contiguous CUDA 2-byte tensor with half-precision bits."""
    assert out.element_size() == 2
    _check(_cuda_lib().synth_gpu_fill_half(k, first, out.numel(), scale_for(sigma), dtype,
                                           out.data_ptr(), _stream_ptr(stream)), "synth fill half")


def gpu_round_half(x, out, dtype: int, stream=None) -> None:
    assert out.element_size() == 2 and out.numel() == x.numel()
    _check(_cuda_lib().synth_gpu_round_half(x.data_ptr(), x.numel(), dtype, out.data_ptr(),
                                            _stream_ptr(stream)), "synth round half")


def gaps(offsets: Sequence[int], numels: Sequence[int], padded: int) -> Tuple[Tuple[int, int], ...]:
    """The [start, end) ranges of a padded flat vector that no tensor covers."""
    out = []
    pos = 0
    for o, n in zip(offsets, numels):
        if o > pos:
            out.append((pos, o))
        pos = max(pos, o + n)
    if padded > pos:
        out.append((pos, padded))
    return tuple(out)
