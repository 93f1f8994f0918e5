"""zero_grad_norm_noalloc against zero_grad_norm and the oracle, through the
C ABI.

The no-allocation entry point serves callers that cannot hand the library a
workspace: C plugins that only receive device pointers, code whose device
memory belongs to a framework's caching allocator, and loops that cannot
afford cudaMalloc's synchronisation.  It keeps the norm's tree in a static
device array instead, and runs the same kernel over the same tree as
zero_grad_norm, so the two give the same bits.  This file is collected last
so that a failure here comes after every other test has run; it also passes
on its own in a fresh process (the first call does the per-device set-up)."""
import ctypes
import struct

import numpy as np
import pytest
import torch

import oracle
import synth
import zero_partitioned_mixed_step_gb300 as zs
from zs_harness import SUMSQ_RTOL

pytestmark = pytest.mark.gpu


def _bits(x: float) -> bytes:
    return struct.pack("<d", x)


def _norm_with_workspace(g, inv_scale):
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    zs.zero_grad_norm(g, inv_scale, out.data_ptr(), zs.new_workspace())
    torch.cuda.synchronize()
    return float(out.item())


def _norm_noalloc(lib, g, inv_scale):
    out = torch.full((1,), -1.0, dtype=torch.float64, device="cuda")
    rc = lib.zero_grad_norm_noalloc(ctypes.c_void_p(g.data_ptr()), g.numel(), inv_scale,
                                    ctypes.c_void_p(out.data_ptr()),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.zero_strerror(rc)
    torch.cuda.synchronize()
    return float(out.item())


def _oracle_sumsq(g, inv_scale):
    h = g.cpu().numpy().copy()
    oracle.unscale(h, oracle.f32(inv_scale))
    return oracle.sumsq_value(oracle.sumsq(h))


@pytest.mark.parametrize("n", [0, 37, 1_000_003, 8 * 256 * 3000 + 5, 300_000_001])
def test_noalloc_norm_matches_workspace_norm(n):
    lib = zs._abi.lib()
    g = torch.empty(n, dtype=torch.float32, device="cuda")
    synth.gpu_fill_f32(synth.key(4242, n), 0, g, 1e-3)
    for inv_scale in (1.0, 2.0 ** -10):
        ref = _norm_with_workspace(g, inv_scale)
        first = _norm_noalloc(lib, g, inv_scale)
        second = _norm_noalloc(lib, g, inv_scale)  # the array keeps the first call's contents
        assert _bits(first) == _bits(second) == _bits(ref), (n, inv_scale, first, second, ref)
        if n <= 10_000_000:
            want = _oracle_sumsq(g, inv_scale)
            assert abs(first - want) <= SUMSQ_RTOL * want, (n, first, want)
        if n == 0:
            assert _bits(first) == _bits(0.0)


def test_noalloc_norm_after_a_larger_call():
    """A short vector after a long one: the long call's tree leaves nothing
    the short one reads (its counters are back at zero)."""
    lib = zs._abi.lib()
    big = torch.empty(50_000_000, dtype=torch.float32, device="cuda")
    synth.gpu_fill_f32(synth.key(7, 1), 0, big, 1.0)
    small = big[:1000].clone()
    _norm_noalloc(lib, big, 1.0)
    got = _norm_noalloc(lib, small, 1.0)
    ref = _norm_with_workspace(small, 1.0)
    assert _bits(got) == _bits(ref)
    want = _oracle_sumsq(small, 1.0)
    assert abs(got - want) <= SUMSQ_RTOL * want
