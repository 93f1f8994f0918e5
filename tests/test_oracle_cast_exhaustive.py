"""The oracle's binary32 -> binary16 / bfloat16 rounding on every one of the
2^32 binary32 bit patterns, against torch's CPU casts (IEEE round to nearest,
ties to even, overflow to infinity).

The step writes the new master weights into the half-precision parameter
buffer ("DeepSpeed ZeRO", ZeRO Stage 1, "权重更新的触发条件": the fp16 copy is
refreshed from the fp32 weights), so the oracle's rounding decides every
parameter bit the GPU is compared with.  The structured pin in
oracle_pins.py covers the rounding-critical patterns quickly; this test
covers all of them (about a minute on 8 cores)."""
import numpy as np
import pytest
import torch

import oracle

BLOCK = 1 << 26


@pytest.mark.slow
@pytest.mark.parametrize("dt", [oracle.F16, oracle.BF16], ids=["fp16", "bf16"])
def test_cast_every_binary32_pattern(dt):
    tdt = torch.float16 if dt == oracle.F16 else torch.bfloat16
    exp_mask, frac_mask = (0x7C00, 0x3FF) if dt == oracle.F16 else (0x7F80, 0x7F)
    for start in range(0, 1 << 32, BLOCK):
        bits = np.arange(BLOCK, dtype=np.uint32) + np.uint32(start)
        x = bits.view(np.float32)
        got = oracle.f32_to_half(x, dt, openmp=True)
        ref = torch.from_numpy(x).to(tdt).view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(x)
        same = (got == ref) | nan
        if not same.all():
            i = int(np.argmin(same))
            raise AssertionError(f"pattern {int(bits[i]):#010x}: oracle {int(got[i]):#06x}, "
                                 f"torch {int(ref[i]):#06x}")
        g = got[nan]
        assert np.all((g & exp_mask) == exp_mask) and np.all(g & frac_mask), start
