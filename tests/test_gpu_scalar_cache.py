"""The step state's scalar cache: the bias-correction scalars of the next step
(lr / (1 - beta1^t), sqrt(1 - beta2^t), each binary64 rounded once to
binary32, as the per-element update of "DeepSpeed ZeRO", 以 AdaW 为例 uses
them) formed ahead by the step before and keyed on every input of their
formula.

  * after every kind of step the entry the next step reads holds exactly the
    oracle's scalars for that step, with their inputs as keys;
  * a learning rate that changes every step, betas changed mid-run, a
    skipped step and caches zeroed, swapped or left over from an earlier
    step all give the oracle's results and the same bits as an untouched
    run (a key that does not match makes the step form its scalars)."""
import json
import os
import struct
import subprocess
import sys

import pytest
import torch

import oracle
from synth.workloads import BF16, CFG1, CFG2, CFG3
import zero_partitioned_mixed_step_gb300 as zs
from zs_harness import Lockstep, gen_grads, state_proper

pytestmark = pytest.mark.gpu

TAG = 0x5A530C01
CACHE_OFF = zs.StepState.scalar_cache.offset


def _entries(st: zs.StepState):
    raw = bytes(st)[CACHE_OFF:CACHE_OFF + 128]
    out = []
    for k in range(2):
        lr, b1, b2, p1, p2, step, rbc2, tag = struct.unpack_from("<5d2fI", raw, 64 * k)
        out.append(dict(lr=lr, beta1=b1, beta2=b2, p1=p1, p2=p2, step=step, rbc2=rbc2, tag=tag))
    return out


def _f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


CASES = {
    # register kernel with the early loads and a lead CTA (2 ranks), Inf in step 2
    "flat-nd2": (CFG1.replace(numels=(300_001,), steps=4, inject_at=((2, 0, 150_000),)), {}),
    # the same with 4 ranks, bf16
    "flat-nd4-bf16": (CFG1.replace(numels=(200_003, 77), world=4, dtype=BF16, steps=4,
                                   inject_at=((3, 2, 100_000),)), {}),
    # staged kernel (16 ranks), dynamic loss scale, Inf in step 3
    "flat-nd16": (CFG3.replace(numels=(1_000_003,), steps=4, inject_every=0,
                               inject_at=((3, 5, 77_777),)), {}),
    # two passes with the fp32 stage, clip on
    "clip-nd8-staged": (CFG2.replace(numels=(400_000, 3_001), steps=4, inject_at=((2, 1, 9),)),
                        {"stage": True}),
}


# Steps whose kernel forms the next step's scalars: the small one-pass steps
# over at most 4 ranks (a lead CTA) and the staged kernel (its last CTA).
# The others leave the cache as it is.
@pytest.mark.parametrize("name", ["flat-nd2", "flat-nd4-bf16", "flat-nd16"])
def test_entry_holds_the_next_steps_scalars(name):
    wl, kw = CASES[name]
    ls = Lockstep(wl, **kw)
    for s in range(1, wl.steps + 1):
        ls.step()
        st = ls.check()
        e = _entries(st)[st.cur]
        want = oracle.step_scalars(ls.ocfg, ls.st)  # the scalars of step t + 1
        assert e["tag"] == TAG, s
        assert (e["lr"], e["beta1"], e["beta2"]) == (ls.ocfg.lr, ls.ocfg.beta1, ls.ocfg.beta2)
        assert (e["p1"], e["p2"]) == (ls.st.bp1, ls.st.bp2) == (st.beta1_pow, st.beta2_pow)
        assert _f32_bits(e["step"]) == _f32_bits(want.step), (s, e["step"], want.step)
        assert _f32_bits(e["rbc2"]) == _f32_bits(want.rbc2), (s, e["rbc2"], want.rbc2)
    assert ls.st.skipped == 1


def _set_cfg(ls, **kw):
    for k, v in kw.items():
        setattr(ls.ocfg, k, v)
        setattr(ls.z.cfg, k, v)


def _poke_cache(ls, how, saved):
    off = CACHE_OFF
    cache = ls.z.state[off:off + 128]
    if how == "zero":
        cache.zero_()
    elif how == "swap":
        a, b = cache[:64].clone(), cache[64:].clone()
        cache[:64].copy_(b)
        cache[64:].copy_(a)
    elif how == "stale" and saved is not None:
        cache.copy_(saved)


@pytest.mark.parametrize("name", list(CASES))
def test_schedules_and_rewritten_caches_match_the_oracle(name):
    """lr changes every step (warm-up then decay), beta1 and beta2 change
    before step 4, one step is skipped; one run keeps its cache, the other
    has it zeroed, swapped or replaced by an older copy before each step.
    Both follow the oracle, and their buffers and states agree bit for bit."""
    wl, kw = CASES[name]
    wl = wl.replace(steps=6)
    keep, poke = Lockstep(wl, **kw), Lockstep(wl, **kw)
    lrs = [2e-4, 6e-4, 1e-3, 1e-3, 7e-4, 3e-4]
    hows = ["zero", "swap", "stale", "none", "stale", "swap"]
    saved = None
    for s in range(1, wl.steps + 1):
        for ls in (keep, poke):
            _set_cfg(ls, lr=lrs[s - 1])
            if s == 4:
                _set_cfg(ls, beta1=0.85, beta2=0.995)
        _poke_cache(poke, hows[s - 1], saved)
        saved = poke.z.state[CACHE_OFF:CACHE_OFF + 128].clone()
        grads = gen_grads(wl, keep.lay, s, keep.st.loss_scale)
        keep.step(grads)
        poke.step(grads)
        a, b = keep.check(), poke.check()
        assert state_proper(a) == state_proper(b), s
        for x, y in zip(keep.z.current(), poke.z.current()):
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), s
    assert keep.st.skipped == 1 and keep.st.t == wl.steps - 1



def _child(name, **env):
    e = dict(os.environ)
    e.pop("ZERO_TEST_MAX_CTAS", None)
    e.update(env)
    here = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, os.path.join(here, "gpu_children.py"), name],
                       capture_output=True, text=True, env=e, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_small_steps_give_the_same_bits_with_and_without_a_lead_cta():
    """The small one-pass steps with their lead CTA (every unit in one wave,
    the next step's scalars formed alongside) and the same steps with every
    grid capped at 7 CTAs (grid-stride, no lead CTA, scalars formed in every
    CTA's prologue) follow the oracle and give the same buffers and state."""
    lead = _child("small_steps")
    capped = _child("small_steps", ZERO_TEST_MAX_CTAS="7")
    assert lead.pop("cap") is None and capped.pop("cap") == "7"
    for name in lead:
        assert lead[name]["digest"] == capped[name]["digest"], name
        assert lead[name]["cache_written"] and not capped[name]["cache_written"], name
