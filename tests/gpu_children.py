"""Programs that GPU tests run in a child process, because the library reads
its test settings (ZERO_TEST_STAGED_WAIT_LIMIT, ZERO_TEST_MAX_CTAS) once per
process.  Usage: python tests/gpu_children.py NAME; prints one JSON line and
exits 0 when the program's own checks pass."""
import hashlib
import json
import os
import struct
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))


def staged_wait():
    """Every mbarrier wait of the staged kernel runs out (the limit and the
    announced extra bytes come from ZERO_TEST_STAGED_WAIT_LIMIT): each step
    records state.error, is skipped with every buffer's current slot
    unchanged bit for bit and the dynamic loss scale backed off, and leaves
    no copy in flight, so the process keeps using the GPU normally."""
    import torch
    import zero_partitioned_mixed_step_gb300 as zs
    from synth.workloads import CFG1
    from zs_harness import Lockstep, gen_grads, to_dev_half
    assert int(os.environ["ZERO_TEST_STAGED_WAIT_LIMIT"]) > 0
    wl = CFG1.replace(numels=(200_001,), world=16, steps=2, inject_at=(), dynamic_scale=True)
    ls = Lockstep(wl)
    before = [t.clone() for t in ls.z.current()]
    S = wl.loss_scale
    for k in range(1, 3):
        grads = gen_grads(wl, ls.lay, k, S)
        ls.z.step([to_dev_half(g, wl.dtype) for g in grads])
        torch.cuda.synchronize()
        st = ls.z.read_state()
        assert (st.error, st.overflow, st.skipped, st.t, st.found_inf) == (1, 1, k, 0, 0), \
            (st.error, st.overflow, st.skipped, st.t, st.found_inf)
        S /= 2
        assert st.loss_scale == S
        for a, b in zip(before, ls.z.current()):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
        off = zs.StepState.error.offset
        ls.z.state[off:off + 4].zero_()  # the caller has handled the error
    x = torch.arange(1 << 20, device="cuda", dtype=torch.int64)
    assert int(x.sum().item()) == (1 << 20) * ((1 << 20) - 1) // 2
    return {"ok": True}


def norm_bits():
    """The clipped step and zero_grad_norm on fixed inputs: the bits of the
    sum of squares and digests of every buffer after two steps."""
    import torch
    import synth
    import zero_partitioned_mixed_step_gb300 as zs
    from gpu_norm_cases import NORM_CASES
    from zs_harness import Lockstep, gen_grads, to_dev_half
    out = {"cap": os.environ.get("ZERO_TEST_MAX_CTAS")}
    for name, (wl, kw) in NORM_CASES.items():
        ls = Lockstep(wl, **kw)
        sums = []
        for s in (1, 2):
            grads = gen_grads(wl, ls.lay, s, ls.st.loss_scale)
            ls.z.step([to_dev_half(g, wl.dtype) for g in grads])
            torch.cuda.synchronize()
            sums.append(struct.pack("<d", ls.z.read_state().sumsq).hex())
        h = hashlib.sha256()
        for t in ls.z.current():
            h.update(t.detach().cpu().contiguous().view(torch.uint8).numpy().tobytes())
        g = torch.empty(3_000_005, dtype=torch.float32, device="cuda")
        synth.gpu_fill_f32(synth.key(99, 3), 0, g, 0.5)
        o = torch.zeros(1, dtype=torch.float64, device="cuda")
        zs.zero_grad_norm(g, 0.25, o.data_ptr(), zs.new_workspace())
        out[name] = {"sumsq": sums, "digest": h.hexdigest(),
                     "norm": struct.pack("<d", float(o.item())).hex()}
    return out


def small_steps():
    """One-pass steps over 2 and 4 ranks (the instances that get a lead CTA
    when their units fit in one wave), four steps each with the learning rate
    changed every step and an Inf in step 2: digests of every buffer and of
    the 64 bytes of state proper, and whether the scalar cache was written."""
    import torch
    from synth.workloads import BF16, CFG1
    from zs_harness import Lockstep, gen_grads, state_proper, to_dev_half
    cases = {
        "nd2-fp16": CFG1.replace(numels=(300_001,), steps=4, inject_at=((2, 0, 150_000),)),
        "nd4-bf16": CFG1.replace(numels=(200_003, 77), world=4, dtype=BF16, steps=4,
                                 inject_at=((2, 3, 100_000),)),
    }
    out = {"cap": os.environ.get("ZERO_TEST_MAX_CTAS")}
    for name, wl in cases.items():
        ls = Lockstep(wl)
        for s, lr in zip(range(1, wl.steps + 1), (2e-4, 6e-4, 1e-3, 5e-4)):
            ls.ocfg.lr = lr
            ls.z.cfg.lr = lr
            ls.step(gen_grads(wl, ls.lay, s, ls.st.loss_scale))
            ls.check()
        h = hashlib.sha256()
        for t in ls.z.current():
            h.update(t.detach().cpu().contiguous().view(torch.uint8).numpy().tobytes())
        st = ls.z.read_state()
        h.update(state_proper(st))
        out[name] = {"digest": h.hexdigest(), "cache_written": any(st.scalar_cache)}
    return out


if __name__ == "__main__":
    result = {"staged_wait": staged_wait, "norm_bits": norm_bits,
              "small_steps": small_steps}[sys.argv[1]]()
    print(json.dumps(result))
