"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
what the pages or the mathematics fix: closed forms, special cases that reduce
to a textbook or library routine (torch's IEEE casts, torch.optim.Adam/AdamW),
invariants (per-element independence, skip invariance) and brute force on tiny
inputs.  ``test_oracle_pins.py`` runs them against the oracle;
``test_oracle_mutations.py`` runs them against copies of the oracle with a
planted mistake and requires that at least one pin fails for every mistake.
"""
from __future__ import annotations

import math
import random
from decimal import ROUND_HALF_UP, Decimal
from fractions import Fraction

import numpy as np
import torch

import oracle
from oracle import memory

U32 = 2.0 ** -24  # unit roundoff of binary32


def _np_half_to_torch(h: np.ndarray, dtype: int) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(h, np.uint16).view(np.int16))
    return t.view(torch.float16 if dtype == oracle.F16 else torch.bfloat16)


# ----------------------------------------------------------------- memory

def pin_memory_closed_forms():
    """The pages print 120 / 31.4 / 16.6 / 1.9 (also 1.88) GB for Psi = 7.5e9,
    N_d = 64, K = 12, and 24 GB for Psi = 1.5e9 (decimal GB).  The values come
    from tests/golden/memory_table.txt."""
    from golden_io import read_table
    for row in read_table("memory_table.txt"):
        psi, nd, stage, printed, digits = (int(row[0]), int(row[1]), row[2], float(row[3]),
                                            int(row[4]))
        fn = {"dp": lambda p, n: memory.plain_dp(p), "zero1": memory.zero1,
              "zero2": memory.zero2, "zero3": memory.zero3}[stage]
        gb = Decimal(fn(psi, nd).numerator) / Decimal(fn(psi, nd).denominator) / Decimal(10 ** 9)
        shown = gb.quantize(Decimal(1).scaleb(-digits), rounding=ROUND_HALF_UP)
        assert shown == Decimal(row[3]), (stage, psi, nd, gb, printed)


# ----------------------------------------------------------------- conversions

def pin_decode_exhaustive():
    """Every binary16 and bfloat16 bit pattern decodes as torch decodes it."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dt in (oracle.F16, oracle.BF16):
        got = oracle.half_to_f32(bits, dt)
        ref = _np_half_to_torch(bits, dt).float().numpy()
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan), dt
        assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32)), dt


def _encode_cases() -> np.ndarray:
    rng = np.random.default_rng(12345)
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x3000, 0x5000, 0x7FFF,
                     0x8000, 0x8001, 0xFFFF], np.uint32)
    parts = [(hi[:, None] | lows[None, :]).ravel(),
             (hi[:, None] | rng.integers(0, 1 << 16, (1 << 16, 4), dtype=np.uint32)).ravel()]
    # binary16 subnormal results: for every fp32 exponent whose values land in
    # the subnormal range, significands exactly at, just below and just above
    # the rounding tie of that exponent (both parities of the kept bit occur
    # among the random upper bits).
    for ex in range(98, 114):
        shift = 126 - ex  # bits of the 24-bit significand that are dropped
        m = rng.integers(0, 1 << 23, 3000, dtype=np.uint32)
        if shift <= 23:
            low = np.uint32((1 << shift) - 1)
            tie = 1 << (shift - 1)
            cands = [(m & ~low) | np.uint32(d) for d in (tie - 1, tie, tie + 1)]
        else:
            cands = [m, np.zeros(1, np.uint32), np.ones(1, np.uint32)]
        for c in cands:
            for sign in (0, 1):
                parts.append(np.uint32(sign << 31) | np.uint32(ex << 23) | (c & np.uint32(0x7FFFFF)))
    parts.append(rng.integers(0, 1 << 32, 1 << 24, dtype=np.uint64).astype(np.uint32))
    return np.concatenate(parts).view(np.float32)


def pin_encode_structured():
    """binary32 -> binary16 / bfloat16 round-to-nearest-even agrees with
    torch's IEEE casts on every sign/exponent/upper-fraction pattern combined
    with the rounding-critical low bits, on ties at every subnormal shift, and
    on 16M random patterns."""
    x = _encode_cases()
    for dt, tdt in ((oracle.F16, torch.float16), (oracle.BF16, torch.bfloat16)):
        got = oracle.f32_to_half(x, dt, openmp=True)
        ref = torch.from_numpy(x).to(tdt).view(torch.int16).numpy().view(np.uint16)
        isn = np.isnan(x)
        assert np.array_equal(got[~isn], ref[~isn]), dt
        exp_mask, frac_mask = (0x7C00, 0x3FF) if dt == oracle.F16 else (0x7F80, 0x7F)
        assert np.all((got[isn] & exp_mask) == exp_mask) and np.all(got[isn] & frac_mask), dt


# ----------------------------------------------------------------- reduce, unscale, flag

def pin_reduce_bruteforce():
    """Reduce-scatter: rank r's slice is the element-wise sum of every rank's
    gradient over that slice.  With values on a coarse grid the binary32 sum
    is exact in any order, so it must equal the exact rational sum."""
    rnd = random.Random(7)
    for world in (1, 2, 3, 4):
        for psi in (1, 7, 64, 65):
            for dt in (oracle.F16, oracle.BF16):
                lay = oracle.layout([psi], world, align=8)
                vals = [[rnd.randint(-100, 100) * 2.0 ** rnd.randint(-12, -4) for _ in range(lay.padded)]
                        for _ in range(world)]
                for q in range(world):
                    for j in range(psi, lay.padded):
                        vals[q][j] = 0.0
                tdt = torch.float16 if dt == oracle.F16 else torch.bfloat16
                grads = [torch.tensor(v, dtype=tdt).view(torch.int16).numpy().view(np.uint16).copy()
                         for v in vals]
                exact = [[Fraction(float(x)) for x in torch.tensor(v, dtype=tdt).double().tolist()]
                         for v in vals]
                for r in range(world):
                    (fs, ln), = lay.segments[r]
                    g = oracle.reduce_sum(grads, dt, fs, ln)
                    for j in range(ln):
                        want = sum(exact[q][fs + j] for q in range(world))
                        assert Fraction(float(g[j])) == want, (world, psi, r, j)


def pin_reduce_order():
    """The sum runs in ascending rank order from +0: with 2^24, 1, -2^24 (in
    rank order) binary32 gives 0 (1 is absorbed), while the reverse order
    gives 1; and -0 + -0 gives +0 because the sum starts from +0."""
    big = np.float32(2.0 ** 24)
    g1 = [torch.tensor([float(big)], dtype=torch.float32).to(torch.bfloat16),
          torch.tensor([1.0]).to(torch.bfloat16), torch.tensor([-float(big)]).to(torch.bfloat16)]
    grads = [t.view(torch.int16).numpy().view(np.uint16).copy() for t in g1]
    assert oracle.reduce_sum(grads, oracle.BF16, 0, 1)[0] == 0.0
    assert oracle.reduce_sum(grads[::-1], oracle.BF16, 0, 1)[0] == 1.0
    negz = np.array([0x8000], np.uint16)
    z = oracle.reduce_sum([negz, negz], oracle.F16, 0, 1)
    assert z.view(np.uint32)[0] == 0


def pin_unscale_exact():
    """Multiplying by 1/S for a power of two S is exact (no underflow here)."""
    rng = np.random.default_rng(3)
    g = rng.standard_normal(4096).astype(np.float32)
    for e in (0, 1, 10, 12, 16):
        h = g.copy()
        oracle.unscale(h, oracle.f32(2.0 ** -e))
        assert np.array_equal(h.astype(np.float64), g.astype(np.float64) / 2.0 ** e)


def pin_overflow_detect():
    """The flag is set by any NaN, +Inf or -Inf, wherever it sits, and never
    by finite values, including the largest finite binary32."""
    g = np.linspace(-1, 1, 1001).astype(np.float32)
    g[3] = np.finfo(np.float32).max
    g[4] = -np.finfo(np.float32).max
    g[5] = np.float32(1e-45)
    assert not oracle.any_nonfinite(g)
    for pos in (0, 500, 1000):
        for bad in (np.inf, -np.inf, np.nan):
            h = g.copy()
            h[pos] = bad
            assert oracle.any_nonfinite(h), (pos, bad)


# ----------------------------------------------------------------- norm and clip

def pin_sumsq():
    """Constant input a: sum of squares n a^2 (exact for a power of two); and
    on random input (sums of 8 bf16 values, the shape of the reduced
    gradients) within 2 ulp of the exactly rounded sum (math.fsum of the exact
    squares), where a plain sequential binary64 sum is already off by ~1e-13;
    chaining over pieces continues the same sum."""
    for a, n in ((0.5, 1000), (2.0 ** -7, 4096), (3.0, 17)):
        g = np.full(n, a, np.float32)
        assert oracle.sumsq_value(oracle.sumsq(g)) == n * a * a
    rng = np.random.default_rng(11)
    g = np.zeros(200_000, np.float32)
    for _ in range(8):
        g += torch.from_numpy((rng.standard_normal(g.size) * 1e-3).astype(np.float32)).to(
            torch.bfloat16).float().numpy()
    exact = math.fsum(float(x) * float(x) for x in g)
    got = oracle.sumsq_value(oracle.sumsq(g))
    assert abs(got - exact) <= 2 * 2.0 ** -52 * exact, (got - exact) / exact
    assert oracle.sumsq(g[777:], oracle.sumsq(g[:777])) == oracle.sumsq(g)


def pin_clip_coef():
    """c = min(1, max_norm / (||g|| + 1e-6)): 1 below the threshold, and
    max_norm / ||g|| (to binary32) above it."""
    assert oracle.clip_coef(0.25, 1.0) == 1.0
    assert oracle.clip_coef(1e-12, 1.0) == 1.0
    c = oracle.clip_coef(100.0, 1.0)
    assert abs(c - 0.1) <= 0.1 * 2e-7
    c = oracle.clip_coef(4e12, 2.0)           # ||g|| = 2e6: the 1e-6 term is negligible
    assert abs(c - 1e-6) <= 1e-6 * 2e-7
    c = oracle.clip_coef(1e-12, 1e-6)         # ||g|| = 1e-6: c = 1e-6 / (1e-6 + 1e-6)
    assert abs(c - 0.5) <= 0.5 * 2e-7


# ----------------------------------------------------------------- Adam closed forms

def _single_rank_step(g_f32: np.ndarray, w, m, v, cfg, st, dtype=oracle.F16):
    """Run the oracle's full step with one rank whose half gradient holds
    exactly g_f32 (which must be representable), loss scale st.loss_scale."""
    n = g_f32.size
    lay = oracle.layout([n], 1, align=1)
    tdt = torch.float16 if dtype == oracle.F16 else torch.bfloat16
    gh = torch.from_numpy(g_f32 * np.float32(st.loss_scale)).to(tdt)
    assert torch.equal(gh.float(), torch.from_numpy(g_f32 * np.float32(st.loss_scale)))
    grads = [gh.view(torch.int16).numpy().view(np.uint16).copy()]
    half = np.zeros(lay.padded, np.uint16)
    oracle.step(grads, dtype, lay, cfg, st, w, m, v, half)
    return half


def _representable_grads(n, seed, lo=-12, hi=-4):
    rnd = random.Random(seed)
    vals = [rnd.choice([-1, 1]) * rnd.randint(1, 1000) * 2.0 ** rnd.randint(lo - 10, hi - 10)
            for _ in range(n)]
    return torch.tensor(vals).to(torch.float16).float().numpy()


def pin_adam_first_step():
    """From zero moments, the bias-corrected first step is
    w1 = w0 (1 - lr wd) - lr g / (|g| + eps)  (m_hat = g, v_hat = g^2),
    including |g| comparable to eps, and for AdamW the decay is decoupled."""
    g = _representable_grads(256, 1)
    g[:8] = np.array([1e-8, -2e-8, 3e-9, 5e-7, -1e-7, 6e-8, 0.0, -0.0], np.float32)
    g = torch.from_numpy(g).to(torch.bfloat16).float().numpy()  # exact in bfloat16
    for wd, adamw in ((0.0, True), (0.01, True), (0.1, True)):
        cfg = oracle.AdamCfg(lr=1e-3, weight_decay=wd, adamw=adamw, eps=1e-8)
        w0 = np.linspace(-0.05, 0.05, g.size).astype(np.float32)
        w, m, v = w0.copy(), np.zeros_like(w0), np.zeros_like(w0)
        _single_rank_step(g, w, m, v, cfg, oracle.State(loss_scale=1.0), oracle.BF16)
        gd = g.astype(np.float64)
        want = w0.astype(np.float64) * (1 - 1e-3 * wd) - 1e-3 * gd / (np.abs(gd) + 1e-8)
        err = np.abs(w - want)
        assert np.all(err <= 4 * U32 * (np.abs(want) + 1e-3)), float(err.max())


def pin_adam_constant_grad():
    """Constant gradient g for T steps: the bias-corrected m_hat = g and
    v_hat = g^2 at every t, so each step moves w by lr g / (|g| + eps) after
    the decoupled decay: w_T = w0 d^T - lr g/(|g|+eps) sum_{k<T} d^k."""
    g = _representable_grads(64, 2)
    cfg = oracle.AdamCfg(lr=1e-3, weight_decay=0.01, eps=1e-8)
    d = 1 - 1e-3 * 0.01
    w0 = np.linspace(-0.1, 0.1, g.size).astype(np.float32)
    w, m, v = w0.copy(), np.zeros_like(w0), np.zeros_like(w0)
    st = oracle.State()
    T = 6
    for _ in range(T):
        _single_rank_step(g, w, m, v, cfg, st)
    gd = g.astype(np.float64)
    want = w0 * d ** T - 1e-3 * gd / (np.abs(gd) + 1e-8) * sum(d ** k for k in range(T))
    assert np.all(np.abs(w - want) <= 40 * U32 * (np.abs(want) + 1e-3)), float(np.abs(w - want).max())
    assert st.t == T


def pin_adam_literal_form():
    """Without bias correction (the formula exactly as the page prints it),
    the first step from zero moments is
    w1 = w0 - lr (1 - b1) g / (sqrt(1 - b2) |g| + eps)."""
    g = _representable_grads(64, 3)
    cfg = oracle.AdamCfg(lr=1e-3, weight_decay=0.0, eps=1e-8, bias_correction=False)
    w0 = np.linspace(-0.1, 0.1, g.size).astype(np.float32)
    w, m, v = w0.copy(), np.zeros_like(w0), np.zeros_like(w0)
    _single_rank_step(g, w, m, v, cfg, oracle.State())
    gd = g.astype(np.float64)
    want = w0 - 1e-3 * 0.1 * gd / (math.sqrt(0.001) * np.abs(gd) + 1e-8)
    assert np.all(np.abs(w - want) <= 8 * U32 * (np.abs(want) + 1e-3))


def _ulp32(x: Fraction) -> Fraction:
    """The binary32 spacing at positive x (normal range)."""
    _, e = math.frexp(float(x))
    return Fraction(2) ** (e - 24)


def pin_step_scalars():
    """The per-step scalars of step t (after t - 1 committed steps) against
    exact rational arithmetic: step = lr / (1 - beta1^t) and
    rbc2 = sqrt(1 - beta2^t), each within one binary32 ulp of the exact value
    (the running binary64 products of the betas stay within about t 2^-53 of
    beta^t, far inside half a binary32 ulp), over 60 committed steps; a
    skipped step changes neither; without bias correction step = lr and
    rbc2 = 1.  ("DeepSpeed ZeRO", 以 AdaW 为例, with the bias correction the
    textbook update adds.)"""
    for lr, b1, b2 in ((1e-3, 0.9, 0.999), (3e-4, 0.85, 0.995), (2.0 ** -10, 0.5, 0.75)):
        cfg = oracle.AdamCfg(lr=lr, beta1=b1, beta2=b2)
        st = oracle.State()
        for t in range(1, 61):
            sc = oracle.step_scalars(cfg, st)
            want = Fraction(lr) / (1 - Fraction(b1) ** t)
            assert abs(Fraction(sc.step) - want) <= _ulp32(want), (lr, t, sc.step)
            y = 1 - Fraction(b2) ** t
            r, u = Fraction(sc.rbc2), _ulp32(Fraction(sc.rbc2))
            assert (r - u) ** 2 <= y <= (r + u) ** 2, (b2, t, sc.rbc2)
            if t % 7 == 0:  # an overflow step in between changes nothing
                oracle.skip(cfg, st)
                assert bytes(oracle.step_scalars(cfg, st)) == bytes(sc)
            oracle.commit(cfg, st)
        assert st.t == 60
    cfg = oracle.AdamCfg(lr=1e-3, bias_correction=False)
    st = oracle.State(t=5, bp1=0.9 ** 5, bp2=0.999 ** 5)
    sc = oracle.step_scalars(cfg, st)
    assert sc.step == np.float32(1e-3) and sc.rbc2 == 1.0


def _torch_reference(g_list, w0, cfg, cls):
    p = torch.nn.Parameter(torch.from_numpy(w0.astype(np.float64)))
    opt = cls([p], lr=cfg.lr, betas=(cfg.beta1, cfg.beta2), eps=cfg.eps,
              weight_decay=cfg.weight_decay, foreach=False)
    for g in g_list:
        p.grad = torch.from_numpy(g.astype(np.float64))
        opt.step()
    s = opt.state[p]
    return p.detach().numpy(), s["exp_avg"].numpy(), s["exp_avg_sq"].numpy()


def pin_vs_torch():
    """With N_d = 1 the step is single-device Adam: AdamW against
    torch.optim.AdamW and coupled-L2 Adam against torch.optim.Adam, both run
    in binary64, over 8 steps with a changing gradient.  The tolerance is a
    few binary32 roundings of each term."""
    n = 512
    for adamw, wd, cls in ((True, 0.01, torch.optim.AdamW), (False, 0.0, torch.optim.Adam),
                           (False, 0.05, torch.optim.Adam)):
        cfg = oracle.AdamCfg(lr=1e-3, weight_decay=wd, adamw=adamw)
        w0 = np.random.default_rng(5).normal(0, 0.02, n).astype(np.float32)
        w, m, v = w0.copy(), np.zeros_like(w0), np.zeros_like(w0)
        st = oracle.State(loss_scale=1024.0)
        gs = []
        for s in range(8):
            g = _representable_grads(n, 100 + s)
            gs.append(g)
            _single_rank_step(g, w, m, v, cfg, st)
        wr, mr, vr = _torch_reference(gs, w0, cfg, cls)
        gmax = max(float(np.abs(g).max()) for g in gs)
        assert np.all(np.abs(m - mr) <= 16 * U32 * gmax), float(np.abs(m - mr).max())
        assert np.all(np.abs(v - vr) <= 16 * U32 * gmax * gmax)
        tol = 8 * U32 * np.abs(wr) + 8 * 16 * U32 * cfg.lr * 10
        assert np.all(np.abs(w - wr) <= tol), float((np.abs(w - wr) / tol).max())


# ----------------------------------------------------------------- partitioning and skip

def _random_problem(world, numels, dtype, seed, align=64, bucket=0, scale=1024.0):
    lay = oracle.layout(numels, world, align=align, bucket=bucket)
    rng = np.random.default_rng(seed)
    tdt = torch.float16 if dtype == oracle.F16 else torch.bfloat16
    grads = []
    for _ in range(world):
        g = (rng.standard_normal(lay.padded) * 1e-3 * scale).astype(np.float32)
        mask = np.zeros(lay.padded, bool)
        for o, n in zip(lay.offsets, lay.numels):
            mask[o:o + n] = True
        g[~mask] = 0
        grads.append(torch.from_numpy(g).to(tdt).view(torch.int16).numpy().view(np.uint16).copy())
    master = rng.normal(0, 0.02, lay.padded).astype(np.float32)
    master[~mask] = 0
    return lay, grads, master


def pin_partition_concat():
    """Per-element independence ("DeepSpeed ZeRO", ZeRO Stage 2 derivation):
    updating every partition on its own and concatenating gives, bit for bit,
    the all-ranks step and the unpartitioned update of the whole vector."""
    for world, numels, bucket, dt in ((4, (1000, 333, 2048), 0, oracle.F16),
                                      (3, (5000, 77), 1536, oracle.BF16),
                                      (2, (4096,), 0, oracle.BF16)):
        lay, grads, master0 = _random_problem(world, numels, dt, world, bucket=bucket)
        cfg = oracle.AdamCfg(weight_decay=0.01)
        # all ranks at once
        w, m, v = master0.copy(), np.zeros_like(master0), np.zeros_like(master0)
        half = np.zeros(lay.padded, np.uint16)
        st = oracle.State(loss_scale=1024.0)
        for _ in range(2):
            oracle.step(grads, dt, lay, cfg, st, w, m, v, half)
        # each rank alone, state in rank-local order
        half_r = np.zeros(lay.padded, np.uint16)
        for r in range(world):
            idx = np.concatenate([np.arange(fs, fs + ln) for fs, ln in lay.segments[r]])
            wr, mr, vr = master0[idx].copy(), np.zeros(idx.size, np.float32), np.zeros(idx.size, np.float32)
            str_ = oracle.State(loss_scale=1024.0)
            for _ in range(2):
                oracle.step(grads, dt, lay, cfg, str_, wr, mr, vr, half_r, rank=r)
            assert np.array_equal(wr.view(np.uint32), w[idx].view(np.uint32))
            assert np.array_equal(mr.view(np.uint32), m[idx].view(np.uint32))
            assert np.array_equal(vr.view(np.uint32), v[idx].view(np.uint32))
            sl = [g[idx].copy() for g in grads]
            wr2, mr2, vr2 = master0[idx].copy(), np.zeros(idx.size, np.float32), np.zeros(idx.size, np.float32)
            st2 = oracle.State(loss_scale=1024.0)
            h2 = np.zeros(lay.padded, np.uint16)
            for _ in range(2):
                oracle.step(sl, dt, lay, cfg, st2, wr2, mr2, vr2, h2, rank=r, grads_are_slices=True)
            assert np.array_equal(wr2.view(np.uint32), wr.view(np.uint32))
        assert np.array_equal(half_r, half)
        # the unpartitioned update of the whole vector
        wu, mu, vu = master0.copy(), np.zeros_like(master0), np.zeros_like(master0)
        stu = oracle.State(loss_scale=1024.0)
        for _ in range(2):
            g = oracle.reduce_sum(grads, dt, 0, lay.padded)
            oracle.unscale(g, oracle.f32(1.0 / stu.loss_scale))
            oracle.adam(g, wu, mu, vu, oracle.step_scalars(cfg, stu))
            oracle.commit(cfg, stu)
        assert np.array_equal(wu.view(np.uint32), w.view(np.uint32))
        assert np.array_equal(oracle.f32_to_half(wu, dt), half)


def pin_skip_invariance():
    """"DeepSpeed ZeRO", ZeRO Stage 1, "权重更新的触发条件": a step whose
    gradients hold NaN/Inf leaves master, moments, half parameters and t
    unchanged (bit for bit); only the dynamic loss scale halves (not below
    min_scale).  The next good step is step t + 1."""
    world = 4
    lay, grads, master0 = _random_problem(world, (3000, 1000), oracle.F16, 9)
    cfg = oracle.AdamCfg(weight_decay=0.01, dynamic_scale=True, min_scale=256.0)
    w, m, v = master0.copy(), np.zeros_like(master0), np.zeros_like(master0)
    half = np.zeros(lay.padded, np.uint16)
    st = oracle.State(loss_scale=1024.0)
    oracle.step(grads, oracle.F16, lay, cfg, st, w, m, v, half)
    P = lay.owned
    last_real = lay.offsets[-1] + lay.numels[-1] - 1
    for rank, idx, bits in ((0, 0, 0x7C00), (1, P - 1, 0xFC00), (2, P, 0x7E00),
                            (3, last_real, 0x7C00), (3, lay.padded - 1, 0x7C01)):
        bad = [g.copy() for g in grads]
        bad[rank][idx] = bits
        before = (w.copy(), m.copy(), v.copy(), half.copy(), st.t, st.bp1, st.bp2)
        s0 = st.loss_scale
        oracle.step(bad, oracle.F16, lay, cfg, st, w, m, v, half)
        for a, b in zip(before[:4], (w, m, v, half)):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), (rank, idx)
        assert (st.t, st.bp1, st.bp2) == before[4:]
        assert st.overflow == 1
        assert st.loss_scale == max(s0 * 0.5, 256.0)
    assert st.loss_scale == 256.0
    # after the skips the next good step equals a fresh run's second step
    w2, m2, v2 = master0.copy(), np.zeros_like(master0), np.zeros_like(master0)
    h2 = np.zeros(lay.padded, np.uint16)
    st2 = oracle.State(loss_scale=1024.0)
    oracle.step(grads, oracle.F16, lay, cfg, st2, w2, m2, v2, h2)
    st2.loss_scale = 256.0
    g256 = [(torch.from_numpy(g.view(np.int16)).view(torch.float16).float() / 4)
            .to(torch.float16).view(torch.int16).numpy().view(np.uint16) for g in grads]
    oracle.step(g256, oracle.F16, lay, cfg, st, w, m, v, half)
    oracle.step(g256, oracle.F16, lay, cfg, st2, w2, m2, v2, h2)
    assert st.t == 2 and st2.t == 2
    assert np.array_equal(w.view(np.uint32), w2.view(np.uint32))


def pin_loss_scale_growth():
    """Dynamic scale doubles after growth_interval good steps in a row, and
    the count restarts after an overflow."""
    lay, grads, master0 = _random_problem(2, (256,), oracle.F16, 4)
    cfg = oracle.AdamCfg(dynamic_scale=True, growth_interval=3)
    w, m, v = master0.copy(), np.zeros_like(master0), np.zeros_like(master0)
    half = np.zeros(lay.padded, np.uint16)
    st = oracle.State(loss_scale=1024.0)
    scales = []
    for s in range(8):
        gs = grads
        if s == 4:
            gs = [g.copy() for g in grads]
            gs[1][3] = 0x7C00
        oracle.step(gs, oracle.F16, lay, cfg, st, w, m, v, half)
        scales.append(st.loss_scale)
    assert scales == [1024, 1024, 2048, 2048, 1024, 1024, 1024, 2048], scales


def pin_clip():
    """With clipping, the first step's moments are m1 = (1 - b1) c g and
    v1 = (1 - b2) (c g)^2 with c = max_norm / ||g||_2, the norm taken over all
    ranks' partitions together."""
    world = 4
    lay, grads, master0 = _random_problem(world, (4000, 100), oracle.BF16, 21, scale=1.0)
    cfg = oracle.AdamCfg(max_grad_norm=0.01)
    w, m, v = master0.copy(), np.zeros_like(master0), np.zeros_like(master0)
    half = np.zeros(lay.padded, np.uint16)
    st = oracle.State()
    oracle.step(grads, oracle.BF16, lay, cfg, st, w, m, v, half)
    full = sum(torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).double() for g in grads).numpy()
    norm = math.sqrt(math.fsum(full * full))
    assert abs(st.sumsq - norm * norm) <= 1e-11 * norm * norm
    c = 0.01 / (norm + 1e-6)
    assert abs(st.coef - c) <= 2 * U32 * c
    assert np.all(np.abs(m - 0.1 * c * full) <= 4 * U32 * np.abs(0.1 * c * full) + 1e-30)
    assert np.all(np.abs(v - 0.001 * (c * full) ** 2) <= 8 * U32 * 0.001 * (c * full) ** 2 + 1e-38)


# ----------------------------------------------------------------- layout

def pin_layout():
    """Special cases and hand-computed sizes: one rank owns the whole
    (aligned) vector; a divisible size needs no padding; partitions cover
    [0, padded) disjointly and start on the alignment; GPT-2 small
    (124,439,808 parameters, all tensor sizes multiples of 64) pads to a
    multiple of 8 * 64; 7.5e9 over 64 ranks is 117,187,500 per rank, padded
    to 117,187,520; the 8B list (8,030,261,248) in 25M buckets is 321 full
    buckets plus 5,261,248 elements."""
    lay = oracle.layout([100], 1)
    assert lay.padded == 128 and lay.segments[0] == ((0, 128),)
    lay = oracle.layout([4096], 4)
    assert lay.padded == 4096 and lay.owned == 1024
    lay = oracle.layout([10, 70, 1], 3, align=64)
    assert lay.offsets == (0, 64, 192)
    assert lay.padded == 384 and lay.owned == 128
    for world, numels, bucket in ((5, (7, 1000, 3), 0), (4, (5000,), 1024), (8, (12345, 6789), 4096)):
        lay = oracle.layout(numels, world, 64, bucket)
        cover = np.zeros(lay.padded, np.int32)
        for r in range(world):
            tot = 0
            for fs, ln in lay.segments[r]:
                cover[fs:fs + ln] += 1
                tot += ln
                assert fs % 8 == 0
            assert tot == lay.owned
        assert np.all(cover == 1)
    from synth.workloads import CFG2, CFG4, CFG5
    lay = oracle.layout(CFG2.numels, 8)
    assert lay.numel == 124_439_808 and lay.flat_end == 124_439_808
    assert lay.padded % 512 == 0 and 0 <= lay.padded - 124_439_808 < 512
    lay = oracle.layout(CFG4.numels, 64)
    assert lay.owned == 117_187_520 and lay.padded == 64 * 117_187_520
    lay = oracle.layout(CFG5.numels, 8, bucket=25_000_000)
    assert lay.numel == 8_030_261_248 and lay.num_buckets == 322
    # the last bucket holds 5,261,248 = 64 * 82,207 elements: padded to the next
    # multiple of 8 * 64 it is 5,261,312, i.e. 657,664 per rank
    assert lay.last_slice == 657_664 and lay.slice == 3_125_000
    assert lay.padded == 321 * 25_000_000 + 5_261_312


# ----------------------------------------------------------------- gradient accumulation

def pin_accumulate_exact():
    """K micro-steps of reduce-scatter into an fp32 accumulator: with values
    on a coarse grid every sum is exact, so the accumulator must equal the
    exact rational sum over micro-steps and ranks (all ranks' partitions and
    one rank's view with slice buffers)."""
    rnd = random.Random(17)
    for world, psi, K in ((3, 200, 3), (4, 65, 5), (1, 8, 2)):
        lay = oracle.layout([psi], world, align=8)
        exact = [Fraction(0)] * lay.padded
        acc = np.zeros(lay.padded, np.float32)
        acc_r = np.zeros(lay.owned, np.float32)
        idx = np.arange(lay.segments[world - 1][0][0], lay.segments[world - 1][0][0] + lay.owned)
        for k in range(K):
            vals = [[rnd.randint(-50, 50) * 2.0 ** rnd.randint(-10, -4) if j < psi else 0.0
                     for j in range(lay.padded)] for _ in range(world)]
            grads = [torch.tensor(v).to(torch.bfloat16).view(torch.int16).numpy()
                     .view(np.uint16).copy() for v in vals]
            for v in vals:
                for j, x in enumerate(v):
                    exact[j] += Fraction(float(torch.tensor(x).to(torch.bfloat16).float()))
            oracle.reduce_scatter_accumulate(grads, oracle.BF16, lay, acc, k > 0)
            oracle.reduce_scatter_accumulate([g[idx].copy() for g in grads], oracle.BF16, lay,
                                             acc_r, k > 0, rank=world - 1, grads_are_slices=True)
        assert all(Fraction(float(acc[j])) == exact[j] for j in range(lay.padded))
        assert np.array_equal(acc_r, acc[idx])


def pin_accumulate_order():
    """A micro-step's ranks are summed first and the sum is added to the
    accumulator once: 2^24 + (1 + 1) = 2^24 + 2 exactly, whereas adding the
    ranks one at a time into the accumulator would lose both ones."""
    lay = oracle.layout([8], 2, align=8)
    acc = np.zeros(lay.padded, np.float32)
    big = [torch.full((lay.padded,), 2.0 ** 24).to(torch.bfloat16), torch.zeros(lay.padded).to(torch.bfloat16)]
    one = [torch.ones(lay.padded).to(torch.bfloat16)] * 2
    for k, gs in enumerate((big, one)):
        grads = [g.view(torch.int16).numpy().view(np.uint16).copy() for g in gs]
        oracle.reduce_scatter_accumulate(grads, oracle.BF16, lay, acc, k > 0)
    assert np.all(acc == np.float32(2.0 ** 24 + 2))


def pin_accumulated_step():
    """One micro-step accumulated and then stepped equals the plain step bit
    for bit (flat, bucketed and one-rank views, with and without the clip); a
    NaN in any micro-step skips the whole step."""
    for world, numels, bucket, rank, clip in ((4, (3000, 100), 0, None, 0.0),
                                               (3, (5000, 77), 1536, None, 0.5),
                                               (4, (4096,), 0, 2, 0.0), (3, (5000, 77), 1536, 1, 0.0)):
        lay, grads, master0 = _random_problem(world, numels, oracle.F16, world + 40, bucket=bucket)
        cfg = oracle.AdamCfg(weight_decay=0.01, max_grad_norm=clip)
        idx = (np.arange(lay.padded) if rank is None else
               np.concatenate([np.arange(fs, fs + ln) for fs, ln in lay.segments[rank]]))
        outs = []
        for accumulated in (False, True):
            w, m, v = master0[idx].copy(), np.zeros(idx.size, np.float32), np.zeros(idx.size, np.float32)
            half = np.zeros(lay.padded, np.uint16)
            st = oracle.State(loss_scale=1024.0)
            for _ in range(2):
                if accumulated:
                    acc = np.zeros(idx.size, np.float32)
                    oracle.reduce_scatter_accumulate(grads, oracle.F16, lay, acc, False, rank=rank)
                    oracle.step_accumulated(acc, oracle.F16, lay, cfg, st, w, m, v, half, rank=rank)
                else:
                    oracle.step(grads, oracle.F16, lay, cfg, st, w, m, v, half, rank=rank)
            outs.append((w, m, v, half, st.t, st.sumsq))
        for a, b in zip(outs[0][:4], outs[1][:4]):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
        assert outs[0][4:] == outs[1][4:]
    lay, grads, master0 = _random_problem(2, (1000,), oracle.F16, 5)
    cfg = oracle.AdamCfg()
    w, m, v = master0.copy(), np.zeros_like(master0), np.zeros_like(master0)
    half = np.zeros(lay.padded, np.uint16)
    st = oracle.State(loss_scale=1024.0)
    acc = np.zeros(lay.padded, np.float32)
    bad = [g.copy() for g in grads]
    bad[1][10] = 0x7E00
    oracle.reduce_scatter_accumulate(bad, oracle.F16, lay, acc, False)
    oracle.reduce_scatter_accumulate(grads, oracle.F16, lay, acc, True)
    before = (w.copy(), m.copy(), v.copy())
    oracle.step_accumulated(acc, oracle.F16, lay, cfg, st, w, m, v, half)
    assert st.overflow == 1 and st.t == 0
    assert all(np.array_equal(a, b) for a, b in zip(before, (w, m, v)))


# ----------------------------------------------------------------- half-precision reduction

def pin_half_reduce():
    """The reduction in the gradient's own half type rounds every partial sum
    to nearest even, in ascending rank order: fp16 against numpy's correctly
    rounded binary64 -> binary16 conversion of each exact partial sum
    (subnormals and overflow included); bf16 on values whose binary32 sums
    are exact, against torch's bf16 rounding; 2048 + 1 + 1 = 2048 in fp16
    (2050 in the reverse order); 60000 + 60000 overflows to Inf in fp16
    although it is finite in binary32."""
    rng = np.random.default_rng(23)
    for world in (1, 2, 3, 5, 8):
        n = 4000
        exps = rng.integers(-24, 16, size=(world, n))
        vals = (rng.integers(-1023, 1024, size=(world, n)) * np.exp2(exps - 10.0)).astype(np.float16)
        grads = [v.view(np.uint16).copy() for v in vals]
        got = oracle.reduce_sum(grads, oracle.F16, 0, n, half_reduce=True)
        acc = np.zeros(n, np.float16)
        for q in range(world):
            acc = (acc.astype(np.float64) + vals[q].astype(np.float64)).astype(np.float16)
        want = acc.astype(np.float32)
        same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
        assert same.all(), world
        # bf16: exponents within a band of 12, so binary32 holds every exact sum
        e = rng.integers(-20, -8, size=(world, n))
        bv = torch.from_numpy((rng.integers(-127, 128, size=(world, n)) * np.exp2(e - 7.0))
                              .astype(np.float32)).to(torch.bfloat16)
        grads = [bv[q].view(torch.int16).numpy().view(np.uint16).copy() for q in range(world)]
        got = oracle.reduce_sum(grads, oracle.BF16, 0, n, half_reduce=True)
        acc = torch.zeros(n, dtype=torch.bfloat16)
        for q in range(world):
            acc = (acc.float() + bv[q].float()).to(torch.bfloat16)
        assert np.array_equal(got.view(np.uint32), acc.float().numpy().view(np.uint32)), world
    order = [np.array([x], np.float16).view(np.uint16) for x in (2048.0, 1.0, 1.0)]
    assert oracle.reduce_sum(order, oracle.F16, 0, 1, half_reduce=True)[0] == 2048.0
    assert oracle.reduce_sum(order[::-1], oracle.F16, 0, 1, half_reduce=True)[0] == 2050.0
    big = [np.array([60000.0], np.float16).view(np.uint16)] * 2
    assert np.isinf(oracle.reduce_sum(big, oracle.F16, 0, 1, half_reduce=True)[0])
    assert oracle.reduce_sum(big, oracle.F16, 0, 1)[0] == 120000.0



# ----------------------------------------------------------------- the windowed path

def _local_of(lay, r, flat):
    local = 0
    for fs, ln in lay.segments[r]:
        if fs <= flat < fs + ln:
            return local + flat - fs
        local += ln
    raise AssertionError("element not owned by the rank")


def _windowed_problems():
    """Small problems for the windowed path, each with its step-by-step
    gradients: (name, layout, dtype, cfg, loss scale, rank, slices,
    half_reduce, master, [grads of step 1, 2, 3])."""
    out = []
    # flat, 16 ranks, fp16 x 4096, dynamic scale; +Inf (rank 5) in step 2
    lay, g1, master = _random_problem(16, (20_003,), oracle.F16, 31, scale=4096.0)
    steps = [g1] + [_random_problem(16, (20_003,), oracle.F16, 31 + s, scale=4096.0)[1]
                    for s in (1, 2)]
    steps[1][5][12_345] = 0x7C00
    out.append(("flat-nd16", lay, oracle.F16,
                oracle.AdamCfg(dynamic_scale=True, max_grad_norm=1e30), 4096.0, None, False,
                False, master, steps))
    # buckets over 3 ranks, bf16, the clip active
    args = (3, (5000, 77, 1200), oracle.BF16)
    lay, g1, master = _random_problem(*args, 41, bucket=1536, scale=1.0)
    steps = [g1] + [_random_problem(*args, 41 + s, bucket=1536, scale=1.0)[1] for s in (1, 2)]
    out.append(("bucketed-clip", lay, oracle.BF16,
                oracle.AdamCfg(weight_decay=0.01, max_grad_norm=0.01), 1.0, None, False, False,
                master, steps))
    # rank 2 of 4 over buckets, gradient buffers holding only rank 2's slices
    args = (4, (4196, 300), oracle.F16)
    lay, g1, master = _random_problem(*args, 51, bucket=4096)
    steps = [g1] + [_random_problem(*args, 51 + s, bucket=4096)[1] for s in (1, 2)]
    idx = np.concatenate([np.arange(fs, fs + ln) for fs, ln in lay.segments[2]])
    steps = [[g[idx].copy() for g in gs] for gs in steps]
    out.append(("rank-view-slices", lay, oracle.F16,
                oracle.AdamCfg(weight_decay=0.01, max_grad_norm=1e30), 1024.0, 2, True, False,
                master[idx].copy(), steps))
    # reduction in bf16, 5 ranks, the clip active
    args = (5, (3000,), oracle.BF16)
    lay, g1, master = _random_problem(*args, 61, scale=1.0)
    steps = [g1] + [_random_problem(*args, 61 + s, scale=1.0)[1] for s in (1, 2)]
    out.append(("half-reduce", lay, oracle.BF16, oracle.AdamCfg(max_grad_norm=0.02), 1.0, None,
                False, True, master, steps))
    # per-rank sums whose binary64 total depends on the rank order: rank 0's
    # sum of squares is 1, ranks 1-3 hold 2^-54 each; in rank order the total
    # is 1, in reverse order 1 + 2^-52
    lay = oracle.layout([256], 4)
    one = torch.tensor([1.0, 2.0 ** -27]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    steps = []
    for _ in range(3):
        g = [np.zeros(lay.padded, np.uint16) for _ in range(4)]
        g[0][0] = one[0]
        for r in (1, 2, 3):
            g[r][r * lay.owned + 3] = one[1]
        steps.append(g)
    out.append(("rank-order", lay, oracle.BF16, oracle.AdamCfg(max_grad_norm=1e30), 1.0, None,
                False, False, np.zeros(lay.padded, np.float32), steps))
    return out


def pin_windowed_matches_step():
    """The full-size parity tests check the GPU against the windowed path:
    ``scan_scalars`` forms the step's overflow flag and sum of squares chunk
    by chunk, and ``window_step`` steps any window of a rank's elements given
    them (the update is element-wise once they are known: "DeepSpeed ZeRO",
    ZeRO Stage 2, the derivation that a rank's optimizer-state shard needs
    only its own gradient slice).  On small problems (16 ranks with an Inf in
    a middle step, buckets with the clip, one rank's view with slice buffers,
    the bf16 reduction, per-rank sums whose total depends on the rank order)
    the flag and the sum of squares equal what ``step`` records, bit for bit,
    and windows that tile every simulated element reproduce master, m, v and
    the half parameters of ``step`` bit for bit over three steps."""
    for (name, lay, dt, cfg, S, rank, slices, hr, master, steps) in _windowed_problems():
        ranks = list(range(lay.world)) if rank is None else [rank]
        n = master.size
        ref = [master.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32),
               np.zeros(lay.padded, np.uint16)]
        win = [master.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32),
               np.zeros(lay.padded, np.uint16)]
        st_ref = oracle.State(loss_scale=S)
        st_win = oracle.State(loss_scale=S)
        lengths = (997, 64, 1500, 8, 333)
        for s, grads in enumerate(steps, 1):
            oracle.step(grads, dt, lay, cfg, st_ref, *ref, rank=rank, grads_are_slices=slices,
                        half_reduce=hr)

            def chunks(r, f0, cnt):
                j = _local_of(lay, r, f0) if slices else f0
                return [g[j:j + cnt] for g in grads]
            flag, total = oracle.scan_scalars(chunks, dt, lay, oracle.f32(1.0 / st_win.loss_scale),
                                              True, ranks=ranks, chunk=1000, half_reduce=hr)
            assert flag == bool(st_ref.overflow), (name, s)
            if not flag:
                assert total == st_ref.sumsq, (name, s, total, st_ref.sumsq)
            k = 0
            for r in ranks:
                local = 0
                for fs, ln in lay.segments[r]:
                    pos = 0
                    while pos < ln:
                        cnt = min(lengths[k % len(lengths)], ln - pos)
                        k += 1
                        si = fs + pos if rank is None else local + pos
                        gi = local + pos if slices else fs + pos
                        gw = [g[gi:gi + cnt].copy() for g in grads]
                        h = oracle.window_step(gw, dt, cfg, st_win, flag, total,
                                               win[0][si:si + cnt], win[1][si:si + cnt],
                                               win[2][si:si + cnt], half_reduce=hr)
                        if h is not None:
                            win[3][fs + pos:fs + pos + cnt] = h
                        pos += cnt
                    local += ln
            oracle.finish_window_step(cfg, st_win, flag, total)
            for a, b in zip(ref, win):
                assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), (name, s)
            assert st_ref == st_win, (name, s, st_ref, st_win)


ALL_PINS = [pin_memory_closed_forms, pin_decode_exhaustive, pin_encode_structured,
            pin_reduce_bruteforce, pin_reduce_order, pin_unscale_exact, pin_overflow_detect,
            pin_sumsq, pin_clip_coef, pin_adam_first_step, pin_adam_constant_grad,
            pin_adam_literal_form, pin_vs_torch, pin_partition_concat, pin_skip_invariance,
            pin_loss_scale_growth, pin_clip, pin_layout, pin_accumulate_exact,
            pin_accumulate_order, pin_accumulated_step, pin_half_reduce,
            pin_windowed_matches_step, pin_step_scalars]
