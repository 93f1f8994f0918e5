"""Plant one plausible mistake at a time in a copy of the oracle (on the CPU)
and check that at least one pin catches it.  This shows the pins constrain
every part of the oracle: a dropped term, a wrong sign, a wrong index or a
transposed operand does not go unnoticed."""
import os
import subprocess

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement)
C_MUTATIONS = [
    ("reduce skips rank 0", "for (int q = 0; q < world; ++q)", "for (int q = 1; q < world; ++q)"),
    ("reduce reads wrong index", "grads[q][offset + j]", "grads[q][j]"),
    ("reduce descending order", "acc = acc + half_to_f32(grads[q][offset + j], dtype);",
     "acc = acc + half_to_f32(grads[world - 1 - q][offset + j], dtype);"),
    ("unscale divides", "g[j] = g[j] * inv_scale;", "g[j] = g[j] / inv_scale;"),
    ("overflow misses Inf", "found |= !isfinite(g[j]);", "found |= isnan(g[j]);"),
    ("sumsq drops square", "double t = d * d;", "double t = d;"),
    ("sumsq drops compensation", "*comp = c;", "*comp = 0.0;"),
    ("momentum uses w", "s->omb1 * g;", "s->omb1 * wj;"),
    ("momentum drops decay", "float mj = s->b1 * m[j] + s->omb1 * g;", "float mj = m[j] + s->omb1 * g;"),
    ("variance not squared", "s->omb2 * (g * g);", "s->omb2 * g;"),
    ("decay dropped", "wj = wj * s->decay;", "wj = wj;"),
    ("bias correction 2 inverted", "sqrtf(vj) / s->rbc2", "sqrtf(vj) * s->rbc2"),
    ("eps sign", "+ s->eps;", "- s->eps;"),
    ("update sign", "wj = wj - s->step * (mj / den);", "wj = wj + s->step * (mj / den);"),
    ("update transposed", "(mj / den)", "(den / mj)"),
    ("coupled L2 dropped", "g = g + s->wd * wj;", "g = g;"),
    ("f16 decode exponent", "ex - 25);", "ex - 24);"),
    ("encode truncates", "double k = rint(q);", "double k = floor(q);"),
    ("encode rounds half up", "double k = rint(q);", "double k = floor(q + 0.5);"),
    ("encode no overflow to Inf", "if (e > emax)", "if (e > emax + 1)"),
    ("bf16 decode shift", "(uint32_t)b << 16;", "(uint32_t)b << 15;"),
    ("accumulate overwrites", "acc[j] = acc[j] + r[j];", "acc[j] = r[j];"),
    ("half reduce rounds only at the end", "acc = (double)half_to_f32(h, dtype);",
     "acc = exact; (void)h;"),
]


def _build_mutant(tmp_path, text, repl, openmp):
    src = open(SRC).read()
    assert src.count(text) >= 1, text
    mutated = src.replace(text, repl)
    path = tmp_path / f"mut{'_omp' if openmp else ''}.c"
    path.write_text(mutated)
    so = tmp_path / f"libmut{'_omp' if openmp else ''}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", *(["-fopenmp"] if openmp else []), str(path), "-o", str(so), "-lm"],
                   check=True)
    return str(so)


def _caught():
    for pin in oracle_pins.ALL_PINS:
        try:
            pin()
        except AssertionError:
            return pin.__name__
    return None


@pytest.mark.parametrize("name,text,repl", C_MUTATIONS, ids=[m[0] for m in C_MUTATIONS])
def test_c_mutation_is_caught(name, text, repl, tmp_path, monkeypatch):
    import ctypes
    libs = {}
    for omp in (False, True):
        lib = ctypes.CDLL(_build_mutant(tmp_path, text, repl, omp))
        libs[omp] = lib
    saved = dict(oracle._LIBS)
    try:
        oracle._LIBS.clear()
        oracle._lib(False)  # sets argtypes on the real libraries' entries
        for omp, lib in libs.items():
            real = saved.get(omp) or oracle._lib(omp)
            for fn in ("orc_f16_to_f32", "orc_bf16_to_f32", "orc_f32_to_f16", "orc_f32_to_bf16",
                       "orc_to_half_array", "orc_from_half_array", "orc_reduce_sum", "orc_unscale",
                       "orc_any_nonfinite", "orc_sumsq", "orc_scale", "orc_adam",
                       "orc_accumulate", "orc_reduce_sum_half"):
                f = getattr(lib, fn)
                f.argtypes = getattr(real, fn).argtypes
                f.restype = getattr(real, fn).restype
            oracle._LIBS[omp] = lib
        assert _caught() is not None, f"mutation not caught: {name}"
    finally:
        oracle._LIBS.clear()
        oracle._LIBS.update(saved)


def _py_mutations():
    import math

    def no_bias_correction(cfg, st):
        return orig_scalars(oracle.AdamCfg(**{**cfg.__dict__, "bias_correction": False}), st)

    def stale_t(cfg, st):
        s = orig_scalars(cfg, st)
        bp1 = st.bp1 if st.t else cfg.beta1
        s.step = oracle.f32(cfg.lr / (1.0 - bp1)) if cfg.bias_correction else s.step
        return s

    def skip_no_backoff(cfg, st):
        st.overflow = 1

    def commit_no_t(cfg, st):
        st.overflow = 0
        st.good_steps += 1

    def clip_no_sqrt(sumsq, max_norm):
        return oracle.f32(min(1.0, max_norm / (sumsq + 1e-6)))

    def layout_floor(numels, world, align=64, bucket=0):
        lay = orig_layout(numels, world, align, bucket)
        if bucket == 0 and world > 1:
            P = lay.flat_end // world  # the floor split: drops the remainder
            segs = tuple(((r * P, P),) for r in range(world))
            return oracle.Layout(lay.numels, world, align, 0, lay.offsets, lay.numel,
                                 lay.flat_end, P * world, P, 1, P, P, segs)
        return lay

    def scan_ranks_reversed(grad_chunks, dtype, lay, inv_scale, want_sumsq, openmp=False,
                            ranks=None, chunk=1 << 24, half_reduce=False):
        order = list(range(lay.world)) if ranks is None else list(ranks)
        return orig_scan(grad_chunks, dtype, lay, inv_scale, want_sumsq, openmp, order[::-1],
                         chunk, half_reduce)

    def scan_unscale_after_flag(grad_chunks, dtype, lay, inv_scale, want_sumsq, openmp=False,
                                ranks=None, chunk=1 << 24, half_reduce=False):
        flag, total = False, 0.0
        for r in (range(lay.world) if ranks is None else ranks):
            acc = (0.0, 0.0)
            for fs, ln in lay.segments[r]:
                for c0 in range(fs, fs + ln, chunk):
                    n = min(chunk, fs + ln - c0)
                    g = oracle.reduce_sum(grad_chunks(r, c0, n), dtype, 0, n, openmp, half_reduce)
                    flag = flag or oracle.any_nonfinite(g, openmp)
                    if want_sumsq:
                        acc = oracle.sumsq(g, acc)
                    oracle.unscale(g, inv_scale, openmp)  # too late
            total = total + oracle.sumsq_value(acc)
        return flag, total

    def window_clip_from_previous_state(grads, dtype, cfg, st, flag, total_sumsq, master, m, v,
                                        half_reduce=False):
        g = oracle.reduce_sum(grads, dtype, 0, master.size, half_reduce=half_reduce)
        oracle.unscale(g, oracle.f32(1.0 / st.loss_scale))
        if flag:
            return None
        if cfg.max_grad_norm > 0 and st.coef < 1.0:  # the last step's coefficient
            oracle.scale(g, st.coef)
        oracle.adam(g, master, m, v, oracle.step_scalars(cfg, st))
        return oracle.f32_to_half(master, dtype)

    orig_scalars = oracle.step_scalars
    orig_layout = oracle.layout
    orig_scan = oracle.scan_scalars
    return [("no bias correction", "step_scalars", no_bias_correction),
            ("stale t in bias correction", "step_scalars", stale_t),
            ("skip keeps loss scale", "skip", skip_no_backoff),
            ("commit forgets t", "commit", commit_no_t),
            ("clip without sqrt", "clip_coef", clip_no_sqrt),
            ("floor partition", "layout", layout_floor),
            ("scan takes the ranks out of order", "scan_scalars", scan_ranks_reversed),
            ("scan unscales after the flag and norm", "scan_scalars", scan_unscale_after_flag),
            ("window clips with the last step's coefficient", "window_step",
             window_clip_from_previous_state)]


@pytest.mark.parametrize("idx", range(9))
def test_python_mutation_is_caught(idx, monkeypatch):
    name, attr, fn = _py_mutations()[idx]
    monkeypatch.setattr(oracle, attr, fn)
    assert _caught() is not None, f"mutation not caught: {name}"
