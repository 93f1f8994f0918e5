"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_openmp_build_matches_single_thread():
    """The OpenMP build only splits independent elements between threads: it
    must give the same bits as the single-threaded build."""
    import numpy as np
    import oracle
    lay, grads, master0 = oracle_pins._random_problem(4, (100_000, 3333), oracle.BF16, 77)
    outs = []
    for omp in (False, True):
        w, m, v = master0.copy(), np.zeros_like(master0), np.zeros_like(master0)
        half = np.zeros(lay.padded, np.uint16)
        st = oracle.State(loss_scale=1024.0)
        cfg = oracle.AdamCfg(weight_decay=0.01, max_grad_norm=0.5)
        for _ in range(3):
            oracle.step(grads, oracle.BF16, lay, cfg, st, w, m, v, half, openmp=omp)
        outs.append((w, m, v, half, st.sumsq))
    for a, b in zip(outs[0][:4], outs[1][:4]):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    assert outs[0][4] == outs[1][4]
