"""The fp64 oracle against closed forms, invariants and brute force (CPU only)."""
import pytest

import oracle
from oracle_pins import ALL_CHECKS


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(lib, check):
    check(lib)


def test_oracle_threads_do_not_change_results(lib):
    """Splitting chains over threads is bookkeeping only: results are bitwise equal."""
    import numpy as np

    r = np.random.default_rng(11)
    b, d, L, N = 3, 7, 33, 5
    args = [r.normal(size=(b, d, L)), r.normal(size=(b, d, L)), r.normal(size=(d, N)),
            r.normal(size=(b, L, N)), r.normal(size=(b, L, N))]
    kw = dict(D=r.normal(size=d), z=r.normal(size=(b, d, L)), delta_bias=r.normal(size=d), lib=lib)
    y1, h1, n1 = oracle.selective_scan(*args, nthreads=1, **kw)
    y4, h4, n4 = oracle.selective_scan(*args, nthreads=4, **kw)
    assert n1 == 1 and n4 == 4
    assert np.array_equal(y1, y4) and np.array_equal(h1, h4)


def test_oracle_empty_sequence(lib):
    """L = 0: no outputs, and the final state is the (zero) initial state."""
    import numpy as np

    y, h, _ = oracle.selective_scan(np.zeros((2, 3, 0)), np.zeros((2, 3, 0)), np.zeros((3, 4)),
                                    np.zeros((2, 0, 4)), np.zeros((2, 0, 4)), lib=lib)
    assert y.shape == (2, 3, 0) and np.all(h == 0.0)


def test_oracle_matches_stored_tiny_fixture(lib):
    """The committed fixture (written by tests/golden/make_golden.py) still matches."""
    import numpy as np

    from golden_io import load_tiny_f32
    from selective_state_space_140_b300 import workloads

    y_ref, h_ref = load_tiny_f32()
    x = workloads.make_config_inputs(workloads.SCAN_CONFIGS["tiny_f32"])
    f = workloads.to_f64
    y, h, _ = oracle.selective_scan(f(x["u"]), f(x["delta"]), f(x["A_log"]), f(x["B"]), f(x["C"]),
                                    D=f(x["D"]), z=f(x["z"]), delta_bias=f(x["delta_bias"]), lib=lib)
    assert np.allclose(y, y_ref, rtol=1e-15, atol=0) and np.allclose(h, h_ref, rtol=1e-15, atol=0)
