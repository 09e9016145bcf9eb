"""The fp64 oracle against what the definition fixes (CPU only)."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.Oracle())


def test_thread_count_changes_only_rounding():
    """One thread and all threads give the same oracle results up to fp64
    rounding (per-thread partial sums are merged in thread order)."""
    import numpy as np
    import workload
    rp, ci = workload.chung_lu(3_000, 2.1, 12.0, 500.0, 5)
    n = len(rp) - 1
    rng = np.random.default_rng(7)
    h = rng.standard_normal((n, 2, 8)).astype(np.float32)
    a_s = (0.1 * rng.standard_normal((2, 8))).astype(np.float32)
    a_d = (0.1 * rng.standard_normal((2, 8))).astype(np.float32)
    dout = rng.standard_normal((n, 2, 8)).astype(np.float32)
    o = oracle.Oracle()
    n_all = o.num_threads()
    try:
        o.set_threads(1)
        assert o.num_threads() == 1
        f1 = o.forward(rp, ci, h, a_s, a_d, 0.2)
        b1 = o.backward(rp, ci, h, a_s, a_d, 0.2, dout)
    finally:
        o.set_threads(n_all)
    f = o.forward(rp, ci, h, a_s, a_d, 0.2)
    b = o.backward(rp, ci, h, a_s, a_d, 0.2, dout)
    for k in ("out", "lse"):
        np.testing.assert_allclose(f[k], f1[k], rtol=1e-12, atol=1e-13, err_msg=k)
    for k in ("dh", "da_src", "da_dst"):
        np.testing.assert_allclose(b[k], b1[k], rtol=1e-12, atol=1e-12, err_msg=k)
