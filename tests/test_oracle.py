"""The oracle against its pins (CPU only).  See tests/pins.py for what each pin
checks and which passage fixes it."""
import numpy as np
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(oracle, pin):
    pin(plant=0)


def test_threads_do_not_change_results(oracle):
    """The OpenMP split over (b, d) is for speed only: 1 and 4 threads agree bit for bit."""
    rng = np.random.default_rng(30)
    x, delta, A, B, C, D, z = pins._rand_inputs(rng, 3, 50, 7, 4, gate=True)
    y1, s1 = oracle.scan_fwd(x, delta, A, B, C, D, z, chunk_len=8, threads=1)
    y4, s4 = oracle.scan_fwd(x, delta, A, B, C, D, z, chunk_len=8, threads=4)
    assert np.array_equal(y1, y4) and np.array_equal(s1, s4)


def test_bad_arguments_rejected(oracle):
    x = np.zeros((1, 4, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.scan_fwd(x, x, np.zeros((3, 2), np.float32), np.zeros((1, 4, 2), np.float32),
                        np.zeros((1, 4, 2), np.float32))
    with pytest.raises(TypeError):
        oracle.scan_fwd(x.astype(np.float64), x, np.zeros((2, 2), np.float32), x, x)
