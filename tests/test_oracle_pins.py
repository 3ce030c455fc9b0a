"""The fp64 oracle against brute force, torch's float64 GroupNorm, closed
forms and invariants (CPU only)."""
import pytest

import oracle
from tests import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_thread_count_does_not_change_results(orc):
    from channels_last_groupnorm_gb300.workloads import make_case
    import numpy as np
    case = make_case(2, 301, 128, 7, mean=2.0, std=0.5)
    y1, m1, r1 = orc.forward(case["x_bits"], case["gamma"], case["beta"], 32, 1e-6, True,
                             nthreads=1)
    y4, m4, r4 = orc.forward(case["x_bits"], case["gamma"], case["beta"], 32, 1e-6, True,
                             nthreads=4)
    assert np.array_equal(y1, y4) and np.array_equal(m1, m4) and np.array_equal(r1, r4)


def test_rejects_bad_geometry(orc):
    import numpy as np
    x = np.zeros((1, 4, 48), np.uint16)
    g = np.ones(48, np.float32)
    with pytest.raises(ValueError):
        orc.forward(x, g, g, 32, 1e-6, True)      # 48 % 32 != 0
