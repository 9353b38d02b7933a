"""The oracle against its pins (CPU only)."""
import pytest

import oracle
from tests import oracle_pins


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(o, pin):
    pin(o)


def test_thread_count_does_not_change_scores(o):
    import numpy as np
    import workloads
    c = workloads.unit_corpus(3000, 200, seed=5)
    q = workloads.unit_queries(1, 200, seed=6)[0]
    n0 = o.num_threads()
    try:
        o.set_num_threads(1)
        a = o.scores(c, q)
        o.set_num_threads(max(2, n0))
        b = o.scores(c, q)
    finally:
        o.set_num_threads(n0)
    assert np.array_equal(a, b)


def test_rejects_bad_arguments(o):
    import numpy as np
    c = np.zeros((4, 3), np.float32)
    q = np.zeros(3, np.float32)
    with pytest.raises(ValueError):
        o.topk(c, q, 5)
    with pytest.raises(ValueError):
        o.topk(c, q, 0)
    with pytest.raises(ValueError):
        o.topk_int32(np.zeros(3, np.int32), 4)
