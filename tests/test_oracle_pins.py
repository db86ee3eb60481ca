"""The committed FP64 oracle against its pins (CPU only)."""
import pytest

from tests import oracle_pins

pytestmark = pytest.mark.cpu


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_thread_count_invariance(orc):
    """Tokens are never split across threads, so any thread count gives the
    same bits."""
    import numpy as np
    rng = np.random.default_rng(12)
    x, L, wgu, wd = oracle_pins.rand_layer(rng, 9, 64, 32, 6)
    a, ia, wa = orc.forward(x, L, wgu, wd, 3, nthreads=1)
    b, ib, wb = orc.forward(x, L, wgu, wd, 3, nthreads=4)
    assert np.array_equal(a, b) and np.array_equal(ia, ib) and np.array_equal(wa, wb)


def test_argument_errors(orc):
    import numpy as np
    with pytest.raises(RuntimeError):
        orc.route(np.zeros((2, 3), np.float32), 4)   # k > E
    with pytest.raises(RuntimeError):
        orc.route(np.zeros((2, 3), np.float32), 0)   # k < 1
    # a selected expert missing from the expert map
    x = np.zeros((1, 4), np.uint16)
    L = np.float32([[1.0, 0.0]])
    wgu = np.zeros((1, 4, 4), np.uint16)
    wd = np.zeros((1, 4, 2), np.uint16)
    with pytest.raises(RuntimeError):
        orc.forward(x, L, wgu, wd, 1, expert_map=np.int32([-1, 0]))
