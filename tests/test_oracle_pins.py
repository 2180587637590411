"""The oracle against its pins (values printed on the pages, closed forms,
invariants, brute force).  CPU only."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def o():
    return oracle.load()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(o, pin):
    pin(o)


def test_threads_do_not_change_results(o):
    p = oracle_pins.Problem(o, [300, 17, 1, 64, 129], 8, 2, 64, True, seed=5)
    a = p.run(0.125, threads=1)
    b = p.run(0.125, threads=4)
    assert (a == b).all()
