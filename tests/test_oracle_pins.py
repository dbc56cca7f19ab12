"""The fp64 oracle against closed forms, an FFT identity, invariants and brute force."""
import pytest

import oracle
from tests.oracle_pins import ALL_PINS


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_uses_threads(orc):
    assert orc.threads() >= 1
