"""The fp64 oracle against closed forms, brute force, invariants and hand cases (CPU)."""
import pytest

import oracle.oracle as orc
from _pins import ALL_PINS


@pytest.fixture(scope="module")
def lib():
    return orc.load()


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(lib, pin):
    pin(lib)
