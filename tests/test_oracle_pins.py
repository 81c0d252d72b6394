"""The fp64 oracle against its pins (closed forms, brute force, library
special cases and invariants); CPU only."""
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(lib, pin):
    pin(lib)


def test_every_oracle_function_pinned():
    assert oracle.UNPINNED == ()
