"""The oracle against its pins (closed forms, invariants, library special case)."""

import pytest

import oracle
import oracle_pins as P


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=[p.__name__ for p in P.ALL_PINS])
def test_pin(lib, pin):
    pin(lib)


def test_validation(lib):
    P.pin_validation(lib)
