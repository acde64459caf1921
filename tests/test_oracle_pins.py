"""The CPU oracle against its pins (closed forms, invariants, finite differences,
hand-worked fixtures, independent float64 library routines).  CPU only."""
import pytest

from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(orc, pin):
    pin(orc)
