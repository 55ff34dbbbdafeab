"""The CPU oracle against its pins (no GPU)."""
import pytest

import oracle
import oracle_pins

NEEDS_SYMPY = {"pin_inv_freq_closed_form", "pin_tables_high_precision"}


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    if pin.__name__ in NEEDS_SYMPY:
        pytest.importorskip("sympy")
    pin(oracle.load())
