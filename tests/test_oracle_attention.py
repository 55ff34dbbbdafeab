"""Pins of the rotary-attention oracle (oracle/attention.py), no GPU.  The pins
themselves are in attention_pins.py, as functions of the oracle module, so the
planted-mistake test can run them on mutants too."""
import pytest

from oracle import attention as A

import attention_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda p: p.__name__)
def test_attention_oracle_pin(pin):
    pin(A)
