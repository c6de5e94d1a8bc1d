"""The CPU oracle against facts fixed outside it (CPU only)."""
import pytest

import oracle as O
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(O.load())
