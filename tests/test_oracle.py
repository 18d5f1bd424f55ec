"""The fp64 oracle against facts fixed by the mathematics and by an
independent library (see oracle_pins for what each pin checks)."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.default())
