"""The CPU oracle against its pins (no GPU needed)."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


@pytest.mark.parametrize("name,overrides", [
    ("c1", {}),
    ("c2", {"B": 1, "Hkv": 2, "Hq": 8, "L": 8192}),
    ("c3", {"Hkv": 2, "Hq": 8, "L": 32768, "k": 20, "needles": 5}),
])
def test_needles_selected(name, overrides):
    P.pin_decode_needles_selected(name, **overrides)
