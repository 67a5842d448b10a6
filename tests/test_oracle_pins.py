"""The oracle against its pins (hand-worked values, library reductions, invariants)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_every_oracle_product_is_pinned():
    names = {f.__name__ for f in oracle_pins.ALL_PINS}
    for prefix in ("pin_wq8_", "pin_wq3_", "pin_wq4_", "pin_w8a8_", "pin_pack", "pin_code3", "pin_scalar",
                   "pin_dequant_"):
        assert any(n.startswith(prefix) for n in names), prefix
