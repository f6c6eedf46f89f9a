"""The CPU oracle against what the mathematics fixes (see tests/pins.py)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(0)


@pytest.mark.parametrize("pin", pins.QUANT_PINS, ids=lambda p: p.__name__)
def test_quantiser_pin(pin):
    pin(0)


@pytest.mark.parametrize("pin", pins.GDN_PINS, ids=lambda p: p.__name__)
def test_gdn_pin(pin):
    pin(0)
