"""The CPU oracle against its pins (no GPU needed)."""
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_mac_count(oracle_counting):
    oracle_pins.pin_mac_count(oracle_counting)


def test_plain_build_reports_no_count(oracle_lib):
    assert oracle_lib.mac_count() == -1
