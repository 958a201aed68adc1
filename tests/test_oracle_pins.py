"""The fp64 oracle against its pins (CPU only)."""
import pytest

import oracle
from oracle.chunked import delta_backward_chunked, delta_forward_chunked
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.lib())


def test_chunked_equals_sequential():
    oracle_pins.pin_chunked_equals_sequential(oracle.lib(), delta_forward_chunked)


def test_chunked_backward_equals_sequential():
    oracle_pins.pin_chunked_backward_equals_sequential(oracle.lib(), delta_backward_chunked)


def test_rejects_bad_nu():
    with pytest.raises(ValueError):
        oracle.dpfp([[1.0, 2.0]], nu=4)
