"""The oracle against its pins (CPU only)."""
import pytest

from pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin, oracle_lib):
    if pin.__name__.startswith("pin_brute_force"):
        pytest.importorskip("mpmath")
    pin(oracle_lib)
