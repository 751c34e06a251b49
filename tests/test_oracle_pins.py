"""The oracle against its pins (CPU only)."""
import pytest

from oracle import oracle as O
import oracle_pins as P

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(O.load())
