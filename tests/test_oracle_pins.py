"""The oracle against its pins (CPU only). See tests/pins.py for what each pin checks."""
import pytest

import oracle as O
from tests import pins

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(O)
