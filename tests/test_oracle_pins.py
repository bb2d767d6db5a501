"""The oracle against what the pages and the mathematics fix (CPU only)."""

import pytest

from oracle import kvsel_oracle as O
from tests import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(O)
