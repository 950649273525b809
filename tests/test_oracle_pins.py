"""CPU tests: the FP64 oracle against its pins (see oracle_pins.py)."""
import pytest

import oracle
from tests import oracle_pins

pytestmark = pytest.mark.timeout(600) if hasattr(pytest.mark, "timeout") else []


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check(oracle.default())
