"""The oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check, oracle_mod):
    check(oracle_mod)
