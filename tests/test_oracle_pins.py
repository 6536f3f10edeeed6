"""CPU pins of the oracle (no GPU): every check in oracle_pins against the real oracle."""
import pytest

import oracle as O
import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(O)
