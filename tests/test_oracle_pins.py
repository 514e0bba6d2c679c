"""The oracle against what the definition, the formats and the pages fix
(no GPU).  The individual checks live in ``oracle_pin_checks.py``."""

import pytest

import oracle
import oracle_pin_checks as pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, check):
    check(orc)
