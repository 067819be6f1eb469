"""The CPU oracle against what the page and the mathematics fix (no GPU)."""
import pytest

import oracle
from tests import oracle_checks


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.mark.parametrize("check", oracle_checks.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(o, check):
    check(o)
