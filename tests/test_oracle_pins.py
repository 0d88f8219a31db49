"""CPU pins of the oracle (see tests/oracle_checks.py for what each pins)."""
import pytest

from tests import oracle_checks as oc


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(oracle_mod, check):
    check(oracle_mod)
