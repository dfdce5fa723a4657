"""The CPU oracle against the pages' worked examples, closed forms and brute force."""
import pytest

from oracle import hashattn_oracle as O
import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(O)
