"""The CPU oracle against its pins (invariants, textbook reductions, closed
forms, derivative definition, brute force, hand-worked examples)."""
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(lib, check):
    check(lib)
