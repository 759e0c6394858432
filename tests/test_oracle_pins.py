"""The CPU oracle against closed forms, an independent O(L^2) formulation,
structural invariants and f64 finite differences (no GPU)."""

import pytest

import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, check):
    check(orc)
