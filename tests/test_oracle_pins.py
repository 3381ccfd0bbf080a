"""The CPU oracle pinned to things other than itself: hand-worked fixtures
(tests/golden), closed forms, torch's dense attention in float64, brute force
on tiny inputs and invariants of the selection rule."""
import pytest

import helpers


@pytest.mark.parametrize("check", helpers.ALL_CHECKS, ids=lambda f: f.__name__[len("check_"):])
def test_oracle_pin(check):
    check()
