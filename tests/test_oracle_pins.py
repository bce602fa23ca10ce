"""The fp64 oracle against its pins (closed forms, brute force, torch float64 SDPA/autograd,
finite differences, hand-worked examples).  CPU only."""
import pytest

from oracle import attention as orc

from tests.pins import ALL_CHECKS


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    ok, msg = check(orc)
    assert ok, msg
