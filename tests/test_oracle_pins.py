"""The CPU oracle against facts fixed outside its code (see pins.py)."""
import numpy as np
import pytest

import pins
from oracle.oracle import Oracle, OracleError


@pytest.fixture(scope="module")
def o():
    return Oracle()


@pytest.mark.parametrize("check", pins.ALL_CHECKS + [pins.check_workload_invariants], ids=lambda c: c.__name__)
def test_pin(o, check):
    check(o)


def test_rejects_values_outside_contract(o):
    for bad in (np.nan, np.inf):
        l = np.zeros((2, 4), np.float32)
        l[1, 2] = bad
        with pytest.raises(OracleError):
            o.route(l, 2)


def test_rejects_bad_sizes(o):
    with pytest.raises(OracleError):
        o.route(np.zeros((2, 3), np.float32), 4)  # k > E
