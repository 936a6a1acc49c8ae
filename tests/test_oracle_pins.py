"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

import oracle
from tests import oracle_checks as oc


@pytest.fixture(scope="module")
def lib():
    return oracle.load(oracle.build())


@pytest.mark.parametrize("name", sorted(oc.ALL_CHECKS))
def test_pin(lib, name):
    oc.ALL_CHECKS[name](lib)


@pytest.mark.parametrize("alpha", [0.3, 0.6, 0.9])
def test_chisq_output_law_is_target(lib, alpha):
    oc.check_chisq(lib, alpha)
