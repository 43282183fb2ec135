"""The fp64 oracle against library routines, closed forms and invariants (CPU)."""
import pytest

import oracle_checks


@pytest.mark.parametrize("check", oracle_checks.ALL_CHECKS, ids=lambda f: f.__name__[6:])
def test_oracle_pin(check):
    check()
