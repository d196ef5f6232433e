"""The fp64 oracle against its pins (CPU only).  See ``pins.py`` for what
each pin checks and which passage of the HYPIC pages it follows."""
import pytest

import pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__[len("check_"):])
def test_pin(oracle_lib, check):
    check()
