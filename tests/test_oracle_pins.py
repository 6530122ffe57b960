"""The committed oracle against its pins (see ``pins.py`` for what each
check compares with).  CPU only."""
import pytest

import pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check, ora):
    check(ora)
