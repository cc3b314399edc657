"""The oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL, ids=lambda c: c.__name__)
def test_oracle_pin(oracle_lib, check):
    failures = check(oracle_lib)
    assert not failures, "\n".join(failures)


def test_backward_fd_wider(oracle_lib):
    """Finite differences on a second, odd shape with t = 3 (non power of two)."""
    failures = oracle_pins.check_backward_fd(oracle_lib, shapes=((2, 5, 9),), ts=(3,))
    assert not failures, "\n".join(failures)
