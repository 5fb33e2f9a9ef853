"""The oracle against its pins (CPU only)."""
import pytest

import oracle
from tests.oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle.lib())


def test_ckpt_count():
    assert oracle.ckpt_count(0, 16) == 0
    assert oracle.ckpt_count(1, 16) == 1
    assert oracle.ckpt_count(16, 16) == 1
    assert oracle.ckpt_count(17, 16) == 2
    assert oracle.ckpt_count(4096, 16) == 256
    assert oracle.ckpt_count(5, 0) == -1
