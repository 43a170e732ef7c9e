"""The CPU oracle against its pins (hand-built words, closed forms, brute force)."""
import pytest

import pins
from oracle import oracle


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


@pytest.mark.parametrize("fmt,ncodes", [(1, 256), (2, 16), (4, 16), (5, 8), (7, 16), (8, 16), (13, 256)])
def test_every_code_value_is_exact_in_f16(orc, fmt, ncodes):
    """The cooperative-matrix reading: the codes of every format are small
    integers or e2m1 values, so each one is exactly an f16 (what lets the
    prefill GEMM decode weights to f16 without rounding)."""
    import numpy as np
    codes = range(-128, 128) if fmt in (1, 13) else range(ncodes)
    for c in codes:
        v = orc.code_value(fmt, c)
        assert float(np.float16(v)) == v, (fmt, c, v)
        assert abs(v) <= 128
