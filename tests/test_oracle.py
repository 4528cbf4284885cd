"""The fp64 oracle against its pins (CPU only)."""
import math

import numpy as np
import pytest

import oracle
from oracle import iomodel
from tests import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ORACLE_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle.get())


def test_page_sizes():
    pins.pin_page_sizes(iomodel)


def test_flop_convention():
    # 4*B*H*N^2*d forward, 2.5x backward, halved when causal
    f, b = iomodel.attention_flops(1, 32, 8192, 128, True)
    assert f == 0.5 * 4 * 32 * 8192**2 * 128
    assert b == 2.5 * f
    f, b = iomodel.attention_flops(2, 16, 4096, 128, False)
    assert math.isclose(f / 1e9, 274.877906944)


def test_fully_masked_row_convention():
    # a row with no allowed key: O = 0, L = -inf, no NaN (online oracle, empty range)
    rng = np.random.default_rng(0)
    k, v = rng.standard_normal((4, 3)), rng.standard_normal((4, 3))
    m, l, acc = oracle.row_partial(rng.standard_normal(3), k, v, 0, 1, 4, True, 1.0, 2)
    assert m == -math.inf and l == 0.0 and not np.isnan(acc).any()


def test_stress_scale_rows():
    # rows with large maxima (Q, K ~ N(0, 4^2)) stay finite and exact in fp64
    rng = np.random.default_rng(11)
    q, k, v = (4 * rng.standard_normal((1, 2, 64, 32)) for _ in range(3))
    o, lse = oracle.fwd(q, k, v, True, 1 / math.sqrt(32))
    o2, l2 = oracle.fwd_online(q, k, v, True, 1 / math.sqrt(32), 16, True)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert np.max(np.abs(o - o2)) < 1e-12 and np.max(np.abs(lse - l2)) < 1e-12
