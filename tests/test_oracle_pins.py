"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import numpy as np
import pytest

import oracle
import oracle_pins
from parity import tolerance


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_golden_fixtures_are_the_pages_values():
    # fill_42 prints 128 values of 42.0; iota prints 0.0 .. 1023.0
    assert np.all(oracle_pins.read_golden("fill_42.txt") == 42.0)
    assert np.array_equal(oracle_pins.read_golden("iota.txt"), np.arange(1024.0))


def test_empty_and_degenerate(oracle_lib):
    # K = 0: an empty sum is zero
    c = oracle.gemm(np.zeros((3, 0), np.float16), np.zeros((0, 4), np.float16), oracle.OUT_F32)
    assert c.shape == (3, 4) and not c.any()
    # M = 0 or N = 0: empty output
    assert oracle.gemm(np.zeros((0, 5), np.float16), np.zeros((5, 4), np.float16)).shape == (0, 4)
    assert oracle.gemm(np.zeros((2, 5), np.float16), np.zeros((5, 0), np.float16)).shape == (2, 0)


def test_bad_arguments_rejected(oracle_lib):
    a = np.zeros((2, 3), np.uint16)
    b = np.zeros((3, 4), np.uint16)
    with pytest.raises(RuntimeError):
        oracle.gemm(a, b, rows=[2])  # row out of range
    with pytest.raises(ValueError):
        oracle.gemm(a, np.zeros((4, 4), np.uint16))


def test_special_values_follow_ieee(oracle_lib):
    inf = np.float16(np.inf)
    a = np.array([[1.0, inf]], np.float16)
    b = np.array([[1.0], [2.0]], np.float16)
    assert np.isinf(oracle.as_values(oracle.gemm(a, b, oracle.OUT_F32), oracle.OUT_F32)).all()
    b0 = np.array([[1.0], [0.0]], np.float16)  # inf * 0 = NaN
    assert np.isnan(oracle.gemm(a, b0, oracle.OUT_F32)).all()
    # overflow of the rounded output: 300 * 300 = 90000 > 65504
    big = oracle.gemm(np.full((1, 1), 300, np.float16), np.full((1, 1), 300, np.float16))
    assert np.isinf(big.view(np.float16)).all()


def test_tolerance_formula():
    # |C - C_ref| <= 2e-3 |C_ref| + 1e-2 sqrt(K / 1024)
    assert tolerance(np.array([0.0]), 1024)[0] == pytest.approx(1e-2)
    assert tolerance(np.array([-100.0]), 4096)[0] == pytest.approx(0.2 + 0.02)
    assert tolerance(np.array([10.0]), 256)[0] == pytest.approx(0.02 + 0.005)
