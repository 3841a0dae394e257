"""Pins of the CPU softmax oracle (oracle/softmax.py) to what the tutorial and
the mathematics fix, without a GPU.

* the tutorial's own check compares against torch.softmax along the rows:
  the oracle must agree with it (fp64, on the CPU) and with scipy's softmax;
* closed forms: a two-entry row is the logistic function, a constant row is
  uniform, a row with one dominant entry is one-hot;
* invariants: rows sum to one, shifting a row changes nothing (exactly
  representable shifts), log-ratios equal differences of the inputs;
* the columns at or past n are not read (NaN there changes nothing);
* IEEE special values follow the definition.
"""
import math

import numpy as np
import pytest
import torch

from dense_fp16_gemm_fp32_gb300 import inputs
from oracle import softmax as osm


def _x(M, n, seed, ld=None):
    return inputs.softmax_inputs(M, n, ld or n, seed).numpy()


@pytest.mark.parametrize("M,n", [(1, 1), (3, 2), (7, 31), (16, 781), (5, 4097)])
def test_matches_torch_softmax_fp64(M, n):
    x = _x(M, n, seed=M * 1000 + n)
    want = torch.softmax(torch.from_numpy(x).double(), dim=1).numpy()
    np.testing.assert_allclose(osm.softmax_rows(x, n), want, rtol=1e-13, atol=0)


def test_matches_scipy_softmax():
    special = pytest.importorskip("scipy.special")
    x = _x(64, 781, seed=3)
    np.testing.assert_allclose(osm.softmax_rows(x, 781), special.softmax(x.astype(np.float64), axis=1),
                               rtol=1e-13, atol=0)


def test_reduces_along_rows_not_columns():
    # a non-square array whose column softmax differs from its row softmax
    x = np.array([[0.0, 1.0, 2.0], [5.0, 5.0, 5.0]], dtype=np.float32)
    y = osm.softmax_rows(x, 3)
    np.testing.assert_allclose(y[1], [1 / 3] * 3, rtol=1e-15)
    e = np.exp([0.0, 1.0, 2.0])
    np.testing.assert_allclose(y[0], e / e.sum(), rtol=1e-15)


def test_two_entry_rows_are_logistic():
    a = np.linspace(-20, 20, 81, dtype=np.float32)
    x = np.stack([a, np.zeros_like(a)], axis=1)
    y = osm.softmax_rows(x, 2)
    for (a0, _), (y0, y1) in zip(x, y):
        want = 1.0 / (1.0 + math.exp(-float(a0)))
        assert y0 == pytest.approx(want, rel=1e-14)
        assert y1 == pytest.approx(1.0 / (1.0 + math.exp(float(a0))), rel=1e-14)


def test_constant_rows_are_uniform_and_dominant_rows_one_hot():
    x = np.full((4, 781), 3.25, dtype=np.float32)
    np.testing.assert_array_equal(osm.softmax_rows(x, 781), np.full((4, 781), 1.0 / 781))
    x = np.zeros((2, 100), dtype=np.float32)
    x[0, 17] = 1000.0               # overflows exp() unless the maximum is subtracted first
    x[1, 99] = 80.0
    y = osm.softmax_rows(x, 100)
    assert y[0, 17] == 1.0 and np.all(y[0, :17] == 0) and np.all(y[0, 18:] == 0)
    assert y[1, 99] == pytest.approx(1.0 / (1.0 + 99 * math.exp(-80.0)), rel=1e-15)


def test_rows_sum_to_one_and_log_ratios():
    x = _x(32, 781, seed=11)
    y = osm.softmax_rows(x, 781)
    for r in range(32):
        assert math.fsum(y[r]) == pytest.approx(1.0, abs=1e-14)
    lr = np.log(y[:, 1:]) - np.log(y[:, :1])
    np.testing.assert_allclose(lr, x[:, 1:].astype(np.float64) - x[:, :1], atol=1e-12)


def test_shift_invariance_with_exact_shifts():
    # small integers: x + 4096 is exact in fp32, and the result must not move
    g = torch.Generator().manual_seed(5)
    x = torch.randint(-8, 9, (8, 300), generator=g).float().numpy()
    y0 = osm.softmax_rows(x, 300)
    for c in (4096.0, -4096.0, 1.0e6):
        np.testing.assert_allclose(osm.softmax_rows(x + np.float32(c), 300), y0, rtol=1e-14)


def test_columns_past_n_are_not_read():
    x = inputs.softmax_inputs(9, 781, 784, seed=2, pad_value=float("nan"))
    assert np.isnan(x[:, 781:]).all()
    y = osm.softmax_rows(x, 781)
    assert y.shape == (9, 781) and np.isfinite(y).all()
    np.testing.assert_array_equal(y, osm.softmax_rows(np.ascontiguousarray(x[:, :781]), 781))
    # a huge pad value would win the maximum if it were read
    x = inputs.softmax_inputs(3, 5, 8, seed=2, pad_value=1.0e30)
    assert np.isfinite(osm.softmax_rows(x, 5)).all()


def test_row_subset_matches_full():
    x = _x(50, 64, seed=7)
    rows = inputs.sample_rows(50, seed=7, count=10)
    np.testing.assert_array_equal(osm.softmax_rows(x, 64, rows=rows.numpy()), osm.softmax_rows(x, 64)[rows.numpy()])


def test_special_values():
    inf, nan = float("inf"), float("nan")
    x = np.array([[0.0, -inf, 1.0, 2.0],
                  [0.0, nan, 1.0, 2.0],
                  [0.0, inf, 1.0, 2.0],
                  [-inf, -inf, -inf, -inf]], dtype=np.float32)
    y = osm.softmax_rows(x, 4)
    e = np.exp([0.0, 1.0, 2.0])
    np.testing.assert_allclose(y[0], [e[0] / e.sum(), 0.0, e[1] / e.sum(), e[2] / e.sum()], rtol=1e-15)
    assert np.isnan(y[1:]).all()
    want = torch.softmax(torch.from_numpy(x).double(), dim=1).numpy()
    np.testing.assert_array_equal(np.isnan(y), np.isnan(want))


def test_degenerate_extents():
    x = np.zeros((0, 8), dtype=np.float32)
    assert osm.softmax_rows(x, 8).shape == (0, 8)
    x = np.zeros((3, 8), dtype=np.float32)
    assert osm.softmax_rows(x, 0).shape == (3, 0)
    np.testing.assert_array_equal(osm.softmax_rows(x, 1), np.ones((3, 1)))


def test_input_recipe():
    x = inputs.softmax_inputs(1823, 781, 784, seed=0)
    assert x.shape == (1823, 784) and x.dtype == torch.float32
    assert torch.all(x[:, 781:] == 0)
    g = torch.Generator().manual_seed(0)
    assert torch.equal(x[:, :781], torch.randn((1823, 781), generator=g))
    w = inputs.SOFTMAX_WORKLOADS_BY_NAME["softmax_1823x781"]
    assert (w.M, w.n, w.ld, w.seed) == (1823, 781, 784, 0)
