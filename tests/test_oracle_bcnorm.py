"""The oracle's B / C normalisation and bias (Mamba-3 summary page, §3.4)
against what fixes it without restating it: a hand-worked example, the
defining property of an RMS norm (unit mean square with a unit scale and no
bias), scale invariance, the axis it normalises over, and where the per-head
bias lands.  CPU only."""
import numpy as np
import pytest

from oracle.bcnorm import bcnorm


def test_worked_example():
    # one head, one rank, N = 2: B = (3, 4) has mean square 12.5, so with
    # eps = 0 it normalises to (3, 4) / sqrt(12.5) = (0.848528..., 1.131370...);
    # scale (2, 1) and bias (0.5, -1) give (2.197056..., 0.131370...)
    B = np.array([3.0, 4.0]).reshape(1, 1, 1, 1, 2)
    out = bcnorm(B, weight=np.array([2.0, 1.0]), bias=np.array([[0.5, -1.0]]), eps=0.0)
    assert out.ravel() == pytest.approx([2.1970562748477141, 0.1313708498984760], rel=1e-15)


def test_unit_mean_square_along_the_state_axis():
    rng = np.random.default_rng(3)
    B = rng.standard_normal((2, 5, 3, 2, 8)) * rng.uniform(0.1, 10.0, (2, 5, 3, 2, 1))
    out = bcnorm(B, np.ones(8), np.zeros((3, 8)), eps=0.0)
    np.testing.assert_allclose((out ** 2).mean(axis=-1), 1.0, rtol=1e-14)
    # normalising over any other axis would not give unit rows
    assert not np.allclose((B / np.sqrt((B ** 2).mean(axis=-2, keepdims=True)) ** 2).mean(axis=-1), 1.0)


def test_scale_invariance_and_bias_per_head():
    rng = np.random.default_rng(4)
    B = rng.standard_normal((1, 4, 3, 2, 6))
    w = rng.standard_normal(6)
    bias = rng.standard_normal((3, 6))
    a = bcnorm(B, w, bias, eps=0.0)
    np.testing.assert_allclose(bcnorm(7.5 * B, w, bias, eps=0.0), a, rtol=1e-13, atol=1e-13)
    # the bias is the output of an all-zero row, per head, shared by the ranks
    Z = np.zeros_like(B)
    out = bcnorm(Z, w, bias, eps=1e-6)
    for h in range(3):
        np.testing.assert_array_equal(out[:, :, h], np.broadcast_to(bias[h], out[:, :, h].shape))


def test_eps_bounds_the_scale_of_a_tiny_row():
    B = np.full((1, 1, 1, 1, 4), 1e-6)
    out = bcnorm(B, np.ones(4), np.zeros((1, 4)), eps=1e-6)
    # mean square 1e-12 << eps: the scale is close to 1 / sqrt(eps) = 1e3
    np.testing.assert_allclose(out.ravel(), 1e-6 / np.sqrt(1e-12 + 1e-6), rtol=1e-15)
