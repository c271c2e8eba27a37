"""The oracle's B / C normalisation and bias (Mamba-3 summary page, §3.4)
against what fixes it without restating it: a hand-worked example, the
defining property of an RMS norm (unit mean square with a unit scale and no
bias), scale invariance, the axis it normalises over, and where the per-head
bias lands.  Plausible mistakes planted in copies of it must each fail one of
these pins.  CPU only."""
import os

import numpy as np
import pytest

import oracle
from oracle.bcnorm import bcnorm


def pin_worked_example(f):
    # one head, one rank, N = 2: B = (3, 4) has mean square 12.5, so with
    # eps = 0 it normalises to (3, 4) / sqrt(12.5) = (0.848528..., 1.131370...);
    # scale (2, 1) and bias (0.5, -1) give (2.197056..., 0.131370...)
    B = np.array([3.0, 4.0]).reshape(1, 1, 1, 1, 2)
    out = f(B, weight=np.array([2.0, 1.0]), bias=np.array([[0.5, -1.0]]), eps=0.0)
    assert out.ravel() == pytest.approx([2.1970562748477141, 0.1313708498984760], rel=1e-15)


def pin_unit_mean_square_along_the_state_axis(f):
    rng = np.random.default_rng(3)
    B = rng.standard_normal((2, 5, 3, 2, 8)) * rng.uniform(0.1, 10.0, (2, 5, 3, 2, 1))
    out = f(B, np.ones(8), np.zeros((3, 8)), eps=0.0)
    np.testing.assert_allclose((out ** 2).mean(axis=-1), 1.0, rtol=1e-14)


def pin_scale_invariance_and_bias_per_head(f):
    rng = np.random.default_rng(4)
    B = rng.standard_normal((1, 4, 3, 2, 6))
    w = rng.standard_normal(6)
    bias = rng.standard_normal((3, 6))
    a = f(B, w, bias, eps=0.0)
    np.testing.assert_allclose(f(7.5 * B, w, bias, eps=0.0), a, rtol=1e-13, atol=1e-13)
    # the bias is the output of an all-zero row, per head, shared by the ranks
    out = f(np.zeros_like(B), w, bias, eps=1e-6)
    for h in range(3):
        np.testing.assert_array_equal(out[:, :, h], np.broadcast_to(bias[h], out[:, :, h].shape))


def pin_eps_bounds_the_scale_of_a_tiny_row(f):
    B = np.full((1, 1, 1, 1, 4), 1e-6)
    out = f(B, np.ones(4), np.zeros((1, 4)), eps=1e-6)
    # mean square 1e-12 << eps: the scale is close to 1 / sqrt(eps) = 1e3
    np.testing.assert_allclose(out.ravel(), 1e-6 / np.sqrt(1e-12 + 1e-6), rtol=1e-15)


PINS = [pin_worked_example, pin_unit_mean_square_along_the_state_axis, pin_scale_invariance_and_bias_per_head,
        pin_eps_bounds_the_scale_of_a_tiny_row]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(bcnorm)


def test_normalising_another_axis_is_not_unit():
    rng = np.random.default_rng(5)
    B = rng.standard_normal((1, 3, 2, 4, 8)) * rng.uniform(0.1, 10.0, (1, 3, 2, 4, 1))
    wrong = B / np.sqrt((B ** 2).mean(axis=-2, keepdims=True))
    assert not np.allclose((wrong ** 2).mean(axis=-1), 1.0)


SRC = open(os.path.join(os.path.dirname(oracle.__file__), "bcnorm.py")).read()

# name -> list of (original snippet, planted replacement)
MUTANTS = {
    "sum_not_mean": [("ms /= N", "ms /= 1")],
    "no_eps": [("np.sqrt(ms + eps)", "np.sqrt(ms)")],
    "no_square_root": [("1.0 / np.sqrt(ms + eps)", "1.0 / (ms + eps)")],
    "scale_after_bias": [("row * scale * weight + bias[idx[2]]", "(row * weight + bias[idx[2]]) * scale")],
    "bias_by_rank": [("bias[idx[2]]", "bias[idx[3] % bias.shape[0]]")],
    "weights_reversed": [("row * scale * weight", "row * scale * weight[::-1]")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name):
    src = SRC
    for old, new in MUTANTS[name]:
        assert old in src, f"{name}: snippet not found: {old}"
        src = src.replace(old, new)
    ns = {}
    exec(compile(src, f"<mutant {name}>", "exec"), ns)
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(ns["bcnorm"])
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passes every pin"
