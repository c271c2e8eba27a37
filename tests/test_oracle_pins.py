"""The fp64 oracle against its pins (closed forms, special cases, the pages'
alternative forms, invariants).  CPU only."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


def _scan(x, dt, A, B, C, lam=None, theta=None, h0=None, prevB=None, prevx=None):
    return oracle.scan(x, dt, A, B, C, lam, theta, h0=h0, prevB=prevB, prevx=prevx)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(_scan)


def test_forms_agree_among_themselves():
    """The alternative forms are mutually consistent too (independent of the C code)."""
    args = pins.random_problem(101, T=16, R=2)
    ref = oracle.forms.rope_frame(*args)
    for f in (oracle.forms.quadratic, oracle.forms.conv_then_euler, oracle.forms.complex_state):
        y, h = f(*args)
        assert pins.rel_err(y, ref[0]) < pins.TOL
        assert pins.rel_err(h, ref[1]) < pins.TOL


def test_step_wrapper_matches_scan():
    x, dt, A, B, C, lam, th = pins.random_problem(7, T=3, R=2)
    y, hT = oracle.scan(x, dt, A, B, C, lam, th)
    state = np.zeros_like(hT)
    pB = np.zeros_like(B[:, 0]); px = np.zeros_like(x[:, 0])
    for t in range(3):
        yt, state = oracle.step(state, x[:, t], dt[:, t], A, B[:, t], C[:, t], lam[:, t], th[:, t], pB, px)
        pB, px = B[:, t], x[:, t]
        assert pins.rel_err(yt, y[:, t]) < pins.TOL
    assert pins.rel_err(state, hT) < pins.TOL


def test_empty_sequence():
    x, dt, A, B, C, lam, th = pins.random_problem(8, T=0)
    y, hT = oracle.scan(x, dt, A, B, C, lam, th)
    assert y.shape[1] == 0 and not np.any(hT)


def test_bad_arguments_rejected(oracle_lib):
    # odd N is rejected by the C entry point
    rc = oracle_lib.oracle_scan_f64(1, 1, 1, 1, 3, 1, *([None] * 12), 1)
    assert rc == -1
