"""The oracle against small examples worked by hand from the pages' equations
(tests/golden/worked_examples.json: each example cites the section, table or
equation it follows and shows its derivation).  CPU only."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import forms

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))["examples"]


def _arrays(ex):
    T = len(ex["x"])
    N, P = ex["N"], ex["P"]
    x = np.array(ex["x"], dtype=np.float64).reshape(1, T, 1, 1, P)
    dt = np.full((1, T, 1), ex["dt"])
    A = np.array([ex["A"]])
    B = np.array(ex["B"], dtype=np.float64).reshape(1, T, 1, 1, N)
    C = np.array(ex["C"], dtype=np.float64).reshape(1, T, 1, 1, N)
    lam = np.full((1, T, 1), ex["lambda"])
    theta = None if ex["theta"] is None else np.array(ex["theta"], dtype=np.float64).reshape(1, T, 1, N // 2)
    return x, dt, A, B, C, lam, theta


@pytest.mark.parametrize("ex", GOLDEN, ids=lambda e: e["name"])
def test_oracle_reproduces_the_worked_example(ex):
    args = _arrays(ex)
    y, h = oracle.scan(*args)
    np.testing.assert_allclose(y.ravel(), ex["y"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(h.reshape(len(ex["final_state"]), -1), ex["final_state"], rtol=0, atol=1e-14)


@pytest.mark.parametrize("ex", GOLDEN, ids=lambda e: e["name"])
def test_alternative_forms_reproduce_the_worked_example(ex):
    args = _arrays(ex)
    for f in (forms.quadratic, forms.conv_then_euler, forms.rope_frame, forms.complex_state):
        y, h = f(*args)
        np.testing.assert_allclose(np.asarray(y).ravel(), ex["y"], rtol=0, atol=1e-14, err_msg=f.__name__)
