"""The fp64 gradient oracle (oracle.scan_bwd) against its pins, and plausible
mistakes planted in copies of it (on the CPU), each of which must fail at least
one pin."""
import os

import numpy as np
import pytest

import oracle
from tests import oracle_bwd_pins as pins


def _bwd(lib=None):
    def bwd(x, dt, A, B, C, lam, theta, dy, dfinal, h0, prevB, prevx):
        return oracle.scan_bwd(x, dt, A, B, C, lam, theta, dy, dfinal, h0=h0, prevB=prevB, prevx=prevx, lib=lib)
    return bwd


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_gradient_oracle_pin(pin):
    pin(_bwd())


def test_gradient_without_optional_inputs():
    """lambda / theta / h0 / prev absent: the same gradients as with lambda = 1,
    theta = 0, zero state and previous token passed explicitly (where defined)."""
    p, up = pins.problem(61, init=False)
    g0 = oracle.scan_bwd(p["x"], p["dt"], p["A"], p["B"], p["C"], None, None, up["dy"], up["dfinal"])
    ones, zeros = np.ones_like(p["dt"]), np.zeros_like(p["theta"])
    g1 = oracle.scan_bwd(p["x"], p["dt"], p["A"], p["B"], p["C"], ones, zeros, up["dy"], up["dfinal"])
    for k in ("dx", "ddt", "dA", "dB", "dC", "dh0"):
        assert np.allclose(g0[k], g1[k], rtol=1e-13, atol=1e-13), k
    assert g0["dlam"] is None and g0["dtheta"] is None and g0["dprevB"] is None


SRC = open(os.path.join(os.path.dirname(oracle.__file__), "m3_oracle_bwd.c")).read()
FWD = os.path.join(os.path.dirname(oracle.__file__), "m3_oracle.c")

MUTANTS = {
    "previous_input_gradient_dropped": [("dup[e] += beta * dz[e];", "")],
    "current_input_gradient_dropped": [("duc[e] += gamma * g[e];", "")],
    "angle_gradient_sign": [("dth += -g0 * w1 + g1 * w0;", "dth += g0 * w1 - g1 * w0;")],
    "adjoint_rotation_not_transposed": [("dz[(2 * k) * P + p] = c * g0 + s * g1;",
                                         "dz[(2 * k) * P + p] = c * g0 - s * g1;"),
                                        ("dz[(2 * k + 1) * P + p] = -s * g0 + c * g1;",
                                         "dz[(2 * k + 1) * P + p] = s * g0 + c * g1;")],
    "angle_gradient_uses_h": [("const double w0 = hc[(2 * k) * P + p] - gamma * uc[(2 * k) * P + p];",
                               "const double w0 = hc[(2 * k) * P + p];"),
                              ("const double w1 = hc[(2 * k + 1) * P + p] - gamma * uc[(2 * k + 1) * P + p];",
                               "const double w1 = hc[(2 * k + 1) * P + p];")],
    "dt_gradient_misses_beta_decay": [("(1.0 + d * A_h)", "1.0")],
    "A_gradient_misses_beta": [("dA_acc += dalpha * alpha * d + dbeta * (1.0 - l) * d * d * alpha;",
                                "dA_acc += dalpha * alpha * d;")],
    "C_gradient_uses_previous_state": [("acc += hc[n * P + p] * dy[(bth * R + r) * P + p];",
                                        "acc += hp[n * P + p] * dy[(bth * R + r) * P + p];")],
    "lambda_gradient_sign": [("dlam[bth] = -dbeta * d * alpha + dgamma * d;",
                              "dlam[bth] = dbeta * d * alpha + dgamma * d;")],
    "x_gradient_uses_C": [("for (int64_t n = 0; n < N; ++n) acc += duc[n * P + p] * Bm[(bth * R + r) * N + n];",
                           "for (int64_t n = 0; n < N; ++n) acc += duc[n * P + p] * Cm[(bth * R + r) * N + n];")],
    "state_gradient_scaled_by_beta": [("g[e] = alpha * dz[e];", "g[e] = beta * dz[e];")],
    "B_gradient_uses_dy": [("for (int64_t p = 0; p < P; ++p) acc += duc[n * P + p] * x[(bth * R + r) * P + p];",
                            "for (int64_t p = 0; p < P; ++p) acc += duc[n * P + p] * dy[(bth * R + r) * P + p];")],
    "previous_B_gradient_uses_current_x": [("acc += dum[n * P + p] * prevx[(unit * R + r) * P + p];",
                                            "acc += dum[n * P + p] * x[(unit * R + r) * P + p];")],
    "readout_gradient_first_rank_only": [
        ("for (int64_t r = 0; r < R; ++r) acc += Cm[(bth * R + r) * N + n] * dy[(bth * R + r) * P + p];",
         "for (int64_t r = 0; r < 1; ++r) acc += Cm[(bth * R + r) * N + n] * dy[(bth * R + r) * P + p];")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_gradient_mutant_is_caught(tmp_path, name):
    src = SRC
    for old, new in MUTANTS[name]:
        assert old in src, f"{name}: snippet not found: {old}"
        src = src.replace(old, new)
    cpath = tmp_path / f"{name}_bwd.c"
    cpath.write_text(src)
    so = oracle.build(FWD, str(tmp_path / f"lib{name}.so"), src_bwd=str(cpath))
    bwd = _bwd(oracle.load(so))
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(bwd)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
