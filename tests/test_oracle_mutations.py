"""Plausible mistakes planted in copies of the oracle (on the CPU) must each
fail at least one pin: the pins are strong enough to catch a dropped term, a
wrong sign, a wrong index or a transposed operand."""
import os

import pytest

import oracle
from tests import oracle_pins as pins

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "m3_oracle.c")).read()

# name -> list of (original snippet, planted replacement)
MUTANTS = {
    "drop_beta_term": [("beta * up0[p]", "0.0 * up0[p]"), ("beta * up1[p]", "0.0 * up1[p]")],
    "rotation_sign": [("h0r[p] = c * z0 - s * z1", "h0r[p] = c * z0 + s * z1")],
    "rotation_transposed": [("h0r[p] = c * z0 - s * z1", "h0r[p] = c * z0 + s * z1"),
                            ("h1r[p] = s * z0 + c * z1", "h1r[p] = -s * z0 + c * z1")],
    "beta_uses_current_input": [("beta * up0[p]", "beta * u0[p]"), ("beta * up1[p]", "beta * u1[p]")],
    "gamma_uses_one_minus_lambda": [("const double gamma = l * d;", "const double gamma = (1.0 - l) * d;")],
    "beta_without_alpha": [("(1.0 - l) * d * alpha", "(1.0 - l) * d")],
    "readout_with_B": [("const double* Ct = Cm + bth", "const double* Ct = Bm + bth")],
    "gamma_term_rotated": [("const double z0 = alpha * h0r[p] + beta * up0[p];",
                            "const double z0 = alpha * h0r[p] + beta * up0[p] + gamma * u0[p];"),
                           ("const double z1 = alpha * h1r[p] + beta * up1[p];",
                            "const double z1 = alpha * h1r[p] + beta * up1[p] + gamma * u1[p];"),
                           ("h0r[p] = c * z0 - s * z1 + gamma * u0[p];", "h0r[p] = c * z0 - s * z1;"),
                           ("h1r[p] = s * z0 + c * z1 + gamma * u1[p];", "h1r[p] = s * z0 + c * z1;")],
    "beta_term_not_rotated": [("const double z0 = alpha * h0r[p] + beta * up0[p];",
                               "const double z0 = alpha * h0r[p];"),
                              ("const double z1 = alpha * h1r[p] + beta * up1[p];",
                               "const double z1 = alpha * h1r[p];"),
                              ("h0r[p] = c * z0 - s * z1 + gamma * u0[p];",
                               "h0r[p] = c * z0 - s * z1 + gamma * u0[p] + beta * up0[p];"),
                              ("h1r[p] = s * z0 + c * z1 + gamma * u1[p];",
                               "h1r[p] = s * z0 + c * z1 + gamma * u1[p] + beta * up1[p];")],
    "mimo_first_column_only": [("for (int64_t r = 0; r < R; ++r) acc += Bt[r * N + n]",
                                "for (int64_t r = 0; r < 1; ++r) acc += Bt[r * N + n]")],
    "previous_input_never_updated": [("memcpy(u_prev, u, (size_t)(N * P) * sizeof(double));", "")],
    "angle_ignores_pair_index": [("theta[bth * K + k]", "theta[bth * K]")],
    "decay_without_dt": [("exp(d * A_h)", "exp(A_h)")],
    "initial_carry_ignored": [("acc += prevB[(unit * R + r) * N + n] * prevx[(unit * R + r) * P + p];",
                               "acc += 0.0;")],
    "readout_index_transposed": [("acc += Ct[r * N + n] * hs[n * P + p];",
                                  "acc += Ct[r * N + n] * hs[p * N + n];")],
}


def _mutant_scan(tmp_path, name):
    src = SRC
    for old, new in MUTANTS[name]:
        assert old in src, f"{name}: snippet not found: {old}"
        src = src.replace(old, new)
    cpath = tmp_path / f"{name}.c"
    cpath.write_text(src)
    so = oracle.build(str(cpath), str(tmp_path / f"lib{name}.so"))
    lib = oracle.load(so)

    def scan(x, dt, A, B, C, lam=None, theta=None, h0=None, prevB=None, prevx=None):
        return oracle.scan(x, dt, A, B, C, lam, theta, h0=h0, prevB=prevB, prevx=prevx, lib=lib)
    return scan


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    scan = _mutant_scan(tmp_path, name)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(scan)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
