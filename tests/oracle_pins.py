"""Pins for the fp64 oracle: checks against what the Mamba-3 pages and plain
mathematics fix, none of which re-types the oracle's own loop.

Every pin takes ``scan(x, dt, A, B, C, lam, theta, h0=None, prevB=None,
prevx=None) -> (y, final_state)`` so that test_oracle_mutations.py can run
the same pins against deliberately broken copies of the oracle.  A pin
raises AssertionError when the scan under test disagrees.
"""
from __future__ import annotations

import numpy as np

from oracle import forms

TOL = 1e-11          # fp64 agreement between two exact forms (relative to max |ref|)


def rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / scale) if a.size else 0.0


def random_problem(seed, b=2, T=24, H=2, P=5, N=6, R=1, lam=True, theta=True, theta_scale=1.0):
    """A small random problem in fp64 with the workloads' distributions."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((b, T, H, R, P))
    B = rng.standard_normal((b, T, H, R, N)) / np.sqrt(N)
    C = rng.standard_normal((b, T, H, R, N)) / np.sqrt(N)
    dt = np.log1p(np.exp(rng.standard_normal((b, T, H)) - 1.0))        # softplus
    A = -np.exp(rng.uniform(0.0, np.log(16.0), H))
    la = 1.0 / (1.0 + np.exp(-rng.standard_normal((b, T, H)))) if lam else None
    th = (dt[..., None] * rng.standard_normal((1, 1, H, N // 2)) * theta_scale) if theta else None
    return x, dt, A, B, C, la, th


def pin_mamba2_reduction(scan):
    """lambda = 1 and theta = 0 give the Mamba-2 (exponential-Euler) update
    h_t = alpha_t h_{t-1} + dt_t B_t x_t^T, y_t = C_t^T h_t
    (Mamba-3 summary page §2.2 and the first special case under eq. (6))."""
    for R in (1, 2):
        x, dt, A, B, C, _, _ = random_problem(11 + R, R=R, lam=False, theta=False)
        b, T, H, _, P = x.shape
        N = B.shape[-1]
        y_ref = np.zeros_like(x)
        h_ref = np.zeros((b, H, N, P))
        for t in range(T):
            a = np.exp(dt[:, t] * A[None, :])
            h_ref = (a[..., None, None] * h_ref
                     + dt[:, t, :, None, None] * np.einsum("bhrn,bhrp->bhnp", B[:, t], x[:, t]))
            y_ref[:, t] = np.einsum("bhrn,bhnp->bhrp", C[:, t], h_ref)
        for lam, th in ((None, None), (np.ones_like(dt), np.zeros(dt.shape + (N // 2,)))):
            y, hT = scan(x, dt, A, B, C, lam, th)
            assert rel_err(y, y_ref) < TOL, ("mamba2 y", rel_err(y, y_ref))
            assert rel_err(hT, h_ref) < TOL, ("mamba2 state", rel_err(hT, h_ref))


def pin_closed_form(scan):
    """Constant dt, lambda, B, C and x with theta = 0: eq. (6) is a geometric
    series, h_t = v [gamma (1 - alpha^(t+1)) + beta (1 - alpha^t)] / (1 - alpha)
    with v = B x^T (v_{-1} = 0)."""
    rng = np.random.default_rng(5)
    b, T, H, R, P, N = 1, 40, 1, 1, 3, 4
    d, lam_v, A_v = 0.07, 0.3, -1.7
    Bv = rng.standard_normal(N)
    Cv = rng.standard_normal(N)
    xv = rng.standard_normal(P)
    x = np.broadcast_to(xv, (b, T, H, R, P)).copy()
    B = np.broadcast_to(Bv, (b, T, H, R, N)).copy()
    C = np.broadcast_to(Cv, (b, T, H, R, N)).copy()
    dt = np.full((b, T, H), d)
    lam = np.full((b, T, H), lam_v)
    A = np.array([A_v])
    y, hT = scan(x, dt, A, B, C, lam, None)
    alpha = np.exp(d * A_v)
    beta = (1 - lam_v) * d * alpha
    gamma = lam_v * d
    v = np.outer(Bv, xv)
    for t in range(T):
        h_t = v * (gamma * (1 - alpha ** (t + 1)) + beta * (1 - alpha ** t)) / (1 - alpha)
        assert rel_err(y[0, t, 0, 0], Cv @ h_t) < 1e-12, ("closed form", t)
    assert rel_err(hT[0, 0], h_t) < 1e-12


def pin_quadratic(scan):
    """Parallel semiseparable form, eq. (7): Y = (L o C~B~^T) X with
    L = decay matrix x two-band matrix, built explicitly (forms.quadratic)."""
    for seed, R in ((21, 1), (22, 2)):
        args = random_problem(seed, T=20, R=R)
        y, hT = scan(*args)
        yq, hq = forms.quadratic(*args)
        assert rel_err(y, yq) < TOL, ("quadratic y", rel_err(y, yq))
        assert rel_err(hT, hq) < TOL, ("quadratic state", rel_err(hT, hq))


def pin_conv(scan):
    """§3.1.2: width-2 convolution of the state input, then the first-order
    recurrence (forms.conv_then_euler)."""
    for seed, R in ((31, 1), (32, 3)):
        args = random_problem(seed, T=30, R=R)
        y, hT = scan(*args)
        yc, hc = forms.conv_then_euler(*args)
        assert rel_err(y, yc) < TOL, ("conv y", rel_err(y, yc))
        assert rel_err(hT, hc) < TOL, ("conv state", rel_err(hT, hc))


def pin_rope(scan):
    """Propositions 3.2.2 / 3.2.3: scalar-decay SSM on B, C rotated by the
    cumulative angles (forms.rope_frame), with large angles too."""
    for seed, scale in ((41, 1.0), (42, 25.0)):
        args = random_problem(seed, T=40, R=2, theta_scale=scale)
        y, hT = scan(*args)
        yr, hr = forms.rope_frame(*args)
        assert rel_err(y, yr) < TOL, ("rope y", rel_err(y, yr))
        assert rel_err(hT, hr) < TOL, ("rope state", rel_err(hT, hr))


def pin_complex(scan):
    """§3.2: the complex-valued SSM with transition exp(dt A + i theta) in
    complex arithmetic (forms.complex_state); fixes the rotation direction."""
    args = random_problem(51, T=33, R=2, N=8)
    y, hT = scan(*args)
    yc, hc = forms.complex_state(*args)
    assert rel_err(y, yc) < TOL, ("complex y", rel_err(y, yc))
    assert rel_err(hT, hc) < TOL, ("complex state", rel_err(hT, hc))


def pin_parity(scan):
    """§3.2: parity needs the rotation h_t = R(pi x_t) h_{t-1}.  With input
    only at t = 0 and angle pi * b_s on every pair at s >= 1,
    y_t = (-1)^(sum_{s=1}^t b_s) (prod_{s=2}^t alpha_s)(alpha_1 gamma_0 + beta_1) C_t^T u_0
    for t >= 1 and y_0 = gamma_0 C_0^T u_0."""
    rng = np.random.default_rng(61)
    b, T, H, R, P, N = 1, 30, 1, 1, 4, 6
    x, dt, A, B, C, lam, _ = random_problem(61, b=b, T=T, H=H, R=R, P=P, N=N)
    x[:, 1:] = 0.0
    bits = rng.integers(0, 2, T)
    bits[0] = 0
    theta = np.broadcast_to((np.pi * bits)[None, :, None, None], (b, T, H, N // 2)).copy()
    y, _ = scan(x, dt, A, B, C, lam, theta)
    alpha = np.exp(dt[0, :, 0] * A[0])
    beta = (1 - lam[0, :, 0]) * dt[0, :, 0] * alpha
    gamma = lam[0, :, 0] * dt[0, :, 0]
    u0 = np.outer(B[0, 0, 0, 0], x[0, 0, 0, 0])
    assert rel_err(y[0, 0, 0, 0], gamma[0] * (C[0, 0, 0, 0] @ u0)) < 1e-12
    for t in range(1, T):
        sign = (-1.0) ** int(bits[1:t + 1].sum())
        coef = sign * np.prod(alpha[2:t + 1]) * (alpha[1] * gamma[0] + beta[1])
        ref = coef * (C[0, t, 0, 0] @ u0)
        assert abs(y[0, t, 0, 0] - ref).max() <= 1e-12 * max(np.abs(ref).max(), 1e-300), ("parity", t)


def pin_norm(scan):
    """Proposition 3.2.1: the transition is a rotation.  With alpha = 1
    (A = 0), lambda = 1 and no input after t = 0 the Frobenius norm of the
    state stays gamma_0 ||u_0||."""
    x, dt, A, B, C, _, theta = random_problem(71, b=1, T=12, H=1, R=1, P=3, N=8, theta_scale=7.0)
    x[:, 1:] = 0.0
    A = np.zeros(1)
    u0 = np.outer(B[0, 0, 0, 0], x[0, 0, 0, 0])
    ref = dt[0, 0, 0] * np.linalg.norm(u0)
    for T in range(1, 12):
        _, hT = scan(x[:, :T], dt[:, :T], A, B[:, :T], C[:, :T], None, theta[:, :T])
        assert abs(np.linalg.norm(hT) - ref) < 1e-12 * ref, ("norm", T)


def pin_mimo(scan):
    """§3.3: a rank-R MIMO SSM equals R^2 coupled SISO systems (summed states,
    per-column readout); also R = 1 MIMO is the SISO scan."""
    args = random_problem(81, T=18, R=3, N=6, P=4)
    y, hT = scan(*args)
    ym, hm = forms.mimo_as_siso(scan, *args)
    assert rel_err(y, ym) < TOL, ("mimo y", rel_err(y, ym))
    assert rel_err(hT, hm) < TOL, ("mimo state", rel_err(hT, hm))


def pin_second_order(scan):
    """§3.1 and Appendix A.2 (Remark 3): with lambda = 1/2 the rule is second
    order (global error / 4 per halving of dt); lambda = 1 (Euler) is first
    order (/2).  Scalar LTI system h' = -h + sin(s), h(0) = 0, exact solution
    h(s) = (sin s - cos s + e^{-s}) / 2, read at s = 2."""
    def err(dt_v, lam_v):
        T = int(round(2.0 / dt_v)) + 1
        s = dt_v * np.arange(T)
        x = np.sin(s).reshape(1, T, 1, 1, 1)
        B = np.zeros((1, T, 1, 1, 2))
        B[..., 0] = 1.0
        C = B.copy()
        dt = np.full((1, T, 1), dt_v)
        lam = np.full((1, T, 1), lam_v)
        y, _ = scan(x, dt, np.array([-1.0]), B, C, lam, None)
        exact = (np.sin(s[-1]) - np.cos(s[-1]) + np.exp(-s[-1])) / 2
        return abs(y[0, -1, 0, 0, 0] - exact)
    e = [err(d, 0.5) for d in (0.1, 0.05, 0.025)]
    r = [e[0] / e[1], e[1] / e[2]]
    assert all(3.5 < v < 4.5 for v in r), ("trapezoid order", r)
    e1 = [err(d, 1.0) for d in (0.1, 0.05, 0.025)]
    r1 = [e1[0] / e1[1], e1[1] / e1[2]]
    assert all(1.7 < v < 2.3 for v in r1), ("euler order", r1)


def pin_split(scan):
    """The state is the whole carry: a scan of T1 + T2 tokens equals a scan of
    T2 tokens started from the first scan's state and last-token (B, x), and
    equals T single steps chained the same way."""
    x, dt, A, B, C, lam, th = random_problem(91, T=15, R=2)
    y, hT = scan(x, dt, A, B, C, lam, th)
    T1 = 6
    y1, h1 = scan(x[:, :T1], dt[:, :T1], A, B[:, :T1], C[:, :T1], lam[:, :T1], th[:, :T1])
    y2, h2 = scan(x[:, T1:], dt[:, T1:], A, B[:, T1:], C[:, T1:], lam[:, T1:], th[:, T1:],
                  h0=h1, prevB=B[:, T1 - 1], prevx=x[:, T1 - 1])
    assert rel_err(np.concatenate([y1, y2], axis=1), y) < TOL
    assert rel_err(h2, hT) < TOL
    h = np.zeros_like(hT)
    for t in range(x.shape[1]):
        pB = B[:, t - 1] if t > 0 else np.zeros_like(B[:, 0])
        px = x[:, t - 1] if t > 0 else np.zeros_like(x[:, 0])
        sl = slice(t, t + 1)
        yt, h = scan(x[:, sl], dt[:, sl], A, B[:, sl], C[:, sl], lam[:, sl], th[:, sl],
                     h0=h, prevB=pB, prevx=px)
        assert rel_err(yt[:, 0], y[:, t]) < TOL, ("steps", t)
    assert rel_err(h, hT) < TOL


ALL_PINS = [pin_mamba2_reduction, pin_closed_form, pin_quadratic, pin_conv, pin_rope,
            pin_complex, pin_parity, pin_norm, pin_mimo, pin_second_order, pin_split]
