"""Alternative forms of the Mamba-3 scan, written independently of m3_oracle.c.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  Each form follows a
different statement on the pages and must agree with the primary sequential
form to rounding; they are the oracle's pins.  All arithmetic is numpy fp64.

Array conventions as in ``oracle.scan``: x [b,T,h,R,P], dt/lam [b,T,h], A [h],
B/C [b,T,h,R,N], theta [b,T,h,N/2].  ``lam=None`` means 1, ``theta=None`` 0.
Every function returns ``(y [b,T,h,R,P], final_state [b,h,N,P])`` with the
final state in the complex frame (the frame the primary form exposes).
"""
from __future__ import annotations

import numpy as np


def _prep(x, dt, A, B, C, lam, theta):
    x, dt, A, B, C = (np.asarray(v, dtype=np.float64) for v in (x, dt, A, B, C))
    b, T, H, R, P = x.shape
    N = B.shape[-1]
    lam = np.ones_like(dt) if lam is None else np.asarray(lam, dtype=np.float64)
    theta = np.zeros((b, T, H, N // 2)) if theta is None else np.asarray(theta, dtype=np.float64)
    # move heads next to batch: [b,h,T,...]
    xs = np.moveaxis(x, 2, 1)
    Bs = np.moveaxis(B, 2, 1)
    Cs = np.moveaxis(C, 2, 1)
    dts = np.moveaxis(dt, 2, 1)
    lams = np.moveaxis(lam, 2, 1)
    ths = np.moveaxis(theta, 2, 1)
    alpha = np.exp(dts * A[None, :, None])          # alpha_t = exp(dt_t A)
    beta = (1.0 - lams) * dts * alpha                # beta_t = (1 - lambda_t) dt_t alpha_t
    gamma = lams * dts                               # gamma_t = lambda_t dt_t
    return xs, Bs, Cs, alpha, beta, gamma, ths, (b, T, H, R, P, N)


def _rot_pairs(v, phi):
    """Rotate the pairs (2k, 2k+1) of the last axis of v by angle phi[..., k]:
    (a, b) -> (a cos - b sin, a sin + b cos)."""
    a = v[..., 0::2]
    c = v[..., 1::2]
    co, si = np.cos(phi), np.sin(phi)
    out = np.empty_like(v)
    out[..., 0::2] = a * co - c * si
    out[..., 1::2] = a * si + c * co
    return out


def _rot_rows(h, phi):
    """Rotate the row pairs (2k, 2k+1) of a state h[..., N, P] by phi[..., k]."""
    a = h[..., 0::2, :]
    c = h[..., 1::2, :]
    co, si = np.cos(phi)[..., None], np.sin(phi)[..., None]
    out = np.empty_like(h)
    out[..., 0::2, :] = a * co - c * si
    out[..., 1::2, :] = a * si + c * co
    return out


def rope_frame(x, dt, A, B, C, lam=None, theta=None):
    """Propositions 3.2.2 / 3.2.3 (Mamba-3 summary page, §3.2): a real scalar-
    decay SSM whose B and C are rotated by the cumulative angle
    Phi_t = sum_{i=0}^{t} theta_i (the product of the transposed rotations):

        h_t = alpha_t h_{t-1} + beta_t B~_{t-1} x_{t-1}^T + gamma_t B~_t x_t^T
        y_t = C~_t^T h_t,     B~_t = R(Phi_t)^T B_t,  C~_t = R(Phi_t)^T C_t.

    The exposed final state is R(Phi_{T-1}) h_{T-1} (back to the complex frame).
    """
    xs, Bs, Cs, alpha, beta, gamma, ths, (b, T, H, R, P, N) = _prep(x, dt, A, B, C, lam, theta)
    Phi = np.cumsum(ths, axis=2)                                   # [b,h,T,K]
    Bt = _rot_pairs(Bs, -Phi[:, :, :, None, :])                    # R(Phi)^T = R(-Phi)
    Ct = _rot_pairs(Cs, -Phi[:, :, :, None, :])
    h = np.zeros((b, H, N, P))
    v_prev = np.zeros((b, H, N, P))
    y = np.zeros((b, H, T, R, P))
    for t in range(T):
        v = np.einsum("bhrn,bhrp->bhnp", Bt[:, :, t], xs[:, :, t])
        h = (alpha[:, :, t, None, None] * h + beta[:, :, t, None, None] * v_prev
             + gamma[:, :, t, None, None] * v)
        y[:, :, t] = np.einsum("bhrn,bhnp->bhrp", Ct[:, :, t], h)
        v_prev = v
    final = _rot_rows(h, Phi[:, :, T - 1]) if T > 0 else h
    return np.moveaxis(y, 1, 2), final


def quadratic(x, dt, A, B, C, lam=None, theta=None):
    """The parallel (semiseparable) form, §2.3 and eq. (7) of the Mamba-3
    summary page: Y = (L o C~ B~^T) X with L = D W, where D is the decay matrix
    D_ij = prod_{k=j+1}^{i} alpha_k (j <= i, else 0) and W the two-band matrix
    with gamma_i on the diagonal and beta_i at (i, i-1).  Both matrices are
    built explicitly (O(T^2) memory: keep T small).  B and C are the rotated
    ones of the RoPE form; the MIMO block is (C~_i[r] . B~_j[r']) x_j[r'].
    """
    xs, Bs, Cs, alpha, beta, gamma, ths, (b, T, H, R, P, N) = _prep(x, dt, A, B, C, lam, theta)
    Phi = np.cumsum(ths, axis=2)
    Bt = _rot_pairs(Bs, -Phi[:, :, :, None, :])
    Ct = _rot_pairs(Cs, -Phi[:, :, :, None, :])
    y = np.zeros((b, H, T, R, P))
    final = np.zeros((b, H, N, P))
    for bi in range(b):
        for hi in range(H):
            a = alpha[bi, hi]
            D = np.zeros((T, T))
            for i in range(T):
                for j in range(i + 1):
                    D[i, j] = np.prod(a[j + 1:i + 1])              # empty product = 1
            W = np.diag(gamma[bi, hi])
            for i in range(1, T):
                W[i, i - 1] = beta[bi, hi, i]
            L = D @ W
            G = np.einsum("irn,jsn->irjs", Ct[bi, hi], Bt[bi, hi])  # C~_i[r] . B~_j[s]
            y[bi, hi] = np.einsum("ij,irjs,jsp->irp", L, G, xs[bi, hi])
            if T > 0:
                v = np.einsum("jsn,jsp->jnp", Bt[bi, hi], xs[bi, hi])   # v~_j
                hT = np.einsum("j,jnp->np", L[T - 1], v)
                final[bi, hi] = _rot_rows(hT, Phi[bi, hi, T - 1])
    return np.moveaxis(y, 1, 2), final


def conv_then_euler(x, dt, A, B, C, lam=None, theta=None):
    """§3.1.2 of the Mamba-3 summary page: the exponential-trapezoidal
    recurrence is a width-2 data-dependent convolution of the state input
    v_t = B~_t x_t^T (w_t = beta_t v_{t-1} + gamma_t v_t, computed for the whole
    sequence first) followed by the plain first-order recurrence
    h_t = alpha_t h_{t-1} + w_t.  Done in the RoPE frame."""
    xs, Bs, Cs, alpha, beta, gamma, ths, (b, T, H, R, P, N) = _prep(x, dt, A, B, C, lam, theta)
    Phi = np.cumsum(ths, axis=2)
    Bt = _rot_pairs(Bs, -Phi[:, :, :, None, :])
    Ct = _rot_pairs(Cs, -Phi[:, :, :, None, :])
    v = np.einsum("bhtrn,bhtrp->bhtnp", Bt, xs)                     # all v_t at once
    v_shift = np.zeros_like(v)
    v_shift[:, :, 1:] = v[:, :, :-1]                                 # v_{t-1}, v_{-1} = 0
    w = beta[..., None, None] * v_shift + gamma[..., None, None] * v   # the convolution
    h = np.zeros((b, H, N, P))
    y = np.zeros((b, H, T, R, P))
    for t in range(T):
        h = alpha[:, :, t, None, None] * h + w[:, :, t]
        y[:, :, t] = np.einsum("bhrn,bhnp->bhrp", Ct[:, :, t], h)
    final = _rot_rows(h, Phi[:, :, T - 1]) if T > 0 else h
    return np.moveaxis(y, 1, 2), final


def complex_state(x, dt, A, B, C, lam=None, theta=None):
    """The complex SSM of §3.2 (Mamba-3 summary page) in complex arithmetic:
    the state has N/2 complex entries per column, the transition is
    exp(dt A + i theta_t) and eq. (5) is applied with that complex factor:

        h_t = e_t h_{t-1} + (1 - lambda_t) dt_t e_t u_{t-1} + lambda_t dt_t u_t,
        e_t = exp(dt_t A + i theta_t),   u_t = sum_r (B_t[r] as complex) x_t[r]^T

    where a real pair (a, b) is the complex number a + i b, and the readout is
    y_t[r] = Re(sum_k conj(c_k) h_k) = C_t[r]^T h_t on the real pairs."""
    x, dt, A, B, C = (np.asarray(v, dtype=np.float64) for v in (x, dt, A, B, C))
    b, T, H, R, P = x.shape
    N = B.shape[-1]
    K = N // 2
    lam = np.ones_like(dt) if lam is None else np.asarray(lam, dtype=np.float64)
    theta = np.zeros((b, T, H, K)) if theta is None else np.asarray(theta, dtype=np.float64)
    Bc = B[..., 0::2] + 1j * B[..., 1::2]                             # [b,T,h,R,K]
    Cc = C[..., 0::2] + 1j * C[..., 1::2]
    h = np.zeros((b, H, K, P), dtype=np.complex128)
    u_prev = np.zeros_like(h)
    y = np.zeros((b, T, H, R, P))
    for t in range(T):
        d = dt[:, t]                                                  # [b,h]
        e = np.exp(d[..., None] * A[None, :, None] + 1j * theta[:, t])  # [b,h,K]
        u = np.einsum("bhrk,bhrp->bhkp", Bc[:, t], x[:, t])
        h = (e[..., None] * h + ((1.0 - lam[:, t]) * d)[..., None, None] * e[..., None] * u_prev
             + (lam[:, t] * d)[..., None, None] * u)
        y[:, t] = np.real(np.einsum("bhrk,bhkp->bhrp", np.conj(Cc[:, t]), h))
        u_prev = u
    final = np.zeros((b, H, N, P))
    final[:, :, 0::2] = h.real
    final[:, :, 1::2] = h.imag
    return y, final


def mimo_as_siso(scan_fn, x, dt, A, B, C, lam=None, theta=None):
    """§3.3 of the Mamba-3 summary page ("MIMO SSM training"): a rank-R MIMO
    SSM is R^2 coupled SISO systems.  Each input column j drives its own SISO
    state h^(j) (same alpha, beta, gamma, theta), the state is the sum
    h = sum_j h^(j), and output column i reads y^(i) = C^(i)^T h.  Here every
    (i, j) pair is run through ``scan_fn`` as a SISO scan with B^(j), x^(j),
    C^(i) and the outputs are summed over j."""
    x, B, C = (np.asarray(v, dtype=np.float64) for v in (x, B, C))
    b, T, H, R, P = x.shape
    N = B.shape[-1]
    y = np.zeros((b, T, H, R, P))
    final = np.zeros((b, H, N, P))
    for j in range(R):
        for i in range(R):
            yij, hj = scan_fn(x[:, :, :, j:j + 1], dt, A, B[:, :, :, j:j + 1],
                              C[:, :, :, i:i + 1], lam, theta)
            y[:, :, :, i] += yij[:, :, :, 0]
            if i == 0:
                final += hj
    return y, final
