"""Pins for the fp64 gradient oracle (oracle.scan_bwd): checks against
mathematics that does not re-type the oracle's reverse loop.

  * central finite differences of the pinned forward oracle (oracle.scan)
    along random directions, for every input;
  * Euler's identity for homogeneous functions: y and the final state are
    linear in (h0, x, prev_x) jointly, in (h0, B, prev_B) jointly, and y is
    linear in C, so <dx, x> + <dh0, h0> + <dprev_x, prev_x> = L, and so on;
  * reverse-mode automatic differentiation (torch, CPU fp64) of the RoPE-frame
    form of the scan (Mamba-3 summary page, Propositions 3.2.2 / 3.2.3), written
    here independently of both oracles.

Every pin takes ``bwd(x, dt, A, B, C, lam, theta, dy, dfinal, h0, prevB, prevx)
-> dict`` so that the mutation tests can run the same pins against broken
copies of the gradient oracle; a pin raises AssertionError on disagreement.
"""
from __future__ import annotations

import numpy as np

import oracle

NAMES = ("x", "dt", "A", "B", "C", "lam", "theta", "h0", "prevB", "prevx")
GRAD = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "lam": "dlam", "theta": "dtheta",
        "h0": "dh0", "prevB": "dprevB", "prevx": "dprevx"}


def problem(seed, b=2, T=17, H=2, P=5, N=6, R=2, init=True):
    """A small fp64 problem with the workloads' distributions, a random
    initial state and previous token, and random upstream gradients."""
    rng = np.random.default_rng(seed)
    p = {
        "x": rng.standard_normal((b, T, H, R, P)),
        "dt": np.log1p(np.exp(rng.standard_normal((b, T, H)) - 1.0)),
        "A": -np.exp(rng.uniform(0.0, np.log(16.0), H)),
        "B": rng.standard_normal((b, T, H, R, N)) / np.sqrt(N),
        "C": rng.standard_normal((b, T, H, R, N)) / np.sqrt(N),
        "lam": 1.0 / (1.0 + np.exp(-rng.standard_normal((b, T, H)))),
        "theta": rng.standard_normal((b, T, H, N // 2)) * 0.7,
        "h0": 0.5 * rng.standard_normal((b, H, N, P)) if init else None,
        "prevB": rng.standard_normal((b, H, R, N)) / np.sqrt(N) if init else None,
        "prevx": rng.standard_normal((b, H, R, P)) if init else None,
    }
    up = {"dy": rng.standard_normal((b, T, H, R, P)), "dfinal": rng.standard_normal((b, H, N, P))}
    return p, up


def loss(p, up):
    y, fs = oracle.scan(p["x"], p["dt"], p["A"], p["B"], p["C"], p["lam"], p["theta"], h0=p["h0"],
                        prevB=p["prevB"], prevx=p["prevx"])
    return float(np.sum(y * up["dy"]) + np.sum(fs * up["dfinal"])), y, fs


def call(bwd, p, up):
    return bwd(p["x"], p["dt"], p["A"], p["B"], p["C"], p["lam"], p["theta"], up["dy"], up["dfinal"], p["h0"],
               p["prevB"], p["prevx"])


def pin_bwd_finite_differences(bwd):
    """<grad, d> equals the central difference of L along d, for two random
    directions d per input (relative to |grad| |d|)."""
    p, up = problem(31)
    g = call(bwd, p, up)
    rng = np.random.default_rng(32)
    for name in NAMES:
        for _ in range(2):
            d = rng.standard_normal(p[name].shape)
            eps = 1e-5
            pp = dict(p, **{name: p[name] + eps * d})
            pm = dict(p, **{name: p[name] - eps * d})
            fd = (loss(pp, up)[0] - loss(pm, up)[0]) / (2 * eps)
            ip = float(np.sum(g[GRAD[name]] * d))
            scale = np.linalg.norm(g[GRAD[name]]) * np.linalg.norm(d) + 1e-300
            assert abs(fd - ip) <= 1e-7 * scale, (name, fd, ip, scale)


def pin_bwd_homogeneity(bwd):
    """Euler's identity: y and the final state are homogeneous of degree 1 in
    (h0, x, prev_x) and in (h0, B, prev_B); y alone is linear in C."""
    for init in (False, True):
        p, up = problem(41 + init, init=init)
        L, y, _ = loss(p, up)
        g = call(bwd, p, up)
        dot = lambda a, b: 0.0 if a is None else float(np.sum(a * b))
        sx = dot(g["dx"], p["x"]) + (dot(g["dh0"], p["h0"]) + dot(g["dprevx"], p["prevx"]) if init else 0.0)
        sb = dot(g["dB"], p["B"]) + (dot(g["dh0"], p["h0"]) + dot(g["dprevB"], p["prevB"]) if init else 0.0)
        sc = dot(g["dC"], p["C"])
        ly = float(np.sum(y * up["dy"]))
        scale = abs(L) + abs(ly) + 1.0
        assert abs(sx - L) <= 1e-11 * scale, ("x", sx, L)
        assert abs(sb - L) <= 1e-11 * scale, ("B", sb, L)
        assert abs(sc - ly) <= 1e-11 * scale, ("C", sc, ly)


def rope_form_torch(t, up):
    """The scan in the rotated frame (B, C rotated by the cumulative angle,
    real decay-and-trapezoid recurrence), torch fp64; returns L."""
    import torch
    x, dt, A, B, C, lam, th = t["x"], t["dt"], t["A"], t["B"], t["C"], t["lam"], t["theta"]
    b, T, H, R, P = x.shape
    N = B.shape[-1]
    phi = torch.cumsum(th, dim=1)                                    # Phi_t = sum_{i<=t} theta_i

    def rot(v, ang, sign):
        a, bb = v[..., 0::2], v[..., 1::2]
        c, s = torch.cos(ang), sign * torch.sin(ang)
        return torch.stack((a * c - bb * s, a * s + bb * c), dim=-1).reshape(v.shape)
    Bt = rot(B, phi[:, :, :, None, :], -1.0)
    Ct = rot(C, phi[:, :, :, None, :], -1.0)
    alpha = torch.exp(dt * A)
    beta = (1.0 - lam) * dt * alpha
    gamma = lam * dt
    h = t["h0"]
    v_prev = torch.einsum("bhrn,bhrp->bhnp", t["prevB"], t["prevx"])
    ys = []
    for i in range(T):
        v = torch.einsum("bhrn,bhrp->bhnp", Bt[:, i], x[:, i])
        h = alpha[:, i, :, None, None] * h + beta[:, i, :, None, None] * v_prev + gamma[:, i, :, None, None] * v
        ys.append(torch.einsum("bhrn,bhnp->bhrp", Ct[:, i], h))
        v_prev = v
    y = torch.stack(ys, 1)
    # final state back in the complex frame: rows rotated by +Phi_{T-1}
    hf = rot(h.transpose(-1, -2), phi[:, T - 1, :, None, :], 1.0).transpose(-1, -2)
    return (y * up["dy"]).sum() + (hf * up["dfinal"]).sum()


def pin_bwd_autograd_rope_form(bwd):
    """Reverse-mode autodiff of the independently written RoPE-frame form gives
    the same gradients, to 1e-10."""
    import torch
    p, up = problem(51, b=1, T=9, H=2, P=3, N=4, R=2)
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in p.items()}
    tu = {k: torch.tensor(v, dtype=torch.float64) for k, v in up.items()}
    L = rope_form_torch(t, tu)
    grads = torch.autograd.grad(L, [t[k] for k in NAMES])
    g = call(bwd, p, up)
    for name, ga in zip(NAMES, grads):
        ref = ga.numpy()
        got = g[GRAD[name]]
        err = float(np.max(np.abs(got - ref)) / (np.max(np.abs(ref)) + 1e-300))
        assert err <= 1e-10, (name, err)


ALL_PINS = [pin_bwd_finite_differences, pin_bwd_homogeneity, pin_bwd_autograd_rope_form]
