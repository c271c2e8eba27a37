"""fp64 CPU oracle for the Mamba-3 selective SSM scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  It shares
no code with the CUDA library (``selective_state_space_131_b300``) and
neither side imports the other; the only module both use is the seeded input
generator ``selective_state_space_131_b300.inputs``, which holds none of the
method's arithmetic.

``scan`` is the primary form: the sequential complex-frame recurrence written
in ``m3_oracle.c``; ``scan_bwd`` is its gradient (reverse mode through the
same recurrence, ``m3_oracle_bwd.c``) (Mamba-3 summary page, §3.1 eq. (5)-(6), §3.2
Proposition 3.2.1, §3.3 MIMO).  ``forms`` holds independently written
alternative forms (RoPE frame, quadratic semiseparable mask, width-2
convolution, MIMO as R^2 SISO systems, complex arithmetic) used as pins.
``bcnorm`` is the B / C normalisation and bias of the Mamba-3 block (§3.4),
applied to B and C before the scan.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "m3_oracle.c")
_SRC_BWD = os.path.join(_HERE, "m3_oracle_bwd.c")
_LIB = os.path.join(_HERE, "libm3oracle.so")
_lib = None


def build(src: str = _SRC, out: str = _LIB, extra_flags=(), src_bwd: str = _SRC_BWD) -> str:
    """Compile the C oracle (forward and gradient) with gcc (plain -O2, IEEE
    arithmetic, OpenMP)."""
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", *extra_flags,
           "-o", out, src, src_bwd, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def load(path: str | None = None):
    """Load (building if needed) the oracle shared library."""
    global _lib
    if path is None:
        if _lib is not None:
            return _lib
        if (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC),
                                                                         os.path.getmtime(_SRC_BWD)):
            build()
        path = _LIB
    lib = ctypes.CDLL(path)
    d = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.oracle_scan_f64.argtypes = [i64] * 6 + [d] * 12 + [ctypes.c_int]
    lib.oracle_scan_f64.restype = ctypes.c_int
    if hasattr(lib, "oracle_scan_bwd_f64"):
        lib.oracle_scan_bwd_f64.argtypes = [i64] * 6 + [d] * 22 + [ctypes.c_int]
        lib.oracle_scan_bwd_f64.restype = ctypes.c_int
    lib.oracle_max_threads.restype = ctypes.c_int
    if path == _LIB:
        _lib = lib
    return lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor (CPU); upcast exactly
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(load().oracle_max_threads())


def scan(x, dt, A, B, C, lam=None, theta=None, h0=None, prevB=None, prevx=None,
         nthreads: int = 0, lib=None):
    """Run the sequential fp64 scan.

    Shapes: x [b,T,h,R,P], dt/lam [b,T,h], A [h], B/C [b,T,h,R,N],
    theta [b,T,h,N/2], h0 [b,h,N,P], prevB [b,h,R,N], prevx [b,h,R,P].
    ``lam``/``theta``/``h0``/``prev*`` may be None (1, 0, 0, 0).
    Inputs of any float dtype are upcast exactly to fp64.
    Returns ``(y [b,T,h,R,P], hT [b,h,N,P])`` as float64 arrays.
    """
    lib = lib or load()
    x, dt, A, B, C = (_f64(v) for v in (x, dt, A, B, C))
    lam, theta, h0, prevB, prevx = (_f64(v) for v in (lam, theta, h0, prevB, prevx))
    b, T, H, R, P = x.shape
    N = B.shape[-1]
    assert dt.shape == (b, T, H) and A.shape == (H,)
    assert B.shape == (b, T, H, R, N) and C.shape == (b, T, H, R, N)
    if lam is not None:
        assert lam.shape == (b, T, H)
    if theta is not None:
        assert theta.shape == (b, T, H, N // 2)
    if h0 is not None:
        assert h0.shape == (b, H, N, P)
    if (prevB is None) != (prevx is None):
        raise ValueError("prevB and prevx go together")
    if prevB is not None:
        assert prevB.shape == (b, H, R, N) and prevx.shape == (b, H, R, P)
    y = np.zeros((b, T, H, R, P), dtype=np.float64)
    hT = np.zeros((b, H, N, P), dtype=np.float64)
    rc = lib.oracle_scan_f64(b, T, H, P, N, R, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                             _ptr(lam), _ptr(theta), _ptr(h0), _ptr(prevB), _ptr(prevx),
                             _ptr(y), _ptr(hT), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_scan_f64 failed with {rc}")
    return y, hT


def step(state, x_t, dt_t, A, B_t, C_t, lam_t, theta_t, prevB=None, prevx=None, lib=None):
    """One decode step from ``state`` (complex frame): the scan with T = 1.

    Shapes: state [b,h,N,P], x_t [b,h,R,P], dt_t/lam_t [b,h], B_t/C_t [b,h,R,N],
    theta_t [b,h,N/2].  Returns ``(y_t [b,h,R,P], new_state [b,h,N,P])``.
    """
    x_t = _f64(x_t)
    add_t = lambda a: None if a is None else _f64(a)[:, None]
    y, hT = scan(x_t[:, None], add_t(dt_t), A, add_t(B_t), add_t(C_t), add_t(lam_t),
                 add_t(theta_t), h0=state, prevB=prevB, prevx=prevx, lib=lib)
    return y[:, 0], hT


def scan_bwd(x, dt, A, B, C, lam, theta, dy, dfinal=None, h0=None, prevB=None, prevx=None,
             nthreads: int = 0, lib=None):
    """Gradient of L = <dy, y> + <dfinal, final_state> of the scan with respect
    to every input (m3_oracle_bwd.c: reverse mode through the sequential
    recurrence, fp64).  Shapes as in ``scan``; dy [b,T,h,R,P], dfinal
    [b,h,N,P] or None.

    Returns a dict of float64 arrays: dx, ddt, dA [h] (summed over b), dB,
    dC, dlam (None without lambda), dtheta (None without theta), dh0, and
    dprevB / dprevx (None without a previous token).
    """
    lib = lib or load()
    x, dt, A, B, C = (_f64(v) for v in (x, dt, A, B, C))
    lam, theta, h0, prevB, prevx = (_f64(v) for v in (lam, theta, h0, prevB, prevx))
    dy, dfinal = _f64(dy), _f64(dfinal)
    b, T, H, R, P = x.shape
    N = B.shape[-1]
    assert dy.shape == x.shape and B.shape == C.shape == (b, T, H, R, N)
    if (prevB is None) != (prevx is None):
        raise ValueError("prevB and prevx go together")
    z = lambda *s: np.zeros(s, dtype=np.float64)
    out = {"dx": z(b, T, H, R, P), "ddt": z(b, T, H), "dB": z(b, T, H, R, N), "dC": z(b, T, H, R, N),
           "dlam": z(b, T, H) if lam is not None else None,
           "dtheta": z(b, T, H, N // 2) if theta is not None else None,
           "dh0": z(b, H, N, P),
           "dprevB": z(b, H, R, N) if prevB is not None else None,
           "dprevx": z(b, H, R, P) if prevB is not None else None}
    dA_bh = z(b, H)
    rc = lib.oracle_scan_bwd_f64(b, T, H, P, N, R, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(lam),
                                 _ptr(theta), _ptr(h0), _ptr(prevB), _ptr(prevx), _ptr(dy), _ptr(dfinal),
                                 _ptr(out["dx"]), _ptr(out["ddt"]), _ptr(out["dB"]), _ptr(out["dC"]),
                                 _ptr(out["dlam"]), _ptr(out["dtheta"]), _ptr(dA_bh), _ptr(out["dh0"]),
                                 _ptr(out["dprevB"]), _ptr(out["dprevx"]), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_scan_bwd_f64 failed with {rc}")
    out["dA"] = dA_bh.sum(axis=0)
    return out
