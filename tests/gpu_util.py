"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
(ctypes binding) and the oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {"f32": 1e-4, "bf16": 2e-2}   # max|gpu - ref| / max|ref|


def max_rel(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30)) if ref.size else 0.0


def dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def gpu_scan(m3, d, chunk, with_state=True, stream=None):
    """Prefill through m3_scan_fwd; returns (y, final_state) device tensors."""
    x = d["x"]
    b, T, H, R, P = x.shape
    N = d["B"].shape[-1]
    y = torch.empty_like(x)
    fs = torch.empty(b, H, N, P, device=x.device, dtype=torch.float32) if with_state else None
    m3.m3_scan_fwd(x, d["dt"], d["A"], d["B"], d["C"], d["lam"], d["theta"], y, fs, chunk=chunk, stream=stream)
    return y, fs


def sub_problem(inp, bsel, hsel):
    """The same inputs restricted to batch rows bsel and heads hsel (CPU)."""
    out = {}
    for k, v in inp.items():
        if v is None:
            out[k] = None
        elif k == "A":
            out[k] = v.cpu()[hsel]
        else:
            out[k] = v.cpu()[bsel][:, :, hsel]
    return out


def oracle_scan(inp, bsel=None, hsel=None, nthreads=0):
    """Oracle on (a subset of) the problem; returns fp64 (y, final_state)."""
    if bsel is not None:
        inp = sub_problem(inp, bsel, hsel)
    return oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["lam"], inp["theta"],
                       nthreads=nthreads)


def pick(t, bsel, hsel):
    t = t.cpu()
    return t[bsel][:, :, hsel] if t.dim() >= 3 and t.shape[2] != 0 else t[bsel]
