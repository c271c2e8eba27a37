"""Seeded synthetic inputs for the Mamba-3 scan (shared by the oracle side and
the CUDA side; holds none of the method's arithmetic -- only the input
distributions).

Distributions (the workloads of the Mamba-3 pages, restated):
  x ~ N(0, 1);  B, C ~ N(0, 1/N);
  dt = softplus(N(0, 1) + b_h), with b_h per head chosen so that softplus(b_h)
       is log-uniform in [1e-3, 1e-1];
  A_h = -exp(U[0, ln 16]) per head;
  lambda = sigmoid(N(0, 1));
  theta_t = dt_t * omega, omega ~ N(0, 1) per (head, rotation pair), fixed
       over batch and time.
Draw order (fixed, from one ``torch.Generator`` seeded with ``seed``):
  b_h, omega, A, x, B, C, dt-noise, lambda-noise.
x, B, C and theta are cast to the requested dtype after drawing; dt, lambda
and A stay fp32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class ScanShape:
    batch: int
    seqlen: int
    heads: int
    headdim: int          # P
    dstate: int           # N (even)
    rank: int = 1         # R
    chunk: int = 64       # Q
    dtype: str = "bf16"   # of x, B, C, theta, y
    with_lambda: bool = True
    with_theta: bool = True


@dataclass(frozen=True)
class DecodeShape:
    batch: int
    heads: int
    headdim: int
    dstate: int
    rank: int = 1
    steps: int = 1024
    dtype: str = "f32"


# The five workloads, by name: four prefill scans and the decode sweep.
TINY = "tiny_siso_f32_b1h2T256P16N16"
SSD_EQUIV = "ssd_equiv_bf16_b8h32T4096P64N128"
SISO = "m3_siso_bf16_b8h32T8192P64N64"
MIMO = "m3_mimo_r4_bf16_b8h32T4096P64N64"
DECODE = "decode_f32_b256h32P64N64"
WORKLOADS = {
    TINY: ScanShape(batch=1, seqlen=256, heads=2, headdim=16, dstate=16, rank=1, chunk=32, dtype="f32"),
    SSD_EQUIV: ScanShape(batch=8, seqlen=4096, heads=32, headdim=64, dstate=128, rank=1, chunk=64, dtype="bf16",
                         with_lambda=False, with_theta=False),
    SISO: ScanShape(batch=8, seqlen=8192, heads=32, headdim=64, dstate=64, rank=1, chunk=64, dtype="bf16"),
    MIMO: ScanShape(batch=8, seqlen=4096, heads=32, headdim=64, dstate=64, rank=4, chunk=64, dtype="bf16"),
    DECODE: DecodeShape(batch=256, heads=32, headdim=64, dstate=64, rank=1, steps=1024, dtype="f32"),
}
# the base seed of each workload's synthetic inputs
WORKLOAD_SEEDS = {TINY: 0, SSD_EQUIV: 1, SISO: 2, MIMO: 3, DECODE: 4}
PREFILL_WORKLOADS = (SSD_EQUIV, SISO, MIMO)


def _head_params(g, heads, K, device):
    s = torch.exp(torch.empty(heads, device=device).uniform_(math.log(1e-3), math.log(1e-1), generator=g))
    b_h = torch.log(torch.expm1(s))                       # softplus(b_h) = s
    omega = torch.randn(heads, K, device=device, generator=g)
    A = -torch.exp(torch.empty(heads, device=device).uniform_(0.0, math.log(16.0), generator=g))
    return b_h, omega, A


def make_scan_inputs(shape: ScanShape, seed: int, device="cpu"):
    """Inputs of one prefill scan as a dict of tensors on ``device``:
    x [b,T,h,R,P], dt [b,T,h], A [h], B, C [b,T,h,R,N], lam [b,T,h] or None,
    theta [b,T,h,N/2] or None."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    b, T, H, P, N, R = shape.batch, shape.seqlen, shape.heads, shape.headdim, shape.dstate, shape.rank
    dt_ = _DTYPES[shape.dtype]
    b_h, omega, A = _head_params(g, H, N // 2, device)
    x = torch.randn(b, T, H, R, P, device=device, generator=g)
    B = torch.randn(b, T, H, R, N, device=device, generator=g) * (1.0 / math.sqrt(N))
    C = torch.randn(b, T, H, R, N, device=device, generator=g) * (1.0 / math.sqrt(N))
    dt = torch.nn.functional.softplus(torch.randn(b, T, H, device=device, generator=g) + b_h)
    lam = torch.sigmoid(torch.randn(b, T, H, device=device, generator=g))
    theta = dt[..., None] * omega[None, None] if shape.with_theta else None
    return {
        "x": x.to(dt_).contiguous(),
        "dt": dt.contiguous(),
        "A": A.contiguous(),
        "B": B.to(dt_).contiguous(),
        "C": C.to(dt_).contiguous(),
        "lam": lam.contiguous() if shape.with_lambda else None,
        "theta": theta.to(dt_).contiguous() if theta is not None else None,
    }


def make_decode_inputs(shape: DecodeShape, seed: int, device="cpu"):
    """Inputs of a decode sweep of ``shape.steps`` tokens: every per-token
    array has a leading axis of steps + 1; token s + 1 is the input of step s
    and token s is its previous token (the carry of the beta term).  Also a
    random N(0, 1) fp32 initial state [b,h,N,P]."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    S, b, H, P, N, R = shape.steps + 1, shape.batch, shape.heads, shape.headdim, shape.dstate, shape.rank
    dt_ = _DTYPES[shape.dtype]
    b_h, omega, A = _head_params(g, H, N // 2, device)
    x = torch.randn(S, b, H, R, P, device=device, generator=g)
    B = torch.randn(S, b, H, R, N, device=device, generator=g) * (1.0 / math.sqrt(N))
    C = torch.randn(S, b, H, R, N, device=device, generator=g) * (1.0 / math.sqrt(N))
    dt = torch.nn.functional.softplus(torch.randn(S, b, H, device=device, generator=g) + b_h)
    lam = torch.sigmoid(torch.randn(S, b, H, device=device, generator=g))
    theta = dt[..., None] * omega[None, None]
    state0 = torch.randn(b, H, N, P, device=device, generator=g)
    return {
        "x": x.to(dt_).contiguous(), "dt": dt.contiguous(), "A": A.contiguous(),
        "B": B.to(dt_).contiguous(), "C": C.to(dt_).contiguous(), "lam": lam.contiguous(),
        "theta": theta.to(dt_).contiguous(), "state0": state0.contiguous(),
    }


def make_bcnorm_params(dstate: int, heads: int, seed: int, device="cpu"):
    """Parameters of the B / C normalisation: per-channel scales norm_B, norm_C
    [N] ~ 1 + 0.1 N(0, 1) and per-head, per-channel biases bias_B, bias_C [h, N]
    ~ 0.1 N(0, 1), all fp32 (the scales of a trained norm stay near 1)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    n = lambda *shape: torch.randn(*shape, device=device, generator=g)
    return {"norm_B": 1.0 + 0.1 * n(dstate), "norm_C": 1.0 + 0.1 * n(dstate),
            "bias_B": 0.1 * n(heads, dstate), "bias_C": 0.1 * n(heads, dstate)}
