"""BC normalisation and biases of the Mamba-3 block -- TEST INFRASTRUCTURE
ONLY (see oracle/__init__.py).  Plain numpy fp64.

Mamba-3 summary page, §3.4 (Mamba-3 architecture; "BC/QK normalisation",
"B, C biases"): an RMS normalisation is applied to the B and C projections
(the role query-key normalisation plays in Transformers), then a learnable
bias per head and per channel is added; the data-dependent RoPE rotation
follows.  The pages fix neither the norm's scale nor its epsilon; the reading
taken here: the usual RMS norm over the state axis N with a learnable scale
w in R^N shared by heads and ranks, and a bias b in R^{H x N} shared by the R
ranks of a head:

    B^[..., h, r, n] = B[..., h, r, n] / sqrt(mean_n' B[..., h, r, n']^2 + eps) * w[n] + b[h, n].
"""
from __future__ import annotations

import numpy as np


def bcnorm(B, weight, bias, eps):
    """B [b,T,h,R,N] (any float dtype, upcast exactly), weight [N], bias [h,N]
    -> fp64 [b,T,h,R,N]."""
    B = np.asarray(B, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    bias = np.asarray(bias, dtype=np.float64)
    N = B.shape[-1]
    assert weight.shape == (N,) and bias.shape == (B.shape[2], N)
    out = np.empty_like(B)
    for idx in np.ndindex(*B.shape[:-1]):
        row = B[idx]
        ms = 0.0
        for v in row:
            ms += v * v
        ms /= N
        scale = 1.0 / np.sqrt(ms + eps)
        out[idx] = row * scale * weight + bias[idx[2]]
    return out
