"""Why the decode state stays fp32: a study on the decode workload's input
distributions (dt = softplus(N(0, 1) + b) with softplus(b) in [1e-3, 1e-1],
A = -exp(U[0, ln 16]), theta_t = dt_t omega), with the fp64 oracle step as the
arithmetic and only the carried state rounded between steps.

With dt as small as 1e-3, a step adds gamma B x^T of order 1e-4 to a state of
order 1, below half a bf16 unit in the last place (2^-9 relative), so round-to-
nearest drops it; the lost increments pile up over the steps.  fp32 carries
them.  So a bf16 state (which would halve the decode bytes) misses the 2e-2
bf16 parity bar within a few hundred tokens, and the decode step keeps its
state in fp32 (the pages fix no state precision for decode).
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_131_b300 import inputs


def _chain_error(round_dtype, steps, R=1):
    shape = inputs.DecodeShape(batch=2, heads=8, headdim=64, dstate=64, rank=R, steps=steps, dtype="f32")
    inp = {k: v.double().numpy() for k, v in inputs.make_decode_inputs(shape, 4).items()}
    exact = inp["state0"].copy()
    rounded = torch.from_numpy(exact).to(round_dtype).double().numpy()
    worst = 0.0
    for s in range(steps):
        args = lambda a: (inp["x"][s + 1], inp["dt"][s + 1], inp["A"], inp["B"][s + 1], inp["C"][s + 1],
                          inp["lam"][s + 1], inp["theta"][s + 1])
        y_ex, exact = oracle.step(exact, *args(None), prevB=inp["B"][s], prevx=inp["x"][s])
        y_rd, nxt = oracle.step(rounded, *args(None), prevB=inp["B"][s], prevx=inp["x"][s])
        rounded = torch.from_numpy(nxt).to(round_dtype).double().numpy()
        worst = max(worst, np.abs(y_rd - y_ex).max() / np.abs(y_ex).max())
    return worst


def test_fp32_state_keeps_decode_within_the_fp32_bar():
    assert _chain_error(torch.float32, 256) <= 1e-4


@pytest.mark.parametrize("R", [1, 4])
def test_bf16_state_drifts_past_the_bf16_bar(R):
    assert _chain_error(torch.bfloat16, 256, R) > 2e-2
