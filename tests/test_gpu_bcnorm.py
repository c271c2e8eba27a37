"""GPU parity of the prefill with the B / C normalisation and biases fused into
its prologue (m3_scan_fwd_bcnorm) against the oracle: the oracle normalises the
same raw bf16 B and C in fp64 (oracle.bcnorm) and runs its scan on them.
Small shapes over several chunks with ragged tails for every (N, R) the
tensor-core kernel takes, with and without theta / lambda, and the SISO
workload at full size on sampled sequences."""
import numpy as np
import pytest
import torch

import oracle
from oracle.bcnorm import bcnorm
from selective_state_space_131_b300 import inputs
from tests.gpu_util import TOL, dev, max_rel, sub_problem

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module")
def m3():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from selective_state_space_131_b300 import m3scan
    return m3scan


def run_and_check(m3, shape, seed, bsel=None, hsel=None, eps=EPS):
    inp = inputs.make_scan_inputs(shape, seed)
    nrm = inputs.make_bcnorm_params(shape.dstate, shape.heads, seed + 1)
    d, nd = dev(inp), dev(nrm)
    x = d["x"]
    y = torch.empty_like(x)
    fs = torch.empty(shape.batch, shape.heads, shape.dstate, shape.headdim, device="cuda")
    m3.m3_scan_fwd_bcnorm(x, d["dt"], d["A"], d["B"], d["C"], d["lam"], d["theta"], nd["norm_B"], nd["norm_C"],
                          nd["bias_B"], nd["bias_C"], eps, y, fs, chunk=shape.chunk)
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    y, fs = y.float().cpu(), fs.cpu()
    if bsel is not None:
        y, fs = y[bsel][:, :, hsel], fs[bsel][:, hsel]
        inp = sub_problem(inp, bsel, hsel)
        nrm = {k: (v[hsel] if k.startswith("bias") else v) for k, v in nrm.items()}
    f64 = lambda t: t.double().numpy()   # exact: the bf16 values as fp64
    Bn = bcnorm(f64(inp["B"]), f64(nrm["norm_B"]), f64(nrm["bias_B"]), eps)
    Cn = bcnorm(f64(inp["C"]), f64(nrm["norm_C"]), f64(nrm["bias_C"]), eps)
    yr, fr = oracle.scan(inp["x"], inp["dt"], inp["A"], Bn, Cn, inp["lam"], inp["theta"])
    ey, ef = max_rel(y, yr), max_rel(fs, fr)
    assert np.isfinite(ey) and np.isfinite(ef)
    assert ey <= TOL["bf16"] and ef <= TOL["bf16"], (ey, ef)
    return ey, ef


SMALL = [
    # (T, N, R, lambda, theta)
    (209, 64, 1, True, True),
    (65, 64, 1, True, True),
    (209, 128, 1, True, True),
    (209, 128, 1, False, False),
    (209, 64, 1, False, False),
    (130, 64, 2, True, False),
    (130, 64, 4, True, True),
    (17, 64, 4, True, True),
    (130, 128, 4, True, True),
]


@pytest.mark.parametrize("T,N,R,lam,th", SMALL, ids=lambda v: str(v))
def test_bcnorm_small(m3, T, N, R, lam, th):
    shape = inputs.ScanShape(batch=2, seqlen=T, heads=3, headdim=64, dstate=N, rank=R, chunk=64 // R, dtype="bf16",
                             with_lambda=lam, with_theta=th)
    ey, ef = run_and_check(m3, shape, 3000 + T + N + R)
    print(f"T{T} N{N} R{R} lam{lam} th{th}: y {ey:.2e} state {ef:.2e}")


def test_bcnorm_siso_workload_full_size(m3):
    """The SISO complex + trapezoidal workload (b8 h32 T8192 P64 N64) with the
    normalisation, on 64 sequences: every batch row, eight heads."""
    ey, ef = run_and_check(m3, inputs.WORKLOADS[inputs.SISO], 2, bsel=list(range(8)), hsel=[0, 4, 9, 13, 18, 22, 27, 31])
    print(f"full size: y {ey:.2e} state {ef:.2e}")


@pytest.mark.parametrize("T,R,th", [(209, 1, True), (209, 1, False), (130, 4, True)], ids=lambda v: str(v))
def test_bcnorm_eps_zero_ragged_tail(m3, T, R, th):
    """eps = 0 with a ragged last chunk: the zero-filled rows past the end of the
    sequence must not turn into NaN (0 / sqrt(0)) and reach y or the state."""
    shape = inputs.ScanShape(batch=2, seqlen=T, heads=3, headdim=64, dstate=64, rank=R, chunk=64 // R,
                             dtype="bf16", with_theta=th)
    ey, ef = run_and_check(m3, shape, 3100 + T + R, eps=0.0)
    print(f"eps 0 T{T} R{R} th{th}: y {ey:.2e} state {ef:.2e}")


def test_bcnorm_empty_sequence(m3):
    shape = inputs.ScanShape(batch=2, seqlen=0, heads=3, headdim=64, dstate=64, rank=1, chunk=64, dtype="bf16")
    nrm = dev(inputs.make_bcnorm_params(64, 3, 5))
    x = torch.empty(2, 0, 3, 1, 64, device="cuda", dtype=torch.bfloat16)
    B = torch.empty(2, 0, 3, 1, 64, device="cuda", dtype=torch.bfloat16)
    fs = torch.full((2, 3, 64, 64), 7.0, device="cuda")
    dims = m3.scan_dims(x, B, 64)
    m3.m3_scan_fwd_bcnorm(None, None, torch.zeros(3, device="cuda"), None, None, None, None, nrm["norm_B"],
                          nrm["norm_C"], nrm["bias_B"], nrm["bias_C"], EPS, None, fs, dims=dims)
    torch.cuda.synchronize()
    assert torch.count_nonzero(fs).item() == 0
