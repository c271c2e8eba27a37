"""GPU parity of the CUDA-core kernels (the chunked prefill, the token-serial
prefill, the generic decode step) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_131_b300 import inputs
from tests.gpu_util import TOL, dev, gpu_scan, max_rel, oracle_scan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m3():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from selective_state_space_131_b300 import m3scan
    return m3scan


def check_scan(m3, shape, seed, expect_algo=None):
    inp = inputs.make_scan_inputs(shape, seed)
    dims = m3.scan_dims(inp["x"], inp["B"], shape.chunk)
    if expect_algo is not None:
        assert m3.m3_scan_algorithm(dims) == expect_algo
    y, fs = gpu_scan(m3, dev(inp), shape.chunk)
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    yr, fr = oracle_scan(inp)
    tol = TOL[shape.dtype]
    ey, ef = max_rel(y.float().cpu(), yr), max_rel(fs.cpu(), fr)
    assert ey <= tol and ef <= tol, (ey, ef)
    return ey, ef


def test_config0_tiny_f32(m3):
    """The tiny SISO fp32 workload (b1 h2 T256 P16 N16, seed 0) at 1e-4, in
    chunks of 32 tokens on the chunked CUDA-core kernel."""
    ey, ef = check_scan(m3, inputs.WORKLOADS[inputs.TINY], 0, m3.M3_ALGO_CHUNKED_SIMT)
    print(f"config0: y {ey:.2e} state {ef:.2e}")


SMALL = [
    dict(batch=2, seqlen=37, heads=3, headdim=8, dstate=6, rank=2),
    dict(batch=1, seqlen=1, heads=1, headdim=4, dstate=2, rank=1),
    dict(batch=1, seqlen=20, heads=2, headdim=64, dstate=128, rank=1),
    dict(batch=2, seqlen=9, heads=1, headdim=16, dstate=16, rank=8),
    dict(batch=1, seqlen=70, heads=2, headdim=32, dstate=64, rank=4),
    dict(batch=1, seqlen=5, heads=1, headdim=256, dstate=32, rank=2),
]


@pytest.mark.parametrize("kw", SMALL, ids=lambda k: "b{batch}T{seqlen}h{heads}P{headdim}N{dstate}R{rank}".format(**k))
@pytest.mark.parametrize("chunk", [16, 32, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_cuda_core_scan_shapes(m3, kw, chunk, dtype):
    shape = inputs.ScanShape(chunk=chunk, dtype=dtype, **kw)
    ey, ef = check_scan(m3, shape, 100 + kw["seqlen"])
    print(f"{kw} Q{chunk} {dtype}: y {ey:.2e} state {ef:.2e}")


def test_no_lambda_no_theta(m3):
    """lambda = NULL and theta = NULL mean 1 and 0 (the Mamba-2 special case)."""
    shape = inputs.ScanShape(batch=1, seqlen=50, heads=2, headdim=16, dstate=8, rank=1, chunk=16, dtype="f32",
                             with_lambda=False, with_theta=False)
    check_scan(m3, shape, 5)


def test_empty_sequence_zero_state(m3):
    x = torch.zeros(2, 0, 3, 1, 8, device="cuda")
    B = torch.zeros(2, 0, 3, 1, 4, device="cuda")
    dt = torch.zeros(2, 0, 3, device="cuda")
    A = -torch.ones(3, device="cuda")
    fs = torch.full((2, 3, 4, 8), 7.0, device="cuda")
    m3.m3_scan_fwd(x, dt, A, B, B, None, None, x, fs, chunk=64)
    torch.cuda.synchronize()
    assert torch.count_nonzero(fs).item() == 0


def _decode_chain(m3, dtype, R, steps, seed=3, b=3, H=2, P=16, N=8):
    shape = inputs.DecodeShape(batch=b, heads=H, headdim=P, dstate=N, rank=R, steps=steps, dtype=dtype)
    inp = inputs.make_decode_inputs(shape, seed)
    d = dev(inp)
    state = d["state0"].clone()
    ys = []
    for s in range(steps):
        y = torch.empty_like(d["x"][s + 1])
        m3.m3_step(state, d["x"][s + 1], d["dt"][s + 1], d["A"], d["B"][s + 1], d["C"][s + 1], d["lam"][s + 1],
                   d["theta"][s + 1], d["B"][s], d["x"][s], y)
        ys.append(y)
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    # oracle: one scan of `steps` tokens from state0 with token 0 as the carry
    tok = lambda a: a[1:].transpose(0, 1)   # [steps, b, ...] -> [b, steps, ...]
    yr, fr = oracle.scan(tok(inp["x"]), tok(inp["dt"]), inp["A"], tok(inp["B"]), tok(inp["C"]),
                         tok(inp["lam"]), tok(inp["theta"]), h0=inp["state0"], prevB=inp["B"][0],
                         prevx=inp["x"][0])
    yg = torch.stack(ys, 1).float().cpu()
    return max_rel(yg, yr), max_rel(state.cpu(), fr)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("R", [1, 4])
def test_decode_chain(m3, dtype, R):
    ey, ef = _decode_chain(m3, dtype, R, steps=25)
    assert ey <= TOL[dtype] and ef <= TOL[dtype], (ey, ef)


def test_decode_without_prev_and_lambda(m3):
    """prev_B = prev_x = NULL (no beta term) and lambda_t = theta_t = NULL."""
    b, H, P, N, R = 2, 3, 8, 4, 2
    g = torch.Generator().manual_seed(9)
    st = torch.randn(b, H, N, P, generator=g)
    x = torch.randn(b, H, R, P, generator=g)
    B = torch.randn(b, H, R, N, generator=g) * 0.5
    C = torch.randn(b, H, R, N, generator=g) * 0.5
    dt = torch.rand(b, H, generator=g) * 0.2
    A = -torch.rand(H, generator=g) * 4
    yr, fr = oracle.step(st, x, dt, A, B, C, None, None)
    dst = st.cuda()
    y = torch.empty(b, H, R, P, device="cuda")
    m3.m3_step(dst, x.cuda(), dt.cuda(), A.cuda(), B.cuda(), C.cuda(), None, None, None, None, y)
    torch.cuda.synchronize()
    assert max_rel(y.cpu(), yr) <= 1e-5 and max_rel(dst.cpu(), fr) <= 1e-5


def test_decode_continues_prefill(m3):
    """Prefill of T tokens, then k decode steps == oracle over T + k tokens."""
    shape = inputs.ScanShape(batch=2, seqlen=40, heads=2, headdim=16, dstate=8, rank=2, chunk=16, dtype="f32")
    inp = inputs.make_scan_inputs(shape, 17)
    d = dev(inp)
    T0 = 30
    pre = {k: (v[:, :T0].contiguous() if (v is not None and k != "A") else v) for k, v in d.items()}
    y0, state = gpu_scan(m3, pre, 16)
    ys = [y0]
    for t in range(T0, 40):
        y = torch.empty_like(d["x"][:, t])
        m3.m3_step(state, d["x"][:, t].contiguous(), d["dt"][:, t].contiguous(), d["A"], d["B"][:, t].contiguous(),
                   d["C"][:, t].contiguous(), d["lam"][:, t].contiguous(), d["theta"][:, t].contiguous(),
                   d["B"][:, t - 1].contiguous(), d["x"][:, t - 1].contiguous(), y)
        ys.append(y[:, None])
    torch.cuda.synchronize()
    yr, fr = oracle_scan(inp)
    assert max_rel(torch.cat(ys, 1).cpu(), yr) <= 1e-4
    assert max_rel(state.cpu(), fr) <= 1e-4


def test_chunked_scan_is_deterministic(m3):
    shape = inputs.ScanShape(batch=2, seqlen=64, heads=2, headdim=32, dstate=16, rank=2, chunk=32, dtype="f32")
    d = dev(inputs.make_scan_inputs(shape, 4))
    y1, f1 = gpu_scan(m3, d, 32)
    y2, f2 = gpu_scan(m3, d, 32)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(f1, f2)
