"""GPU parity of the continued prefill (m3_scan_fwd_from) against the fp64
oracle: a prefill started from a state and the previous token's (B, x), on
the tensor-core kernel, the chunked CUDA-core kernel and the token-serial
kernel; a sequence split into two
prefills equals one prefill; prefill -> decode steps -> prefill equals the
oracle over the whole sequence; T = 0 passes the state through."""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_131_b300 import inputs
from tests.gpu_util import TOL, max_rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m3():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from selective_state_space_131_b300 import m3scan
    return m3scan


def cut(inp, t0, t1):
    return {k: (v if (v is None or k == "A") else v[:, t0:t1].contiguous()) for k, v in inp.items()}


def dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_from(m3, d, h0, pB, px, chunk):
    b, T, H, R, P = d["x"].shape
    N = d["B"].shape[-1]
    y = torch.empty_like(d["x"])
    fs = torch.empty(b, H, N, P, device="cuda")
    m3.m3_scan_fwd_from(d["x"], d["dt"], d["A"], d["B"], d["C"], d["lam"], d["theta"], h0, pB, px, y, fs,
                        chunk=chunk)
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    return y, fs


TC, SIMT, SEQ = 1, 2, 0   # M3_ALGO_CHUNKED_TC, M3_ALGO_CHUNKED_SIMT, M3_ALGO_SEQUENTIAL
CASES = [
    # (dtype, T, N, R, chunk, lambda, theta, with_h0, with_prev, algorithm)
    ("bf16", 130, 64, 1, 64, True, True, True, True, TC),
    ("bf16", 37, 64, 1, 64, True, True, True, True, TC),
    ("bf16", 1, 64, 1, 64, True, True, True, True, TC),
    ("bf16", 64, 64, 1, 64, True, True, True, True, TC),
    ("bf16", 200, 128, 1, 64, True, True, True, True, TC),
    ("bf16", 130, 64, 2, 32, True, True, True, True, TC),
    ("bf16", 130, 64, 4, 16, True, True, True, True, TC),
    ("bf16", 130, 128, 4, 16, True, False, True, True, TC),
    ("bf16", 130, 64, 1, 64, False, False, True, True, TC),
    ("bf16", 130, 64, 1, 64, True, True, True, False, TC),
    ("bf16", 130, 64, 1, 64, True, True, False, True, TC),
    ("bf16", 130, 64, 2, 64, True, True, True, True, SIMT),
    ("bf16", 130, 64, 1, 32, True, True, True, False, SIMT),
    ("f32", 70, 16, 2, 32, True, True, True, True, SIMT),
    ("f32", 33, 64, 1, 16, True, True, True, False, SIMT),
    ("f32", 33, 8, 4, 64, True, True, False, True, SIMT),
    ("f32", 40, 8, 8, 128, True, True, True, True, SEQ),
]


@pytest.mark.parametrize("dtype,T,N,R,chunk,lam,th,wh,wp,algo", CASES, ids=lambda v: str(v))
def test_continued_prefill_matches_oracle(m3, dtype, T, N, R, chunk, lam, th, wh, wp, algo):
    P = 64 if dtype == "bf16" else 16
    if algo == SEQ:
        P = 64
    shape = inputs.ScanShape(batch=2, seqlen=T + 1, heads=3, headdim=P, dstate=N, rank=R, chunk=chunk, dtype=dtype,
                             with_lambda=lam, with_theta=th)
    full = inputs.make_scan_inputs(shape, 500 + T + N + R)
    prev = cut(full, 0, 1)                    # token 0 is the previous token
    seq = cut(full, 1, T + 1)
    assert m3.m3_scan_algorithm(m3.scan_dims(seq["x"], seq["B"], chunk)) == algo
    g = torch.Generator().manual_seed(T + N)
    h0 = (0.3 * torch.randn(2, 3, N, P, generator=g)) if wh else None
    pB = prev["B"][:, 0] if wp else None
    px = prev["x"][:, 0] if wp else None
    d = dev(seq)
    y, fs = run_from(m3, d, h0.cuda() if wh else None, pB.cuda() if wp else None, px.cuda() if wp else None, chunk)
    yr, fr = oracle.scan(seq["x"], seq["dt"], seq["A"], seq["B"], seq["C"], seq["lam"], seq["theta"],
                         h0=h0, prevB=pB, prevx=px)
    ey, ef = max_rel(y.float().cpu(), yr), max_rel(fs.cpu(), fr)
    assert ey <= TOL[dtype] and ef <= TOL[dtype], (ey, ef)


@pytest.mark.parametrize("dtype,N,R,chunk", [("bf16", 64, 1, 64), ("bf16", 128, 2, 32), ("bf16", 64, 2, 64),
                                             ("f32", 16, 1, 32)])
def test_split_prefill_equals_one_prefill(m3, dtype, N, R, chunk):
    """prefill(T1) then prefill_from(T2, state, last token) == prefill(T1 + T2)."""
    P = 64 if dtype == "bf16" else 16
    T1, T2 = 150, 97
    shape = inputs.ScanShape(batch=2, seqlen=T1 + T2, heads=2, headdim=P, dstate=N, rank=R, chunk=chunk, dtype=dtype)
    full = inputs.make_scan_inputs(shape, 31)
    d1, d2 = dev(cut(full, 0, T1)), dev(cut(full, T1, T1 + T2))
    y1, s1 = run_from(m3, d1, None, None, None, chunk)
    y2, s2 = run_from(m3, d2, s1, d1["B"][:, T1 - 1].contiguous(), d1["x"][:, T1 - 1].contiguous(), chunk)
    yr, fr = oracle.scan(full["x"], full["dt"], full["A"], full["B"], full["C"], full["lam"], full["theta"])
    y = torch.cat([y1, y2], 1).float().cpu()
    assert max_rel(y, yr) <= TOL[dtype] and max_rel(s2.cpu(), fr) <= TOL[dtype]


def test_prefill_decode_prefill(m3):
    """The serving loop: prefill, decode steps, prefill again, all in one frame."""
    T1, K, T2 = 100, 5, 70
    shape = inputs.ScanShape(batch=2, seqlen=T1 + K + T2, heads=2, headdim=64, dstate=64, rank=1, chunk=64,
                             dtype="bf16")
    full = inputs.make_scan_inputs(shape, 77)
    d = dev(full)
    ys = []
    y1, state = run_from(m3, dev(cut(full, 0, T1)), None, None, None, 64)
    ys.append(y1.float())
    for t in range(T1, T1 + K):
        y = torch.empty_like(d["x"][:, t])
        m3.m3_step(state, d["x"][:, t].contiguous(), d["dt"][:, t].contiguous(), d["A"], d["B"][:, t].contiguous(),
                   d["C"][:, t].contiguous(), d["lam"][:, t].contiguous(), d["theta"][:, t].contiguous(),
                   d["B"][:, t - 1].contiguous(), d["x"][:, t - 1].contiguous(), y)
        ys.append(y[:, None].float())
    t = T1 + K
    y3, state3 = run_from(m3, dev(cut(full, t, t + T2)), state, d["B"][:, t - 1].contiguous(),
                          d["x"][:, t - 1].contiguous(), 64)
    ys.append(y3.float())
    yr, fr = oracle.scan(full["x"], full["dt"], full["A"], full["B"], full["C"], full["lam"], full["theta"])
    assert max_rel(torch.cat(ys, 1).cpu(), yr) <= 2e-2
    assert max_rel(state3.cpu(), fr) <= 2e-2


def test_empty_continuation_passes_state_through(m3):
    h0 = torch.randn(2, 3, 8, 16, device="cuda")
    x = torch.zeros(2, 0, 3, 1, 16, device="cuda")
    B = torch.zeros(2, 0, 3, 1, 8, device="cuda")
    dt = torch.zeros(2, 0, 3, device="cuda")
    A = -torch.ones(3, device="cuda")
    fs = torch.zeros_like(h0)
    m3.m3_scan_fwd_from(x, dt, A, B, B, None, None, h0, None, None, x, fs, chunk=64)
    torch.cuda.synchronize()
    assert torch.equal(fs, h0)
