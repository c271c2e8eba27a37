"""GPU parity of the multi-token decode step (m3_step_k: k tokens per launch,
the state read and written once) against the fp64 oracle, through the C ABI:
the fast kernel's shapes with fp32 and bf16 inputs for several k (and launches
of up to 70 tokens), missing
optional inputs, equality with k single steps, the generic fallback (shapes the
kernel does not take, and element-aligned inputs), and the decode workload
(b256 h32 P64 N64 fp32) over 1024 tokens as 128 launches of 8, checked every
64 tokens on sampled units."""
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


def make_case(b, H, P, N, R, k, dtype, seed, lam=True, theta=True):
    """k tokens in the prefill's token-major layout, plus a random state and the
    token before the first (token 0 of a k + 1 token draw)."""
    shape = inputs.ScanShape(batch=b, seqlen=k + 1, heads=H, headdim=P, dstate=N, rank=R, dtype=dtype,
                             with_lambda=lam, with_theta=theta)
    full = inputs.make_scan_inputs(shape, seed)
    cut = lambda v: None if v is None else v[:, 1:].contiguous()
    toks = {key: (v if key == "A" else cut(v)) for key, v in full.items()}
    g = torch.Generator().manual_seed(seed + 7)
    state0 = torch.randn(b, H, N, P, generator=g)
    return toks, state0, full["B"][:, 0].contiguous(), full["x"][:, 0].contiguous()


def run_k(m3, toks, state0, pB, pX, with_prev=True):
    d = {key: (None if v is None else v.cuda()) for key, v in toks.items()}
    state = state0.cuda().clone()
    y = torch.empty_like(d["x"])
    m3.m3_step_k(state, d["x"], d["dt"], d["A"], d["B"], d["C"], d["lam"], d["theta"],
                 pB.cuda() if with_prev else None, pX.cuda() if with_prev else None, y)
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    return y.float().cpu(), state.cpu()


def oracle_k(toks, state0, pB, pX, with_prev=True):
    return oracle.scan(toks["x"], toks["dt"], toks["A"], toks["B"], toks["C"], toks["lam"], toks["theta"],
                       h0=state0, prevB=pB if with_prev else None, prevx=pX if with_prev else None)


@pytest.mark.parametrize("P,N", [(64, 64), (32, 8), (128, 16), (32, 64)], ids=lambda v: str(v))
@pytest.mark.parametrize("R", [1, 2, 4])
@pytest.mark.parametrize("k", [1, 3, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_step_k_matches_oracle(m3, P, N, R, k, dtype):
    toks, s0, pB, pX = make_case(3, 5, P, N, R, k, dtype, 700 + P + N + R + k)
    y, st = run_k(m3, toks, s0, pB, pX)
    yr, fr = oracle_k(toks, s0, pB, pX)
    ey, es = max_rel(y, yr), max_rel(st, fr)
    assert ey <= TOL[dtype] and es <= TOL[dtype], (ey, es)


@pytest.mark.parametrize("k", [31, 32, 33, 70])
@pytest.mark.parametrize("R,dtype", [(1, "f32"), (4, "f32"), (2, "bf16")])
def test_step_k_long_launches(m3, k, R, dtype):
    """Launches longer than one group of 8 staged tokens, ragged and not: the
    next group loads while one runs, the state stays in registers across
    groups.  Same bar."""
    toks, s0, pB, pX = make_case(3, 5, 64, 64, R, k, dtype, 770 + k + R)
    y, st = run_k(m3, toks, s0, pB, pX)
    yr, fr = oracle_k(toks, s0, pB, pX)
    assert max_rel(y, yr) <= TOL[dtype] and max_rel(st, fr) <= TOL[dtype]


@pytest.mark.parametrize("prev,lam,theta", [(False, True, True), (True, False, True), (True, True, False),
                                            (False, False, False)])
def test_step_k_optional_inputs(m3, prev, lam, theta):
    toks, s0, pB, pX = make_case(2, 3, 64, 64, 2, 5, "f32", 731, lam=lam, theta=theta)
    y, st = run_k(m3, toks, s0, pB, pX, with_prev=prev)
    yr, fr = oracle_k(toks, s0, pB, pX, with_prev=prev)
    assert max_rel(y, yr) <= 1e-4 and max_rel(st, fr) <= 1e-4


@pytest.mark.parametrize("R", [1, 4])
def test_step_k_equals_single_steps(m3, R):
    """One launch of k = 6 tokens gives what six m3_step calls give."""
    k = 6
    toks, s0, pB, pX = make_case(4, 4, 64, 64, R, k, "f32", 740 + R)
    yk, sk = run_k(m3, toks, s0, pB, pX)
    d = {key: (None if v is None else v.cuda()) for key, v in toks.items()}
    state = s0.cuda().clone()
    ys = []
    for j in range(k):
        y = torch.empty_like(d["x"][:, j])
        prevB = pB.cuda() if j == 0 else d["B"][:, j - 1].contiguous()
        prevx = pX.cuda() if j == 0 else d["x"][:, j - 1].contiguous()
        m3.m3_step(state, d["x"][:, j].contiguous(), d["dt"][:, j].contiguous(), d["A"], d["B"][:, j].contiguous(),
                   d["C"][:, j].contiguous(), d["lam"][:, j].contiguous(), d["theta"][:, j].contiguous(), prevB,
                   prevx, y)
        ys.append(y)
    torch.cuda.synchronize()
    y1 = torch.stack(ys, 1).cpu()
    assert max_rel(yk, y1) <= 1e-6 and max_rel(sk, state.cpu()) <= 1e-6


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_step_k_generic_shapes(m3, dtype):
    """Shapes outside the kernel's (P = 16, N = 6, R = 3) run the continued
    prefill on the state in place; same bar."""
    toks, s0, pB, pX = make_case(2, 3, 16, 6, 3, 7, dtype, 750)
    y, st = run_k(m3, toks, s0, pB, pX)
    yr, fr = oracle_k(toks, s0, pB, pX)
    assert max_rel(y, yr) <= TOL[dtype] and max_rel(st, fr) <= TOL[dtype]


def test_step_k_element_aligned_inputs(m3):
    """x only element-aligned: the generic path, still exact to the bar."""
    toks, s0, pB, pX = make_case(2, 2, 64, 64, 1, 4, "f32", 760)
    d = {key: (None if v is None else v.cuda()) for key, v in toks.items()}
    xbuf = torch.empty(d["x"].numel() + 1, device="cuda")
    x1 = xbuf[1:].view_as(d["x"])
    x1.copy_(d["x"])
    state = s0.cuda().clone()
    y = torch.empty_like(d["x"])
    m3.m3_step_k(state, x1, d["dt"], d["A"], d["B"], d["C"], d["lam"], d["theta"], pB.cuda(), pX.cuda(), y)
    torch.cuda.synchronize()
    yr, fr = oracle_k(toks, s0, pB, pX)
    assert max_rel(y.cpu(), yr) <= 1e-4 and max_rel(state.cpu(), fr) <= 1e-4


def test_step_k_zero_tokens_is_a_no_op(m3):
    state = torch.randn(2, 3, 64, 64, device="cuda")
    ref = state.clone()
    x = torch.empty(2, 0, 3, 1, 64, device="cuda")
    B = torch.empty(2, 0, 3, 1, 64, device="cuda")
    m3.m3_step_k(state, x, torch.empty(2, 0, 3, device="cuda"), torch.zeros(3, device="cuda"), B, B, None, None,
                 None, None, x)
    torch.cuda.synchronize()
    assert torch.equal(state, ref)


@pytest.mark.parametrize("R", [1, 4])
def test_step_k_decode_workload_1024_tokens(m3, R):
    """The decode workload (b256 h32 P64 N64, fp32) over 1024 tokens as 128
    launches of k = 8 (the bench's multi-token line), from an N(0, 1) state;
    y and the state checked after every 64 tokens on 12 sampled units."""
    k, launches, seg = 8, 128, 64
    steps = k * launches
    shape = inputs.DecodeShape(**{**inputs.WORKLOADS[inputs.DECODE].__dict__, "rank": R, "steps": steps})
    dec = inputs.make_decode_inputs(shape, 40 + R, device="cuda")
    b, H = shape.batch, shape.heads
    # tokens 1..steps in launch-major, token-major order: [launch, b, k, h, ...]
    lay = lambda a: a[1:].reshape(launches, k, b, H, *a.shape[3:]).transpose(1, 2).contiguous()
    X, DT, Bm, Cm, LAM, TH = (lay(dec[key]) for key in ("x", "dt", "B", "C", "lam", "theta"))
    state = dec["state0"].clone()
    Y = torch.empty_like(X)
    snaps = []
    for i in range(launches):
        prevB = dec["B"][0] if i == 0 else Bm[i - 1][:, k - 1].contiguous()
        prevx = dec["x"][0] if i == 0 else X[i - 1][:, k - 1].contiguous()
        m3.m3_step_k(state, X[i], DT[i], dec["A"], Bm[i], Cm[i], LAM[i], TH[i], prevB, prevx, Y[i])
        if (i + 1) * k % seg == 0:
            snaps.append(state.clone())
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    bsel, hsel = [0, 37, 128, 255], [0, 11, 31]
    sel = lambda a: a[:, bsel][:, :, hsel].cpu()          # [S, b, h, ...] -> sampled units
    x, dt, B, C, lam, th = (sel(dec[key]) for key in ("x", "dt", "B", "C", "lam", "theta"))
    A = dec["A"][hsel].cpu()
    h = dec["state0"][bsel][:, hsel].cpu()
    # y back to [S, b', h', R, P]
    yg = Y.transpose(1, 2).reshape(steps, b, H, R, -1)[:, bsel][:, :, hsel].cpu()
    for s in range(steps // seg):
        t0, t1 = s * seg + 1, (s + 1) * seg + 1
        tok = lambda a: a[t0:t1].transpose(0, 1)
        yr, h = oracle.scan(tok(x), tok(dt), A, tok(B), tok(C), tok(lam), tok(th), h0=h, prevB=B[t0 - 1],
                            prevx=x[t0 - 1])
        ey = max_rel(yg[t0 - 1:t1 - 1].transpose(0, 1), yr)
        es = max_rel(snaps[s][bsel][:, hsel].cpu(), h)
        assert ey <= 1e-4 and es <= 1e-4, (s, ey, es)


@pytest.mark.parametrize("kind", ["fast_decay", "a_zero", "lambda_zero", "lambda_one", "tiny_dt", "large_phi"])
@pytest.mark.parametrize("R", [1, 4])
def test_step_k_edges(m3, kind, R):
    """The forced edge cases of test_gpu_edges over a 12-token launch (fp32)."""
    from tests.test_gpu_edges import apply_edge
    toks, s0, pB, pX = make_case(3, 4, 64, 64, R, 12, "f32", 770 + R)
    toks = apply_edge(toks, kind, 771 + R, "f32", R)
    y, st = run_k(m3, toks, s0, pB, pX)
    yr, fr = oracle_k(toks, s0, pB, pX)
    assert max_rel(y, yr) <= 1e-4 and max_rel(st, fr) <= 1e-4, kind
