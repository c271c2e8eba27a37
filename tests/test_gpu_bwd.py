"""GPU parity of the backward pass (m3_scan_bwd) against the fp64 gradient
oracle (oracle.scan_bwd, itself pinned by finite differences of the forward
oracle): every gradient -- dx, ddt, dA, dB, dC, dlambda, dtheta -- on small
shapes over several chunks with ragged tails, fp32 at 1e-4 and bf16 at 2e-2,
with and without lambda / theta / dfinal; chunk invariance; the SISO workload
(b8 h32 T8192 P64 N64, bf16) at full size on sampled heads; determinism."""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_131_b300 import inputs
from tests.gpu_util import TOL, max_rel

pytestmark = pytest.mark.gpu

GRADS = ("dx", "ddt", "dA", "dB", "dC", "dlam", "dtheta")


@pytest.fixture(scope="module")
def m3():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from selective_state_space_131_b300 import m3scan
    return m3scan


def upstream(shape, seed, with_dfinal=True):
    g = torch.Generator().manual_seed(seed)
    b, T, H, R, P, N = shape.batch, shape.seqlen, shape.heads, shape.rank, shape.headdim, shape.dstate
    cast = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    dy = torch.randn(b, T, H, R, P, generator=g).to(cast)
    dfinal = torch.randn(b, H, N, P, generator=g) if with_dfinal else None
    return dy, dfinal


def gpu_bwd(m3, inp, dy, dfinal, chunk):
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    x, B = d["x"], d["B"]
    dims = m3.scan_dims(x, B, chunk)
    ws_bytes = m3.m3_scan_bwd_workspace_size(dims)
    assert ws_bytes > 0
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = {"dx": torch.empty_like(x), "ddt": torch.empty_like(d["dt"]),
           "dA": torch.empty_like(d["A"]), "dB": torch.empty_like(B), "dC": torch.empty_like(d["C"]),
           "dlam": torch.empty_like(d["lam"]) if d["lam"] is not None else None,
           "dtheta": torch.empty_like(d["theta"]) if d["theta"] is not None else None}
    m3.m3_scan_bwd(x, d["dt"], d["A"], B, d["C"], d["lam"], d["theta"], dy.cuda(),
                   None if dfinal is None else dfinal.cuda(), out["dx"], out["ddt"], out["dA"], out["dB"],
                   out["dC"], out["dlam"], out["dtheta"], ws, ws_bytes, dims=dims)
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    return {k: (None if v is None else v.float().cpu()) for k, v in out.items()}


def compare(got, ref, tol, label=""):
    errs = {}
    for k in GRADS:
        if ref.get(k) is None:
            assert got.get(k) is None, k
            continue
        if not np.any(ref[k]):
            # an identically zero gradient (dA with a single token: no earlier state
            # to decay): the fp32 sums leave rounding noise only
            e = float(np.max(np.abs(got[k].numpy())))
            assert e <= 1e-6, (label, k, e)
        else:
            e = max_rel(got[k], ref[k])
            assert np.isfinite(e) and e <= tol, (label, k, e)
        errs[k] = e
    return errs


def run_case(m3, shape, seed, with_dfinal=True, chunk=None):
    inp = inputs.make_scan_inputs(shape, seed)
    dy, dfinal = upstream(shape, seed + 1, with_dfinal)
    got = gpu_bwd(m3, inp, dy, dfinal, chunk or shape.chunk)
    ref = oracle.scan_bwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["lam"], inp["theta"], dy, dfinal)
    return compare(got, ref, TOL[shape.dtype], str(shape))


SMALL = [
    # (dtype, T, P, N, R, chunk, lambda, theta)
    ("f32", 100, 16, 16, 1, 32, True, True),
    ("f32", 37, 16, 8, 2, 16, True, True),
    ("f32", 130, 32, 32, 4, 16, True, True),
    ("f32", 64, 16, 16, 1, 64, True, True),
    ("f32", 1, 8, 4, 1, 16, True, True),
    ("f32", 90, 16, 16, 1, 32, False, False),
    ("f32", 90, 16, 16, 1, 32, True, False),
    ("f32", 90, 16, 16, 1, 32, False, True),
    ("f32", 70, 64, 64, 1, 64, True, True),
    ("bf16", 209, 64, 64, 1, 64, True, True),
    ("bf16", 130, 64, 64, 4, 16, True, True),
    ("bf16", 150, 64, 128, 1, 32, True, True),
    ("bf16", 100, 32, 16, 2, 32, True, False),
    # the tensor-core path on sequences of one partial chunk, exactly one chunk and
    # one chunk plus a token (the gradient tiles' TMA stores clip the rows past T)
    ("bf16", 5, 64, 64, 1, 64, True, True),
    ("bf16", 32, 64, 64, 2, 32, True, True),
    ("bf16", 17, 64, 64, 4, 16, True, True),
    # the tensor-core path without theta and / or lambda (no rotation: the checkpoint
    # run loads B and x in one part)
    ("bf16", 150, 64, 64, 1, 64, False, False),
    ("bf16", 130, 64, 64, 2, 32, True, False),
    ("bf16", 77, 64, 64, 4, 16, False, True),
    # state sizes that leave a partial 4-wide register tile (N % 4 == 2), narrow heads
    ("f32", 77, 12, 6, 1, 16, True, True),
    ("f32", 50, 4, 2, 2, 16, True, True),
    ("f32", 90, 8, 10, 4, 16, True, True),
    ("bf16", 81, 12, 6, 2, 32, True, True),
]


@pytest.mark.parametrize("dtype,T,P,N,R,chunk,lam,th", SMALL, ids=lambda v: str(v))
def test_bwd_matches_gradient_oracle(m3, dtype, T, P, N, R, chunk, lam, th):
    shape = inputs.ScanShape(batch=2, seqlen=T, heads=3, headdim=P, dstate=N, rank=R, chunk=chunk, dtype=dtype,
                             with_lambda=lam, with_theta=th)
    errs = run_case(m3, shape, 800 + T + P + N + R)
    print(dtype, T, P, N, R, chunk, {k: f"{v:.1e}" for k, v in errs.items()})


def test_bwd_without_dfinal(m3):
    shape = inputs.ScanShape(batch=2, seqlen=75, heads=2, headdim=16, dstate=16, rank=2, chunk=16, dtype="f32")
    run_case(m3, shape, 870, with_dfinal=False)


def test_bwd_chunk_invariance_f32(m3):
    """Chunks of 16, 32 and 64 tokens: each within 1e-4 of the gradient oracle."""
    shape = inputs.ScanShape(batch=2, seqlen=200, heads=2, headdim=16, dstate=16, rank=1, chunk=16, dtype="f32")
    inp = inputs.make_scan_inputs(shape, 880)
    dy, dfinal = upstream(shape, 881)
    ref = oracle.scan_bwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["lam"], inp["theta"], dy, dfinal)
    for q in (16, 32, 64):
        compare(gpu_bwd(m3, inp, dy, dfinal, q), ref, TOL["f32"], f"Q{q}")


def test_bwd_deterministic(m3):
    shape = inputs.ScanShape(batch=2, seqlen=150, heads=2, headdim=64, dstate=64, rank=1, chunk=64, dtype="bf16")
    inp = inputs.make_scan_inputs(shape, 890)
    dy, dfinal = upstream(shape, 891)
    a = gpu_bwd(m3, inp, dy, dfinal, 64)
    b = gpu_bwd(m3, inp, dy, dfinal, 64)
    for k in GRADS:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("R", [1, 4])
def test_bwd_repeated_runs_write_every_gradient_the_same(m3, R):
    """30 backward passes of the tensor-core path into gradient buffers pre-filled
    with NaN (and a NaN-filled workspace): every element written and every run
    bit-identical to the first -- a check on the checkpoint and gradient tiles
    that leave through shared memory by TMA stores."""
    shape = inputs.ScanShape(batch=2, seqlen=150, heads=3, headdim=64, dstate=64, rank=R, chunk=64 // R, dtype="bf16")
    inp = inputs.make_scan_inputs(shape, 895 + R)
    dy, dfinal = upstream(shape, 896 + R)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    dims = m3.scan_dims(d["x"], d["B"], 64 // R)
    wsb = m3.m3_scan_bwd_workspace_size(dims)
    dyc, dfc = dy.cuda(), dfinal.cuda()
    ref = None
    for it in range(30):
        ws = torch.full((wsb // 4,), float("nan"), device="cuda")
        out = {"dx": d["x"], "ddt": d["dt"], "dA": d["A"], "dB": d["B"], "dC": d["C"], "dlam": d["lam"],
               "dtheta": d["theta"]}
        out = {k: torch.full_like(v, float("nan")) for k, v in out.items()}
        m3.m3_scan_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["lam"], d["theta"], dyc, dfc, out["dx"],
                       out["ddt"], out["dA"], out["dB"], out["dC"], out["dlam"], out["dtheta"], ws, wsb, dims=dims)
        if ref is None:
            torch.cuda.synchronize()
            for k, v in out.items():
                assert not torch.isnan(v.float()).any(), k
            ref = out
        else:
            for k in out:
                assert torch.equal(out[k], ref[k]), (it, k)
    assert m3.m3_device_status() == m3.M3_OK


def test_bwd_siso_workload_full_size(m3):
    """The SISO complex + trapezoidal workload (b8 h32 T8192 P64 N64, bf16) at
    full size -- the launch the bench times -- checked on three heads for every
    batch row (24 sequences; dA[h] sums all eight rows of a head)."""
    shape = inputs.WORKLOADS[inputs.SISO]
    inp = inputs.make_scan_inputs(shape, 2)
    dy, dfinal = upstream(shape, 892)
    got = gpu_bwd(m3, inp, dy, dfinal, 64)
    hs = [0, 17, 31]
    sub = {k: (None if v is None else (v[hs] if k == "A" else v[:, :, hs])) for k, v in inp.items()}
    ref = oracle.scan_bwd(sub["x"], sub["dt"], sub["A"], sub["B"], sub["C"], sub["lam"], sub["theta"],
                          dy[:, :, hs], dfinal[:, hs], nthreads=4)
    pick = {k: (None if v is None else (v[hs] if k == "dA" else v[:, :, hs])) for k, v in got.items()}
    errs = compare(pick, ref, TOL["bf16"], "full size")
    print({k: f"{v:.1e}" for k, v in errs.items()})


def test_bwd_empty_sequence(m3):
    x = torch.empty(2, 0, 3, 1, 16, device="cuda")
    B = torch.empty(2, 0, 3, 1, 8, device="cuda")
    dims = m3.scan_dims(x, B, 16)
    dA = torch.full((3,), 5.0, device="cuda")
    m3.m3_scan_bwd(None, None, torch.zeros(3, device="cuda"), None, None, None, None, None, None, None, None, dA,
                   None, None, None, None, None, 0, dims=dims)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dA).item() == 0


EDGE_KINDS = ["fast_decay", "a_zero", "lambda_zero", "lambda_one", "tiny_dt", "mixed", "large_phi"]


@pytest.mark.parametrize("kind", EDGE_KINDS)
@pytest.mark.parametrize("dtype,P,N,R,chunk", [("bf16", 64, 64, 1, 64), ("bf16", 64, 64, 4, 16),
                                               ("f32", 16, 16, 2, 32)], ids=lambda v: str(v))
def test_bwd_edges(m3, kind, dtype, P, N, R, chunk):
    """The forced edge cases of test_gpu_edges through the backward pass: the
    tensor-core path (bf16 N = P = 64) and the CUDA-core path (fp32)."""
    from tests.test_gpu_edges import apply_edge
    shape = inputs.ScanShape(batch=2, seqlen=150, heads=3, headdim=P, dstate=N, rank=R, chunk=chunk, dtype=dtype)
    inp = apply_edge(inputs.make_scan_inputs(shape, 950 + R), kind, 951 + R, dtype, R)
    dy, dfinal = upstream(shape, 952)
    got = gpu_bwd(m3, inp, dy, dfinal, chunk)
    ref = oracle.scan_bwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["lam"], inp["theta"], dy, dfinal)
    for k in GRADS:
        if got[k] is not None:
            assert torch.isfinite(got[k]).all(), k
    errs = compare(got, ref, TOL[dtype], kind)
    print(kind, dtype, R, {k: f"{v:.1e}" for k, v in errs.items()})
