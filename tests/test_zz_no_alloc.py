"""The backward pass without a workspace argument (m3_scan_bwd_noalloc), for
callers that cannot allocate device memory -- a host whose allocator belongs to
another runtime or framework, a process held to a fixed memory budget, code
that must not touch the allocator inside a serving loop.  It uses the
library's fixed 32 MiB scratch array instead of a caller's workspace.

Checked through the C ABI against the entry point that takes a workspace
(m3_scan_bwd), within the tolerance the other tests use, on two calls in a row
with different inputs (the scratch keeps the first call's contents, which must
not matter); and sizes beyond the scratch are refused before anything runs.
This file is collected last so that a run stopping at the first failure has
already run every other test."""
import pytest
import torch

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


def case(shape, seed):
    inp = {k: (None if v is None else v.cuda()) for k, v in inputs.make_scan_inputs(shape, seed).items()}
    g = torch.Generator().manual_seed(seed + 1)
    b, T, H, R, P, N = shape.batch, shape.seqlen, shape.heads, shape.rank, shape.headdim, shape.dstate
    dy = torch.randn(b, T, H, R, P, generator=g).to(inp["x"].dtype).cuda()
    dfinal = torch.randn(b, H, N, P, generator=g).cuda()
    return inp, dy, dfinal


def outputs(inp):
    return {"dx": torch.empty_like(inp["x"]), "ddt": torch.empty_like(inp["dt"]), "dA": torch.empty_like(inp["A"]),
            "dB": torch.empty_like(inp["B"]), "dC": torch.empty_like(inp["C"]),
            "dlam": torch.empty_like(inp["lam"]) if inp["lam"] is not None else None,
            "dtheta": torch.empty_like(inp["theta"]) if inp["theta"] is not None else None}


def with_workspace(m3, inp, dy, dfinal, dims):
    out = outputs(inp)
    wsb = m3.m3_scan_bwd_workspace_size(dims)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    m3.m3_scan_bwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["lam"], inp["theta"], dy, dfinal,
                   *[out[k] for k in GRADS], ws, wsb, dims=dims)
    return out


def without_workspace(m3, inp, dy, dfinal, dims):
    out = outputs(inp)
    m3.m3_scan_bwd_noalloc(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["lam"], inp["theta"], dy, dfinal,
                           *[out[k] for k in GRADS], dims=dims)
    return out


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_noalloc_matches_workspace_entry_on_two_calls(m3, dtype):
    P = 16 if dtype == "f32" else 64
    shape = inputs.ScanShape(batch=2, seqlen=150, heads=3, headdim=P, dstate=P, rank=1, chunk=32, dtype=dtype)
    for call, seed in enumerate((910, 911)):
        inp, dy, dfinal = case(shape, seed)
        dims = m3.scan_dims(inp["x"], inp["B"], shape.chunk)
        ref = with_workspace(m3, inp, dy, dfinal, dims)
        got = without_workspace(m3, inp, dy, dfinal, dims)
        torch.cuda.synchronize()
        assert m3.m3_device_status() == m3.M3_OK
        for k in GRADS:
            e = max_rel(got[k].float().cpu(), ref[k].float().cpu())
            assert e <= TOL[dtype], (call, k, e)


def test_noalloc_refuses_sizes_beyond_its_scratch(m3):
    """b8 h32 T8192 P64 N64 needs a 545 MB workspace: refused with
    M3_ERR_WORKSPACE before any launch (the buffers below are only the size of
    a small problem, and are never touched)."""
    small = inputs.ScanShape(batch=1, seqlen=64, heads=1, headdim=64, dstate=64, rank=1, chunk=64, dtype="bf16")
    inp, dy, dfinal = case(small, 920)
    big = m3.make_dims(8, 8192, 32, 64, 64, 1, 64, m3.M3_BF16)
    assert m3.m3_scan_bwd_workspace_size(big) > (32 << 20)
    out = outputs(inp)
    with pytest.raises(m3.M3Error) as e:
        m3.m3_scan_bwd_noalloc(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["lam"], inp["theta"], dy,
                               dfinal, *[out[k] for k in GRADS], dims=big)
    assert e.value.status == m3.M3_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
