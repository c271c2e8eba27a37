"""GPU checks of the host-buffer prefill (m3_scan_fwd_host): inputs and
outputs in page-locked host memory, the batch in slices staged through a device
workspace, copies overlapping the scans.  Every (b, h) sequence is independent,
so its y and final state must equal, bit for bit, those of m3_scan_fwd on the
whole batch in device memory; one case is also checked against the fp64
oracle."""
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


def pinned(t):
    return None if t is None else t.contiguous().pin_memory()


def device_reference(m3, inp, chunk, with_fs=True):
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    b, T, H, R, P = d["x"].shape
    fs = torch.empty(b, H, d["B"].shape[-1], P, device="cuda") if with_fs else None
    m3.m3_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["lam"], d["theta"], y, fs, chunk=chunk)
    torch.cuda.synchronize()
    return y.cpu(), (fs.cpu() if with_fs else None)


def host_run(m3, inp, chunk, slice_rows, with_fs=True, repeat=1):
    h = {k: pinned(v) for k, v in inp.items()}
    b, T, H, R, P = h["x"].shape
    y = torch.empty_like(h["x"]).pin_memory()
    fs = torch.empty(b, H, h["B"].shape[-1], P).pin_memory() if with_fs else None
    dims = m3.scan_dims(h["x"], h["B"], chunk)
    wsb = m3.m3_scan_fwd_host_workspace_size(dims, slice_rows)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    for _ in range(repeat):
        m3.m3_scan_fwd_host(h["x"], h["dt"], h["A"], h["B"], h["C"], h["lam"], h["theta"], y, fs, ws, wsb,
                            slice=slice_rows, stream=stream, dims=dims)
    stream.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    return y, fs


CASES = [
    # (dtype, batch, T, heads, P, N, R, chunk, slice)
    ("bf16", 5, 200, 3, 64, 64, 1, 64, 2),     # tensor cores; ragged last slice and last chunk
    ("bf16", 5, 200, 3, 64, 64, 4, 16, 0),     # default slice (one row each)
    ("bf16", 3, 130, 2, 64, 128, 1, 64, 7),    # slice larger than the batch: one slice
    ("f32", 4, 77, 2, 32, 16, 2, 32, 1),       # the chunked CUDA-core kernel
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_host_prefill_equals_device_prefill(m3, case):
    dtype, b, T, H, P, N, R, chunk, sl = case
    shape = inputs.ScanShape(batch=b, seqlen=T, heads=H, headdim=P, dstate=N, rank=R, chunk=chunk, dtype=dtype)
    inp = inputs.make_scan_inputs(shape, 1300 + b + T)
    y_ref, fs_ref = device_reference(m3, inp, chunk)
    y, fs = host_run(m3, inp, chunk, sl)
    assert torch.equal(y, y_ref)
    assert torch.equal(fs, fs_ref)


def test_host_prefill_against_oracle_and_optional_inputs(m3):
    shape = inputs.ScanShape(batch=4, seqlen=150, heads=2, headdim=64, dstate=64, rank=1, chunk=64, dtype="bf16",
                             with_lambda=False, with_theta=False)
    inp = inputs.make_scan_inputs(shape, 1400)
    assert inp["lam"] is None and inp["theta"] is None
    y, fs = host_run(m3, inp, 64, 3)
    yr, fr = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], None, None)
    assert max_rel(y.float(), yr) <= TOL["bf16"] and max_rel(fs, fr) <= TOL["bf16"]
    # without a final state: y alone, the same bits
    y2, fs2 = host_run(m3, inp, 64, 3, with_fs=False)
    assert fs2 is None and torch.equal(y2, y)


def test_host_prefill_repeated_calls_reuse_the_workspace(m3):
    """Back-to-back calls on one stream with one workspace: the second call's
    copies into the staging sets wait for the first call's read-backs."""
    shape = inputs.ScanShape(batch=6, seqlen=256, heads=4, headdim=64, dstate=64, rank=1, chunk=64, dtype="bf16")
    inp = inputs.make_scan_inputs(shape, 1500)
    y_ref, fs_ref = device_reference(m3, inp, 64)
    y, fs = host_run(m3, inp, 64, 1, repeat=3)
    assert torch.equal(y, y_ref) and torch.equal(fs, fs_ref)


def test_host_prefill_empty_sequence_writes_zero_state(m3):
    shape = inputs.ScanShape(batch=3, seqlen=0, heads=2, headdim=64, dstate=64, rank=1, chunk=64, dtype="bf16")
    inp = inputs.make_scan_inputs(shape, 1600)
    h = {k: pinned(v) for k, v in inp.items()}
    fs = torch.full((3, 2, 64, 64), 7.0).pin_memory()
    y = torch.empty_like(h["x"]).pin_memory()
    dims = m3.scan_dims(h["x"], h["B"], 64)
    wsb = m3.m3_scan_fwd_host_workspace_size(dims, 2)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
    m3.m3_scan_fwd_host(h["x"], h["dt"], h["A"], h["B"], h["C"], h["lam"], h["theta"], y, fs, ws, wsb, slice=2,
                        dims=dims)
    torch.cuda.synchronize()
    assert torch.count_nonzero(fs) == 0

