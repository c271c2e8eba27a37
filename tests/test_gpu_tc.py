"""GPU parity of the chunked tensor-core prefill (M3_ALGO_CHUNKED_TC) against
the fp64 oracle: small shapes spanning several chunks and a ragged tail, the
three bf16 workloads at full size on sampled (batch, head) sequences, chunk
invariance, prefill -> decode continuation and determinism."""
import numpy as np
import pytest
import torch

from selective_state_space_131_b300 import inputs
from tests.gpu_util import TOL, dev, gpu_scan, max_rel, oracle_scan, sub_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m3():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from selective_state_space_131_b300 import m3scan
    return m3scan


def run_and_check(m3, shape, seed, bsel=None, hsel=None, tol=None):
    inp = inputs.make_scan_inputs(shape, seed)
    dims = m3.scan_dims(inp["x"], inp["B"], shape.chunk)
    assert m3.m3_scan_algorithm(dims) == m3.M3_ALGO_CHUNKED_TC
    y, fs = gpu_scan(m3, dev(inp), shape.chunk)
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    y, fs = y.float().cpu(), fs.cpu()
    if bsel is not None:
        y = y[bsel][:, :, hsel]
        fs = fs[bsel][:, hsel]
    yr, fr = oracle_scan(inp, bsel, hsel)
    ey, ef = max_rel(y, yr), max_rel(fs, fr)
    tol = tol or TOL[shape.dtype]
    assert np.isfinite(ey) and np.isfinite(ef)
    assert ey <= tol and ef <= tol, (ey, ef)
    return ey, ef


SMALL = [
    # (T, N, R, lambda, theta): several chunks, ragged tails, one token, exactly
    # one chunk, every (N, R) the tensor-core kernel takes, with and without
    # lambda / theta.  The chunk is the kernel's 64-row tile: 64 / R tokens.
    (209, 64, 1, True, True),
    (64, 64, 1, True, True),
    (65, 64, 1, True, True),
    (1, 64, 1, True, True),
    (37, 64, 1, True, True),
    (209, 128, 1, True, True),
    (209, 128, 1, False, False),
    (209, 64, 1, False, False),
    (209, 64, 1, True, False),
    (209, 64, 1, False, True),
    (130, 64, 2, True, True),
    (130, 64, 4, True, True),
    (17, 64, 4, True, True),
    (130, 128, 2, True, True),
    (130, 128, 4, True, False),
    (130, 128, 4, True, True),
    (513, 64, 1, True, True),
]


@pytest.mark.parametrize("T,N,R,lam,th", SMALL, ids=lambda v: str(v))
def test_tc_small(m3, T, N, R, lam, th):
    shape = inputs.ScanShape(batch=2, seqlen=T, heads=3, headdim=64, dstate=N, rank=R, chunk=64 // R, dtype="bf16",
                             with_lambda=lam, with_theta=th)
    ey, ef = run_and_check(m3, shape, 1000 + T + N + R)
    print(f"T{T} N{N} R{R} lam{lam} th{th}: y {ey:.2e} state {ef:.2e}")


# Full-size units checked: every (batch, head) sequence of the SSD-equivalent and
# SISO workloads; for the MIMO workload every batch row on 17 of the 32 heads
# (136 of 256 sequences).  With 256 CTAs on 148 SMs some SMs run one CTA and
# others two, so both placements are among the units checked.
FULL_SEL = {inputs.SSD_EQUIV: (list(range(8)), list(range(32))),
            inputs.SISO: (list(range(8)), list(range(32))),
            inputs.MIMO: (list(range(8)), list(range(0, 32, 2)) + [31])}


@pytest.mark.parametrize("name", list(inputs.PREFILL_WORKLOADS))
def test_tc_full_size_workloads(m3, name):
    """The bf16 workloads at full size, in the launch configuration the bench
    times (the tensor-core kernel; for the MIMO workload its 16-token chunk, the
    64-row tile at R = 4), checked against the oracle on the units of FULL_SEL."""
    shape = inputs.WORKLOADS[name]
    shape = inputs.ScanShape(**{**shape.__dict__, "chunk": 64 // shape.rank})
    bsel, hsel = FULL_SEL[name]
    ey, ef = run_and_check(m3, shape, inputs.WORKLOAD_SEEDS[name], bsel, hsel)
    print(f"{name}: y {ey:.2e} state {ef:.2e}")


def test_chunk_invariance_across_kernels(m3):
    """The result does not depend on the chunk beyond rounding: the same bf16
    inputs through the tensor-core kernel (chunk 64) and the chunked CUDA-core
    kernel at chunks 16, 32 and 128 -- four executions that really tile the
    sequence differently -- each match the oracle, and each other."""
    shape = inputs.ScanShape(batch=2, seqlen=300, heads=2, headdim=64, dstate=64, rank=1, chunk=64, dtype="bf16")
    inp = inputs.make_scan_inputs(shape, 5)
    d = dev(inp)
    yr, fr = oracle_scan(inp)
    outs = {}
    for q, algo in [(64, m3.M3_ALGO_CHUNKED_TC), (16, m3.M3_ALGO_CHUNKED_SIMT), (32, m3.M3_ALGO_CHUNKED_SIMT),
                    (128, m3.M3_ALGO_CHUNKED_SIMT)]:
        assert m3.m3_scan_algorithm(m3.scan_dims(d["x"], d["B"], q)) == algo
        y, f = gpu_scan(m3, d, q)
        torch.cuda.synchronize()
        outs[q] = (y.float().cpu(), f.cpu())
        assert max_rel(outs[q][0], yr) <= 2e-2 and max_rel(outs[q][1], fr) <= 2e-2, q
    for q in (16, 32, 128):
        assert max_rel(outs[q][0], outs[64][0]) <= 2e-2
        assert max_rel(outs[q][1], outs[64][1]) <= 2e-2


def test_tc_prefill_then_decode(m3):
    """Prefill (tensor cores) then bf16 decode steps continue the same sequence."""
    shape = inputs.ScanShape(batch=2, seqlen=150, heads=2, headdim=64, dstate=64, rank=2, chunk=64, dtype="bf16")
    inp = inputs.make_scan_inputs(shape, 23)
    d = dev(inp)
    T0 = 140
    pre = {k: (v[:, :T0].contiguous() if (v is not None and k != "A") else v) for k, v in d.items()}
    y0, state = gpu_scan(m3, pre, 64)
    ys = [y0.float()]
    for t in range(T0, 150):
        y = torch.empty_like(d["x"][:, t])
        m3.m3_step(state, d["x"][:, t].contiguous(), d["dt"][:, t].contiguous(), d["A"], d["B"][:, t].contiguous(),
                   d["C"][:, t].contiguous(), d["lam"][:, t].contiguous(), d["theta"][:, t].contiguous(),
                   d["B"][:, t - 1].contiguous(), d["x"][:, t - 1].contiguous(), y)
        ys.append(y[:, None].float())
    torch.cuda.synchronize()
    yr, fr = oracle_scan(inp)
    assert max_rel(torch.cat(ys, 1).cpu(), yr) <= 2e-2
    assert max_rel(state.cpu(), fr) <= 2e-2


def test_tc_deterministic(m3):
    shape = inputs.ScanShape(batch=2, seqlen=257, heads=2, headdim=64, dstate=64, rank=1, chunk=64, dtype="bf16")
    d = dev(inputs.make_scan_inputs(shape, 6))
    y1, f1 = gpu_scan(m3, d, 64)
    y2, f2 = gpu_scan(m3, d, 64)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(f1, f2)


@pytest.mark.parametrize("N,R", [(64, 1), (64, 4), (128, 1), (128, 4)], ids=lambda v: str(v))
def test_tc_repeated_runs_write_every_output_the_same(m3, N, R):
    """100 runs of one small prefill into buffers pre-filled with NaN, with other
    device work between some of them: every y and final-state element written,
    and every run bit-identical to the first (a check on the warpgroups' buffer
    hand-offs, whose races show up as rare wrong or unwritten chunks)."""
    shape = inputs.ScanShape(batch=2, seqlen=130, heads=3, headdim=64, dstate=N, rank=R, chunk=64 // R,
                             dtype="bf16")
    d = dev(inputs.make_scan_inputs(shape, 1100 + N + R))
    b, T, H, _, P = d["x"].shape
    junk = torch.empty(8 << 20, dtype=torch.uint8, device="cuda")
    ref = None
    for it in range(100):
        y = torch.full_like(d["x"], float("nan"))
        fs = torch.full((b, H, N, P), float("nan"), device="cuda")
        m3.m3_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["lam"], d["theta"], y, fs, chunk=64 // R)
        if it % 3 == 0:
            junk.random_(0, 255)
        if ref is None:
            torch.cuda.synchronize()
            assert not torch.isnan(y.float()).any() and not torch.isnan(fs).any()
            ref = (y, fs)
        else:
            assert torch.equal(y, ref[0]) and torch.equal(fs, ref[1]), it
    assert m3.m3_device_status() == m3.M3_OK


def test_tc_without_final_state(m3):
    shape = inputs.ScanShape(batch=1, seqlen=100, heads=2, headdim=64, dstate=64, rank=1, chunk=64, dtype="bf16")
    inp = inputs.make_scan_inputs(shape, 8)
    y, _ = gpu_scan(m3, dev(inp), 64, with_state=False)
    torch.cuda.synchronize()
    yr, _ = oracle_scan(inp)
    assert max_rel(y.float().cpu(), yr) <= 2e-2
