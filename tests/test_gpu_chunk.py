"""GPU parity of the chunked CUDA-core prefill (M3_ALGO_CHUNKED_SIMT), which
executes exactly the chunk the caller asks for, against the fp64 oracle:

  * chunk invariance in fp32 at the 1e-4 bar: one input through chunks of 16,
    32, 64 and 128 tokens, each matching the oracle (the chunked algebra -- the
    folded trapezoid mask and the augmented carry -- checked without bf16
    rounding in the way);
  * the MIMO R = 4 workload at its stated chunk of 64 tokens (256-row chunks)
    at full size, on sampled sequences;
  * the forced edge cases of test_gpu_edges in fp32;
  * the token-serial kernel, which takes chunks too large for shared memory.
"""
import pytest
import torch

from selective_state_space_131_b300 import inputs
from tests.gpu_util import TOL, dev, gpu_scan, max_rel, oracle_scan
from tests.test_gpu_edges import apply_edge

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m3():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from selective_state_space_131_b300 import m3scan
    return m3scan


def run(m3, inp, chunk, expect_algo):
    d = dev(inp)
    assert m3.m3_scan_algorithm(m3.scan_dims(d["x"], d["B"], chunk)) == expect_algo
    y, fs = gpu_scan(m3, d, chunk)
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    return y.float().cpu(), fs.cpu()


# (N = 6 and 10 leave a partial 4-wide register tile of state rows; P = 12 and 4
# give 3 and 1 column tiles)
@pytest.mark.parametrize("R,N,P", [(1, 16, 16), (2, 64, 32), (4, 32, 64), (1, 6, 12), (2, 10, 4)],
                         ids=lambda v: str(v))
def test_chunk_invariance_f32(m3, R, N, P):
    """Chunks of 16, 32, 64, 128 tokens over T = 300 (ragged for every chunk):
    each within 1e-4 of the oracle, so within 2e-4 of each other."""
    shape = inputs.ScanShape(batch=2, seqlen=300, heads=3, headdim=P, dstate=N, rank=R, chunk=16, dtype="f32")
    inp = inputs.make_scan_inputs(shape, 600 + R + N)
    yr, fr = oracle_scan(inp)
    ran = 0
    for q in (16, 32, 64, 128):
        if m3.m3_scan_algorithm(m3.scan_dims(inp["x"], inp["B"], q)) != m3.M3_ALGO_CHUNKED_SIMT:
            continue   # a chunk whose rows do not fit in shared memory
        y, fs = run(m3, inp, q, m3.M3_ALGO_CHUNKED_SIMT)
        ey, ef = max_rel(y, yr), max_rel(fs, fr)
        assert ey <= TOL["f32"] and ef <= TOL["f32"], (q, ey, ef)
        print(f"R{R} N{N} P{P} Q{q}: y {ey:.2e} state {ef:.2e}")
        ran += 1
    assert ran >= 3


@pytest.mark.parametrize("kind", ["fast_decay", "a_zero", "lambda_zero", "lambda_one", "tiny_dt", "mixed",
                                  "large_phi"])
@pytest.mark.parametrize("R", [1, 4])
def test_chunked_simt_edges_f32(m3, kind, R):
    shape = inputs.ScanShape(batch=2, seqlen=209, heads=4, headdim=32, dstate=32, rank=R, chunk=32, dtype="f32")
    inp = apply_edge(inputs.make_scan_inputs(shape, 4300 + R), kind, 4301 + R, "f32", R)
    yr, fr = oracle_scan(inp)
    y, fs = run(m3, inp, 32, m3.M3_ALGO_CHUNKED_SIMT)
    assert torch.isfinite(y).all() and torch.isfinite(fs).all()
    ey, ef = max_rel(y, yr), max_rel(fs, fr)
    assert ey <= TOL["f32"] and ef <= TOL["f32"], (kind, ey, ef)


def test_large_cumulative_angle_f32(m3):
    """Per-step angles of ~1.2 rad over T = 8192 in fp32: |Phi| ~ 1e4 rad, and
    the 1e-4 bar still holds (the running angle is reduced mod 2 pi in fp64)."""
    shape = inputs.ScanShape(batch=1, seqlen=8192, heads=2, headdim=16, dstate=16, rank=1, chunk=64, dtype="f32")
    inp = apply_edge(inputs.make_scan_inputs(shape, 4400), "large_phi", 4401, "f32")
    assert inp["theta"].sum(1).abs().max().item() > 8e3
    yr, fr = oracle_scan(inp)
    y, fs = run(m3, inp, 64, m3.M3_ALGO_CHUNKED_SIMT)
    ey, ef = max_rel(y, yr), max_rel(fs, fr)
    assert ey <= TOL["f32"] and ef <= TOL["f32"], (ey, ef)


def test_mimo_workload_chunk64_full_size(m3):
    """The MIMO R = 4 workload (b8 h32 T4096 P64 N64, bf16) at its stated chunk
    of 64 tokens: 256-row chunks on the chunked CUDA-core kernel, checked on
    every batch row for eight heads (64 sequences)."""
    shape = inputs.WORKLOADS[inputs.MIMO]
    assert shape.chunk == 64 and shape.rank == 4
    inp = inputs.make_scan_inputs(shape, 3)
    y, fs = run(m3, inp, 64, m3.M3_ALGO_CHUNKED_SIMT)
    bsel, hsel = list(range(8)), [0, 4, 9, 13, 18, 22, 27, 31]
    yr, fr = oracle_scan(inp, bsel, hsel)
    ey, ef = max_rel(y[bsel][:, :, hsel], yr), max_rel(fs[bsel][:, hsel], fr)
    assert ey <= TOL["bf16"] and ef <= TOL["bf16"], (ey, ef)
    print(f"MIMO chunk 64: y {ey:.2e} state {ef:.2e}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_token_serial_fallback(m3, dtype):
    """R = 8 with chunks of 128 tokens (1024 rows) does not fit in shared memory:
    the token-serial kernel runs it, at the same bar."""
    shape = inputs.ScanShape(batch=2, seqlen=150, heads=2, headdim=64, dstate=64, rank=8, chunk=128, dtype=dtype)
    inp = inputs.make_scan_inputs(shape, 4500)
    yr, fr = oracle_scan(inp)
    y, fs = run(m3, inp, 128, m3.M3_ALGO_SEQUENTIAL)
    ey, ef = max_rel(y, yr), max_rel(fs, fr)
    assert ey <= TOL[dtype] and ef <= TOL[dtype], (ey, ef)
