"""The C-ABI library on the host: it loads, exports every entry point the
header declares, and rejects bad arguments before any launch.  No kernel
runs here (no GPU needed)."""
import ctypes
import os
import re

import pytest

from selective_state_space_131_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m3():
    if not build.up_to_date():
        build.build()
    from selective_state_space_131_b300 import m3scan
    return m3scan


def declared_symbols():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            names += re.findall(r"M3_API[^;(]*?\b(m3_\w+)\s*\(", src)
    return names


def test_every_declared_symbol_is_exported(m3):
    names = declared_symbols()
    assert {"m3_scan_fwd", "m3_scan_bwd", "m3_step", "m3_step_k", "m3_scan_workspace_size",
            "m3_status_string"} <= set(names)
    lib = ctypes.CDLL(m3.LIBRARY_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(m3):
    for code in range(-9, 1):
        assert m3.m3_status_string(code) != "unknown status"
    assert m3.m3_status_string(-99) == "unknown status"


def _dims(m3, **kw):
    base = dict(batch=2, seqlen=100, heads=4, headdim=64, dstate=64, rank=1, chunk=64, dtype=m3.M3_BF16)
    base.update(kw)
    return m3.make_dims(**base)


FAKE = 0x7f0000000000  # never dereferenced: every call below fails validation first


def _scan_ptrs(**over):
    p = dict(x=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, lam=FAKE, theta=FAKE, y=FAKE, fs=FAKE, ws=None, wsb=0)
    p.update(over)
    return [p[k] for k in ("x", "dt", "A", "B", "C", "lam", "theta", "y", "fs", "ws", "wsb")]


def test_scan_validation(m3):
    assert m3.raw_scan_fwd(_dims(m3), _scan_ptrs(x=None)) == m3.M3_ERR_NULL
    assert m3.raw_scan_fwd(_dims(m3), _scan_ptrs(C=None)) == m3.M3_ERR_NULL
    assert m3.raw_scan_fwd(_dims(m3, dstate=63), _scan_ptrs()) == m3.M3_ERR_SHAPE
    assert m3.raw_scan_fwd(_dims(m3, headdim=62), _scan_ptrs()) == m3.M3_ERR_SHAPE
    assert m3.raw_scan_fwd(_dims(m3, rank=9), _scan_ptrs()) == m3.M3_ERR_SHAPE
    assert m3.raw_scan_fwd(_dims(m3, chunk=48), _scan_ptrs()) == m3.M3_ERR_SHAPE
    assert m3.raw_scan_fwd(_dims(m3, heads=0), _scan_ptrs()) == m3.M3_ERR_SHAPE
    assert m3.raw_scan_fwd(_dims(m3, seqlen=-1), _scan_ptrs()) == m3.M3_ERR_SHAPE
    assert m3.raw_scan_fwd(_dims(m3, dtype=7), _scan_ptrs()) == m3.M3_ERR_DTYPE
    assert m3.raw_scan_fwd(_dims(m3), _scan_ptrs(y=FAKE + 1)) == m3.M3_ERR_ALIGN
    assert m3.raw_scan_fwd(_dims(m3, dtype=m3.M3_F32), _scan_ptrs(theta=FAKE + 2)) == m3.M3_ERR_ALIGN
    assert m3.raw_scan_fwd(_dims(m3), _scan_ptrs(dt=FAKE + 2)) == m3.M3_ERR_ALIGN
    assert m3.raw_scan_fwd(_dims(m3), _scan_ptrs(fs=FAKE + 8)) == m3.M3_ERR_ALIGN
    d = _dims(m3)
    d.reserved = 1
    assert m3.raw_scan_fwd(d, _scan_ptrs()) == m3.M3_ERR_SHAPE
    # an empty batch is valid and launches nothing
    assert m3.raw_scan_fwd(_dims(m3, batch=0), _scan_ptrs(x=None, y=None)) == m3.M3_OK


def _step_ptrs(**over):
    p = dict(state=FAKE, x=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, lam=FAKE, theta=FAKE, pB=FAKE, px=FAKE, y=FAKE)
    p.update(over)
    return [p[k] for k in ("state", "x", "dt", "A", "B", "C", "lam", "theta", "pB", "px", "y")]


def test_step_validation(m3):
    assert m3.raw_step(_dims(m3), _step_ptrs(state=None)) == m3.M3_ERR_NULL
    assert m3.raw_step(_dims(m3), _step_ptrs(pB=None)) == m3.M3_ERR_NULL    # prev_B and prev_x go together
    assert m3.raw_step(_dims(m3, dstate=5), _step_ptrs()) == m3.M3_ERR_SHAPE
    assert m3.raw_step(_dims(m3), _step_ptrs(px=FAKE + 1)) == m3.M3_ERR_ALIGN
    assert m3.raw_step(_dims(m3), _step_ptrs(state=FAKE + 4)) == m3.M3_ERR_ALIGN
    assert m3.raw_step(_dims(m3, batch=0), _step_ptrs()) == m3.M3_OK


def test_algorithm_selection(m3):
    assert m3.m3_scan_algorithm(_dims(m3, dstate=63)) == m3.M3_ALGO_NONE
    # the tensor-core kernel takes bf16, P = 64, N in {64, 128}, R in {1, 2, 4} when
    # the chunk is its 64-row tile (chunk * R == 64)
    for n in (64, 128):
        for r in (1, 2, 4):
            assert m3.m3_scan_algorithm(_dims(m3, dstate=n, rank=r, chunk=64 // r)) == m3.M3_ALGO_CHUNKED_TC
    # any other chunk is executed as given by the chunked CUDA-core kernel
    assert m3.m3_scan_algorithm(_dims(m3, chunk=32)) == m3.M3_ALGO_CHUNKED_SIMT
    assert m3.m3_scan_algorithm(_dims(m3, chunk=128)) == m3.M3_ALGO_CHUNKED_SIMT
    assert m3.m3_scan_algorithm(_dims(m3, rank=4, chunk=64)) == m3.M3_ALGO_CHUNKED_SIMT
    assert m3.m3_scan_algorithm(_dims(m3, dtype=m3.M3_F32)) == m3.M3_ALGO_CHUNKED_SIMT
    assert m3.m3_scan_algorithm(_dims(m3, headdim=16, dstate=16, chunk=32, dtype=m3.M3_F32)) == \
        m3.M3_ALGO_CHUNKED_SIMT
    # a chunk too large for shared memory falls back to the token-serial kernel
    assert m3.m3_scan_algorithm(_dims(m3, rank=8, chunk=128, dtype=m3.M3_F32)) == m3.M3_ALGO_SEQUENTIAL
    assert m3.m3_scan_workspace_size(_dims(m3)) == 0


def test_launch_without_gpu_reports_cuda_error(m3):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: fake pointers must not reach a kernel")
    assert m3.raw_scan_fwd(_dims(m3, dtype=m3.M3_F32), _scan_ptrs()) == m3.M3_ERR_CUDA
    assert m3.raw_step(_dims(m3), _step_ptrs()) == m3.M3_ERR_CUDA


def _from_ptrs(**over):
    p = dict(x=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, lam=FAKE, theta=FAKE, h0=FAKE, pB=FAKE, px=FAKE, y=FAKE,
             fs=FAKE, ws=None, wsb=0)
    p.update(over)
    return [p[k] for k in ("x", "dt", "A", "B", "C", "lam", "theta", "h0", "pB", "px", "y", "fs", "ws", "wsb")]


def test_scan_from_validation(m3):
    assert m3.raw_scan_fwd_from(_dims(m3), _from_ptrs(pB=None)) == m3.M3_ERR_NULL   # prev_B / prev_x pair
    assert m3.raw_scan_fwd_from(_dims(m3), _from_ptrs(px=None)) == m3.M3_ERR_NULL
    assert m3.raw_scan_fwd_from(_dims(m3), _from_ptrs(h0=FAKE + 4)) == m3.M3_ERR_ALIGN
    assert m3.raw_scan_fwd_from(_dims(m3), _from_ptrs(pB=FAKE + 1)) == m3.M3_ERR_ALIGN
    assert m3.raw_scan_fwd_from(_dims(m3, dstate=7), _from_ptrs()) == m3.M3_ERR_SHAPE
    assert m3.raw_scan_fwd_from(_dims(m3, batch=0), _from_ptrs(x=None, y=None)) == m3.M3_OK


def _bcnorm_ptrs(**over):
    p = dict(x=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, lam=FAKE, theta=FAKE, wB=FAKE, wC=FAKE, bB=FAKE, bC=FAKE,
             y=FAKE, fs=FAKE, ws=None, wsb=0)
    p.update(over)
    return [p[k] for k in ("x", "dt", "A", "B", "C", "lam", "theta", "wB", "wC", "bB", "bC", "y", "fs", "ws", "wsb")]


def test_scan_bcnorm_validation(m3):
    d = _dims(m3)
    for k in ("wB", "wC", "bB", "bC"):
        assert m3.raw_scan_fwd_bcnorm(d, _bcnorm_ptrs(**{k: None}), 1e-6) == m3.M3_ERR_NULL
        assert m3.raw_scan_fwd_bcnorm(d, _bcnorm_ptrs(**{k: FAKE + 2}), 1e-6) == m3.M3_ERR_ALIGN
    for eps in (-1e-6, float("inf"), float("nan")):
        assert m3.raw_scan_fwd_bcnorm(d, _bcnorm_ptrs(), eps) == m3.M3_ERR_VALUE
    # only the tensor-core kernel's shapes and chunk take the fused normalisation
    assert m3.raw_scan_fwd_bcnorm(_dims(m3, dtype=m3.M3_F32), _bcnorm_ptrs(), 1e-6) == m3.M3_ERR_UNSUPPORTED
    assert m3.raw_scan_fwd_bcnorm(_dims(m3, chunk=32), _bcnorm_ptrs(), 1e-6) == m3.M3_ERR_UNSUPPORTED
    assert m3.raw_scan_fwd_bcnorm(_dims(m3, headdim=32), _bcnorm_ptrs(), 1e-6) == m3.M3_ERR_UNSUPPORTED
    assert m3.raw_scan_fwd_bcnorm(_dims(m3, dstate=7), _bcnorm_ptrs(), 1e-6) == m3.M3_ERR_SHAPE
    assert m3.raw_scan_fwd_bcnorm(_dims(m3, batch=0), _bcnorm_ptrs(x=None, y=None), 1e-6) == m3.M3_OK


def test_selftest_wait_timeout_validation(m3):
    assert m3.m3_selftest_wait_timeout(0, 0) == m3.M3_ERR_VALUE
    assert m3.m3_selftest_wait_timeout(-5, 0) == m3.M3_ERR_VALUE
    assert m3.m3_selftest_wait_timeout(5_000_000_000, 0) == m3.M3_ERR_VALUE


def test_binding_rejects_strided_tensors(m3):
    import torch
    t = torch.zeros(4, 6)
    assert m3._ptr(t) == t.data_ptr()
    with pytest.raises(ValueError):
        m3._ptr(t.t())                  # a transposed view is not C-contiguous
    with pytest.raises(ValueError):
        m3._ptr(torch.zeros(3, 5, 2)[:, 1])


def test_step_k_validation(m3):
    # pointers in the order (state, x, dt, A, B, C, lam, theta, pB, px, y)
    d = _dims(m3, seqlen=8)
    assert m3.raw_step_k(d, _step_ptrs(state=None)) == m3.M3_ERR_NULL
    assert m3.raw_step_k(d, _step_ptrs(x=None)) == m3.M3_ERR_NULL
    assert m3.raw_step_k(d, _step_ptrs(pB=None)) == m3.M3_ERR_NULL    # prev_B and prev_x go together
    assert m3.raw_step_k(_dims(m3, seqlen=8, dstate=5), _step_ptrs()) == m3.M3_ERR_SHAPE
    assert m3.raw_step_k(_dims(m3, seqlen=-1), _step_ptrs()) == m3.M3_ERR_SHAPE
    assert m3.raw_step_k(d, _step_ptrs(px=FAKE + 1)) == m3.M3_ERR_ALIGN
    assert m3.raw_step_k(d, _step_ptrs(state=FAKE + 4)) == m3.M3_ERR_ALIGN
    # no token or no batch row: nothing to do, nothing launched
    assert m3.raw_step_k(_dims(m3, seqlen=0), _step_ptrs()) == m3.M3_OK
    assert m3.raw_step_k(_dims(m3, seqlen=8, batch=0), _step_ptrs()) == m3.M3_OK


def _bwd_ptrs(**over):
    names = ("x", "dt", "A", "B", "C", "lam", "theta", "dy", "dfinal", "dx", "ddt", "dA", "dB", "dC", "dlam",
             "dtheta", "ws", "wsb")
    p = {k: FAKE for k in names}
    p.update(wsb=1 << 40)
    p.update(over)
    return [p[k] for k in names]


def test_bwd_validation(m3):
    d = _dims(m3)
    need = m3.m3_scan_bwd_workspace_size(d)
    # chunk states of every (b, h): (ceil(100 / 64) + 1) x 64 x 64 fp32 each, and more
    assert need >= 2 * 4 * 3 * 64 * 64 * 4
    assert m3.raw_scan_bwd(d, _bwd_ptrs(dx=None)) == m3.M3_ERR_NULL
    assert m3.raw_scan_bwd(d, _bwd_ptrs(dA=None)) == m3.M3_ERR_NULL
    assert m3.raw_scan_bwd(d, _bwd_ptrs(dlam=None)) == m3.M3_ERR_NULL        # lambda given, no dlambda
    assert m3.raw_scan_bwd(d, _bwd_ptrs(dtheta=None)) == m3.M3_ERR_NULL      # theta given, no dtheta
    assert m3.raw_scan_bwd(d, _bwd_ptrs(dx=FAKE + 1)) == m3.M3_ERR_ALIGN
    assert m3.raw_scan_bwd(d, _bwd_ptrs(ws=None)) == m3.M3_ERR_WORKSPACE
    assert m3.raw_scan_bwd(d, _bwd_ptrs(wsb=need - 1)) == m3.M3_ERR_WORKSPACE
    assert m3.raw_scan_bwd(d, _bwd_ptrs(ws=FAKE + 16)) == m3.M3_ERR_ALIGN    # workspace: 256-byte aligned
    # more than 64 rows per chunk is not taken (nor a workspace size given for it)
    assert m3.raw_scan_bwd(_dims(m3, chunk=128), _bwd_ptrs()) == m3.M3_ERR_UNSUPPORTED
    assert m3.raw_scan_bwd(_dims(m3, rank=2, chunk=64), _bwd_ptrs()) == m3.M3_ERR_UNSUPPORTED
    assert m3.m3_scan_bwd_workspace_size(_dims(m3, chunk=128)) == 0
    assert m3.raw_scan_bwd(_dims(m3, dstate=7), _bwd_ptrs()) == m3.M3_ERR_SHAPE


def test_scan_fwd_host_validation(m3):
    """The host-buffer prefill: its workspace size and the arguments it rejects
    before touching a stream (no GPU here)."""
    d = _dims(m3)    # b2 T100 h4 P64 N64 R1 bf16
    per_row = 100 * 4 * (64 * 2 * 2 + 4 + 64 * 2 * 2 + 4 + 32 * 2)   # x, dt, B, C, lambda, theta, y of one row
    one = m3.m3_scan_fwd_host_workspace_size(d, 1)
    two = m3.m3_scan_fwd_host_workspace_size(d, 2)
    assert one >= 2 * (per_row + 4 * 64 * 64 * 4) and 1.9 * one < two < 2 * one
    assert m3.m3_scan_fwd_host_workspace_size(d, 0) == one            # default: ceil(2 / 8) = 1 row
    assert m3.m3_scan_fwd_host_workspace_size(d, 50) == two           # at most the batch
    assert m3.m3_scan_fwd_host_workspace_size(d, -1) == 0
    assert m3.m3_scan_fwd_host_workspace_size(_dims(m3, batch=0), 1) == 0
    assert m3.m3_scan_fwd_host_workspace_size(_dims(m3, dstate=63), 1) == 0
    ok = dict(ws=FAKE, wsb=one)
    assert m3.raw_scan_fwd_host(d, _scan_ptrs(**ok), slice=-1) == m3.M3_ERR_VALUE
    assert m3.raw_scan_fwd_host(d, _scan_ptrs(x=None, **ok)) == m3.M3_ERR_NULL
    assert m3.raw_scan_fwd_host(d, _scan_ptrs(A=None, **ok)) == m3.M3_ERR_NULL
    assert m3.raw_scan_fwd_host(d, _scan_ptrs(y=FAKE + 1, **ok)) == m3.M3_ERR_ALIGN
    assert m3.raw_scan_fwd_host(d, _scan_ptrs(ws=FAKE, wsb=one - 1)) == m3.M3_ERR_WORKSPACE
    assert m3.raw_scan_fwd_host(d, _scan_ptrs(ws=None, wsb=one)) == m3.M3_ERR_WORKSPACE
    assert m3.raw_scan_fwd_host(d, _scan_ptrs(ws=FAKE + 16, wsb=one)) == m3.M3_ERR_ALIGN
    assert m3.raw_scan_fwd_host(_dims(m3, dstate=63), _scan_ptrs(**ok)) == m3.M3_ERR_SHAPE
    assert m3.raw_scan_fwd_host(_dims(m3, batch=0), _scan_ptrs(x=None, y=None, ws=None, wsb=0)) == m3.M3_OK
