"""ctypes binding of libm3scan.so with the C ABI's entry-point names.

Argument marshalling only: sizes are read from the tensors' shapes, pointers
from ``data_ptr()`` and the stream from torch's current CUDA stream; every
step of the computation runs in the library's CUDA kernels.  Importing this
module loads the library and raises ImportError when it has not been built
(``python -m selective_state_space_131_b300.build``): there is no CPU path.

Tensor arguments may also be given as raw integer device addresses (or None
for an optional pointer), in which case ``dims`` must be passed explicitly.
"""
from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libm3scan.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libm3scan.so is not built ({_LIB_PATH}); run "
                      "`python -m selective_state_space_131_b300.build` (needs nvcc)")
_lib = ctypes.CDLL(_LIB_PATH)

M3_F32, M3_BF16 = 0, 1
M3_OK = 0
M3_ERR_NULL, M3_ERR_SHAPE, M3_ERR_DTYPE, M3_ERR_ALIGN = -1, -2, -3, -4
M3_ERR_CUDA, M3_ERR_UNSUPPORTED, M3_ERR_DEVICE, M3_ERR_WORKSPACE = -5, -6, -7, -8
M3_ERR_VALUE = -9
M3_ALGO_NONE, M3_ALGO_SEQUENTIAL, M3_ALGO_CHUNKED_TC, M3_ALGO_CHUNKED_SIMT = -1, 0, 1, 2


class m3_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("heads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("dstate", ctypes.c_int64), ("rank", ctypes.c_int64),
                ("chunk", ctypes.c_int64), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_vp = ctypes.c_void_p
_dp = ctypes.POINTER(m3_dims)
_lib.m3_scan_workspace_size.argtypes = [_dp]
_lib.m3_scan_workspace_size.restype = ctypes.c_size_t
_lib.m3_scan_algorithm.argtypes = [_dp]
_lib.m3_scan_algorithm.restype = ctypes.c_int
_lib.m3_scan_fwd.argtypes = [_dp] + [_vp] * 10 + [ctypes.c_size_t, _vp]
_lib.m3_scan_fwd.restype = ctypes.c_int
_lib.m3_scan_fwd_from.argtypes = [_dp] + [_vp] * 13 + [ctypes.c_size_t, _vp]
_lib.m3_scan_fwd_from.restype = ctypes.c_int
_lib.m3_scan_fwd_bcnorm.argtypes = [_dp] + [_vp] * 11 + [ctypes.c_float] + [_vp] * 3 + [ctypes.c_size_t, _vp]
_lib.m3_scan_fwd_bcnorm.restype = ctypes.c_int
_lib.m3_scan_fwd_host_workspace_size.argtypes = [_dp, ctypes.c_int64]
_lib.m3_scan_fwd_host_workspace_size.restype = ctypes.c_size_t
_lib.m3_scan_fwd_host.argtypes = [_dp] + [_vp] * 9 + [ctypes.c_int64, _vp, ctypes.c_size_t, _vp]
_lib.m3_scan_fwd_host.restype = ctypes.c_int
_lib.m3_step.argtypes = [_dp] + [_vp] * 11 + [_vp]
_lib.m3_step.restype = ctypes.c_int
_lib.m3_scan_bwd_workspace_size.argtypes = [_dp]
_lib.m3_scan_bwd_workspace_size.restype = ctypes.c_size_t
_lib.m3_scan_bwd.argtypes = [_dp] + [_vp] * 17 + [ctypes.c_size_t, _vp]
_lib.m3_scan_bwd.restype = ctypes.c_int
_lib.m3_scan_bwd_noalloc.argtypes = [_dp] + [_vp] * 16 + [_vp]
_lib.m3_scan_bwd_noalloc.restype = ctypes.c_int
_lib.m3_step_k.argtypes = [_dp] + [_vp] * 11 + [_vp]
_lib.m3_step_k.restype = ctypes.c_int
_lib.m3_selftest_wait_timeout.argtypes = [ctypes.c_longlong, _vp]
_lib.m3_selftest_wait_timeout.restype = ctypes.c_int
_lib.m3_device_status.argtypes = [_vp]
_lib.m3_device_status.restype = ctypes.c_int
_lib.m3_status_string.argtypes = [ctypes.c_int]
_lib.m3_status_string.restype = ctypes.c_char_p

LIBRARY_PATH = _LIB_PATH


class M3Error(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {m3_status_string(status)} ({status})")
        self.status = status


def m3_status_string(status: int) -> str:
    return _lib.m3_status_string(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        # the C ABI takes C-contiguous buffers; a strided view would be read as one
        raise ValueError(f"tensor of shape {tuple(t.shape)} is not contiguous; pass .contiguous()")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return M3_F32
    if t.dtype == torch.bfloat16:
        return M3_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def make_dims(batch, seqlen, heads, headdim, dstate, rank=1, chunk=64, dtype=M3_BF16) -> m3_dims:
    return m3_dims(int(batch), int(seqlen), int(heads), int(headdim), int(dstate), int(rank), int(chunk),
                   int(dtype), 0)


def scan_dims(x, B, chunk: int) -> m3_dims:
    """Dims of a prefill from x [b,T,h,R,P] and B [b,T,h,R,N]."""
    b, T, H, R, P = x.shape
    return make_dims(b, T, H, P, B.shape[-1], R, chunk, _dtype_code(x))


def step_dims(x_t, B_t) -> m3_dims:
    """Dims of a decode step from x_t [b,h,R,P] and B_t [b,h,R,N]."""
    b, H, R, P = x_t.shape
    return make_dims(b, 1, H, P, B_t.shape[-1], R, 64, _dtype_code(x_t))


def m3_scan_workspace_size(dims: m3_dims) -> int:
    return int(_lib.m3_scan_workspace_size(ctypes.byref(dims)))


def m3_scan_algorithm(dims: m3_dims) -> int:
    return int(_lib.m3_scan_algorithm(ctypes.byref(dims)))


def m3_scan_fwd(x, dt, A, B, C, lam, theta, y, final_state, chunk: int = 64, workspace=None,
                workspace_bytes: int = 0, stream=None, dims: m3_dims | None = None) -> None:
    """Chunked prefill; writes y (and final_state if given).  Raises M3Error."""
    if dims is None:
        dims = scan_dims(x, B, chunk)
    rc = _lib.m3_scan_fwd(ctypes.byref(dims), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(lam),
                          _ptr(theta), _ptr(y), _ptr(final_state), _ptr(workspace), int(workspace_bytes),
                          _stream(stream))
    if rc != M3_OK:
        raise M3Error(rc, "m3_scan_fwd")


def m3_scan_fwd_host_workspace_size(dims: m3_dims, slice: int = 0) -> int:
    """Device workspace bytes of m3_scan_fwd_host for these sizes and slice."""
    return int(_lib.m3_scan_fwd_host_workspace_size(ctypes.byref(dims), int(slice)))


def m3_scan_fwd_host(x, dt, A, B, C, lam, theta, y, final_state, workspace, workspace_bytes: int, slice: int = 0,
                     chunk: int = 64, stream=None, dims: m3_dims | None = None) -> None:
    """Prefill with every tensor in host memory (CPU tensors, page-locked for the
    copies to overlap), the batch in slices of `slice` rows staged through the
    device `workspace`; y / final_state are complete once `stream` is.  Raises
    M3Error."""
    if dims is None:
        dims = scan_dims(x, B, chunk)
    rc = _lib.m3_scan_fwd_host(ctypes.byref(dims), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(lam),
                               _ptr(theta), _ptr(y), _ptr(final_state), int(slice), _ptr(workspace),
                               int(workspace_bytes), _stream(stream))
    if rc != M3_OK:
        raise M3Error(rc, "m3_scan_fwd_host")


def m3_scan_fwd_from(x, dt, A, B, C, lam, theta, initial_state, prev_B, prev_x, y, final_state, chunk: int = 64,
                     workspace=None, workspace_bytes: int = 0, stream=None, dims: m3_dims | None = None) -> None:
    """Prefill continuing a sequence from initial_state [b,h,N,P] (fp32, complex
    frame; None for zero) and the previous token's prev_B [b,h,R,N] / prev_x
    [b,h,R,P] (both None for no previous token).  Raises M3Error."""
    if dims is None:
        dims = scan_dims(x, B, chunk)
    rc = _lib.m3_scan_fwd_from(ctypes.byref(dims), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(lam),
                               _ptr(theta), _ptr(initial_state), _ptr(prev_B), _ptr(prev_x), _ptr(y),
                               _ptr(final_state), _ptr(workspace), int(workspace_bytes), _stream(stream))
    if rc != M3_OK:
        raise M3Error(rc, "m3_scan_fwd_from")


def m3_scan_fwd_bcnorm(x, dt, A, B, C, lam, theta, norm_B, norm_C, bias_B, bias_C, eps: float, y, final_state,
                       chunk: int = 64, workspace=None, workspace_bytes: int = 0, stream=None,
                       dims: m3_dims | None = None) -> None:
    """Prefill with the B / C normalisation and biases fused into the prologue:
    norm_B / norm_C [N] fp32 scales, bias_B / bias_C [h, N] fp32 biases, eps >= 0.
    Raises M3Error."""
    if dims is None:
        dims = scan_dims(x, B, chunk)
    rc = _lib.m3_scan_fwd_bcnorm(ctypes.byref(dims), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(lam),
                                 _ptr(theta), _ptr(norm_B), _ptr(norm_C), _ptr(bias_B), _ptr(bias_C), float(eps),
                                 _ptr(y), _ptr(final_state), _ptr(workspace), int(workspace_bytes), _stream(stream))
    if rc != M3_OK:
        raise M3Error(rc, "m3_scan_fwd_bcnorm")


def raw_scan_fwd_bcnorm(dims: m3_dims, ptrs, eps: float, stream=None) -> int:
    """Direct call with raw addresses (x, dt, A, B, C, lam, theta, norm_B, norm_C,
    bias_B, bias_C, y, final_state, workspace, workspace_bytes) and eps; returns
    the status code."""
    *p, ws_bytes = ptrs
    return int(_lib.m3_scan_fwd_bcnorm(ctypes.byref(dims), *p[:11], ctypes.c_float(eps), *p[11:], int(ws_bytes),
                                       stream))


def m3_step(state, x_t, dt_t, A, B_t, C_t, lam_t, theta_t, prev_B, prev_x, y_t, stream=None,
            dims: m3_dims | None = None) -> None:
    """One decode step; updates state in place and writes y_t.  Raises M3Error."""
    if dims is None:
        dims = step_dims(x_t, B_t)
    rc = _lib.m3_step(ctypes.byref(dims), _ptr(state), _ptr(x_t), _ptr(dt_t), _ptr(A), _ptr(B_t), _ptr(C_t),
                      _ptr(lam_t), _ptr(theta_t), _ptr(prev_B), _ptr(prev_x), _ptr(y_t), _stream(stream))
    if rc != M3_OK:
        raise M3Error(rc, "m3_step")


def m3_scan_bwd_workspace_size(dims: m3_dims) -> int:
    return int(_lib.m3_scan_bwd_workspace_size(ctypes.byref(dims)))


def m3_scan_bwd(x, dt, A, B, C, lam, theta, dy, dfinal, dx, ddt, dA, dB, dC, dlam, dtheta, workspace,
                workspace_bytes: int, chunk: int = 64, stream=None, dims: m3_dims | None = None) -> None:
    """Backward pass of the prefill: writes dx, ddt, dA [h], dB, dC, dlam (if
    lam is given) and dtheta (if theta is given) from the upstream dy and
    dfinal (or None).  workspace: a device buffer of at least
    m3_scan_bwd_workspace_size(dims) bytes.  Raises M3Error."""
    if dims is None:
        dims = scan_dims(x, B, chunk)
    rc = _lib.m3_scan_bwd(ctypes.byref(dims), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(lam), _ptr(theta),
                          _ptr(dy), _ptr(dfinal), _ptr(dx), _ptr(ddt), _ptr(dA), _ptr(dB), _ptr(dC), _ptr(dlam),
                          _ptr(dtheta), _ptr(workspace), int(workspace_bytes), _stream(stream))
    if rc != M3_OK:
        raise M3Error(rc, "m3_scan_bwd")


def raw_scan_bwd(dims: m3_dims, ptrs, stream=None) -> int:
    """Direct call with raw addresses (x, dt, A, B, C, lam, theta, dy, dfinal, dx,
    ddt, dA, dB, dC, dlam, dtheta, workspace, workspace_bytes); returns the
    status code."""
    *p, ws_bytes = ptrs
    return int(_lib.m3_scan_bwd(ctypes.byref(dims), *p, int(ws_bytes), stream))


def m3_scan_bwd_noalloc(x, dt, A, B, C, lam, theta, dy, dfinal, dx, ddt, dA, dB, dC, dlam, dtheta,
                        chunk: int = 64, stream=None, dims: m3_dims | None = None) -> None:
    """m3_scan_bwd without a workspace argument, for callers that cannot
    allocate device memory: the library's fixed 32 MiB scratch serves instead
    (sizes needing more raise M3Error with M3_ERR_WORKSPACE; calls that overlap
    on the GPU share that scratch and must be ordered).  Raises M3Error."""
    if dims is None:
        dims = scan_dims(x, B, chunk)
    rc = _lib.m3_scan_bwd_noalloc(ctypes.byref(dims), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(lam),
                                  _ptr(theta), _ptr(dy), _ptr(dfinal), _ptr(dx), _ptr(ddt), _ptr(dA), _ptr(dB),
                                  _ptr(dC), _ptr(dlam), _ptr(dtheta), _stream(stream))
    if rc != M3_OK:
        raise M3Error(rc, "m3_scan_bwd_noalloc")


def m3_step_k(state, x, dt, A, B, C, lam, theta, prev_B, prev_x, y, stream=None,
              dims: m3_dims | None = None) -> None:
    """k decode steps in one launch: x [b,k,h,R,P], dt / lam [b,k,h],
    B / C [b,k,h,R,N], theta [b,k,h,N/2] (token-major, as for the prefill);
    updates state [b,h,N,P] in place and writes y [b,k,h,R,P].  Raises M3Error."""
    if dims is None:
        dims = scan_dims(x, B, 64)
    rc = _lib.m3_step_k(ctypes.byref(dims), _ptr(state), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(lam),
                        _ptr(theta), _ptr(prev_B), _ptr(prev_x), _ptr(y), _stream(stream))
    if rc != M3_OK:
        raise M3Error(rc, "m3_step_k")


def raw_step_k(dims: m3_dims, ptrs, stream=None) -> int:
    """Direct call with raw addresses (state, x, dt, A, B, C, lam, theta, prev_B,
    prev_x, y); returns the status code."""
    return int(_lib.m3_step_k(ctypes.byref(dims), *ptrs, stream))


def m3_selftest_wait_timeout(budget_cycles: int, stream=None) -> int:
    """Launch the bounded-wait self-test (a wait that nothing satisfies, given
    up after budget_cycles); returns the launch status.  The device status word
    then reports the timeout through m3_device_status()."""
    return int(_lib.m3_selftest_wait_timeout(int(budget_cycles), _stream(stream)))


def m3_device_status(stream=None) -> int:
    return int(_lib.m3_device_status(_stream(stream)))


def raw_scan_fwd(dims: m3_dims, ptrs, stream=None) -> int:
    """Direct call with raw addresses (x, dt, A, B, C, lam, theta, y, final_state,
    workspace, workspace_bytes); returns the status code."""
    *p, ws_bytes = ptrs
    return int(_lib.m3_scan_fwd(ctypes.byref(dims), *p, int(ws_bytes), stream))


def raw_scan_fwd_host(dims: m3_dims, ptrs, slice: int = 0, stream=None) -> int:
    """Direct call with raw addresses (x, dt, A, B, C, lam, theta, y, final_state,
    workspace, workspace_bytes) and the slice; returns the status code."""
    *p, ws, ws_bytes = ptrs
    return int(_lib.m3_scan_fwd_host(ctypes.byref(dims), *p, int(slice), ws, int(ws_bytes), stream))


def raw_scan_fwd_from(dims: m3_dims, ptrs, stream=None) -> int:
    """Direct call with raw addresses (x, dt, A, B, C, lam, theta, initial_state,
    prev_B, prev_x, y, final_state, workspace, workspace_bytes); returns the
    status code."""
    *p, ws_bytes = ptrs
    return int(_lib.m3_scan_fwd_from(ctypes.byref(dims), *p, int(ws_bytes), stream))


def raw_step(dims: m3_dims, ptrs, stream=None) -> int:
    """Direct call with raw addresses (state, x_t, dt_t, A, B_t, C_t, lam_t, theta_t,
    prev_B, prev_x, y_t); returns the status code."""
    return int(_lib.m3_step(ctypes.byref(dims), *ptrs, stream))
