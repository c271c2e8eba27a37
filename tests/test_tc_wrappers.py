"""GPU unit tests of the hand-written tcgen05 / TMA wrappers the tensor-core
scan is built on: shared-memory descriptors (128-byte swizzle, K-major and
MN-major operands), the instruction descriptor, TMEM allocation and
tcgen05.ld lane mapping, and a TMA load with the 128-byte swizzle."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "csrc", "tc_probe.cu")
LIB = os.path.join(ROOT, "tests", "csrc", "libtcprobe.so")
CSRC = os.path.join(ROOT, "selective_state_space_131_b300", "csrc")


def build_probe():
    deps = [SRC, os.path.join(CSRC, "ptx_sm100.cuh")]
    if os.path.exists(LIB) and all(os.path.getmtime(d) <= os.path.getmtime(LIB) for d in deps):
        return LIB
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-I", CSRC, "-o", LIB, SRC, "-lcudart"], check=True)
    return LIB


@pytest.fixture(scope="module")
def probe():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    lib = ctypes.CDLL(build_probe())
    lib.probe_umma.argtypes = [ctypes.c_int] * 6 + [ctypes.c_void_p] * 4
    lib.probe_tma.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 5 + [ctypes.c_void_p] * 2
    return lib


def run_umma(lib, M, N, K, a_mn, b_mn, seed=0, half_split=0):
    import torch
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    dA, dB = A.cuda(), B.cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.probe_umma(M, N, K, a_mn, b_mn, half_split, dA.data_ptr(), dB.data_ptr(), D.data_ptr(),
                        st.data_ptr())
    assert rc == 0, rc
    assert int(st.item()) == 0, "mbarrier wait timed out"
    ref = A.double().numpy() @ B.double().numpy().T
    return D.cpu().double().numpy(), ref


@pytest.mark.gpu
@pytest.mark.parametrize("a_mn", [0, 1])
@pytest.mark.parametrize("b_mn", [0, 1])
@pytest.mark.parametrize("N,K", [(64, 64), (128, 128), (256, 64)])
def test_umma_m128(probe, a_mn, b_mn, N, K):
    D, ref = run_umma(probe, 128, N, K, a_mn, b_mn)
    err = np.abs(D - ref).max() / np.abs(ref).max()
    assert err < 1e-5, err


def m64_lane(i):
    """TMEM lane of accumulator row i for an M = 64 MMA: rows 16w..16w+15 sit
    in lanes 32w..32w+15 of each warp's quarter."""
    return (i // 16) * 32 + i % 16


@pytest.mark.gpu
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 1), (0, 1)])
def test_umma_m64_layout(probe, a_mn, b_mn):
    D, ref = run_umma(probe, 64, 64, 64, a_mn, b_mn, seed=3)
    lanes = [m64_lane(i) for i in range(64)]
    got = D[lanes]
    err = np.abs(got - ref).max() / np.abs(ref).max()
    ident = np.abs(D[:64] - ref).max() / np.abs(ref).max()
    print(f"M=64 layout: quarter-16 err {err:.3g}, identity err {ident:.3g}")
    assert err < 1e-5, (err, ident)


@pytest.mark.gpu
@pytest.mark.parametrize("rows,c1,c2", [(64, 0, 0), (64, 3, 1), (128, 40, 2)])
def test_tma_sw128(probe, rows, c1, c2):
    import torch
    d1, d2 = 150, 3
    g = torch.Generator().manual_seed(rows + c1)
    src = torch.randn(d2, d1, 64, generator=g).to(torch.bfloat16)
    out = torch.zeros(rows * 128, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dsrc = src.cuda()
    rc = probe.probe_tma(dsrc.data_ptr(), d1, d2, rows, c1, c2, out.data_ptr(), st.data_ptr())
    assert rc == 0 and int(st.item()) == 0
    img = out.cpu().numpy().view(np.uint16).reshape(rows, 64)
    bits = src.view(torch.int16).numpy().view(np.uint16)
    exp = np.zeros((rows, 64), dtype=np.uint16)
    for r in range(rows):
        if c1 + r < d1:
            for col in range(64):
                chunk = (col // 8) ^ (r % 8)
                exp[r, chunk * 8 + col % 8] = bits[c2, c1 + r, col]
    assert np.array_equal(img, exp)


@pytest.mark.gpu
@pytest.mark.parametrize("N", [64, 128])
def test_tmem_ld_16x32bx2(probe, N):
    """The 16x32bx2 TMEM load spreads an M = 64 accumulator over all 32
    threads of a warp: thread t < 16 gets row 16w + t, columns [c, c+32);
    thread t >= 16 the same row, columns [c+32, c+64)."""
    D, ref = run_umma(probe, 64, N, 64, 0, 1, seed=5, half_split=1)
    err = np.abs(D[:64] - ref).max() / np.abs(ref).max()
    assert err < 1e-5, err


@pytest.mark.gpu
@pytest.mark.parametrize("M", [64, 128])
def test_umma_b_mn_major_sw64(probe, M):
    """A 32-wide MN-major B operand in the 64-byte swizzle (the layout TMA's
    64-byte swizzle writes for a [K][32] bf16 tile)."""
    D, ref = run_umma(probe, M, 32, 64, 0, 2, seed=11)
    if M == 64:
        lanes = [m64_lane(i) for i in range(64)]
        D = D[lanes]
    err = np.abs(D[:M] - ref).max() / np.abs(ref).max()
    assert err < 1e-5, err
