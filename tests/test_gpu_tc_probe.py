"""Unit test of the tcgen05 layouts and descriptors (csrc/ptx.cuh) the chunk kernels use:
K-major tf32 and bf16 operands in 128-byte-swizzled shared memory, tf32 A operands in TMEM,
and the bf16 MN-major operand layouts, accumulated in TMEM and read back with tcgen05.ld."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("probe") / "probe.so")
    src = os.path.join(ROOT, "tests", "gpu_probe", "mma_probe.cu")
    inc = os.path.join(ROOT, "linear_attention_state_kda_gb300", "csrc")
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                           "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I", inc, src,
                           "-o", out])
    L = ctypes.CDLL(out)
    L.probe_mma.restype = ctypes.c_int
    L.probe_mma.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                            ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    return L


def _tf32(x):
    return (x.view(torch.int32) & ~0x1FFF).view(torch.float32)


# (mode, N, K). Modes 4 and 5 are the bf16 MN-major layouts; mode 5 at N = 64, K = 64 is the
# one the prep kernel uses (U0^T = V^T TB^T reads the bf16 v staging itself as an MN-major A
# operand, two 64-channel column groups 8 KiB apart). tf32 operands are only ever K-major.
CASES = [(0, 64, 128), (0, 32, 64), (3, 64, 128), (6, 64, 64), (6, 128, 128), (6, 32, 64),
         (4, 128, 64), (5, 64, 64), (5, 32, 64)]


@pytest.mark.parametrize("mode,N,K", CASES)
def test_mma_layouts(probe, mode, N, K):
    g = torch.Generator().manual_seed(100 + mode * 7 + N + K)
    A = torch.randn(128, K, generator=g)
    B = torch.randn(N, K, generator=g)
    Bin = B.t().contiguous() if mode == 4 else B          # mode 4: B given as [K][N]
    Ain = A.t().contiguous() if mode == 5 else A          # mode 5: A given as [K][128]
    if mode in (3, 4, 5):
        ref = A.bfloat16().double() @ B.bfloat16().double().t()
    else:
        ref = _tf32(A).double() @ _tf32(B).double().t()
    dA, dB = Ain.cuda(), Bin.cuda()
    dD = torch.zeros(128, N, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.probe_mma(mode, dA.data_ptr(), dB.data_ptr(), dD.data_ptr(), N, K,
                         err.data_ptr())
    torch.cuda.synchronize()
    assert rc == 0 and err.item() == 0
    D = dD.cpu().double()
    rel = (D - ref).abs().max() / ref.abs().max()
    # bf16 products are exact in fp32 accumulation up to summation order; tf32 operands: the
    # reference truncates to 10 mantissa bits (rounding would also pass)
    assert rel < (1e-5 if mode in (3, 4, 5) else 3e-3), (mode, N, K, float(rel))
