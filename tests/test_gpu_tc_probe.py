"""Unit probe of the tcgen05 layouts and descriptors (csrc/ptx.cuh) the chunk kernel uses:
K-major x K-major, K-major x MN-major and MN-major x K-major operands in 128-byte-swizzled
shared memory, tf32 and bf16, accumulated in TMEM and read back with tcgen05.ld."""
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


CASES = [(0, 64, 128), (0, 32, 64), (3, 64, 128), (6, 64, 64), (6, 128, 128), (6, 32, 64)]
# MN-major operand layouts (modes 1, 2 tf32; 4, 5 bf16) are probed for information only: the
# chunk kernel keeps every operand K-major (tf32 MN-major read back as zeros on sm_103a).
INFO = [(1, 128, 64), (2, 32, 64), (4, 128, 64), (5, 32, 64)]


@pytest.mark.parametrize("mode,N,K", CASES + INFO)
def test_mma_layouts(probe, mode, N, K):
    g = torch.Generator().manual_seed(100 + mode * 7 + N + K)
    A = torch.randn(128, K, generator=g)
    B = torch.randn(N, K, generator=g)
    if mode in (1, 4):
        Bin = B.t().contiguous()          # given as [K][N]
    else:
        Bin = B
    Ain = A.t().contiguous() if mode in (2, 5) else A   # given as [K][128]
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
    # tf32 operands: the reference truncates to 10 mantissa bits; rounding would also pass
    ok = rel < (1e-5 if mode in (3, 4, 5) else 3e-3)
    if (mode, N, K) in INFO:
        print(f"MN-major probe mode {mode} N {N} K {K}: rel {float(rel):.3e} "
              f"({'matches' if ok else 'does not match'})")
        return
    assert ok, (mode, N, K, float(rel))
