"""kda_package_scan_noalloc (the scan with the library's built-in scratch array, for callers
that cannot allocate device memory) against kda_package_scan with a caller workspace.

Called through the C ABI twice in a row on different packages, so that a result left in the
shared scratch by the first call cannot pass for the second call's answer. This file is
collected last (its name sorts after every other test file)."""
import ctypes

import pytest
import torch

from linear_attention_state_kda_gb300 import kda
from kda_testutil import TOL_F32, rel_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _packages(seed, P, H, d):
    g = torch.Generator(device=DEV).manual_seed(seed)
    M = torch.randn(P, H, d, d, generator=g, device=DEV) * (0.9 / d ** 0.5)
    D = torch.randn(P, H, d, d, generator=g, device=DEV)
    init = torch.randn(2, H, d, d, generator=g, device=DEV) * 0.02
    return M, D, init


def _noalloc_via_abi(M, D, seq_seg, max_segs, init, seg_init, fin):
    L = kda.lib()
    P, H, dk, dv = D.shape
    st = L.kda_package_scan_noalloc(seq_seg.numel() - 1, P, seq_seg.data_ptr(), max_segs, H,
                                    dk, dv, M.data_ptr(), D.data_ptr(), init.data_ptr(),
                                    seg_init.data_ptr(), fin.data_ptr(), None,
                                    torch.cuda.current_stream().cuda_stream)
    assert st == kda.KDA_OK, kda.last_error()


@pytest.mark.parametrize("d", [128, 64])
def test_noalloc_scan_matches_workspace_scan_twice(d):
    H = 4
    seq_seg = torch.tensor([0, 5, 8], dtype=torch.int32, device=DEV)  # 2 sequences, 5 + 3
    for call, seed in enumerate([7, 8]):
        M, D, init = _packages(seed, 8, H, d)
        ref_si, ref_fin = kda.package_scan(M, D, seq_seg, 5, init_state=init)
        si = torch.full_like(ref_si, float("nan"))
        fin = torch.full_like(ref_fin, float("nan"))
        _noalloc_via_abi(M, D, seq_seg, 5, init, si, fin)
        torch.cuda.synchronize()
        assert rel_gpu(si, ref_si) <= TOL_F32, (call, rel_gpu(si, ref_si))
        assert rel_gpu(fin, ref_fin) <= TOL_F32, (call, rel_gpu(fin, ref_fin))


def test_noalloc_scan_rejects_oversize():
    L = kda.lib()
    # 4 sequences x 16 segments x 32 heads at d = 128 needs 384 MiB of scratch (> 64 MiB)
    st = L.kda_package_scan_noalloc(4, 64, 4096, 16, 32, 128, 128, 4096, 4096, None, 4096,
                                    None, None, None)
    assert st == kda.KDA_ERR_WORKSPACE
    assert "64" in kda.last_error() or "67108864" in kda.last_error()
