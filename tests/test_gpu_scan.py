"""kda_package_scan on its own, against the oracle's left fold, for both of its schedules at
dk = dv = 128: the sequential chain (sequences of at most 256 segments) and the Blelloch tree
(selected by a larger max_segs_per_seq). The packages are synthetic: M with spectral norm
below one (a contraction, as a segment's transition is) and D, S_init of order 0.1, so every
segment's prefix reaches the entry states of the later ones.

Cases: sequences of 3, 0 (empty), 1, 17 and 64 segments side by side, three heads, with and
without an entry state, with and without the final state; then offsets that decrease.
fp32 packages: entry and exit states within 1e-4 (normwise per head and per key-channel row).
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_kda_gb300 import kda
from kda_testutil import TOL_F32, f64, rel_s, rows_s

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
COUNTS = [3, 0, 1, 17, 64]
H = 3
D_ = 128


def _packages(seed, counts=COUNTS, h=H, d=D_):
    gen = torch.Generator().manual_seed(seed)
    P = sum(counts)
    # an i.i.d. N(0, s^2) d x d matrix has spectral norm about 2 s sqrt(d): s = 0.45 / sqrt(d)
    # keeps it near 0.9
    M = torch.randn(P, h, d, d, generator=gen) * (0.45 / d ** 0.5)
    D = torch.randn(P, h, d, d, generator=gen) * 0.1
    init = torch.randn(len(counts), h, d, d, generator=gen) * 0.1
    so = torch.zeros(len(counts) + 1, dtype=torch.int32)
    so[1:] = torch.cumsum(torch.tensor(counts), 0).to(torch.int32)
    return M, D, init, so


def _check(si, fin, rsi, rfin, tol=TOL_F32):
    e_si, e_fin = rel_s(f64(si), rsi), rel_s(f64(fin), rfin)
    r_si, r_fin = rows_s(f64(si), rsi)[0], rows_s(f64(fin), rfin)[0]
    print(f"seg_init {e_si:.2e} (rows {r_si:.2e}), final {e_fin:.2e} (rows {r_fin:.2e})")
    assert e_si < tol and e_fin < tol and r_si < tol and r_fin < tol


@pytest.mark.parametrize("with_init", [True, False])
@pytest.mark.parametrize("max_segs", [64, 300], ids=["sequential", "tree"])
def test_scan_vs_oracle(with_init, max_segs):
    M, D, init, so = _packages(71)
    init = init if with_init else None
    rsi, rfin = oracle.scan(M.numpy(), D.numpy(), so.numpy().astype(np.int64),
                            None if init is None else init.numpy())
    dev = lambda t: None if t is None else t.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    si, fin = kda.package_scan(dev(M), dev(D), dev(so), max_segs, init_state=dev(init),
                               status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    _check(si, fin, rsi, rfin)
    # the empty sequence passes its entry state (or zeros) through: a copy in the sequential
    # chain, the identity package applied in 3xTF32 in the tree (within 2^-20 of it)
    want = init[1] if init is not None else torch.zeros(H, D_, D_)
    if max_segs <= 256:
        assert torch.equal(fin[1].cpu(), want)
    else:
        assert torch.allclose(fin[1].cpu(), want, rtol=2e-6, atol=1e-9)


def test_sequential_and_tree_agree_without_final():
    M, D, init, so = _packages(72)
    args = (M.to(DEV), D.to(DEV), so.to(DEV))
    si_a, fin_a = kda.package_scan(*args, 64, init_state=init.to(DEV), want_final=False)
    si_b, _ = kda.package_scan(*args, 300, init_state=init.to(DEV))
    torch.cuda.synchronize()
    assert fin_a is None
    assert rel_s(f64(si_a), f64(si_b)) < 1e-5


def test_scan_decreasing_offsets_flagged():
    M, D, init, so = _packages(73, counts=[2, 3])
    bad = torch.tensor([0, 4, 3], dtype=torch.int32)  # sequence 1 ends before it starts
    for max_segs in (4, 300):
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        si = torch.zeros(5, H, D_, D_, device=DEV)
        _, fin = kda.package_scan(M.to(DEV), D.to(DEV), bad.to(DEV), max_segs,
                                  init_state=init.to(DEV), seg_init=si, status=status)
        torch.cuda.synchronize()
        assert status.item() & kda.STATUS_BAD_OFFSETS
        # the malformed sequence is treated as empty: its exit state is its entry state
        assert torch.allclose(fin[1].cpu(), init[1], rtol=2e-6, atol=1e-9)
