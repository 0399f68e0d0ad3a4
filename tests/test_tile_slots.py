"""Host-side check of the tile placement the chunk and short-conv kernels share: tile j of
sequence s sits in slot floor(cu[s] / R) + s + j, a launch has floor(T / R) + n_seqs slots,
and a CTA finds its sequence as the largest s with floor(cu[s] / R) + s <= slot (the same
binary search the kernels run). Every sequence, empty ones included, owns a tile 0 (where
the per-sequence state work happens); no two tiles share a slot; every tile fits the grid."""
import numpy as np
import pytest


def _find(cu, R, slot):
    lo, hi = 0, len(cu) - 2
    while lo < hi:
        mid = (lo + hi + 1) >> 1
        if cu[mid] // R + mid <= slot:
            lo = mid
        else:
            hi = mid - 1
    return lo


@pytest.mark.parametrize("R", [16, 32, 64])
def test_tile_slots_unique_and_found(R):
    rng = np.random.default_rng(R)
    for trial in range(300):
        n = int(rng.integers(1, 12))
        lens = rng.integers(0, 4 * R, n)
        lens[rng.random(n) < 0.25] = 0                    # empty sequences
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        T = int(cu[-1])
        n_slots = T // R + n
        owner = {}
        for s in range(n):
            L = int(cu[s + 1] - cu[s])
            for j in range(max(1, -(-L // R))):            # tile 0 always exists
                slot = int(cu[s] // R + s + j)
                assert slot < n_slots, (lens, s, j)
                assert slot not in owner, (lens, s, j)
                owner[slot] = (s, j)
        for slot in range(n_slots):
            s = _find(cu, R, slot)
            j = slot - (cu[s] // R + s)
            if slot in owner:
                assert owner[slot] == (s, j)
            else:                                           # an unused slot exits early
                L = int(cu[s + 1] - cu[s])
                assert j > 0 and j * R >= L
