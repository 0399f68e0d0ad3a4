"""Verify windows with a state fork (kda_decode_window) and the slot utilities
(kda_slot_zero, kda_slot_copy), through the C ABI, against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_kda_gb300 import inputs, kda
from kda_testutil import f64, rel_o, rel_s, tols

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _ids(t):
    return t.cpu().numpy().astype(np.int64)


def _beta(w, logit):
    return w.beta_logit if logit else w.beta


@pytest.mark.parametrize("dkv,dtype,W,logit", [(128, "bf16", 4, True), (128, "bf16", 16, False),
                                               (64, "bf16", 3, True), (128, "f32", 5, True),
                                               (64, "f32", 1, False), (128, "f32", 16, False)])
def test_window_small_pool(dkv, dtype, W, logit):
    """Outputs of every window token and every column's snapshot against the oracle; the read
    slots (not written) and every slot not named stay bit-identical."""
    B, H, n_slots = 9, 3, 9 * (W + 1) + 7
    w = inputs.make_window(B, W, H, dkv, dkv, n_slots, dtype=dtype, seed=51 + W, device=DEV)
    # row 0 stores its last column back into its own read slot (in place)
    w.write_slots[0, -1] = w.read_slots[0]
    pool0 = f64(w.pool)
    o = kda.decode_window(w.q, w.k, w.v, w.g, _beta(w, logit), w.read_slots, w.write_slots,
                          w.pool, scale=0.75, beta_is_logit=logit)
    torch.cuda.synchronize()
    host = pool0.copy()
    o_ref, bad = oracle.decode_window(f64(w.q), f64(w.k), f64(w.v), f64(w.g),
                                      f64(_beta(w, logit)), _ids(w.read_slots),
                                      _ids(w.write_slots), host, scale=0.75,
                                      beta_is_logit=logit)
    assert bad == 0
    to, ts = tols(w.q.dtype)
    assert rel_o(f64(o), o_ref) < to
    written = sorted(set(_ids(w.write_slots).reshape(-1).tolist()))
    assert rel_s(f64(w.pool[written]), host[written]) < ts
    others = [s for s in range(n_slots) if s not in set(written)]
    assert np.array_equal(f64(w.pool[others]), pool0[others])


def test_window_one_column_is_decode_step():
    """window = 1 with write slots = read slots is the decode step (same arithmetic order)."""
    d = inputs.make_decode(64, 4, 128, 128, 200, seed=52, device=DEV)
    pool_a = d.pool.clone()
    o_a = kda.decode_step(d.q, d.k, d.v, d.g, d.beta, d.slot_ids, pool_a)
    pool_b = d.pool.clone()
    o_b = kda.decode_window(d.q, d.k, d.v, d.g, d.beta, d.slot_ids,
                            d.slot_ids.reshape(-1, 1).contiguous(), pool_b)
    torch.cuda.synchronize()
    assert rel_o(f64(o_b), f64(o_a)) < 1e-6
    sl = d.slot_ids.long()
    assert rel_s(f64(pool_b[sl]), f64(pool_a[sl])) < 1e-6
    print("bit-identical to the decode step:", torch.equal(o_a, o_b) and
          torch.equal(pool_a, pool_b))


def test_window_padding_bad_slots_and_rollback():
    """Padding / out-of-range read slots zero the window's outputs and store nothing; a
    negative write slot stores nothing; an out-of-range write slot raises the status bit;
    resuming from an accepted column's snapshot reproduces the rest of the window."""
    B, W, H, n_slots = 5, 4, 2, 40
    w = inputs.make_window(B, W, H, 128, 128, n_slots, seed=53, device=DEV)
    w.read_slots[1] = -1
    w.read_slots[3] = n_slots + 5
    w.write_slots[2, 1] = -1
    w.write_slots[4, 3] = n_slots
    pool0 = f64(w.pool)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = kda.decode_window(w.q, w.k, w.v, w.g, w.beta_logit, w.read_slots, w.write_slots,
                          w.pool, beta_is_logit=True, status=status)
    torch.cuda.synchronize()
    assert status.item() & kda.STATUS_BAD_SLOT
    host = pool0.copy()
    o_ref, bad = oracle.decode_window(f64(w.q), f64(w.k), f64(w.v), f64(w.g),
                                      f64(w.beta_logit), _ids(w.read_slots),
                                      _ids(w.write_slots), host, beta_is_logit=True)
    assert bad == 2
    for b in (1, 3):
        assert torch.count_nonzero(o[b * W:(b + 1) * W]).item() == 0
    to, ts = tols(w.q.dtype)
    assert rel_o(f64(o), o_ref) < to
    assert rel_s(f64(w.pool), host) < ts
    for b in (1, 3):  # skipped rows stored nothing
        for s in _ids(w.write_slots[b]):
            if 0 <= s < n_slots:
                assert np.array_equal(f64(w.pool[s]), pool0[s])
    # rollback: row 0 accepted n = 2 tokens; resume from column 1 with the rest of its window
    n = 2
    rest = slice(n, W)
    wr = torch.tensor([[-1] * (W - n)], dtype=torch.int32, device=DEV)
    wr[0, -1] = int(w.read_slots[0])
    o2 = kda.decode_window(w.q[rest].contiguous(), w.k[rest].contiguous(),
                           w.v[rest].contiguous(), w.g[rest].contiguous(),
                           w.beta_logit[rest].contiguous(), w.write_slots[0, 1:2].contiguous(),
                           wr, w.pool, beta_is_logit=True)
    torch.cuda.synchronize()
    assert torch.equal(o2, o[rest])  # same state, same tokens, same kernel: bit-identical
    assert torch.equal(w.pool[int(w.read_slots[0])], w.pool[int(w.write_slots[0, W - 1])])


def test_window_full_256x4():
    """The 256-row, 4-token window workload over the 4096-slot pool (8.6 GB): parity on a
    sample of rows (all heads), untouched slots bit-identical."""
    w = inputs.make_workload("window_256x4", device=DEV)
    B, W = w.write_slots.shape
    rows = [0, 1, 77, 128, 200, 255]
    rs = w.read_slots.long()
    read0 = f64(w.pool[rs[rows]])
    touched = torch.zeros(w.pool.shape[0], dtype=torch.bool, device=DEV)
    touched[w.write_slots.long().reshape(-1)] = True
    untouched_ref = w.pool[~touched].clone()
    o = kda.decode_window(w.q, w.k, w.v, w.g, w.beta_logit, w.read_slots, w.write_slots,
                          w.pool, beta_is_logit=True)
    torch.cuda.synchronize()
    assert torch.equal(w.pool[~touched], untouched_ref)
    toks = np.concatenate([np.arange(r * W, (r + 1) * W) for r in rows])
    sel = lambda t: f64(t[torch.as_tensor(toks, device=DEV)])
    host = np.ascontiguousarray(read0)                         # compacted: slot i = row i
    wr = np.arange(len(rows), len(rows) * (W + 1)).reshape(len(rows), W)
    host = np.concatenate([host, np.zeros((len(rows) * W,) + host.shape[1:])])
    o_ref, bad = oracle.decode_window(sel(w.q), sel(w.k), sel(w.v), sel(w.g),
                                      sel(w.beta_logit), np.arange(len(rows)), wr, host,
                                      beta_is_logit=True)
    assert bad == 0
    to, ts = tols(w.q.dtype)
    assert rel_o(sel(o), o_ref) < to
    got = f64(w.pool[w.write_slots[rows].long().reshape(-1)])
    assert rel_s(got, host[len(rows):]) < ts


@pytest.mark.parametrize("H,d", [(3, 64), (4, 128)])
def test_slot_zero_and_copy(H, d):
    """Zero, checkpoint image and restore: bit-exact against the oracle's slot operations."""
    n_slots = 50
    gen = torch.Generator(device=DEV)
    gen.manual_seed(54)
    pool = torch.randn(n_slots, H, d, d, generator=gen, device=DEV)
    pool0 = pool.cpu().numpy()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids = torch.tensor([7, -1, 3, 49, 60], dtype=torch.int32, device=DEV)
    kda.slot_zero(pool, ids, status=status)
    torch.cuda.synchronize()
    ref = pool0.copy()
    assert oracle.slot_zero(ref, ids.cpu().numpy()) == 1
    assert status.item() & kda.STATUS_BAD_SLOT
    assert np.array_equal(pool.cpu().numpy(), ref)
    # checkpoint image of 6 slots into a compact buffer, then restore it elsewhere
    src_ids = torch.tensor([10, 11, 0, 25, 49, 31], dtype=torch.int32, device=DEV)
    image = torch.zeros(6, H, d, d, device=DEV)
    kda.slot_copy(pool, src_ids, image, None)
    img_ref = np.zeros((6, H, d, d), dtype=np.float32)
    assert oracle.slot_copy(ref, src_ids.cpu().numpy(), img_ref, None) == 0
    torch.cuda.synchronize()
    assert np.array_equal(image.cpu().numpy(), img_ref)
    status.zero_()
    dst_ids = torch.tensor([40, 41, -1, 42, 43, 99], dtype=torch.int32, device=DEV)
    kda.slot_copy(image, None, pool, dst_ids, status=status)
    assert oracle.slot_copy(img_ref, None, ref, dst_ids.cpu().numpy()) == 1
    torch.cuda.synchronize()
    assert status.item() & kda.STATUS_BAD_SLOT
    assert np.array_equal(pool.cpu().numpy(), ref)


def test_slot_copy_full_pool_256():
    """A checkpoint image of the 256 slots of the decode workload's 4096-slot pool (512 MiB),
    zeroed slots, and the restore: bit-exact."""
    dec = inputs.make_workload("decode_256", device=DEV)
    before = dec.pool[dec.slot_ids.long()].clone()
    image = torch.empty_like(before)
    kda.slot_copy(dec.pool, dec.slot_ids, image, None)
    kda.slot_zero(dec.pool, dec.slot_ids)
    torch.cuda.synchronize()
    assert torch.equal(image, before)
    assert torch.count_nonzero(dec.pool[dec.slot_ids.long()]).item() == 0
    kda.slot_copy(image, None, dec.pool, dec.slot_ids)
    torch.cuda.synchronize()
    assert torch.equal(dec.pool[dec.slot_ids.long()], before)
