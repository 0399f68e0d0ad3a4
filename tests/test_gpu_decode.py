"""Decode step (kda_decode_step) over the slot-addressed pool, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_kda_gb300 import inputs, kda
from kda_testutil import f64, rel_o, rel_s, tols

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _oracle_steps(d, pool_rows, steps, scale=1.0):
    """Runs `steps` decode steps in the oracle on host copies of the touched slots only."""
    slots = d.slot_ids.cpu().numpy().astype(np.int64)
    n_slots = d.pool.shape[0]
    valid = (slots >= 0) & (slots < n_slots)
    compact = np.where(valid, np.arange(len(slots)), np.where(slots < 0, -1, 1 << 40))
    host = pool_rows.copy()
    outs = []
    for _ in range(steps):
        o, _ = oracle.decode(f64(d.q), f64(d.k), f64(d.v), f64(d.g), f64(d.beta), compact, host,
                             scale=scale)
        outs.append(o)
    return outs, host


@pytest.mark.parametrize("dkv,dtype", [(128, "bf16"), (64, "bf16"), (128, "f32"), (64, "f32")])
def test_small_pool(dkv, dtype):
    d = inputs.make_decode(37, 3, dkv, dkv, 101, dtype=dtype, seed=41, device=DEV)
    slots = d.slot_ids.long()
    rows0 = f64(d.pool[slots])
    for step in range(3):
        o = kda.decode_step(d.q, d.k, d.v, d.g, d.beta, d.slot_ids, d.pool, scale=0.5)
    torch.cuda.synchronize()
    outs, host = _oracle_steps(d, rows0, 3, scale=0.5)
    to, ts = tols(d.q.dtype)
    assert rel_o(f64(o), outs[-1]) < to
    assert rel_s(f64(d.pool[slots]), host) < ts


def test_padding_and_bad_slots():
    d = inputs.make_decode(6, 2, 128, 128, 16, seed=42, device=DEV)
    d.slot_ids[:] = torch.tensor([3, -1, 15, 16, 99, 0], dtype=torch.int32, device=DEV)
    before = d.pool.clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = kda.decode_step(d.q, d.k, d.v, d.g, d.beta, d.slot_ids, d.pool, status=status)
    torch.cuda.synchronize()
    assert status.item() & kda.STATUS_BAD_SLOT
    for b in [1, 3, 4]:
        assert torch.count_nonzero(o[b]).item() == 0
    touched = {3, 15, 0}
    for s in range(16):
        if s not in touched:
            assert torch.equal(d.pool[s], before[s])
    assert not torch.equal(d.pool[3], before[3])


def test_full_pool_256x32_slot_bit_exact():
    """The 256-row, 32-head decode over the 4096-slot pool (8.6 GB): parity with the oracle
    on the touched slots after 1 and 3 steps; decoding through the random slot table is
    bit-identical to decoding the same states compacted into slots 0..255; untouched slots
    stay bit-identical."""
    d = inputs.make_workload("decode_256", device=DEV)
    slots = d.slot_ids.long()
    rows0 = d.pool[slots].clone()
    compact_pool = rows0.clone()                     # states at slots 0..255
    compact_ids = torch.arange(256, dtype=torch.int32, device=DEV)
    untouched = torch.ones(d.pool.shape[0], dtype=torch.bool, device=DEV)
    untouched[slots] = False
    ref_untouched = d.pool[untouched].clone()

    o1 = kda.decode_step(d.q, d.k, d.v, d.g, d.beta, d.slot_ids, d.pool)
    oc = kda.decode_step(d.q, d.k, d.v, d.g, d.beta, compact_ids, compact_pool)
    torch.cuda.synchronize()
    assert torch.equal(o1, oc)
    assert torch.equal(d.pool[slots], compact_pool)
    outs, host = _oracle_steps(d, f64(rows0), 1)
    to, ts = tols(d.q.dtype)
    assert rel_o(f64(o1), outs[0]) < to
    assert rel_s(f64(d.pool[slots]), host) < ts
    for _ in range(2):
        o3 = kda.decode_step(d.q, d.k, d.v, d.g, d.beta, d.slot_ids, d.pool)
    torch.cuda.synchronize()
    outs, host = _oracle_steps(d, f64(rows0), 3)
    assert rel_o(f64(o3), outs[-1]) < to
    assert rel_s(f64(d.pool[slots]), host) < ts
    assert torch.equal(d.pool[untouched], ref_untouched)
