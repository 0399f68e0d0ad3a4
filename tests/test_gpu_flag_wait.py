"""The bounded-wait error path of the tensor-core state walk, run without any fault.

In a fused prefill the walk waits for each record's ready flag, which the prep CTAs publish.
kda_debug_flag_wait runs the same walk over prepared records with the caller's flags and a
short wait limit. Published flags: the walk equals kda_segment_replay_prepared bit for bit.
Flags that nothing ever sets: each walk gives up after the limit, raises KDA_STATUS_TIMEOUT,
drains its own copies and tensor-core work, frees its tensor memory and returns, and the
next ordinary call on the device still matches the reference. A walk that finds its flags
missing part way through has written the outputs of the chunks it finished before that.
"""
import time

import pytest
import torch

from linear_attention_state_kda_gb300 import inputs, kda

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
H, D = 4, 128


@pytest.fixture(scope="module")
def prepared():
    lens = [1000, 300]
    x = inputs.make_prefill(lens, H=H, dk=D, dv=D, dtype="bf16", seed=61, device=DEV)
    offs = torch.tensor([0, 700, 1000, 1300], dtype=torch.int32, device=DEV)
    P, T = offs.numel() - 1, x.T
    g = torch.Generator(device=DEV).manual_seed(62)
    seg_init = torch.randn(P, H, D, D, generator=g, device=DEV) * 0.05
    ws = kda.chunk_prepare(x.q, x.k, x.v, x.g, x.beta, offs)
    o_ref, f_ref = kda.segment_replay_prepared(ws, offs, seg_init, T, H, D, D, want_final=True)
    torch.cuda.synchronize()
    return dict(ws=ws, offs=offs, seg_init=seg_init, T=T, P=P, o_ref=o_ref, f_ref=f_ref)


def _walk(r, limit_ns, status):
    return kda.debug_flag_wait(r["ws"], r["offs"], r["seg_init"], r["T"], H, D, D, limit_ns,
                               want_final=True, status=status)


def test_published_flags_match_the_prepared_walk(prepared):
    r = prepared
    kda.record_flags(r["ws"], r["P"], r["T"], H).fill_(1)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, f = _walk(r, int(1e9), status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(o, r["o_ref"]) and torch.equal(f, r["f_ref"])


def test_unpublished_flags_time_out_and_the_device_recovers(prepared):
    r = prepared
    kda.record_flags(r["ws"], r["P"], r["T"], H).zero_()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    o, _ = _walk(r, int(5e7), status)          # 50 ms limit
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert status.item() & kda.STATUS_TIMEOUT
    assert elapsed < 1.5, elapsed               # one limit per walk, all walks side by side
    assert torch.count_nonzero(o).item() == 0   # nothing was loaded, nothing was written
    # the context is intact: an ordinary call still matches
    o2, f2 = kda.segment_replay_prepared(r["ws"], r["offs"], r["seg_init"], r["T"], H, D, D,
                                         want_final=True)
    torch.cuda.synchronize()
    assert torch.equal(o2, r["o_ref"]) and torch.equal(f2, r["f_ref"])


def test_flags_missing_part_way(prepared):
    """Segment 0's first four chunks are published, nothing else: that walk gives up while
    its copies and products for chunks 2 and 3 are in flight, after finishing chunks 0 and 1."""
    r = prepared
    flags = kda.record_flags(r["ws"], r["P"], r["T"], H)
    flags.zero_()
    flags[:4 * H] = 1                           # chunk slots 0..3 of segment 0, every head
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, _ = _walk(r, int(5e7), status)
    torch.cuda.synchronize()
    assert status.item() & kda.STATUS_TIMEOUT
    assert torch.equal(o[:128], r["o_ref"][:128])
    o2, f2 = kda.segment_replay_prepared(r["ws"], r["offs"], r["seg_init"], r["T"], H, D, D,
                                         want_final=True)
    torch.cuda.synchronize()
    assert torch.equal(o2, r["o_ref"]) and torch.equal(f2, r["f_ref"])
