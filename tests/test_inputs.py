"""Host logic of the seeded workload generators (no GPU, no method arithmetic)."""
import torch

from linear_attention_state_kda_gb300 import inputs


def test_seeded_and_deterministic():
    a = inputs.make_prefill([100, 28], 2, 16, 8, "bf16", seed=7)
    b = inputs.make_prefill([100, 28], 2, 16, 8, "bf16", seed=7)
    for x, y in zip([a.q, a.k, a.v, a.g, a.beta], [b.q, b.k, b.v, b.g, b.beta]):
        assert torch.equal(x, y)
    assert a.cu_seqlens.tolist() == [0, 100, 128]
    assert a.q.dtype == torch.bfloat16 and a.g.dtype == torch.float32
    assert (a.g <= 0).all() and (a.beta > 0).all() and (a.beta < 1).all()
    kn = a.k.float().norm(dim=-1)
    assert (kn - 1).abs().max() < 1e-2          # normalised in fp32 before the bf16 cast


def test_decode_slots_unique():
    d = inputs.make_decode(64, 2, 16, 16, 500, seed=3)
    s = d.slot_ids.tolist()
    assert len(set(s)) == len(s) and min(s) >= 0 and max(s) < 500


def test_window_slots_disjoint_and_logits():
    w = inputs.make_window(16, 4, 2, 16, 16, 100, seed=3)
    r, ws = w.read_slots.tolist(), w.write_slots.reshape(-1).tolist()
    assert w.write_slots.shape == (16, 4) and w.q.shape == (64, 2, 16)
    assert len(set(r + ws)) == len(r) + len(ws)
    assert min(r + ws) >= 0 and max(r + ws) < 100
    assert torch.equal(w.beta, torch.sigmoid(w.beta_logit))
    # the q, k, v, g, beta draws come first, in the same order as the other workloads
    p = inputs.make_prefill([64], 2, 16, 16, "bf16", seed=3)
    assert torch.equal(w.q, p.q) and torch.equal(w.g, p.g) and torch.equal(w.beta, p.beta)


def test_conv_inputs():
    c = inputs.make_conv([5, 0, 9], 16, 4, seed=2, n_slots=10)
    assert c.x.shape == (14, 16) and c.weight.shape == (16, 4) and c.state.shape == (10, 3, 16)
    assert c.cu_seqlens.tolist() == [0, 5, 5, 14]
    ids = c.read_slots.tolist() + c.write_slots.tolist()
    assert len(set(ids)) == 6 and min(ids) >= 0 and max(ids) < 10
    d = inputs.make_conv([5, 0, 9], 16, 4, seed=2, n_slots=10)
    assert torch.equal(c.x, d.x) and torch.equal(c.state, d.state)


def test_leveled_split_rule():
    for length, n in [(131072, 16), (65536, 16), (32768, 8), (8192, 4)]:
        segs = inputs.gang_split(length)
        assert len(segs) == n, (length, segs)
        assert sum(segs) == length
        assert min(segs) >= inputs.SEGMENT_FLOOR
        assert all(s % 64 == 0 for s in segs[:-1])
        # deeper segments are not longer (leveling), up to the 64-token rounding
        assert all(segs[i] + 64 >= segs[i + 1] for i in range(len(segs) - 2))
    assert inputs.gang_split(8192) == [2048] * 4
    segs = inputs.workload_segments("varlen_long")
    assert sum(len(s) for s in segs) == 44
    offs, seq = inputs.segment_offsets([131072, 65536, 32768, 8192], segs)
    assert offs[-1].item() == 237568 and seq.tolist() == [0, 16, 32, 40, 44]


def test_gang_split_too_short_is_one_segment():
    assert inputs.gang_split(3000) == [3000]
    assert inputs.gang_split(4096) == [2048, 2048]
