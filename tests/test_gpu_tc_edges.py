"""Edge cases of the tensor-core chunk path, element by element against the oracle.

Every case here has a shape the tensor-core kernels take (bf16 q/k/v, dk = dv = 128, H a
multiple of 4; `tc_path` asserts it), so partial chunks, empty and one-token ranges, a query
scale, nonzero entry states, strong coupling across segments (packages whose M is far from
zero) and the prepared walks are all checked on the hot-path kernels themselves, not on the
CUDA-core kernel that serves the other shapes.

Tolerances are the bf16 ones: outputs 2e-2, fp32 states and packages 5e-3, asserted both
normwise per head and row by row (`rows_o`: every token row of an output against its own
magnitude; `rows_s`: every key-channel row of a state), so that an error confined to a few
rows, such as the tail rows of a partial chunk, cannot hide under a head's maximum. The
element-wise figure (floor 1e-6 of the head's maximum) is printed beside them; it is not a
bound for bf16 arithmetic, where an element whose true value nearly cancels carries the
absolute error of its larger terms.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_kda_gb300 import inputs, kda
from kda_testutil import (TOL_BF16_O, TOL_BF16_S, f64, oracle_inputs, rel_gpu, rel_o, rel_s,
                          rows_o, rows_s, tc_path)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
H = 4
D = 128
SCALE = D ** -0.5


def _forward_oracle(x, scale=1.0, init=True):
    d = oracle_inputs(x)
    return oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                          d["init_state"] if init else None, scale=scale)


def _assert_o(go, ro, what):
    e = rel_o(go, ro)
    rows, elems = rows_o(go, ro)
    print(f"{what}: o normwise {e:.2e}, rows {rows:.2e}, elements {elems:.2e}")
    assert e < TOL_BF16_O, (what, e)
    assert rows < TOL_BF16_O, (what, rows)


def _assert_s(gs, rs, what):
    e = rel_s(gs, rs)
    rows, elems = rows_s(gs, rs)
    print(f"{what}: state normwise {e:.2e}, rows {rows:.2e}, elements {elems:.2e}")
    assert e < TOL_BF16_S, (what, e)
    assert rows < TOL_BF16_S, (what, rows)


def test_ragged_varlen_partial_chunks_on_tc_path():
    """Six packed sequences: 15 full chunks + a 40-token tail, an empty one, one token, 63
    tokens, 2 chunks + 2 tokens, 64 chunks + 1 token; nonzero entry states; scale 1/sqrt(d)."""
    lens = [1000, 0, 1, 63, 130, 4097]
    x = inputs.make_prefill(lens, H=H, dk=D, dv=D, dtype="bf16", seed=41, device=DEV,
                            init_std=0.05)
    assert tc_path(len(lens), x.T, H)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, fin = kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                               init_state=x.init_state, scale=SCALE, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    ro, rf = _forward_oracle(x, scale=SCALE)
    _assert_o(f64(o), ro, "ragged varlen")
    _assert_s(f64(fin), rf, "ragged varlen")
    # every sequence's own tokens (the tails included) on their own
    cu = x.cu_seqlens.cpu().tolist()
    for s in range(len(lens)):
        a, b = cu[s], cu[s + 1]
        if b > a:
            assert rel_o(f64(o[a:b]), ro[a:b]) < TOL_BF16_O, s
    # the last 40 tokens of the first sequence: the partial chunk's rows
    assert rel_o(f64(o[960:1000]), ro[960:1000]) < TOL_BF16_O
    # an empty sequence leaves its entry state untouched, bit for bit
    assert torch.equal(fin[1], x.init_state[1])


def test_strong_coupling_16k_on_tc_path():
    """16,384 tokens with slow decay and small write strengths, so that the state carries
    information across the whole prompt (tf32 rounding has 256 chunks to accumulate)."""
    x = inputs.make_prefill([16384], H=H, dk=D, dv=D, dtype="bf16", seed=42, device=DEV,
                            init_std=0.3, **inputs.STRONG_COUPLING)
    assert tc_path(1, x.T, H)
    o, fin = kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta, init_state=x.init_state,
                               scale=SCALE)
    torch.cuda.synchronize()
    ro, rf = _forward_oracle(x, scale=SCALE)
    _assert_o(f64(o), ro, "strong coupling 16k")
    _assert_s(f64(fin), rf, "strong coupling 16k")


def _strong_segments():
    lens = [9000, 7384]
    segs = [[1000, 3000, 0, 64, 1, 4935], [2048, 5336]]   # none but one a multiple of 64
    x = inputs.make_prefill(lens, H=H, dk=D, dv=D, dtype="bf16", seed=43, device=DEV,
                            init_std=0.3, **inputs.STRONG_COUPLING)
    offs, seq_seg = inputs.segment_offsets(lens, segs)
    return x, offs.to(DEV), seq_seg.to(DEV), max(len(s) for s in segs)


def test_segment_path_strong_coupling_ragged_on_tc_path():
    """Packages of ragged segments (an empty one and a one-token one among them) of two
    sequences with entry states, where the packages' M is of order one: M, D, the scanned
    entry states, the exit states and the replayed outputs all against the oracle."""
    x, offs, seq_seg, max_segs = _strong_segments()
    P = offs.numel() - 1
    assert tc_path(P, x.T, H)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    M, Dp = kda.segment_package(x.k, x.v, x.g, x.beta, offs, status=status)
    seg_init, fin = kda.package_scan(M, Dp, seq_seg, max_segs, init_state=x.init_state)
    o, seg_final = kda.segment_replay(x.q, x.k, x.v, x.g, x.beta, offs, seg_init, scale=SCALE,
                                      want_final=True, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    d = oracle_inputs(x)
    offs_h = offs.cpu().numpy().astype(np.int64)
    rM, rD = oracle.package(d["k"], d["v"], d["g"], d["beta"], offs_h)
    rsi, rfin = oracle.scan(rM, rD, seq_seg.cpu().numpy().astype(np.int64), d["init_state"])
    # the packages carry the prefix: M is far from zero (not a vacuous test of the M tile)
    assert max(np.linalg.norm(rM[p, 0], 2) for p in range(P)) > 0.5
    _assert_s(f64(M), rM, "package M")
    _assert_s(f64(Dp), rD, "package D")
    _assert_s(f64(seg_init), rsi, "scanned entry states")
    _assert_s(f64(fin), rfin, "exit states")
    # the empty segment's package is the identity map, bit for bit
    assert torch.equal(M[2], torch.eye(D, device=DEV).expand(H, D, D))
    assert torch.equal(Dp[2], torch.zeros(H, D, D, device=DEV))
    ro, rf = _forward_oracle(x, scale=SCALE)
    _assert_o(f64(o), ro, "replayed outputs")
    _assert_s(f64(fin), rf, "exit states vs single pass (oracle)")
    # each sequence's last replayed segment ends in that sequence's exit state
    _assert_s(f64(seg_final[[5, 7]]), rf, "last segments' exit states")
    # and the GPU's own single pass agrees with the segment path
    o1, f1 = kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                               init_state=x.init_state, scale=SCALE)
    torch.cuda.synchronize()
    assert rel_gpu(o, o1) < TOL_BF16_O
    assert rel_gpu(fin, f1) < TOL_BF16_S


def test_prepared_walks_strong_coupling_ragged():
    """The same segments through kda_chunk_prepare and the two prepared walks: identical to
    the unprepared calls, bit for bit, and so to the oracle."""
    x, offs, seq_seg, max_segs = _strong_segments()
    T = x.T
    M, Dp = kda.segment_package(x.k, x.v, x.g, x.beta, offs)
    seg_init, _ = kda.package_scan(M, Dp, seq_seg, max_segs, init_state=x.init_state)
    o, sf = kda.segment_replay(x.q, x.k, x.v, x.g, x.beta, offs, seg_init, scale=SCALE,
                               want_final=True)
    ws = kda.chunk_prepare(x.q, x.k, x.v, x.g, x.beta, offs, scale=SCALE)
    M2, D2 = kda.segment_package_prepared(ws, offs, T, H, D, D)
    o2, sf2 = kda.segment_replay_prepared(ws, offs, seg_init, T, H, D, D, want_final=True)
    ws_k = kda.chunk_prepare(None, x.k, x.v, x.g, x.beta, offs)
    M3, D3 = kda.segment_package_prepared(ws_k, offs, T, H, D, D)
    torch.cuda.synchronize()
    assert torch.equal(M2, M) and torch.equal(D2, Dp)
    assert torch.equal(M3, M) and torch.equal(D3, Dp)
    assert torch.equal(o2, o) and torch.equal(sf2, sf)


def test_single_token_and_single_chunk_sequences():
    """Many tiny sequences (1, 2, 63, 64, 65 tokens, and empties between them) in one call."""
    lens = [1, 0, 2, 63, 64, 65, 0, 1, 127, 128, 129]
    x = inputs.make_prefill(lens, H=8, dk=D, dv=D, dtype="bf16", seed=44, device=DEV,
                            init_std=0.1)
    assert tc_path(len(lens), x.T, 8)
    o, fin = kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                               init_state=x.init_state, scale=SCALE)
    torch.cuda.synchronize()
    ro, rf = _forward_oracle(x, scale=SCALE)
    _assert_o(f64(o), ro, "tiny sequences")
    _assert_s(f64(fin), rf, "tiny sequences")
    assert torch.equal(fin[1], x.init_state[1]) and torch.equal(fin[6], x.init_state[6])


def test_few_sequences_walked_in_turn_by_one_cta_per_head():
    """Six ragged sequences at 8 heads: 48 walks are more than a quarter of the SMs, so the fused
    launch gives each head one walk CTA that takes the six ranges in turn (an empty one and a
    one-token one among them) while the prep CTAs produce their records. Against the oracle on
    all heads, and against the same walks run from two separate launches (prepare, then a
    replay from the entry states), bit for bit."""
    lens = [1000, 0, 1, 63, 130, 4097]
    h8 = 8
    x = inputs.make_prefill(lens, H=h8, dk=D, dv=D, dtype="bf16", seed=47, device=DEV,
                            init_std=0.05)
    assert tc_path(len(lens), x.T, h8)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, fin = kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                               init_state=x.init_state, scale=SCALE, status=status)
    ws = kda.chunk_prepare(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, scale=SCALE)
    o2, fin2 = kda.segment_replay_prepared(ws, x.cu_seqlens, x.init_state, x.T, h8, D, D,
                                           want_final=True)
    torch.cuda.synchronize()
    assert status.item() == 0
    ro, rf = _forward_oracle(x, scale=SCALE)
    _assert_o(f64(o), ro, "ranges in turn")
    _assert_s(f64(fin), rf, "ranges in turn")
    assert torch.equal(o, o2) and torch.equal(fin, fin2)
    assert torch.equal(fin[1], x.init_state[1])  # the empty sequence
