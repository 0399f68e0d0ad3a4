"""Segment path (kda_segment_package -> kda_package_scan -> kda_segment_replay) against the
oracle and against the single chunked pass, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_kda_gb300 import inputs, kda
from kda_testutil import f64, oracle_inputs, rel_gpu, rel_o, rel_s, tols

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _segment_path(x, seg_lens_per_seq, want_seg_final=False):
    offs, seq_seg = inputs.segment_offsets(x.lens, seg_lens_per_seq)
    offs, seq_seg = offs.to(DEV), seq_seg.to(DEV)
    max_segs = max(len(s) for s in seg_lens_per_seq)
    M, D = kda.segment_package(x.k, x.v, x.g, x.beta, offs)
    seg_init, fin = kda.package_scan(M, D, seq_seg, max_segs, init_state=x.init_state)
    o, seg_final = kda.segment_replay(x.q, x.k, x.v, x.g, x.beta, offs, seg_init,
                                      want_final=want_seg_final)
    torch.cuda.synchronize()
    return dict(offs=offs, seq_seg=seq_seg, M=M, D=D, seg_init=seg_init, fin=fin, o=o,
                seg_final=seg_final)


def _oracle_segment(x, r, heads=None):
    d = oracle_inputs(x, heads)
    offs = r["offs"].cpu().numpy().astype(np.int64)
    sso = r["seq_seg"].cpu().numpy().astype(np.int64)
    M, D = oracle.package(d["k"], d["v"], d["g"], d["beta"], offs)
    seg_init, fin = oracle.scan(M, D, sso, d["init_state"])
    return M, D, seg_init, fin


def test_tiny_fp32_segments():
    x = inputs.make_workload("tiny_fp32", device=DEV)
    segs = inputs.workload_segments("tiny_fp32")
    r = _segment_path(x, segs, want_seg_final=True)
    M, D, seg_init, fin = _oracle_segment(x, r)
    tol = 1e-4
    assert rel_s(f64(r["M"]), M) < tol
    assert rel_s(f64(r["D"]), D) < tol
    assert rel_s(f64(r["seg_init"]), seg_init) < tol
    assert rel_s(f64(r["fin"]), fin) < tol
    d = oracle_inputs(x)
    ro, rf = oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
    assert rel_o(f64(r["o"]), ro) < tol
    # the last segment's replayed exit state is the sequence's exit state
    assert rel_s(f64(r["seg_final"][-1:]), rf) < tol
    # segment path agrees with the single pass on the GPU
    o1, f1 = kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta)
    assert rel_o(f64(r["o"]), f64(o1)) < tol and rel_s(f64(r["fin"]), f64(f1)) < tol


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ragged_segments_strong_coupling(dtype):
    """Short, ragged segments and slow decay: the prefix state dominates every segment."""
    lens = [777, 300]
    segs = [[64, 200, 13, 500], [300]]
    x = inputs.make_prefill(lens, H=2, dk=64, dv=64, dtype=dtype, seed=31, device=DEV,
                            init_std=0.3, **inputs.STRONG_COUPLING)
    r = _segment_path(x, segs)
    M, D, seg_init, fin = _oracle_segment(x, r)
    to, ts = tols(x.q.dtype)
    assert np.abs(M).max() > 0.1          # packages carry the prefix (not a vacuous test)
    assert rel_s(f64(r["M"]), M) < ts
    assert rel_s(f64(r["D"]), D) < ts
    assert rel_s(f64(r["seg_init"]), seg_init) < ts
    assert rel_s(f64(r["fin"]), fin) < ts
    d = oracle_inputs(x)
    ro, rf = oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                            d["init_state"])
    assert rel_o(f64(r["o"]), ro) < to
    assert rel_s(f64(r["fin"]), rf) < ts


def test_segments_8x2048_vs_single_pass():
    """Segment-parallel prefill of the 16k workload (8 x 2048) against the single chunked
    pass on the GPU (all heads) and against the oracle (two sampled heads)."""
    x = inputs.make_workload("segments_8x2048", device=DEV)
    segs = inputs.workload_segments("segments_8x2048")
    r = _segment_path(x, segs)
    o1, f1 = kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta)
    torch.cuda.synchronize()
    to, ts = tols(x.q.dtype)
    assert rel_gpu(r["o"], o1) < to
    assert rel_gpu(r["fin"], f1) < ts
    heads = [3, 30]
    M, D, seg_init, fin = _oracle_segment(x, r, heads)
    assert rel_s(f64(r["D"][:, heads]), D) < ts
    assert rel_s(f64(r["seg_init"][:, heads]), seg_init) < ts
    assert rel_s(f64(r["fin"][:, heads]), fin) < ts


def test_segments_8x2048_strong_coupling_vs_oracle():
    x = inputs.make_prefill([16384], H=2, dk=128, dv=128, dtype="bf16", seed=1001,
                            device=DEV, **inputs.STRONG_COUPLING)
    r = _segment_path(x, [[2048] * 8])
    M, D, seg_init, fin = _oracle_segment(x, r)
    to, ts = tols(x.q.dtype)
    assert np.linalg.norm(M[0, 0], 2) > 0.3
    assert rel_s(f64(r["M"]), M) < ts
    assert rel_s(f64(r["seg_init"]), seg_init) < ts
    assert rel_s(f64(r["fin"]), fin) < ts
    d = oracle_inputs(x)
    ro, _ = oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
    assert rel_o(f64(r["o"]), ro) < to


def test_varlen_long_leveled_sampled_head():
    """The long varlen workload (4 sequences, 237,568 tokens, 44 leveled segments, nonzero
    entry states): single pass and segment path on all heads; the oracle on one head."""
    x = inputs.make_workload("varlen_long", device=DEV)
    segs = inputs.workload_segments("varlen_long")
    r = _segment_path(x, segs)
    o1, f1 = kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                               init_state=x.init_state)
    torch.cuda.synchronize()
    to, ts = tols(x.q.dtype)
    assert rel_gpu(r["o"], o1) < to
    assert rel_gpu(r["fin"], f1) < ts
    heads = [11]
    d = oracle_inputs(x, heads)
    ro, rf = oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                            d["init_state"])
    assert rel_o(f64(o1[:, heads]), ro) < to
    assert rel_s(f64(f1[:, heads]), rf) < ts
    assert rel_o(f64(r["o"][:, heads]), ro) < to


def test_prepared_records_serve_package_and_replay():
    """One kda_chunk_prepare feeds both walks: identical to the unprepared calls."""
    x = inputs.make_workload("segments_8x2048", device=DEV)
    segs = inputs.workload_segments("segments_8x2048")
    r = _segment_path(x, segs, want_seg_final=True)
    T, H, dk = x.k.shape
    dv = x.v.shape[2]
    ws = kda.chunk_prepare(x.q, x.k, x.v, x.g, x.beta, r["offs"])
    M, D = kda.segment_package_prepared(ws, r["offs"], T, H, dk, dv)
    o, seg_final = kda.segment_replay_prepared(ws, r["offs"], r["seg_init"], T, H, dk, dv,
                                               want_final=True)
    torch.cuda.synchronize()
    assert torch.equal(M, r["M"]) and torch.equal(D, r["D"])
    assert torch.equal(o, r["o"]) and torch.equal(seg_final, r["seg_final"])
    # records prepared without q still serve the package walk
    ws2 = kda.chunk_prepare(None, x.k, x.v, x.g, x.beta, r["offs"])
    M2, D2 = kda.segment_package_prepared(ws2, r["offs"], T, H, dk, dv)
    torch.cuda.synchronize()
    assert torch.equal(M2, r["M"]) and torch.equal(D2, r["D"])


def test_fused_prefill_matches_two_kernel_walk():
    """The 16k single-sequence prefill runs as one cooperative launch (walks next to the prep
    work, records handed over through per-record flags); the same walk over the same records
    from two separate launches (prepare, then a one-segment replay from a zero state) must give
    bit-identical outputs and final states, every time."""
    x = inputs.make_workload("prefill_16k", device=DEV)
    T, H, dk = x.k.shape
    dv = x.v.shape[2]
    offs = torch.tensor([0, T], dtype=torch.int32, device=DEV)
    zero = torch.zeros(1, H, dk, dv, dtype=torch.float32, device=DEV)
    ws = kda.chunk_prepare(x.q, x.k, x.v, x.g, x.beta, offs)
    o_ref, f_ref = kda.segment_replay_prepared(ws, offs, zero, T, H, dk, dv, want_final=True)
    for _ in range(3):
        o, f = kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref)
        assert torch.equal(f, f_ref)
