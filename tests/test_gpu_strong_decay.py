"""Strong per-channel decay on the chunked paths, against the oracle: exact for every g <= 0.

The recurrence holds for any log-decay g <= 0 (a = e^g in [0, 1]). The chunk kernels share one
exponent frame per channel and chunk only while the channel decays by at most 160 nats over
the chunk; a channel beyond that is computed frame-free. These cases put many channels, one
channel, or one token of one channel past that bound, on the tensor-core kernels (bf16,
dk = dv = 128, H = 4) and on the CUDA-core kernel (fp32 at d = 64 and d = 128, bf16 with
H = 3), through the single pass and the segment path:

  * heavy: g = -20 softplus(N(0, 1)) on every channel (about 1000 nats per chunk);
  * one channel at g = -30 on every token, the others at the workloads' decay;
  * one channel with almost no decay (g = -1e-3) except a single drop of 500 nats in the
    middle of a chunk: the pairs of tokens across the drop vanish, those on either side are
    of order one, and the cumulative sums after the drop are large (a precision trap for a
    difference of cumulative sums);
  * decay exactly 0 (a = 1) on some channels next to those, so both extremes meet.

The status word must stay 0: nothing is out of range.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_kda_gb300 import inputs, kda
from kda_testutil import (TOL_F32, f64, oracle_inputs, rel_gpu, rel_o, rel_s, rows_s, tc_path,
                          tols)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _strong_inputs(lens, H, d, dtype, seed, kind):
    x = inputs.make_prefill(lens, H=H, dk=d, dv=d, dtype=dtype, seed=seed, device=DEV,
                            init_std=0.1, decay_scale=20.0 if kind == "heavy" else 1.0)
    if kind == "mixed":
        g = x.g
        g[:, :, 3] = -30.0                  # one channel at -30 nats on every token
        g[:, :, 5] = -1e-3                  # almost no decay ...
        g[x.T // 2 + 5, :, 5] = -500.0      # ... but one drop of 500 nats mid-chunk
        g[:, :, 6] = 0.0                    # no decay at all
        g[:, 1::2, 9] = -200.0              # every token, every other head
    return x


def _check_single_pass(x, scale):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, fin = kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                               init_state=x.init_state, scale=scale, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    d = oracle_inputs(x)
    ro, rf = oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                            d["init_state"], scale=scale)
    to, ts = tols(x.q.dtype)
    eo, es = rel_o(f64(o), ro), rel_s(f64(fin), rf)
    rows = rows_s(f64(fin), rf)[0]
    print(f"single pass: o {eo:.2e}, state {es:.2e}, state rows {rows:.2e}")
    assert eo < to and es < ts and rows < ts, (eo, es, rows)
    return o, fin


@pytest.mark.parametrize("kind", ["heavy", "mixed"])
def test_strong_decay_tc_single_pass(kind):
    x = _strong_inputs([700, 0, 1, 300], 4, 128, "bf16", 51, kind)
    assert tc_path(4, x.T, 4)
    _check_single_pass(x, 128 ** -0.5)


@pytest.mark.parametrize("kind", ["heavy", "mixed"])
@pytest.mark.parametrize("d,dtype,H", [(64, "f32", 2), (128, "f32", 2), (128, "bf16", 3)])
def test_strong_decay_cuda_core_single_pass(kind, d, dtype, H):
    x = _strong_inputs([300, 90], H, d, dtype, 52, kind)
    assert not tc_path(2, x.T, H, d, d)
    _check_single_pass(x, d ** -0.5)


@pytest.mark.parametrize("kind", ["heavy", "mixed"])
@pytest.mark.parametrize("H,dtype", [(4, "bf16"), (2, "f32")])
def test_strong_decay_segment_path(kind, H, dtype):
    """Packages, scan and replay under strong decay against the oracle, and against the
    GPU's single pass."""
    lens = [1000, 333]
    segs = [[64, 500, 1, 435], [333]]
    x = _strong_inputs(lens, H, 128, dtype, 53, kind)
    offs, sso = inputs.segment_offsets(lens, segs)
    offs, sso = offs.to(DEV), sso.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    M, Dp = kda.segment_package(x.k, x.v, x.g, x.beta, offs, status=status)
    si, fin = kda.package_scan(M, Dp, sso, 4, init_state=x.init_state)
    o, _ = kda.segment_replay(x.q, x.k, x.v, x.g, x.beta, offs, si, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    d = oracle_inputs(x)
    rM, rD = oracle.package(d["k"], d["v"], d["g"], d["beta"],
                            offs.cpu().numpy().astype(np.int64))
    rsi, rfin = oracle.scan(rM, rD, sso.cpu().numpy().astype(np.int64), d["init_state"])
    ro, rf = oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                            d["init_state"])
    to, ts = tols(x.q.dtype)
    for name, got, ref in [("M", M, rM), ("D", Dp, rD), ("seg_init", si, rsi),
                           ("fin", fin, rfin)]:
        e = rel_s(f64(got), ref)
        print(f"segment path {name}: {e:.2e}")
        assert e < ts, (name, e)
    assert rel_s(f64(fin), rf) < ts
    assert rel_o(f64(o), ro) < to
    o1, f1 = kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                               init_state=x.init_state)
    torch.cuda.synchronize()
    assert rel_gpu(o, o1) < to and rel_gpu(fin, f1) < ts


def test_strong_decay_mixed_chunks_fused_16k():
    """A 16k-token prompt where only a few chunks hold a strong channel, in the fused launch
    the benchmark times (heads 0 and 3 against the oracle): the items with and without strong
    channels share the persistent prep CTAs."""
    x = inputs.make_prefill([16384], H=32, dk=128, dv=128, dtype="bf16", seed=54, device=DEV)
    x.g[5000:5064, 3, 17] = -4.0            # one chunk of head 3: 256 nats in channel 17
    x.g[9001, 0, 100] = -300.0              # one token of head 0
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, fin = kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    heads = [0, 3]
    d = oracle_inputs(x, heads)
    ro, rf = oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
    assert rel_o(f64(o[:, heads]), ro) < 2e-2
    assert rel_s(f64(fin[:, heads]), rf) < 5e-3
