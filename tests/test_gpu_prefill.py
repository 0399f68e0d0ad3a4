"""Chunked prefill (kda_chunk_prefill) against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_kda_gb300 import inputs, kda
from kda_testutil import f64, oracle_inputs, rel_o, rel_s, tols

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _check(x, heads=None, scale=1.0):
    o, fin = kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                               init_state=x.init_state, scale=scale)
    torch.cuda.synchronize()
    d = oracle_inputs(x, heads)
    ro, rf = oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                            d["init_state"], scale=scale)
    go = f64(o) if heads is None else f64(o[:, heads])
    gf = f64(fin) if heads is None else f64(fin[:, heads])
    to, ts = tols(x.q.dtype)
    eo, es = rel_o(go, ro), rel_s(gf, rf)
    assert eo < to and es < ts, (eo, es)
    return o, fin, eo, es


def test_tiny_fp32_workload():
    x = inputs.make_workload("tiny_fp32", device=DEV)
    _check(x)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ragged_tail_and_scale(d, dtype):
    # 1000 = 15 full chunks and a 40-token tail
    x = inputs.make_prefill([1000], H=3, dk=d, dv=d, dtype=dtype, seed=21, device=DEV,
                            init_std=0.1)
    _check(x, scale=d ** -0.5)


def test_varlen_with_empty_and_short_sequences():
    x = inputs.make_prefill([130, 0, 64, 700, 1, 63], H=2, dk=128, dv=128, dtype="bf16",
                            seed=22, device=DEV, init_std=0.05)
    o, fin, _, _ = _check(x)
    # the empty sequence's exit state is its entry state
    assert torch.equal(fin[1], x.init_state[1])


def test_strong_coupling_variant():
    x = inputs.make_prefill([2048], H=2, dk=128, dv=128, dtype="bf16", seed=23, device=DEV,
                            init_std=0.5, **inputs.STRONG_COUPLING)
    _check(x)


def test_full_prefill_16k_sampled_heads():
    """The 16k-token, 32-head workload in the launch configuration the benchmark times;
    the oracle checks two sampled heads (heads are independent)."""
    x = inputs.make_workload("prefill_16k", device=DEV)
    _check(x, heads=[0, 17])
