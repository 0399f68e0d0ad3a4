"""Short causal depthwise convolution with per-sequence history windows (kda_short_conv),
through the C ABI, against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_kda_gb300 import inputs, kda
from kda_testutil import f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

# fp32 inputs: fp32 arithmetic against double (<= 4 products per output). bf16 inputs: the
# output is rounded to bf16 (relative 2^-9), so the normwise bound is 2^-8.
TOL = {"f32": 1e-5, "bf16": 4e-3}


def _rel(x, y):
    return float(np.abs(x - y).max() / max(np.abs(y).max(), 1e-30))


def _ids(t):
    return None if t is None else t.cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("silu", [False, True])
def test_varlen_with_history(dtype, W, silu):
    """Packed sequences (empty, shorter than the window, spanning several tiles, ragged) and a
    channel count that leaves a partial channel block: outputs and stored windows against the
    oracle; the read slots and every slot not written stay bit-identical."""
    lens = [0, 2, 37, 100, 1, 64]
    C = 520
    cv = inputs.make_conv(lens, C, W, dtype=dtype, seed=60 + W, device=DEV, n_slots=16)
    state0 = f64(cv.state)
    out = kda.short_conv(cv.x, cv.weight, cv.cu_seqlens, silu=silu, read_slots=cv.read_slots,
                         write_slots=cv.write_slots, conv_state=cv.state)
    torch.cuda.synchronize()
    host = state0.copy()
    ref, bad = oracle.short_conv(f64(cv.x), f64(cv.weight), _ids(cv.cu_seqlens), silu=silu,
                                 read_slots=_ids(cv.read_slots), write_slots=_ids(cv.write_slots),
                                 pool=host)
    assert bad == 0
    assert _rel(f64(out), ref) < TOL[dtype]
    # the stored windows are copies of inputs: bit-exact
    assert np.array_equal(f64(cv.state), host)


def test_in_place_window_and_bad_slots():
    """read slot = write slot updates in place (a short sequence keeps part of its old window);
    negative and out-of-range ids; a padding sequence with no history."""
    lens = [2, 70, 0, 5]
    C, W = 1024, 4
    cv = inputs.make_conv(lens, C, W, seed=64, device=DEV, n_slots=8)
    cv.read_slots[:] = torch.tensor([2, 5, 6, -1], dtype=torch.int32, device=DEV)
    cv.write_slots[:] = torch.tensor([2, 5, 9, 7], dtype=torch.int32, device=DEV)
    state0 = f64(cv.state)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = kda.short_conv(cv.x, cv.weight, cv.cu_seqlens, silu=True, read_slots=cv.read_slots,
                         write_slots=cv.write_slots, conv_state=cv.state, status=status)
    torch.cuda.synchronize()
    assert status.item() & kda.STATUS_BAD_SLOT
    host = state0.copy()
    ref, bad = oracle.short_conv(f64(cv.x), f64(cv.weight), _ids(cv.cu_seqlens), silu=True,
                                 read_slots=_ids(cv.read_slots), write_slots=_ids(cv.write_slots),
                                 pool=host)
    assert bad == 1
    assert _rel(f64(out), ref) < TOL["bf16"]
    assert np.array_equal(f64(cv.state), host)


def test_no_slots_and_split_continuation():
    """Without slot tables the history is zero; running a sequence in two calls with the
    window carried through a slot gives the one-call outputs bit for bit."""
    C, W = 2048, 4
    cv = inputs.make_conv([300], C, W, seed=65, device=DEV, n_slots=4)
    out0 = kda.short_conv(cv.x, cv.weight, silu=True)
    torch.cuda.synchronize()
    ref0, _ = oracle.short_conv(f64(cv.x), f64(cv.weight), silu=True)
    assert _rel(f64(out0), ref0) < TOL["bf16"]
    rs = torch.tensor([0], dtype=torch.int32, device=DEV)
    ws = torch.tensor([1], dtype=torch.int32, device=DEV)
    full = kda.short_conv(cv.x, cv.weight, silu=True, read_slots=rs, write_slots=ws,
                          conv_state=cv.state)
    for t in (1, 2, 63, 64, 65, 170):
        st = cv.state.clone()
        a = kda.short_conv(cv.x[:t].contiguous(), cv.weight, silu=True, read_slots=rs,
                           write_slots=torch.tensor([2], dtype=torch.int32, device=DEV),
                           conv_state=st)
        b = kda.short_conv(cv.x[t:].contiguous(), cv.weight, silu=True,
                           read_slots=torch.tensor([2], dtype=torch.int32, device=DEV),
                           write_slots=torch.tensor([3], dtype=torch.int32, device=DEV),
                           conv_state=st)
        torch.cuda.synchronize()
        assert torch.equal(torch.cat([a, b]), full), t
        assert torch.equal(st[3], cv.state[1])


def test_full_conv_16k_sampled_channels():
    """The 16k-token, 12288-channel workload (width 4, SiLU): oracle on sampled channel
    blocks (all tokens), the stored window exact."""
    cv = inputs.make_workload("conv_16k", device=DEV)
    out = kda.short_conv(cv.x, cv.weight, cv.cu_seqlens, silu=True, read_slots=cv.read_slots,
                         write_slots=cv.write_slots, conv_state=cv.state)
    torch.cuda.synchronize()
    cols = np.r_[0:16, 4096:4104, 12280:12288]
    sel = torch.as_tensor(cols, device=DEV)
    r = int(cv.read_slots[0])
    hist = f64(cv.state[r][:, sel])[None]
    ref, _ = oracle.short_conv(f64(cv.x[:, sel]), f64(cv.weight[sel]), silu=True,
                               read_slots=[0], pool=np.ascontiguousarray(hist))
    assert _rel(f64(out[:, sel]), ref) < TOL["bf16"]
    w = int(cv.write_slots[0])
    assert torch.equal(cv.state[w], cv.x[-3:])


@pytest.mark.parametrize("dtype,W", [("bf16", 4), ("f32", 3)])
def test_many_sequences_more_tiles_than_ctas(dtype, W):
    """Two hundred ragged sequences (empty, shorter than the window, multiples of the tile,
    a few hundred tokens), so that each persistent CTA takes many tiles in turn, holes in the
    tile numbering between them: every output and every stored window against the oracle."""
    rng = np.random.default_rng(71)
    lens = [int(v) for v in rng.integers(0, 300, size=200)]
    lens[:8] = [0, 1, 2, 3, 32, 64, 16, 0]
    C = 1024
    cv = inputs.make_conv(lens, C, W, dtype=dtype, seed=72 + W, device=DEV)
    state0 = f64(cv.state)
    out = kda.short_conv(cv.x, cv.weight, cv.cu_seqlens, silu=True, read_slots=cv.read_slots,
                         write_slots=cv.write_slots, conv_state=cv.state)
    torch.cuda.synchronize()
    host = state0.copy()
    ref, bad = oracle.short_conv(f64(cv.x), f64(cv.weight), _ids(cv.cu_seqlens), silu=True,
                                 read_slots=_ids(cv.read_slots), write_slots=_ids(cv.write_slots),
                                 pool=host)
    assert bad == 0
    assert _rel(f64(out), ref) < TOL[dtype]
    assert np.array_equal(f64(cv.state), host)


def test_more_channel_blocks_than_ctas():
    """240,000 channels: 469 blocks of 512 channels (the last one 384 wide), more than the
    persistent grid's CTAs, so that a CTA changes channel block from one tile to the next and
    reloads its taps: outputs and stored windows against the oracle."""
    lens = [40, 30]
    C, W = 240000, 4
    cv = inputs.make_conv(lens, C, W, seed=77, device=DEV)
    state0 = f64(cv.state)
    out = kda.short_conv(cv.x, cv.weight, cv.cu_seqlens, silu=True, read_slots=cv.read_slots,
                         write_slots=cv.write_slots, conv_state=cv.state)
    torch.cuda.synchronize()
    host = state0.copy()
    ref, bad = oracle.short_conv(f64(cv.x), f64(cv.weight), _ids(cv.cu_seqlens), silu=True,
                                 read_slots=_ids(cv.read_slots), write_slots=_ids(cv.write_slots),
                                 pool=host)
    assert bad == 0
    assert _rel(f64(out), ref) < TOL["bf16"]
    assert np.array_equal(f64(cv.state), host)
