"""The C-ABI library builds, loads and exports every declared symbol; host-side argument
checks reject bad calls before any launch (no GPU needed: no call here reaches CUDA)."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from linear_attention_state_kda_gb300 import build as libbuild
    libbuild.build()
    from linear_attention_state_kda_gb300 import kda
    return kda.lib()


def _declared():
    with open(os.path.join(ROOT, "include", "kda.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", src)))


def test_header_symbols_exported(L):
    names = _declared()
    assert len(names) >= 8, names
    for n in names:
        assert hasattr(L, n), f"{n} not exported"
    for n in ["kda_chunk_prefill", "kda_segment_package", "kda_package_scan",
              "kda_segment_replay", "kda_decode_step"]:
        assert n in names


def test_version(L):
    from linear_attention_state_kda_gb300 import kda
    assert "sm_103a" in kda.version()


def test_workspace_query(L):
    from linear_attention_state_kda_gb300 import kda
    w = kda.package_scan_workspace(4, 16, 32, 128, 128)
    # 4 sequences x (16 + 8) tree nodes x 32 heads x (128*128 + 128*128) fp32
    assert w >= 4 * 24 * 32 * 2 * 128 * 128 * 4
    assert kda.package_scan_workspace(1, 3, 2, 64, 64) == \
        kda.package_scan_workspace(1, 4, 2, 64, 64)
    assert kda.package_scan_workspace(0, 4, 2, 64, 64) == 0


def _prefill(L, dt=1, n=1, T=64, cu=None, H=2, dk=128, dv=128, chunk=64, ptr=4096):
    p = ptr
    return L.kda_chunk_prefill(dt, n, T, cu, H, dk, dv, chunk, 1.0, p, p, p, p, p, None, p,
                               None, None, 0, None, None)


def test_prefill_argument_checks(L):
    from linear_attention_state_kda_gb300 import kda
    assert _prefill(L, dk=96, dv=96) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill(L, dk=128, dv=64) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill(L, chunk=32) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill(L, dt=7) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill(L, H=0) == kda.KDA_ERR_INVALID_ARG
    assert _prefill(L, T=-1) == kda.KDA_ERR_INVALID_ARG
    assert _prefill(L, n=2, cu=None) == kda.KDA_ERR_INVALID_ARG
    assert "cu_seqlens" in kda.last_error()
    assert _prefill(L, ptr=4098) == kda.KDA_ERR_INVALID_ARG      # misaligned
    assert "aligned" in kda.last_error()
    # null inputs with tokens to process
    assert L.kda_chunk_prefill(1, 1, 64, None, 2, 128, 128, 64, 1.0, None, None, None, None,
                               None, None, None, None, None, 0, None,
                               None) == kda.KDA_ERR_INVALID_ARG
    # nothing to do is OK and launches nothing
    assert _prefill(L, n=0) == kda.KDA_OK
    # the tensor-core shapes need the caller's workspace (checked before any launch)
    assert _prefill(L, H=4) == kda.KDA_ERR_WORKSPACE
    assert "workspace" in kda.last_error()
    need = kda.chunk_workspace(torch.bfloat16, 1, 64, 4, 128, 128)
    assert L.kda_chunk_prefill(1, 1, 64, None, 4, 128, 128, 64, 1.0, 4096, 4096, 4096, 4096,
                               4096, None, 4096, None, 4096, need - 1, None,
                               None) == kda.KDA_ERR_WORKSPACE
    assert L.kda_chunk_prefill(1, 1, 64, None, 4, 128, 128, 64, 1.0, 4096, 4096, 4096, 4096,
                               4096, None, 4096, None, 4096 + 16, need, None,
                               None) == kda.KDA_ERR_WORKSPACE


def test_chunk_workspace_query(L):
    from linear_attention_state_kda_gb300 import kda
    bf, f32 = torch.bfloat16, torch.float32
    # one record of 147,968 bytes per (chunk slot, head), slots = T // 64 + ranges, then a
    # 4-byte flag per record rounded up to 256 bytes
    def need(items):
        return items * 147968 + (items * 4 + 255) // 256 * 256
    assert kda.chunk_workspace(bf, 1, 16384, 32, 128, 128) == need((256 + 1) * 32)
    assert kda.chunk_workspace(bf, 8, 16384, 32, 128, 128) == need((256 + 8) * 32)
    assert kda.chunk_workspace(bf, 3, 100, 4, 128, 128) == need((1 + 3) * 4)
    # paths that need none: fp32, d = 64, H not a multiple of 4, nothing to do
    assert kda.chunk_workspace(f32, 1, 16384, 32, 128, 128) == 0
    assert kda.chunk_workspace(bf, 1, 16384, 32, 64, 64) == 0
    assert kda.chunk_workspace(bf, 1, 16384, 6, 128, 128) == 0
    assert kda.chunk_workspace(bf, 1, 0, 32, 128, 128) == 0
    assert kda.chunk_workspace(bf, 0, 64, 32, 128, 128) == 0


def test_scan_and_package_checks(L):
    from linear_attention_state_kda_gb300 import kda
    p = 4096
    assert L.kda_package_scan(1, 2, p, 2, 2, 128, 128, p, p, None, p, None, None, 0, None,
                              None) == kda.KDA_ERR_WORKSPACE
    assert L.kda_package_scan(1, 2, p, 0, 2, 128, 128, p, p, None, p, None, p, 1 << 40, None,
                              None) == kda.KDA_ERR_INVALID_ARG
    assert L.kda_package_scan(1, 2, p, 2, 2, 96, 96, p, p, None, p, None, p, 1 << 40, None,
                              None) == kda.KDA_ERR_UNSUPPORTED
    assert L.kda_segment_package(1, 2, 128, None, 2, 128, 128, 64, p, p, p, p, p, p, None, 0,
                                 None, None) == kda.KDA_ERR_INVALID_ARG
    assert L.kda_segment_replay(1, 2, 128, None, 2, 128, 128, 64, 1.0, p, p, p, p, p, p, p,
                                None, None, 0, None, None) == kda.KDA_ERR_INVALID_ARG
    assert "kda_segment_replay" in kda.last_error()


def test_decode_checks(L):
    from linear_attention_state_kda_gb300 import kda
    p = 4096
    assert L.kda_decode_step(1, 4, 2, 128, 128, 1.0, p, p, p, p, p, p, p, 0, p, None,
                             None) == kda.KDA_ERR_INVALID_ARG
    assert L.kda_decode_step(1, 4, 2, 128, 128, 1.0, p, p, p, p, p, p, p + 8, 10, p, None,
                             None) == kda.KDA_ERR_INVALID_ARG
    assert L.kda_decode_step(1, 4, 2, 32, 32, 1.0, p, p, p, p, p, p, p, 10, p, None,
                             None) == kda.KDA_ERR_UNSUPPORTED
    assert L.kda_decode_step(1, 0, 2, 128, 128, 1.0, p, p, p, p, p, p, p, 10, p, None,
                             None) == kda.KDA_OK
    assert L.kda_decode_step(1, 1 << 30, 2, 128, 128, 1.0, p, p, p, p, p, p, p, 10, p, None,
                             None) == kda.KDA_ERR_INVALID_ARG   # batch * H > 2^30


def test_window_checks(L):
    from linear_attention_state_kda_gb300 import kda
    p = 4096
    win = lambda batch=4, window=4, dk=128, flags=0, n_slots=10, pool=p, ws=p: \
        L.kda_decode_window(1, batch, window, 2, dk, dk, 1.0, p, p, p, p, p, flags, p, ws, pool,
                            n_slots, p, None, None)
    assert win(window=kda.MAX_WINDOW + 1) == kda.KDA_ERR_UNSUPPORTED
    assert "window" in kda.last_error()
    assert win(dk=96) == kda.KDA_ERR_UNSUPPORTED
    assert win(flags=2) == kda.KDA_ERR_INVALID_ARG
    assert win(n_slots=0) == kda.KDA_ERR_INVALID_ARG
    assert win(pool=p + 8) == kda.KDA_ERR_INVALID_ARG       # the pool must be 16-byte aligned
    assert win(ws=None) == kda.KDA_ERR_INVALID_ARG
    assert win(batch=-1) == kda.KDA_ERR_INVALID_ARG
    assert win(batch=(1 << 27) + 1) == kda.KDA_ERR_INVALID_ARG  # batch * window * H > 2^30
    assert win(batch=0) == kda.KDA_OK                      # nothing to do launches nothing
    assert win(window=0) == kda.KDA_OK


def test_slot_checks(L):
    from linear_attention_state_kda_gb300 import kda
    p = 4096
    assert L.kda_slot_zero(4, p, p, 10, 6, None, None) == kda.KDA_ERR_INVALID_ARG  # 6 % 4
    assert L.kda_slot_zero(4, p, p + 4, 10, 8, None, None) == kda.KDA_ERR_INVALID_ARG
    assert L.kda_slot_zero(11, None, p, 10, 8, None, None) == kda.KDA_ERR_INVALID_ARG
    assert L.kda_slot_zero(0, p, p, 10, 8, None, None) == kda.KDA_OK
    assert L.kda_slot_copy(4, p, p, 10, None, p, 10, 8, None, None) == kda.KDA_ERR_INVALID_ARG
    assert L.kda_slot_copy(5, p, None, 4, p, p, 10, 8, None, None) == kda.KDA_ERR_INVALID_ARG
    assert L.kda_slot_copy(4, p, p, 0, p, p, 10, 8, None, None) == kda.KDA_ERR_INVALID_ARG
    assert L.kda_slot_copy(0, p, p, 10, p, p, 10, 8, None, None) == kda.KDA_OK


def test_short_conv_checks(L):
    from linear_attention_state_kda_gb300 import kda
    p = 4096
    def conv(dt=1, n=1, T=64, cu=None, C=64, W=4, x=p, flags=0, rs=None, ws=None, st=None,
             ns=0, out=p + 4096):
        return L.kda_short_conv(dt, n, T, cu, C, W, x, p, flags, rs, ws, st, ns, out, None,
                                None)

    assert conv(W=5) == kda.KDA_ERR_UNSUPPORTED
    assert conv(W=0) == kda.KDA_ERR_UNSUPPORTED
    assert conv(dt=7) == kda.KDA_ERR_UNSUPPORTED
    assert conv(C=12) == kda.KDA_ERR_INVALID_ARG               # not a multiple of 8
    assert conv(n=2) == kda.KDA_ERR_INVALID_ARG                # two sequences need cu_seqlens
    assert conv(flags=2) == kda.KDA_ERR_INVALID_ARG
    assert conv(rs=p) == kda.KDA_ERR_INVALID_ARG               # slot tables need a state pool
    assert conv(x=p + 8) == kda.KDA_ERR_INVALID_ARG            # misaligned
    assert conv(out=p) == kda.KDA_ERR_INVALID_ARG              # out aliases x
    assert conv(x=None) == kda.KDA_ERR_INVALID_ARG
    assert conv(n=0) == kda.KDA_OK                             # nothing to do launches nothing


def test_beta_alignment_fails_loudly(L):
    """beta offset by 4 bytes (a view one head into a [T, H] array, say) is rejected before
    any launch, on the tensor-core shapes and the CUDA-core ones alike: no call quietly runs
    another implementation."""
    from linear_attention_state_kda_gb300 import kda
    p, pb = 4096, 4096 + 4
    need = kda.chunk_workspace(torch.bfloat16, 1, 64, 4, 128, 128)
    assert need > 0
    for H, ws, nb in [(4, p, need), (2, None, 0)]:
        assert L.kda_chunk_prefill(1, 1, 64, None, H, 128, 128, 64, 1.0, p, p, p, p, pb, None,
                                   p, None, ws, nb, None, None) == kda.KDA_ERR_INVALID_ARG
        assert "beta" in kda.last_error()
        assert L.kda_segment_package(1, 1, 64, p, H, 128, 128, 64, p, p, p, pb, p, p, ws, nb,
                                     None, None) == kda.KDA_ERR_INVALID_ARG
        assert "beta" in kda.last_error()
        assert L.kda_segment_replay(1, 1, 64, p, H, 128, 128, 64, 1.0, p, p, p, p, pb, None, p,
                                    None, ws, nb, None, None) == kda.KDA_ERR_INVALID_ARG
        assert kda.last_error().startswith("kda_segment_replay")
