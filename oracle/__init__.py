"""CPU oracle for the KDA gated delta-rule recurrence (double precision).

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()`` and by the
benchmark's ``cpu_baseline`` / reference leg. The product path (the CUDA library and its
Python binding) never imports this package, and this package imports nothing from it.

Each function wraps one C entry point of ``kda_oracle.cpp`` (see its header for the
mathematics and its source on the pages). Arrays are numpy float64, C-contiguous, in the
token-major layouts

    q, k, g: [T, H, dk]    v, o: [T, H, dv]    beta: [T, H]    states: [N, H, dk, dv]

The oracle is pinned against closed forms, exact rational arithmetic and invariants in
tests/test_oracle_pins.py.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(_build.build()))
    return _lib


def _bind(lib):
    """Declares the C signatures of the oracle's entry points on a loaded library."""
    d = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.POINTER(ctypes.c_int64)
    c_int, c_dbl, c_i64 = ctypes.c_int, ctypes.c_double, ctypes.c_int64
    lib.kda_ref_forward.argtypes = [c_int, i64, c_int, c_int, c_int, c_dbl, d, d, d, d, d,
                                    d, d, d, c_int]
    lib.kda_ref_forward.restype = c_int
    lib.kda_ref_package.argtypes = [c_int, i64, c_int, c_int, c_int, d, d, d, d, d, d,
                                    c_int]
    lib.kda_ref_package.restype = c_int
    lib.kda_ref_compose.argtypes = [c_int, c_int, d, d, d, d, d, d]
    lib.kda_ref_compose.restype = None
    lib.kda_ref_scan.argtypes = [c_int, i64, c_int, c_int, c_int, d, d, d, d, d, c_int]
    lib.kda_ref_scan.restype = c_int
    lib.kda_ref_decode.argtypes = [c_int, c_int, c_int, c_int, c_dbl, d, d, d, d, d, i64,
                                   d, c_i64, d, c_int]
    lib.kda_ref_decode.restype = c_int
    lib.kda_ref_decode_window.argtypes = [c_int, c_int, c_int, c_int, c_int, c_dbl, d, d, d,
                                          d, d, c_int, i64, i64, d, c_i64, d, c_int]
    lib.kda_ref_decode_window.restype = c_int
    lib.kda_ref_short_conv.argtypes = [c_int, i64, c_int, c_int, d, d, c_int, i64, i64, d,
                                       c_i64, d, c_int]
    lib.kda_ref_short_conv.restype = c_int
    return lib


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _ptr(a, typ=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(typ))


def threads_default():
    return os.cpu_count() or 1


def forward(q, k, v, g, beta, cu_seqlens=None, init_state=None, scale=1.0, threads=0,
            want_o=True):
    """Token-by-token recurrence. Returns (o [T,H,dv] or None, final_state [N,H,dk,dv])."""
    lib = _load()
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    T, H, dk = k.shape
    dv = v.shape[2]
    cu = _i64([0, T] if cu_seqlens is None else cu_seqlens)
    n = len(cu) - 1
    init = None if init_state is None else _f64(init_state)
    if init is not None:
        assert init.shape == (n, H, dk, dv)
    o = np.zeros((T, H, dv)) if want_o else None
    fin = np.zeros((n, H, dk, dv))
    rc = lib.kda_ref_forward(n, _ptr(cu, ctypes.c_int64), H, dk, dv, float(scale), _ptr(q),
                             _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init), _ptr(o),
                             _ptr(fin), int(threads))
    if rc < 0:
        raise ValueError("kda_ref_forward: bad arguments")
    return o, fin


def package(k, v, g, beta, seg_offsets, threads=0):
    """(M [P,H,dk,dk], D [P,H,dk,dv]) per segment [seg_offsets[p], seg_offsets[p+1])."""
    lib = _load()
    k, v, g, beta = _f64(k), _f64(v), _f64(g), _f64(beta)
    T, H, dk = k.shape
    dv = v.shape[2]
    so = _i64(seg_offsets)
    P = len(so) - 1
    M = np.zeros((P, H, dk, dk))
    D = np.zeros((P, H, dk, dv))
    rc = lib.kda_ref_package(P, _ptr(so, ctypes.c_int64), H, dk, dv, _ptr(k), _ptr(v),
                             _ptr(g), _ptr(beta), _ptr(M), _ptr(D), int(threads))
    if rc < 0:
        raise ValueError("kda_ref_package: bad arguments")
    return M, D


def compose(M2, D2, M1, D1):
    """(M2, D2) o (M1, D1) = (M2 M1, M2 D1 + D2) for one head (2-D arrays)."""
    lib = _load()
    M2, D2, M1, D1 = _f64(M2), _f64(D2), _f64(M1), _f64(D1)
    dk, dv = D2.shape
    M = np.zeros((dk, dk))
    D = np.zeros((dk, dv))
    lib.kda_ref_compose(dk, dv, _ptr(M2), _ptr(D2), _ptr(M1), _ptr(D1), _ptr(M), _ptr(D))
    return M, D


def scan(M, D, seq_seg_offsets, init_state=None, threads=0):
    """Segmented exclusive prefix. Returns (seg_init [P,H,dk,dv], final [N,H,dk,dv])."""
    lib = _load()
    M, D = _f64(M), _f64(D)
    P, H, dk, dv = D.shape
    so = _i64(seq_seg_offsets)
    n = len(so) - 1
    init = None if init_state is None else _f64(init_state)
    seg_init = np.zeros((P, H, dk, dv))
    fin = np.zeros((n, H, dk, dv))
    rc = lib.kda_ref_scan(n, _ptr(so, ctypes.c_int64), H, dk, dv, _ptr(M), _ptr(D), _ptr(init),
                          _ptr(seg_init), _ptr(fin), int(threads))
    if rc < 0:
        raise ValueError("kda_ref_scan: bad arguments")
    return seg_init, fin


def decode(q, k, v, g, beta, slot_ids, pool, scale=1.0, threads=0):
    """One decode token per row over pool [n_slots,H,dk,dv] (a float64 copy, updated in
    place). Returns (o [B,H,dv], number of slot ids >= n_slots)."""
    lib = _load()
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    B, H, dk = k.shape
    dv = v.shape[2]
    assert pool.dtype == np.float64 and pool.flags["C_CONTIGUOUS"]
    n_slots = pool.shape[0]
    sl = _i64(slot_ids)
    o = np.zeros((B, H, dv))
    rc = lib.kda_ref_decode(B, H, dk, dv, float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                            _ptr(beta), _ptr(sl, ctypes.c_int64), _ptr(pool), n_slots, _ptr(o),
                            int(threads))
    if rc < 0:
        raise ValueError("kda_ref_decode: bad arguments")
    return o, rc


def decode_window(q, k, v, g, beta, read_slots, write_slots, pool, scale=1.0,
                  beta_is_logit=False, threads=0):
    """Verify window with a state fork over pool [n_slots,H,dk,dv] (a float64 copy, updated
    in place): row b reads slot read_slots[b], runs the W tokens of its window (token b*W + j,
    arrays [B*W, H, *]) and stores the state after token j into slot write_slots[b, j].
    Returns (o [B*W,H,dv], number of slot ids >= n_slots)."""
    lib = _load()
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    rs = _i64(read_slots)
    ws = _i64(write_slots)
    B = rs.shape[0]
    W = ws.size // B if B else 0
    assert ws.size == B * W
    n_tok, H, dk = k.shape
    assert n_tok == B * W
    dv = v.shape[2]
    assert pool.dtype == np.float64 and pool.flags["C_CONTIGUOUS"]
    o = np.zeros((n_tok, H, dv))
    rc = lib.kda_ref_decode_window(B, W, H, dk, dv, float(scale), _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(g), _ptr(beta), int(bool(beta_is_logit)),
                                   _ptr(rs, ctypes.c_int64), _ptr(ws.reshape(-1), ctypes.c_int64),
                                   _ptr(pool), pool.shape[0], _ptr(o), int(threads))
    if rc < 0:
        raise ValueError("kda_ref_decode_window: bad arguments")
    return o, rc


def slot_zero(pool, slot_ids):
    """Sets pool[s] = 0 for every listed slot s (pool [n_slots, ...], updated in place).
    Negative ids are skipped; ids >= n_slots are skipped and counted. Returns the count."""
    n = pool.shape[0]
    bad = 0
    for s in np.asarray(slot_ids, dtype=np.int64).reshape(-1):
        if s >= n:
            bad += 1
        elif s >= 0:
            pool[s] = 0
    return bad


def slot_copy(src, src_ids, dst, dst_ids):
    """Copies slot src[src_ids[i]] into dst[dst_ids[i]] for each i (dst updated in place);
    None for an id list means 0..n-1. A pair with a negative id is skipped; a pair with an
    id past its pool's end is skipped and counted. Returns the count."""
    n = len(src_ids) if src_ids is not None else len(dst_ids)
    si = np.arange(n) if src_ids is None else np.asarray(src_ids, dtype=np.int64).reshape(-1)
    di = np.arange(n) if dst_ids is None else np.asarray(dst_ids, dtype=np.int64).reshape(-1)
    bad = 0
    for a, b in zip(si, di):
        if a >= src.shape[0] or b >= dst.shape[0]:
            bad += 1
        elif a >= 0 and b >= 0:
            dst[b] = src[a]
    return bad


def short_conv(x, w, cu_seqlens=None, silu=False, read_slots=None, write_slots=None,
               pool=None, threads=0):
    """Short causal depthwise convolution over packed sequences (x [T, C], w [C, W]) with a
    per-sequence history of W - 1 inputs in pool [n_slots, W-1, C] (a float64 copy, updated
    in place when write_slots is given). Returns (out [T, C], number of slot ids >= n_slots)."""
    lib = _load()
    x, w = _f64(x), _f64(w)
    T, C = x.shape
    W = w.shape[1]
    cu = _i64([0, T] if cu_seqlens is None else cu_seqlens)
    n = len(cu) - 1
    rs = None if read_slots is None else _i64(read_slots)
    ws = None if write_slots is None else _i64(write_slots)
    if pool is not None:
        assert pool.dtype == np.float64 and pool.flags["C_CONTIGUOUS"]
    n_slots = 0 if pool is None else pool.shape[0]
    out = np.zeros((T, C))
    rc = lib.kda_ref_short_conv(n, _ptr(cu, ctypes.c_int64), C, W, _ptr(x), _ptr(w),
                                int(bool(silu)), _ptr(rs, ctypes.c_int64),
                                _ptr(ws, ctypes.c_int64), _ptr(pool), n_slots, _ptr(out),
                                int(threads))
    if rc < 0:
        raise ValueError("kda_ref_short_conv: bad arguments")
    return out, rc

